// Prologue of the attention step: split qkv, RMSNorm + RoPE on K (and on Q
// when a Q output is given), write K and V to the cache (and the prepared Q).
//
// Zero-to-sglang Ch.3 code walkthrough, section 3.3: AttentionLayer.forward
// splits the merged projection into Q, K and V, applies RMSNorm to each Q/K
// head's last dimension and RoPE at each token's position (V is not rotated);
// transformer-basics "Prefill vs Decode": the new K/V are appended to the
// per-layer cache (past_key_values.update).  One pass: every (token, head)
// vector of D bf16 values is read once with 16-byte loads by a group of D/16
// lanes, reduced with warp shuffles, and written once.
#include "kernels.cuh"

namespace gb300 {

namespace {

constexpr int kWarpsPerBlock = 8;  // each warp takes one run of (token, step) units
constexpr int kThreads = kWarpsPerBlock * 32;
#ifndef PROLOGUE_BATCH
#define PROLOGUE_BATCH 6
#endif
#ifndef PROLOGUE_BATCH_F8
#define PROLOGUE_BATCH_F8 4
#endif
#ifndef PROLOGUE_MIN_BLOCKS
#define PROLOGUE_MIN_BLOCKS 2
#endif
// steps whose loads are issued before processing (bf16 cache, E4M3 cache):
// as many as fit in the registers two blocks per SM allow
constexpr int kBatchBf16 = PROLOGUE_BATCH;
constexpr int kBatchF8 = PROLOGUE_BATCH_F8;
constexpr int kMinBlocks = PROLOGUE_MIN_BLOCKS;  // resident blocks per SM the registers allow

struct ProloguePar {
  const uint16_t* __restrict__ qkv;        // [N, W] bf16
  const uint16_t* __restrict__ q_norm_w;   // [D] bf16 (used when q_out != NULL)
  const uint16_t* __restrict__ k_norm_w;   // [D] bf16
  uint16_t* __restrict__ q_out;            // [N, Hq, D] bf16 or NULL
  const int32_t* cu_seqlens;  // [B+1] or NULL: token b is request b (decode)
  void* __restrict__ k_cache;  // bf16, or E4M3 codes (one byte per entry)
  void* __restrict__ v_cache;
  float inv_k, inv_v;          // E4M3: fp32(1 / scale), rounded on the host
  KvIndex kv;
  int32_t* status;
  int32_t B, N, Hq, Hkv;
  int64_t steps_per_warp;  // each warp takes this many consecutive (token, step) units
  float eps;
  RopeFreqs freqs;
};

// One warp per token.  A head vector (D bf16) is held by L = D/16 lanes, lane
// li taking the 8 values at 8*li and the 8 values at D/2 + 8*li: the two
// members of each rotation pair (i, i + D/2) sit in the same lane, so RoPE
// needs no data exchange and the norm's sum of squares needs log2(L) shuffles.
// HPI = 32 / L head vectors are taken per step; each load instruction reads
// HPI runs of 128 contiguous bytes and each store writes whole runs.  cos/sin
// of the token's D/2 rotation angles are computed once (D/64 per lane) and
// handed to the lanes that need them with shuffles.  F8: the cache holds E4M3
// codes.
template <int D, bool F8>
__global__ void __launch_bounds__(kThreads, kMinBlocks) kv_append_kernel(const ProloguePar p) {
  constexpr int L = D / 16;     // lanes per head vector
  constexpr int HPI = 32 / L;   // head vectors per warp-wide step
  constexpr int H2 = D / 2;     // offset of the second member of a rotation pair
  constexpr int kBatch = F8 ? kBatchF8 : kBatchBf16;
  const int lane = threadIdx.x & 31;
  launch_dependents();  // the attention kernel after this one may be scheduled as CTAs finish

  const bool with_q = p.q_out != nullptr;
  const int hd0 = with_q ? 0 : p.Hq;               // first head handled (Q heads only with q_out)
  const int nhead = p.Hq + 2 * p.Hkv - hd0;
  const int nstep = (nhead + HPI - 1) / HPI;
  const int64_t W = (int64_t)(p.Hq + 2 * p.Hkv) * D;
  const int li = lane % L;
  const int sub = lane / L;                        // head slot within a step

  uint4 qw[2], kw[2];  // norm weights of this lane's 16 values, bf16 pairs
  {
    const uint16_t* wk = p.k_norm_w + li * 8;
    const uint16_t* wq = with_q ? p.q_norm_w + li * 8 : wk;
    kw[0] = __ldg(reinterpret_cast<const uint4*>(wk));
    kw[1] = __ldg(reinterpret_cast<const uint4*>(wk + H2));
    qw[0] = __ldg(reinterpret_cast<const uint4*>(wq));
    qw[1] = __ldg(reinterpret_cast<const uint4*>(wq + H2));
  }

  // this warp's units: steps [u0, u_end) of the N x nstep (token, step) grid,
  // the same count for every warp so that all of them finish together
  int64_t u0 = ((int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5)) * p.steps_per_warp;
  const int64_t u_end = min((int64_t)p.N * nstep, u0 + p.steps_per_warp);
  if (u0 >= u_end) return;
  int t = (int)(u0 / nstep);
  int s_begin = (int)(u0 - (int64_t)t * nstep);
  for (;;) {
    const int s_end = (int)min((int64_t)nstep, s_begin + (u_end - u0));
    const uint16_t* row = p.qkv + (int64_t)t * W + (int64_t)hd0 * D + li * 8;

    // first batch of loads before anything that depends on the request lookup
    uint4 raw_a[kBatch], raw_b[kBatch];  // values 8*li.. and D/2 + 8*li.. of a head
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int hd = (s_begin + k) * HPI + sub;
      const bool in = s_begin + k < s_end && hd < nhead;
      const uint16_t* src = row + (int64_t)hd * D;
      raw_a[k] = in ? __ldg(reinterpret_cast<const uint4*>(src)) : make_uint4(0, 0, 0, 0);
      raw_b[k] = in ? __ldg(reinterpret_cast<const uint4*>(src + H2)) : make_uint4(0, 0, 0, 0);
    }

    // request of this token: 0 = none, 1 = Q only (region too small), 2 = Q and cache
    int ok = 0;
    int64_t slot = 0;
    float pos = 0.f;
    {
      int b = t, j = 0, n = 1;
      bool seq_ok = true;
      if (p.cu_seqlens) {
        int lo = 0, hi = p.B;  // largest b with cu[b] <= t
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (__ldg(p.cu_seqlens + mid) <= t) lo = mid; else hi = mid;
        }
        b = lo;
        const int c0 = __ldg(p.cu_seqlens + b);
        j = t - c0;
        n = __ldg(p.cu_seqlens + b + 1) - c0;
        seq_ok = j >= 0 && j < n;
        if (!seq_ok && lane == 0) set_status(p.status, ATTN_STATUS_SEQLENS);
        if (t == 0 && lane == 0 && __ldg(p.cu_seqlens + p.B) != p.N) set_status(p.status, ATTN_STATUS_SEQLENS);
      }
      if (seq_ok) {
        const ReqInfo r = load_request(p.kv, b, n);
        ok = 1;
        pos = (float)(r.cached + j);
        slot = r.valid ? cache_slot(p.kv, r, r.cached + j) : -1;
        if (slot >= 0)
          ok = 2;
        else if (lane == 0)
          set_status(p.status, ATTN_STATUS_CAPACITY);
      }
    }
    if (ok != 0) {  // warp-uniform

      // cos/sin of the 8 rotation pairs 8*li .. 8*li + 7 this lane's values belong to
      float cs[8], sn[8];
      pair_angles<D>(pos, p.freqs, lane, cs, sn);
      uint16_t* q_row = with_q ? p.q_out + (int64_t)t * p.Hq * D + li * 8 : nullptr;
      const int64_t cache_row = slot * p.Hkv * D + li * 8;

      for (int base = s_begin; base < s_end; base += kBatch) {
        if (base > s_begin) {
#pragma unroll
          for (int k = 0; k < kBatch; ++k) {
            const int hd = (base + k) * HPI + sub;
            const bool in = base + k < s_end && hd < nhead;
            const uint16_t* src = row + (int64_t)hd * D;
            raw_a[k] = in ? __ldg(reinterpret_cast<const uint4*>(src)) : make_uint4(0, 0, 0, 0);
            raw_b[k] = in ? __ldg(reinterpret_cast<const uint4*>(src + H2)) : make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          if (base + k >= s_end) break;  // warp-uniform
          const int hd = hd0 + (base + k) * HPI + sub;  // head index in the qkv row
          const bool live = hd < p.Hq + 2 * p.Hkv;
          const bool is_q = hd < p.Hq;
          const bool is_v = hd >= p.Hq + p.Hkv;
          // steps made only of V heads: bit copies into the cache
          const bool step_all_v = hd0 + (base + k) * HPI >= p.Hq + p.Hkv;
          if (step_all_v) {
            if (live && ok == 2) {
              const int64_t e0 = cache_row + (int64_t)(hd - p.Hq - p.Hkv) * D;
              if constexpr (F8) {
                float y[8];
                uint8_t* dst = static_cast<uint8_t*>(p.v_cache) + e0;
                unpack_bf16x8(raw_a[k], y);
                *reinterpret_cast<uint2*>(dst) = e4m3x8(y, p.inv_v);
                unpack_bf16x8(raw_b[k], y);
                *reinterpret_cast<uint2*>(dst + H2) = e4m3x8(y, p.inv_v);
              } else {
                uint16_t* dst = static_cast<uint16_t*>(p.v_cache) + e0;
                *reinterpret_cast<uint4*>(dst) = raw_a[k];
                *reinterpret_cast<uint4*>(dst + H2) = raw_b[k];
              }
            }
            continue;
          }
          float ra[8], rb[8];
          norm_rope_pair<D>(raw_a[k], raw_b[k], is_q ? qw[0] : kw[0], is_q ? qw[1] : kw[1], cs, sn, p.eps, ra, rb);
          if (!live) continue;
          const int64_t e0 = cache_row + (int64_t)(hd - (is_v ? p.Hq + p.Hkv : p.Hq)) * D;
          if (F8 && !is_q) {
            if (ok == 2) {
              uint8_t* dst = static_cast<uint8_t*>(is_v ? p.v_cache : p.k_cache) + e0;
              const float r = is_v ? p.inv_v : p.inv_k;
              float ya[8], yb[8];
              if (is_v) {
                unpack_bf16x8(raw_a[k], ya);
                unpack_bf16x8(raw_b[k], yb);
              }
              *reinterpret_cast<uint2*>(dst) = e4m3x8(is_v ? ya : ra, r);
              *reinterpret_cast<uint2*>(dst + H2) = e4m3x8(is_v ? yb : rb, r);
            }
            continue;
          }
          // the prepared Q is f16 next to an E4M3 cache (the prefill kernel's operand type), else bf16
          uint4 va, vb;
          if (is_v) {
            va = raw_a[k];
            vb = raw_b[k];
          } else if (F8) {
            va = make_uint4(pack_f16(ra[0], ra[1]), pack_f16(ra[2], ra[3]), pack_f16(ra[4], ra[5]), pack_f16(ra[6], ra[7]));
            vb = make_uint4(pack_f16(rb[0], rb[1]), pack_f16(rb[2], rb[3]), pack_f16(rb[4], rb[5]), pack_f16(rb[6], rb[7]));
          } else {
            va = make_uint4(pack_bf16(ra[0], ra[1]), pack_bf16(ra[2], ra[3]), pack_bf16(ra[4], ra[5]),
                            pack_bf16(ra[6], ra[7]));
            vb = make_uint4(pack_bf16(rb[0], rb[1]), pack_bf16(rb[2], rb[3]), pack_bf16(rb[4], rb[5]),
                            pack_bf16(rb[6], rb[7]));
          }
          uint16_t* dst = is_q ? q_row + (int64_t)hd * D
                               : static_cast<uint16_t*>(is_v ? p.v_cache : p.k_cache) + e0;
          if (is_q || ok == 2) {
            *reinterpret_cast<uint4*>(dst) = va;
            *reinterpret_cast<uint4*>(dst + H2) = vb;
          }
        }
      }
    }  // ok != 0
    u0 += s_end - s_begin;
    if (u0 >= u_end) break;
    ++t;
    s_begin = 0;
  }
}

}  // namespace

cudaError_t launch_prologue(const PrologueArgs& a, cudaStream_t stream) {
  if (a.N <= 0) return cudaSuccess;
  ProloguePar p;
  p.qkv = static_cast<const uint16_t*>(a.qkv);
  p.q_norm_w = static_cast<const uint16_t*>(a.q_norm_w);
  p.k_norm_w = static_cast<const uint16_t*>(a.k_norm_w);
  p.q_out = static_cast<uint16_t*>(a.q_out);
  p.cu_seqlens = a.cu_seqlens;
  p.k_cache = a.kv.k_cache;
  p.v_cache = a.kv.v_cache;
  const bool f8 = a.kv.kv_dtype == ATTN_KV_E4M3;
  p.inv_k = f8 ? 1.0f / a.kv.k_scale : 1.0f;
  p.inv_v = f8 ? 1.0f / a.kv.v_scale : 1.0f;
  p.kv = kv_index(a.kv);
  p.status = a.status;
  p.B = a.B;
  p.N = a.N;
  p.Hq = a.cfg.num_q_heads;
  p.Hkv = a.cfg.num_kv_heads;
  p.eps = a.cfg.rms_eps;
  p.freqs = a.freqs;
  // (token, step) units: a step covers 32 / (D/16) head vectors of a token.
  // Warps take equal runs of consecutive units, cut across token boundaries:
  // with more units than the resident warps (kMinBlocks blocks per SM) every
  // resident warp takes one run, else every unit gets a warp of its own (a
  // decode append is latency-bound: its steps run side by side).
  const int hpi = 512 / a.cfg.head_dim;
  const int nstep = (a.cfg.num_q_heads * (a.q_out ? 1 : 0) + 2 * a.cfg.num_kv_heads + hpi - 1) / hpi;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidDevice;
  const int64_t units = (int64_t)a.N * nstep;
  const int64_t resident = (int64_t)sms * kMinBlocks * kWarpsPerBlock;
  p.steps_per_warp = (units + resident - 1) / resident;
  const int64_t warps = (units + p.steps_per_warp - 1) / p.steps_per_warp;
  const dim3 grid((unsigned)((warps + kWarpsPerBlock - 1) / kWarpsPerBlock));
  if (a.cfg.head_dim == 128) {
    if (f8) kv_append_kernel<128, true><<<grid, kThreads, 0, stream>>>(p);
    else kv_append_kernel<128, false><<<grid, kThreads, 0, stream>>>(p);
  } else {
    if (f8) kv_append_kernel<64, true><<<grid, kThreads, 0, stream>>>(p);
    else kv_append_kernel<64, false><<<grid, kThreads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace gb300
