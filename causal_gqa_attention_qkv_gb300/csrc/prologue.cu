// Prologue of the attention step: split qkv, RMSNorm + RoPE on K (and on Q
// when a Q output is given), write K and V to the cache (and the prepared Q).
//
// Zero-to-sglang Ch.3 code walkthrough, section 3.3: AttentionLayer.forward
// splits the merged projection into Q, K and V, applies RMSNorm to each Q/K
// head's last dimension and RoPE at each token's position (V is not rotated);
// transformer-basics "Prefill vs Decode": the new K/V are appended to the
// per-layer cache (past_key_values.update).  One pass: every (token, head)
// vector of D bf16 values is read once with 16-byte loads by a group of D/8
// lanes, reduced with warp shuffles, and written once.
#include "kernels.cuh"

namespace gb300 {

namespace {

constexpr int kTokPerBlock = 8;
constexpr int kThreads = 256;

struct ProloguePar {
  const uint16_t* __restrict__ qkv;        // [N, W] bf16
  const uint16_t* __restrict__ q_norm_w;   // [D] bf16 (used when q_out != NULL)
  const uint16_t* __restrict__ k_norm_w;   // [D] bf16
  uint16_t* __restrict__ q_out;            // [N, Hq, D] bf16 or NULL
  const int32_t* cu_seqlens;  // [B+1] or NULL: token b is request b (decode)
  uint16_t* __restrict__ k_cache;
  uint16_t* __restrict__ v_cache;
  const int64_t* slot_base;
  const int32_t* cache_lens;
  const int32_t* slot_capacity;
  int64_t num_slots;
  int32_t* status;
  int32_t B, N, Hq, Hkv;
  float eps;
  RopeFreqs freqs;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 4) kv_append_kernel(const ProloguePar p) {
  constexpr int L = D / 8;     // lanes per head vector (8 bf16 = 16 bytes each)
  constexpr int HALF = D / 2;  // rotation pairs
  constexpr int kGroups = kThreads / L;
  __shared__ float s_cos[kTokPerBlock][HALF];
  __shared__ float s_sin[kTokPerBlock][HALF];
  __shared__ int64_t s_slot[kTokPerBlock];
  __shared__ float s_pos[kTokPerBlock];
  __shared__ int s_ok[kTokPerBlock];  // 1: token exists; 2: it may also write the cache

  const int t0 = blockIdx.x * kTokPerBlock;
  if (threadIdx.x < kTokPerBlock) {
    const int tk = threadIdx.x, t = t0 + tk;
    int ok = 0;
    int64_t slot = 0;
    float pos = 0.f;
    if (t < p.N) {
      int b = t, j = 0, n = 1;
      bool seq_ok = true;
      if (p.cu_seqlens) {
        int lo = 0, hi = p.B;  // largest b with cu[b] <= t
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (p.cu_seqlens[mid] <= t) lo = mid; else hi = mid;
        }
        b = lo;
        j = t - p.cu_seqlens[b];
        n = p.cu_seqlens[b + 1] - p.cu_seqlens[b];
        seq_ok = j >= 0 && j < n;
        if (!seq_ok) set_status(p.status, ATTN_STATUS_SEQLENS);
      }
      if (seq_ok) {
        const ReqInfo r = load_request(p.slot_base + b, p.cache_lens + b, p.slot_capacity + b,
                                       p.num_slots, n);
        ok = 1;
        pos = (float)(r.cached + j);
        if (r.valid) {
          ok = 2;
          slot = r.slot0 + r.cached + j;
        } else {
          set_status(p.status, ATTN_STATUS_CAPACITY);
        }
      }
    }
    if (p.cu_seqlens && t == 0 && p.cu_seqlens[p.B] != p.N) set_status(p.status, ATTN_STATUS_SEQLENS);
    s_ok[tk] = ok;
    s_slot[tk] = slot;
    s_pos[tk] = pos;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kTokPerBlock * HALF; i += kThreads) {
    const int tk = i / HALF, pr = i % HALF;
    float c, s;
    rope_angle(s_pos[tk], p.freqs.hi[pr], p.freqs.lo[pr], p.freqs, &c, &s);
    s_cos[tk][pr] = c;
    s_sin[tk][pr] = s;
  }
  __syncthreads();

  const int64_t W = (int64_t)(p.Hq + 2 * p.Hkv) * D;
  const int lane = threadIdx.x & 31;
  const int li = lane % L;  // lane within the head group
  const int group = threadIdx.x / L;
  const unsigned gmask = (L == 32) ? 0xffffffffu : (((1u << L) - 1u) << (lane - li));
  const bool first_half = li < L / 2;
  const int pair0 = (first_half ? li : li - L / 2) * 8;  // first rotation pair of this lane
  const uint4 kw4 = __ldg(reinterpret_cast<const uint4*>(p.k_norm_w + li * 8));
  const uint4 qw4 = p.q_out ? __ldg(reinterpret_cast<const uint4*>(p.q_norm_w + li * 8)) : kw4;

  // heads of a token handled here: K heads, V heads, then (with q_out) Q heads
  const int nq = p.q_out ? p.Hq : 0;
  const int nhead = 2 * p.Hkv + nq;
  const int ntask = kTokPerBlock * nhead;
  constexpr int kMaxTasks = 6;  // tasks per group held in flight (loads issued first)
  for (int base = 0; base < ntask; base += kGroups * kMaxTasks) {
    uint4 raw[kMaxTasks];
#pragma unroll
    for (int k = 0; k < kMaxTasks; ++k) {
      const int task = base + group + k * kGroups;
      raw[k] = make_uint4(0, 0, 0, 0);
      if (task < ntask) {
        const int tk = task / nhead, hd = task % nhead;
        // Q heads are prepared even for a request whose cache region is too
        // small (s_ok == 1): only the cache writes are withheld there
        const int col = hd < 2 * p.Hkv ? p.Hq + hd : hd - 2 * p.Hkv;
        if (s_ok[tk] == 2 || (s_ok[tk] == 1 && hd >= 2 * p.Hkv))
          raw[k] = __ldg(reinterpret_cast<const uint4*>(p.qkv + (int64_t)(t0 + tk) * W +
                                                          (int64_t)col * D + li * 8));
      }
    }
#pragma unroll
    for (int k = 0; k < kMaxTasks; ++k) {
      const int task = base + group + k * kGroups;  // whole groups move together
      if (task >= ntask) break;
      const int tk = task / nhead, hd = task % nhead;
      const bool is_q = hd >= 2 * p.Hkv;
      if (s_ok[tk] == 0 || (!is_q && s_ok[tk] != 2)) continue;
      const bool is_k = hd < p.Hkv;
      const int kvh = is_k ? hd : hd - p.Hkv;
      const int64_t dst = is_q ? ((int64_t)(t0 + tk) * p.Hq + (hd - 2 * p.Hkv)) * D + li * 8
                               : (s_slot[tk] * p.Hkv + kvh) * D + li * 8;
      if (!is_k && !is_q) {  // V: bit copy into the cache
        *reinterpret_cast<uint4*>(p.v_cache + dst) = raw[k];
        continue;
      }
      float x[8];
      const uint32_t* rw = reinterpret_cast<const uint32_t*>(&raw[k]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[2 * e] = bf16_lo(rw[e]);
        x[2 * e + 1] = bf16_hi(rw[e]);
      }
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
      for (int off = L / 2; off >= 1; off >>= 1) ss += __shfl_xor_sync(gmask, ss, off);
      const float inv = rsqrtf(ss * (1.0f / D) + p.eps);
      const uint32_t* ww = reinterpret_cast<const uint32_t*>(is_q ? &qw4 : &kw4);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[2 * e] = bf16_lo(ww[e]) * (x[2 * e] * inv);
        x[2 * e + 1] = bf16_hi(ww[e]) * (x[2 * e + 1] * inv);
      }
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const float y0 = x[e], y1 = x[e + 1];
        const float q0 = __shfl_xor_sync(gmask, y0, L / 2);
        const float q1 = __shfl_xor_sync(gmask, y1, L / 2);
        const float c0 = s_cos[tk][pair0 + e], s0 = s_sin[tk][pair0 + e];
        const float c1 = s_cos[tk][pair0 + e + 1], s1 = s_sin[tk][pair0 + e + 1];
        float r0, r1;
        if (first_half) {
          r0 = y0 * c0 - q0 * s0;
          r1 = y1 * c1 - q1 * s1;
        } else {
          r0 = y0 * c0 + q0 * s0;
          r1 = y1 * c1 + q1 * s1;
        }
        o[e / 2] = pack_bf16(r0, r1);
      }
      *reinterpret_cast<uint4*>((is_q ? p.q_out : p.k_cache) + dst) = make_uint4(o[0], o[1], o[2], o[3]);
    }
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
  p.k_cache = static_cast<uint16_t*>(a.kv.k_cache);
  p.v_cache = static_cast<uint16_t*>(a.kv.v_cache);
  p.slot_base = a.kv.slot_base;
  p.cache_lens = a.kv.cache_lens;
  p.slot_capacity = a.kv.slot_capacity;
  p.num_slots = a.kv.num_slots;
  p.status = a.status;
  p.B = a.B;
  p.N = a.N;
  p.Hq = a.cfg.num_q_heads;
  p.Hkv = a.cfg.num_kv_heads;
  p.eps = a.cfg.rms_eps;
  p.freqs = a.freqs;
  const dim3 grid((a.N + kTokPerBlock - 1) / kTokPerBlock);
  if (a.cfg.head_dim == 128)
    kv_append_kernel<128><<<grid, kThreads, 0, stream>>>(p);
  else
    kv_append_kernel<64><<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gb300
