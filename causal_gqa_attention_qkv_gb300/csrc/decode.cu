// Decode: one new query token per request against its KV cache.
//
// Concept chapter section 4.2/4.3: decode reads the cached history for every
// new token and is memory-bandwidth bound; transformer-basics "Prefill vs
// Decode": attention of the new token to the cache is one more row of the
// lower-triangular attention matrix.  The grid is (split, KV head, request):
// each CTA streams one contiguous slice of one KV head's cache through shared
// memory exactly once (TMA, mbarrier pipeline of 3 bf16 or 6 E4M3 stages) and
// applies it to all Hq/Hkv query heads of the group at the same time, so
// every cached byte is read from HBM once per step.  Partial results (running max, sum, unscaled
// output) of the splits are merged by log-sum-exp in a second kernel.
// With k_norm_w set, the kernel also appends the new token's K and V: the CTA
// of each (request, KV head) whose split holds position c_b writes them (K
// normed and rotated, with the prologue kernel's arithmetic) before it loads
// its first tile, so the whole decode step is one launch (two with a merge).
#include "kernels.cuh"

namespace gb300 {

namespace {

constexpr int kKeysPerTile = 64;
#ifndef DECODE_F8_STAGES
#define DECODE_F8_STAGES 6
#endif
#ifndef DECODE_F8_MIN_BLOCKS
#define DECODE_F8_MIN_BLOCKS 2  // resident CTAs per SM the registers must allow
#endif
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;


struct DecodePar {
  const uint16_t* qkv;       // [B, W]
  const uint16_t* q_norm_w;  // [D]
  const uint16_t* k_norm_w;  // [D], or NULL: the cache already holds the new K/V
  void* k_cache;             // written only with k_norm_w
  void* v_cache;
  float inv_k, inv_v;        // E4M3: fp32(1 / scale), rounded on the host
  RopeFreqs freqs;
  float eps;
  int32_t W;
  uint16_t* out;
  float* part_o;
  float* part_ml;
  KvIndex kv;
  int32_t* status;
  int32_t Hq, Hkv, G, split_len, max_splits;
  float scale_log2;  // log2(e) / sqrt(D), times k_scale for an E4M3 cache
  float v_scale;     // 1, or v_scale for an E4M3 cache
};

// One K or V tile: 64 keys.  bf16: D / 64 boxes of 64 rows x 128 bytes
// (128-byte swizzled).  E4M3: one box of 64 rows x D bytes, 128-byte
// swizzled when D = 128, plain rows of 64 bytes when D = 64.
template <int D, bool F8>
struct DecodeLayout {
  static constexpr int kRegions = F8 ? 1 : D / 64;
  static constexpr int kRegionBytes = kKeysPerTile * (F8 ? D : 128);
  static constexpr int kTileBytes = kRegions * kRegionBytes;     // 64 keys x D entries
  // bytes in flight per CTA: 3 x 32 KB (bf16, D = 128) or 6 x 16 KB (E4M3),
  // two CTAs per SM either way
  static constexpr int kStages = F8 ? DECODE_F8_STAGES : 3;
  static constexpr int kStageBytes = 2 * kTileBytes;             // K + V
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kSmemBytes = kBarOffset + 2 * kStages * 8 + 1024;  // + alignment slack
};

// Byte offset of 16-byte chunk `chunk` of key row `key` in an E4M3 tile.
template <int D>
__device__ __forceinline__ uint32_t f8_off(uint32_t key, uint32_t chunk) {
  return D == 128 ? sw128(key, chunk) : key * (uint32_t)D + (chunk << 4);
}

__device__ __forceinline__ void named_sync_consumers() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// The new token of request b (position c_b): its K and V of KV head kh
// written to the cache by one warp in the prologue kernel's pair layout and
// arithmetic (lanes [0, D/16) K, lanes [D/16, D/8) V).  Each writer then
// orders its stores before later async-proxy (TMA) reads, and the
// __syncwarp hands that order to the lane that issues the tile loads.
template <int D, bool F8>
__device__ __forceinline__ void append_new_kv(const DecodePar& p, const ReqInfo& r, int b, int kh, int lane) {
  constexpr int L = D / 16, H2 = D / 2;
  const int li = lane % L, which = lane / L;  // 0: K, 1: V, else idle
  const int64_t slot = cache_slot(p.kv, r, r.cached);
  uint4 xa = make_uint4(0, 0, 0, 0), xb = xa;
  if (which < 2) {
    const uint16_t* src = p.qkv + (int64_t)b * p.W + (int64_t)(p.Hq + which * p.Hkv + kh) * D + li * 8;
    xa = __ldg(reinterpret_cast<const uint4*>(src));
    xb = __ldg(reinterpret_cast<const uint4*>(src + H2));
  }
  float cs[8], sn[8];
  pair_angles<D>((float)r.cached, p.freqs, lane, cs, sn);
  const uint4 wa = __ldg(reinterpret_cast<const uint4*>(p.k_norm_w + li * 8));
  const uint4 wb = __ldg(reinterpret_cast<const uint4*>(p.k_norm_w + li * 8 + H2));
  float ra[8], rb[8];
  norm_rope_pair<D>(xa, xb, wa, wb, cs, sn, p.eps, ra, rb);
  if (which < 2 && slot >= 0) {
    const int64_t e0 = (slot * p.Hkv + kh) * D + li * 8;
    if constexpr (F8) {
      uint8_t* dst = static_cast<uint8_t*>(which == 0 ? p.k_cache : p.v_cache) + e0;
      if (which == 0) {
        *reinterpret_cast<uint2*>(dst) = e4m3x8(ra, p.inv_k);
        *reinterpret_cast<uint2*>(dst + H2) = e4m3x8(rb, p.inv_k);
      } else {
        float y[8];
        unpack_bf16x8(xa, y);
        *reinterpret_cast<uint2*>(dst) = e4m3x8(y, p.inv_v);
        unpack_bf16x8(xb, y);
        *reinterpret_cast<uint2*>(dst + H2) = e4m3x8(y, p.inv_v);
      }
    } else {
      uint16_t* dst = static_cast<uint16_t*>(which == 0 ? p.k_cache : p.v_cache) + e0;
      if (which == 0) {
        xa = make_uint4(pack_bf16(ra[0], ra[1]), pack_bf16(ra[2], ra[3]), pack_bf16(ra[4], ra[5]),
                        pack_bf16(ra[6], ra[7]));
        xb = make_uint4(pack_bf16(rb[0], rb[1]), pack_bf16(rb[2], rb[3]), pack_bf16(rb[4], rb[5]),
                        pack_bf16(rb[6], rb[7]));
      }
      *reinterpret_cast<uint4*>(dst) = xa;
      *reinterpret_cast<uint4*>(dst + H2) = xb;
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }
  if (lane == 0 && slot < 0) set_status(p.status, ATTN_STATUS_CAPACITY);
  __syncwarp();
}

// F8: the cache holds E4M3 codes.  The tiles are converted to f16 in
// registers (exact) and the products run as f16 mma.sync.  Each lane then
// reads contiguous bytes: for Q.K^T, quad member c takes the columns
// [c D/4, (c+1) D/4) of its key row (the query fragments use the same column
// order); for P.V, lane (g, c) takes columns [g D/8, (g+1) D/8) of its four
// keys 2c, 2c+1, 2c+8, 2c+9, byte-interleaved in pairs of keys, so n-tile t
// of the output holds column g D/8 + t.
template <int D, bool F8>
__global__ void __launch_bounds__(kThreads, F8 ? DECODE_F8_MIN_BLOCKS : 0)
    decode_split_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodePar p) {
  using Lay = DecodeLayout<D, F8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kBarOffset);
  uint64_t* empty = full + Lay::kStages;
  __shared__ int s_abort;       // written by the producer only
  __shared__ int s_cons_abort;  // written by consumers only, read after their barrier

  const int split = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  launch_dependents();  // the merge kernel may be scheduled as CTAs finish
  const ReqInfo r = load_request(p.kv, b, 1);  // request facts: written by the caller, not by a kernel
  const bool append = p.k_norm_w != nullptr;
  if (!r.valid) {  // nothing written (with the append kernel before this one: flagged there)
    if (append && split == 0 && kh == 0 && threadIdx.x == 0) set_status(p.status, ATTN_STATUS_CAPACITY);
    return;
  }
  const int kv_len = r.cached + 1;
  const int n_splits = (kv_len + p.split_len - 1) / p.split_len;
  if (n_splits > p.max_splits) {  // max_cache_len below this request's length
    if (split == 0 && kh == 0 && threadIdx.x == 0) set_status(p.status, ATTN_STATUS_BOUNDS);
    if (append && split == p.max_splits - 1 && threadIdx.x < 32) {  // the new K/V are still appended
      grid_dependency_wait();
      append_new_kv<D, F8>(p, r, b, kh, threadIdx.x);
    }
    return;
  }
  if (split >= n_splits) return;
  const int k0 = split * p.split_len;
  const int k1 = min(k0 + p.split_len, kv_len);
  const int ntiles = (k1 - k0 + kKeysPerTile - 1) / kKeysPerTile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Lay::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    s_abort = 0;
    s_cons_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  grid_dependency_wait();  // the append kernel's cache entries, earlier kernels' reads of the outputs

  if (warp == kConsumerWarps) {  // producer warp: one thread issues all TMA loads
    if (append && split == n_splits - 1) append_new_kv<D, F8>(p, r, b, kh, lane);  // before the last tile's load
    if (lane == 0) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % Lay::kStages;
        if (i >= Lay::kStages && !mbar_wait(&empty[st], ((i / Lay::kStages) - 1) & 1)) {
          s_abort = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[st], Lay::kStageBytes);
        uint8_t* kt = smem + st * Lay::kStageBytes;
        uint8_t* vt = kt + Lay::kTileBytes;
        // a 64-key tile lies in one page; a page outside the cache reads as zeros
        int64_t slot = cache_slot(p.kv, r, k0 + i * kKeysPerTile);
        if (slot < 0) {
          set_status(p.status, ATTN_STATUS_CAPACITY);
          slot = 0;
        }
#pragma unroll
        for (int rg = 0; rg < Lay::kRegions; ++rg) {  // x: 64 bf16 (128 B) per box, or 0
          tma_load_3d(kt + rg * Lay::kRegionBytes, &kmap, &full[st], rg * 64, kh, (int)slot);
          tma_load_3d(vt + rg * Lay::kRegionBytes, &vmap, &full[st], rg * 64, kh, (int)slot);
        }
        issued = i + 1;
      }
      __syncwarp(1);
      // After a failed wait, let the copies still in flight land before exit.
      if (s_abort) {
        for (int i = max(0, issued - Lay::kStages); i < issued; ++i)
          (void)mbar_wait(&full[i % Lay::kStages], (i / Lay::kStages) & 1);
        set_status(p.status, ATTN_STATUS_TIMEOUT);
      }
    }
    return;
  }

  // ---------------- consumer warps: warp w owns keys [16w, 16w + 16) of each tile
  const int G = p.G;
  const int h0 = kh * G;
  const int qrow = lane >> 2;  // A/C fragment row of this thread (rows >= G are padding)
  uint32_t qa[D / 16][2];  // rows 0-7 of the A fragment; rows 8-15 are zero
  if constexpr (F8)
    q_row_frags_quarters<D>(p.qkv + (int64_t)b * p.W + (int64_t)(h0 + min(qrow, G - 1)) * D, qrow < G,
                            p.q_norm_w, p.eps, (float)r.cached, p.freqs, qa);
  else
    q_row_frags<D>(p.qkv + (int64_t)b * p.W + (int64_t)(h0 + min(qrow, G - 1)) * D, qrow < G,
                   p.q_norm_w, p.eps, (float)r.cached, p.freqs, qa);
  const int qc = lane & 3;  // quad member
  // E4M3: transposed products, O^T = V^T P^T and S^T = K Q^T: the warp's 16
  // keys of a tile are the M dimension and the group's heads the N dimension
  // (8, heads >= G are zero padding), so one m16n8k16 covers 16 keys.  The
  // d order inside a product is free as long as both operands agree: for
  // S^T, quad member q takes d in [q D/4, (q+1) D/4) (the Q fragments use
  // the same order); for O^T, lane (g, q) holds d in [g D/8, (g+1) D/8) of
  // heads 2q, 2q+1.  Every lane reads contiguous codes from shared memory.
  constexpr int MT = D / 16;   // m-tiles of O^T
  float o[F8 ? MT : D / 8][4];
#pragma unroll
  for (int i = 0; i < (F8 ? MT : D / 8); ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m = kNegInf, l = 0.f;
  float mh[2] = {kNegInf, kNegInf}, lh[2] = {0.f, 0.f};  // E4M3: heads 2q, 2q+1
  bool ok = true;

  if constexpr (F8) {
    constexpr int S = Lay::kStages;
    constexpr int KW = D / 16;  // 32-bit code words of a key per quad member
    const int g = qrow;
    // two 64-key tiles per pass: one softmax reduction and one O rescale per 128 keys
    for (int i = 0; i < ntiles; i += 2) {
      const bool two = i + 1 < ntiles;
      const int st0 = i % S, st1 = (i + 1) % S;
      if (!mbar_wait(&full[st0], (i / S) & 1) || (two && !mbar_wait(&full[st1], ((i + 1) / S) & 1))) {
        ok = false;
        break;
      }
      // Without a second tile, stage st1 holds an older tile or nothing and no
      // copy is in flight into it; all of its keys lie past k1 and are masked.
      const uint32_t kb[2] = {smem_u32(smem + st0 * Lay::kStageBytes), smem_u32(smem + st1 * Lay::kStageBytes)};
      float s[2][4];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        // codes of keys g and g + 8, columns [q D/4, (q+1) D/4)
        uint32_t kw[2][KW];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int hc = 0; hc < D / 64; ++hc) {
            const uint4 raw = lds128(kb[t] + f8_off<D>(warp * 16 + g + 8 * r, qc * (D / 64) + hc));
            kw[r][4 * hc] = raw.x;
            kw[r][4 * hc + 1] = raw.y;
            kw[r][4 * hc + 2] = raw.z;
            kw[r][4 * hc + 3] = raw.w;
          }
        s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KW; ++ks) {
          uint32_t a[4];  // rows g, g + 8; columns 2q, 2q + 1 (a0, a1) and 2q + 8, 2q + 9 (a2, a3)
          e4m3x4_to_f16(kw[0][ks], a[0], a[2]);
          e4m3x4_to_f16(kw[1][ks], a[1], a[3]);
          mma_f16_16816(s[t], a, qa[ks][0], qa[ks][1]);
        }
      }
      // s[t]: key g (c0: head 2q, c1: head 2q + 1) and key g + 8 (c2, c3)
      float sc[2][4];
      int kg[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        kg[t] = k0 + (i + t) * kKeysPerTile + warp * 16 + g;
        sc[t][0] = kg[t] < k1 ? s[t][0] * p.scale_log2 : kNegInf;
        sc[t][1] = kg[t] < k1 ? s[t][1] * p.scale_log2 : kNegInf;
        sc[t][2] = kg[t] + 8 < k1 ? s[t][2] * p.scale_log2 : kNegInf;
        sc[t][3] = kg[t] + 8 < k1 ? s[t][3] * p.scale_log2 : kNegInf;
      }
      float alpha[2], m_use[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {  // head 2q + e: maximum over the warp's keys
        float mx = fmaxf(fmaxf(sc[0][e], sc[0][2 + e]), fmaxf(sc[1][e], sc[1][2 + e]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float m_new = fmaxf(mh[e], mx);
        m_use[e] = m_new == kNegInf ? 0.f : m_new;
        alpha[e] = fast_exp2(mh[e] - m_use[e]);
        mh[e] = m_new;
      }
      float pr[2][4], rs[2] = {0.f, 0.f};
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pr[t][e] = fast_exp2(sc[t][e] - m_use[e & 1]);
          rs[e & 1] += pr[t][e];
        }
#pragma unroll
      for (int e = 0; e < 2; ++e) lh[e] = lh[e] * alpha[e] + rs[e];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        o[mt][0] *= alpha[0];
        o[mt][1] *= alpha[1];
        o[mt][2] *= alpha[0];
        o[mt][3] *= alpha[1];
      }
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        // P^T as the B operand: the 8 x 8 blocks (keys g | g + 8, heads 2q, 2q + 1) transposed
        uint32_t pb0, pb1;
        asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(pb0) : "r"(pack_f16(pr[t][0], pr[t][1])));
        asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(pb1) : "r"(pack_f16(pr[t][2], pr[t][3])));
        // V codes of keys 2q, 2q + 1, 2q + 8, 2q + 9, columns [g D/8, (g+1) D/8)
        const uint32_t vb = kb[t] + Lay::kTileBytes;
        constexpr int VW = D / 32;  // 32-bit words per key
        uint32_t v4[4][VW];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int key = warp * 16 + 2 * qc + (q4 & 1) + (q4 >> 1) * 8;
          if constexpr (D == 128) {
            const uint4 v = lds128(vb + f8_off<D>(key, g));
            v4[q4][0] = v.x; v4[q4][1] = v.y; v4[q4][2] = v.z; v4[q4][3] = v.w;
          } else {
            const uint2 v = lds64(vb + key * (uint32_t)D + g * 8);
            v4[q4][0] = v.x; v4[q4][1] = v.y;
          }
        }
        // keys past the end hold arbitrary bits: zero their V entries so 0 * NaN cannot occur
        const int kq = k0 + (i + t) * kKeysPerTile + warp * 16 + 2 * qc;
        const bool partial = k0 + (i + t) * kKeysPerTile + warp * 16 + 16 > k1;
        const uint32_t mAB = (kq < k1 ? 0x0000FFFFu : 0u) | (kq + 1 < k1 ? 0xFFFF0000u : 0u);
        const uint32_t mCD = (kq + 8 < k1 ? 0x0000FFFFu : 0u) | (kq + 9 < k1 ? 0xFFFF0000u : 0u);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          // rows g / g + 8 of m-tile mt: d = g D/8 + 2 mt and + 1 (bytes 2 mt, 2 mt + 1 of the run)
          const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
          uint32_t a[4];
          e4m3x4_to_f16(prmt(v4[0][mt >> 1], v4[1][mt >> 1], sel), a[0], a[1]);
          e4m3x4_to_f16(prmt(v4[2][mt >> 1], v4[3][mt >> 1], sel), a[2], a[3]);
          if (partial) {
            a[0] &= mAB;
            a[1] &= mAB;
            a[2] &= mCD;
            a[3] &= mCD;
          }
          mma_f16_16816(o[mt], a, pb0, pb1);
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&empty[st0]);
        if (two) mbar_arrive(&empty[st1]);
      }
    }
  } else
  for (int i = 0; i < ntiles; ++i) {
    const int st = i % Lay::kStages;
    if (!mbar_wait(&full[st], (i / Lay::kStages) & 1)) {
      ok = false;
      break;
    }
    const uint32_t kb = smem_u32(smem + st * Lay::kStageBytes);
    const uint32_t vb = kb + Lay::kTileBytes;
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int mi = lane >> 3;
        const int key = warp * 16 + (mi >> 1) * 8 + (lane & 7);
        const int chunk = 2 * ks + (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + (chunk >> 3) * Lay::kRegionBytes + sw128(key, chunk & 7), b0, b1, b2, b3);
        const uint32_t a[4] = {qa[ks][0], 0u, qa[ks][1], 0u};
        mma_bf16_16816(s[0], a, b0, b1);
        mma_bf16_16816(s[1], a, b2, b3);
      }
    }
    const int kfirst = k0 + i * kKeysPerTile + warp * 16;  // first key of this warp's slice
    const int kA = kfirst + 2 * (lane & 3);
    float sc[4];
    sc[0] = kA < k1 ? s[0][0] * p.scale_log2 : kNegInf;
    sc[1] = kA + 1 < k1 ? s[0][1] * p.scale_log2 : kNegInf;
    sc[2] = kA + 8 < k1 ? s[1][0] * p.scale_log2 : kNegInf;
    sc[3] = kA + 9 < k1 ? s[1][1] * p.scale_log2 : kNegInf;
    float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m, mx);
    const float m_use = m_new == kNegInf ? 0.f : m_new;
    const float alpha = fast_exp2(m - m_use);
    float pr[4], rs = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      pr[e] = fast_exp2(sc[e] - m_use);
      rs += pr[e];
    }
    l = l * alpha + rs;
    m = m_new;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
      o[dt][0] *= alpha;
      o[dt][1] *= alpha;
    }
    // keys past the end hold arbitrary bits: zero their V entries so 0 * NaN cannot occur
    const bool partial = kfirst + 16 > k1;
    const uint32_t mA = (kA < k1 ? 0x0000FFFFu : 0u) | (kA + 1 < k1 ? 0xFFFF0000u : 0u);
    const uint32_t mB = (kA + 8 < k1 ? 0x0000FFFFu : 0u) | (kA + 9 < k1 ? 0xFFFF0000u : 0u);
    {
    const uint32_t pa[4] = {pack_bf16(pr[0], pr[1]), 0u, pack_bf16(pr[2], pr[3]), 0u};
#pragma unroll
    for (int dp = 0; dp < D / 16; ++dp) {
      const int mi = lane >> 3;
      const int key = warp * 16 + (mi & 1) * 8 + (lane & 7);
      const int chunk = 2 * dp + (mi >> 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vb + (chunk >> 3) * Lay::kRegionBytes + sw128(key, chunk & 7), b0, b1, b2, b3);
      if (partial) {
        b0 &= mA; b2 &= mA;
        b1 &= mB; b3 &= mB;
      }
      mma_bf16_16816(o[2 * dp], pa, b0, b1);
      mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
    }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
  if (!ok) {
    s_cons_abort = 1;
    set_status(p.status, ATTN_STATUS_TIMEOUT);
  }
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
#pragma unroll
  for (int e = 0; e < 2; ++e) {  // E4M3: the head's sum over the warp's keys
    lh[e] += __shfl_xor_sync(0xffffffffu, lh[e], 4);
    lh[e] += __shfl_xor_sync(0xffffffffu, lh[e], 8);
    lh[e] += __shfl_xor_sync(0xffffffffu, lh[e], 16);
  }

  // ---------------- merge the four warps' partial softmax states
  named_sync_consumers();  // every consumer is done with the stage buffers
  if (s_cons_abort) return;  // same value for every consumer thread
  float* mo = reinterpret_cast<float*>(smem);                 // [warps][G][D]
  float* mm = mo + kConsumerWarps * G * D;                      // [warps][G]
  float* ml = mm + kConsumerWarps * G;                          // [warps][G]
  if constexpr (F8) {
    // lane (g, q): heads 2q, 2q + 1, d in [g D/8, (g+1) D/8)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int head = 2 * qc + e;
      if (head < G) {
        float* dst = mo + (warp * G + head) * D + qrow * (D / 8);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          dst[2 * mt] = o[mt][e] * p.v_scale;
          dst[2 * mt + 1] = o[mt][2 + e] * p.v_scale;
        }
        if (qrow == 0) {
          mm[warp * G + head] = mh[e];
          ml[warp * G + head] = lh[e];
        }
      }
    }
  } else if (qrow < G) {
    float* dst = mo + (warp * G + qrow) * D;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
      dst[dt * 8 + 2 * qc] = o[dt][0];
      dst[dt * 8 + 2 * qc + 1] = o[dt][1];
    }
    if ((lane & 3) == 0) {
      mm[warp * G + qrow] = m;
      ml[warp * G + qrow] = l;
    }
  }
  named_sync_consumers();
  const bool direct = n_splits == 1;
  for (int idx = threadIdx.x; idx < G * D; idx += kConsumerWarps * 32) {
    const int row = idx / D, d = idx % D;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mm[w * G + row]);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float sw = fast_exp2(mm[w * G + row] - M);
      L += sw * ml[w * G + row];
      acc += sw * mo[(w * G + row) * D + d];
    }
    const int64_t hrow = (int64_t)b * p.Hq + h0 + row;
    if (direct) {
      const __nv_bfloat16 v = __float2bfloat16_rn(acc / L);
      p.out[hrow * D + d] = *reinterpret_cast<const uint16_t*>(&v);
    } else {
      const int64_t prow = hrow * p.max_splits + split;
      p.part_o[prow * D + d] = acc;
      if (d == 0) {
        p.part_ml[prow * 2] = M;
        p.part_ml[prow * 2 + 1] = L;
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const DecodePar p) {
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  grid_dependency_wait();  // the split kernel's partial results
  const ReqInfo r = load_request(p.kv, b, 1);
  if (!r.valid) return;
  const int n = (r.cached + 1 + p.split_len - 1) / p.split_len;
  if (n <= 1 || n > p.max_splits) return;  // written directly / flagged by the split kernel
  const int64_t row = (int64_t)b * p.Hq + h;
  const float* ml = p.part_ml + row * p.max_splits * 2;
  float M = kNegInf;
  for (int s = 0; s < n; ++s) M = fmaxf(M, ml[2 * s]);
  float L = 0.f, acc = 0.f;
  for (int s = 0; s < n; ++s) {
    const float w = fast_exp2(ml[2 * s] - M);
    L += w * ml[2 * s + 1];
    acc += w * p.part_o[(row * p.max_splits + s) * D + d];
  }
  const __nv_bfloat16 v = __float2bfloat16_rn(acc / L);
  p.out[row * D + d] = *reinterpret_cast<const uint16_t*>(&v);
}

template <int D, bool F8>
int launch_decode_t(const DecodeArgs& a, cudaStream_t stream) {
  using Lay = DecodeLayout<D, F8>;
  CacheMaps maps;
  if (make_cache_maps(a.kv, a.cfg.num_kv_heads, D, kKeysPerTile, &maps) != 0) return ATTN_ELAUNCH;
  DecodePar p;
  p.qkv = static_cast<const uint16_t*>(a.qkv);
  p.q_norm_w = static_cast<const uint16_t*>(a.q_norm_w);
  p.k_norm_w = static_cast<const uint16_t*>(a.k_norm_w);
  p.k_cache = a.kv.k_cache;
  p.v_cache = a.kv.v_cache;
  p.inv_k = F8 ? 1.0f / a.kv.k_scale : 1.0f;
  p.inv_v = F8 ? 1.0f / a.kv.v_scale : 1.0f;
  p.freqs = a.freqs;
  p.eps = a.cfg.rms_eps;
  p.W = (a.cfg.num_q_heads + 2 * a.cfg.num_kv_heads) * D;
  p.out = static_cast<uint16_t*>(a.out);
  p.part_o = a.part_o;
  p.part_ml = a.part_ml;
  p.kv = kv_index(a.kv);
  p.status = a.status;
  p.Hq = a.cfg.num_q_heads;
  p.Hkv = a.cfg.num_kv_heads;
  p.G = a.cfg.num_q_heads / a.cfg.num_kv_heads;
  p.split_len = a.split_len;
  p.max_splits = a.max_splits;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)D) * (F8 ? a.kv.k_scale : 1.0f);
  p.v_scale = F8 ? a.kv.v_scale : 1.0f;
  if (cudaFuncSetAttribute(decode_split_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Lay::kSmemBytes) != cudaSuccess)
    return ATTN_ELAUNCH;
  dim3 grid(a.max_splits, a.cfg.num_kv_heads, a.B);
  if (launch_dependent(decode_split_kernel<D, F8>, grid, dim3(kThreads), Lay::kSmemBytes, stream, maps.k, maps.v,
                       p) != cudaSuccess)
    return ATTN_ELAUNCH;
  if (a.max_splits > 1 && launch_dependent(decode_combine_kernel<D>, dim3(a.cfg.num_q_heads, a.B), dim3(D), 0,
                                           stream, p) != cudaSuccess)
    return ATTN_ELAUNCH;
  return ATTN_OK;
}

}  // namespace

// Keys per split: enough CTAs to fill 152 SMs several times over when every
// request is at its longest, at least 256 keys, and at most 16 splits.
int decode_split_len(int B, int Hkv, int max_kv_len, int* max_splits) {
  const int64_t target_ctas = 2048;
  int64_t len = ((int64_t)max_kv_len * B * Hkv + target_ctas - 1) / target_ctas;
  len = std::max<int64_t>(len, 256);
  len = std::max<int64_t>(len, ((int64_t)max_kv_len + 15) / 16);
  len = (len + 63) / 64 * 64;
  *max_splits = (int)std::max<int64_t>(1, ((int64_t)max_kv_len + len - 1) / len);
  return (int)len;
}

int launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.B <= 0) return ATTN_OK;
  const bool f8 = a.kv.kv_dtype == ATTN_KV_E4M3;
  if (a.cfg.head_dim == 128) return f8 ? launch_decode_t<128, true>(a, stream) : launch_decode_t<128, false>(a, stream);
  return f8 ? launch_decode_t<64, true>(a, stream) : launch_decode_t<64, false>(a, stream);
}

}  // namespace gb300
