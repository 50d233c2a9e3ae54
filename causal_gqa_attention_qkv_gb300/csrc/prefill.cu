// Prefill: causal grouped-query attention over ragged packed sequences.
//
// Code walkthrough section 3.3 teaching snippet and transformer-basics
// "Attention calculation: part 1": scores q.k / sqrt(D) against the KV head
// h / (Hq/Hkv), future positions masked, softmax in fp32, weights times V;
// concept chapter section 2.6: computed the I/O-aware way (flash attention),
// never materialising the score matrix.  A CTA owns 64 query rows packed as
// (token, group head) pairs of one KV head, so each K/V tile it loads serves
// all Hq/Hkv query heads of the group; KV tiles beyond the last row's causal
// limit are never loaded.
#include "kernels.cuh"

namespace gb300 {

namespace {

constexpr int kKeysPerTile = 64;
constexpr int kRowsPerCta = 64;
constexpr int kStages = 3;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;


struct PrefillPar {
  const uint16_t* qkv;       // [N, W]
  const uint16_t* q_norm_w;  // [D]
  RopeFreqs freqs;
  float eps;
  int32_t W;
  uint16_t* out;
  const int32_t* cu_seqlens;
  const int64_t* slot_base;
  const int32_t* cache_lens;
  const int32_t* slot_capacity;
  int64_t num_slots;
  int32_t* status;
  int32_t Hq, log2G, N;
  float scale_log2;
};

template <int D>
struct PrefillLayout {
  static constexpr int kRegions = D / 64;
  static constexpr int kRegionBytes = kKeysPerTile * 128;
  static constexpr int kTileBytes = kRegions * kRegionBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kSmemBytes = kBarOffset + 2 * kStages * 8 + 1024;
};

template <int D>
__global__ void __launch_bounds__(kThreads)
    prefill_sync_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const PrefillPar p) {
  using Lay = PrefillLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kBarOffset);
  uint64_t* empty = full + kStages;
  __shared__ int s_abort;

  const int kh = blockIdx.y, b = blockIdx.z;
  const int tokbase = p.cu_seqlens[b];
  const int n_b = p.cu_seqlens[b + 1] - tokbase;
  if (n_b <= 0) return;
  if (tokbase < 0 || tokbase + n_b > p.N) {  // flagged by kv_append as well
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) set_status(p.status, ATTN_STATUS_SEQLENS);
    return;
  }
  const ReqInfo r = load_request(p.slot_base + b, p.cache_lens + b, p.slot_capacity + b,
                                 p.num_slots, n_b);
  if (!r.valid) return;  // flagged by the prologue
  const int G = 1 << p.log2G;
  const int tok_per_cta = kRowsPerCta >> p.log2G;
  const int ntile_b = (n_b + tok_per_cta - 1) / tok_per_cta;
  if (ntile_b > (int)gridDim.x) {  // max_seqlen below this sequence's length
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) set_status(p.status, ATTN_STATUS_BOUNDS);
    return;
  }
  if ((int)blockIdx.x >= ntile_b) return;
  const int t0 = (ntile_b - 1 - blockIdx.x) * tok_per_cta;  // heaviest tiles first
  const int t_hi = min(t0 + tok_per_cta, n_b);
  const int kv_total = r.cached + n_b;
  const int nk = (r.cached + t_hi + kKeysPerTile - 1) / kKeysPerTile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int st = i % kStages;
        if (i >= kStages && !mbar_wait(&empty[st], ((i / kStages) - 1) & 1)) {
          s_abort = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[st], Lay::kStageBytes);
        uint8_t* kt = smem + st * Lay::kStageBytes;
        uint8_t* vt = kt + Lay::kTileBytes;
        const int slot = (int)(r.slot0 + i * kKeysPerTile);
#pragma unroll
        for (int rg = 0; rg < Lay::kRegions; ++rg) {
          tma_load_3d(kt + rg * Lay::kRegionBytes, &kmap, &full[st], rg * 64, kh, slot);
          tma_load_3d(vt + rg * Lay::kRegionBytes, &vmap, &full[st], rg * 64, kh, slot);
        }
        issued = i + 1;
      }
      if (s_abort) {
        for (int i = max(0, issued - kStages); i < issued; ++i)
          (void)mbar_wait(&full[i % kStages], (i / kStages) & 1);
        set_status(p.status, ATTN_STATUS_TIMEOUT);
      }
    }
    return;
  }

  // ---------------- consumers: warp w owns query rows [16w, 16w + 16) of the CTA
  const int rA = warp * 16 + (lane >> 2), rB = rA + 8;
  const int tokA = t0 + (rA >> p.log2G), tokB = t0 + (rB >> p.log2G);
  const int hA = kh * G + (rA & (G - 1)), hB = kh * G + (rB & (G - 1));
  // Largest key each row may see: its own position (rows past the sequence
  // end are computed against every key and discarded).
  const int limA = tokA < n_b ? r.cached + tokA : kv_total - 1;
  const int limB = tokB < n_b ? r.cached + tokB : kv_total - 1;

  uint32_t qa[D / 16][4];
  {
    const bool vA = tokA < n_b, vB = tokB < n_b;
    uint32_t fa[D / 16][2], fb[D / 16][2];
    q_row_frags<D>(p.qkv + (int64_t)(tokbase + (vA ? tokA : 0)) * p.W + (int64_t)hA * D, vA,
                   p.q_norm_w, p.eps, (float)(r.cached + tokA), p.freqs, fa);
    q_row_frags<D>(p.qkv + (int64_t)(tokbase + (vB ? tokB : 0)) * p.W + (int64_t)hB * D, vB,
                   p.q_norm_w, p.eps, (float)(r.cached + tokB), p.freqs, fb);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qa[ks][0] = fa[ks][0];
      qa[ks][1] = fb[ks][0];
      qa[ks][2] = fa[ks][1];
      qa[ks][3] = fb[ks][1];
    }
  }
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mA = kNegInf, mB = kNegInf, lA = 0.f, lB = 0.f;
  bool ok = true;
  const int cta_min_lim = r.cached + t0;  // smallest limit of any row of the CTA

  for (int i = 0; i < nk; ++i) {
    const int st = i % kStages;
    if (!mbar_wait(&full[st], (i / kStages) & 1)) {
      ok = false;
      break;
    }
    const uint32_t kb = smem_u32(smem + st * Lay::kStageBytes);
    const uint32_t vb = kb + Lay::kTileBytes;
    const int kv0 = i * kKeysPerTile;
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int mi = lane >> 3;
        const int key = np * 16 + (mi >> 1) * 8 + (lane & 7);
        const int chunk = 2 * ks + (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + (chunk >> 3) * Lay::kRegionBytes + sw128(key, chunk & 7), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * np], qa[ks], b0, b1);
        mma_bf16_16816(s[2 * np + 1], qa[ks], b2, b3);
      }
    }
    const bool masked = kv0 + kKeysPerTile - 1 > cta_min_lim;
    float mxA = kNegInf, mxB = kNegInf;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const int key = kv0 + n * 8 + 2 * (lane & 3);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float a = s[n][e] * p.scale_log2, c = s[n][2 + e] * p.scale_log2;
        if (masked) {
          a = key + e <= limA ? a : kNegInf;
          c = key + e <= limB ? c : kNegInf;
        }
        s[n][e] = a;
        s[n][2 + e] = c;
        mxA = fmaxf(mxA, a);
        mxB = fmaxf(mxB, c);
      }
    }
    mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
    mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
    mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
    mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
    const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
    const float uA = nA == kNegInf ? 0.f : nA, uB = nB == kNegInf ? 0.f : nB;
    const float alA = fast_exp2(mA - uA), alB = fast_exp2(mB - uB);
    mA = nA;
    mB = nB;
    float rsA = 0.f, rsB = 0.f;
    uint32_t pa[4][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const float p0 = fast_exp2(s[n][0] - uA), p1 = fast_exp2(s[n][1] - uA);
      const float p2 = fast_exp2(s[n][2] - uB), p3 = fast_exp2(s[n][3] - uB);
      rsA += p0 + p1;
      rsB += p2 + p3;
      pa[n >> 1][(n & 1) * 2] = pack_bf16(p0, p1);
      pa[n >> 1][(n & 1) * 2 + 1] = pack_bf16(p2, p3);
    }
    lA = lA * alA + rsA;
    lB = lB * alB + rsB;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
      o[dt][0] *= alA;
      o[dt][1] *= alA;
      o[dt][2] *= alB;
      o[dt][3] *= alB;
    }
    const bool tail = kv0 + kKeysPerTile > kv_total;  // keys past the end: arbitrary bits
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int kA2 = kv0 + kk * 16 + 2 * (lane & 3);
      const uint32_t m0 = (kA2 < kv_total ? 0x0000FFFFu : 0u) | (kA2 + 1 < kv_total ? 0xFFFF0000u : 0u);
      const uint32_t m1 = (kA2 + 8 < kv_total ? 0x0000FFFFu : 0u) | (kA2 + 9 < kv_total ? 0xFFFF0000u : 0u);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        const int mi = lane >> 3;
        const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
        const int chunk = 2 * dp + (mi >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + (chunk >> 3) * Lay::kRegionBytes + sw128(key, chunk & 7), b0, b1, b2, b3);
        if (tail) {
          b0 &= m0; b2 &= m0;
          b1 &= m1; b3 &= m1;
        }
        mma_bf16_16816(o[2 * dp], pa[kk], b0, b1);
        mma_bf16_16816(o[2 * dp + 1], pa[kk], b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
  if (!ok) {
    set_status(p.status, ATTN_STATUS_TIMEOUT);
    return;
  }
  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);
  const float iA = 1.f / lA, iB = 1.f / lB;
  const int64_t ostride = (int64_t)p.Hq * D;
  if (tokA < n_b) {
    uint16_t* dst = p.out + (int64_t)(tokbase + tokA) * ostride + (int64_t)hA * D + 2 * (lane & 3);
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt)
      *reinterpret_cast<uint32_t*>(dst + dt * 8) = pack_bf16(o[dt][0] * iA, o[dt][1] * iA);
  }
  if (tokB < n_b) {
    uint16_t* dst = p.out + (int64_t)(tokbase + tokB) * ostride + (int64_t)hB * D + 2 * (lane & 3);
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt)
      *reinterpret_cast<uint32_t*>(dst + dt * 8) = pack_bf16(o[dt][2] * iB, o[dt][3] * iB);
  }
}

template <int D>
int launch_prefill_t(const PrefillArgs& a, cudaStream_t stream) {
  using Lay = PrefillLayout<D>;
  CacheMaps maps;
  if (make_cache_maps(a.kv, a.cfg.num_kv_heads, D, kKeysPerTile, &maps) != 0) return ATTN_ELAUNCH;
  PrefillPar p;
  p.qkv = static_cast<const uint16_t*>(a.qkv);
  p.q_norm_w = static_cast<const uint16_t*>(a.q_norm_w);
  p.freqs = a.freqs;
  p.eps = a.cfg.rms_eps;
  p.W = (a.cfg.num_q_heads + 2 * a.cfg.num_kv_heads) * D;
  p.out = static_cast<uint16_t*>(a.out);
  p.cu_seqlens = a.cu_seqlens;
  p.slot_base = a.kv.slot_base;
  p.cache_lens = a.kv.cache_lens;
  p.slot_capacity = a.kv.slot_capacity;
  p.num_slots = a.kv.num_slots;
  p.status = a.status;
  p.Hq = a.cfg.num_q_heads;
  p.N = a.N;
  const int G = a.cfg.num_q_heads / a.cfg.num_kv_heads;
  p.log2G = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  if (cudaFuncSetAttribute(prefill_sync_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Lay::kSmemBytes) != cudaSuccess)
    return ATTN_ELAUNCH;
  const int tok_per_cta = kRowsPerCta / G;
  dim3 grid((a.max_seqlen + tok_per_cta - 1) / tok_per_cta, a.cfg.num_kv_heads, a.B);
  prefill_sync_kernel<D><<<grid, kThreads, Lay::kSmemBytes, stream>>>(maps.k, maps.v, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ELAUNCH;
}

}  // namespace

int launch_prefill_sync(const PrefillArgs& a, cudaStream_t stream) {
  if (a.B <= 0 || a.N <= 0 || a.max_seqlen <= 0) return ATTN_OK;
  return a.cfg.head_dim == 128 ? launch_prefill_t<128>(a, stream) : launch_prefill_t<64>(a, stream);
}

}  // namespace gb300
