// Prefill attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Code walkthrough section 3.3 teaching snippet and transformer-basics
// "Attention calculation: part 1": scores q.k / sqrt(D) against KV head
// h / (Hq/Hkv), future positions masked, softmax in fp32, P rounded to the
// input type, P times V; concept chapter section 2.6: computed the I/O-aware
// way (flash attention), never materialising the score matrix.
//
// One CTA computes 128 query rows packed as (token, group head) pairs of one
// KV head (128/G tokens x G heads), so every K/V tile it loads serves the
// whole GQA group.  Roles (192 threads):
//   warps 0-3  softmax: thread r owns row r = TMEM lane r.  Normalise and
//              rotate Q in shared memory, then per KV tile: read S from
//              TMEM, mask, online softmax in fp32 (exp2 domain), rescale O in
//              TMEM when the row max grows, write P (bf16) to shared memory.
//   warp 4     TMA producer: Q tile once, then K and V tiles (128 keys,
//              128-byte swizzle) through a 2-stage ring.
//   warp 5     MMA issuer (one thread) and TMEM owner: S = Q K^T into one
//              of two TMEM buffers, O += P V into TMEM.
// TMEM: columns [0,128) and [128,256) hold S (fp32), [256, 256+D) hold O.
// KV tiles past the causal limit of the CTA's last row are never loaded.
#include "kernels.cuh"
#include "tcgen05.cuh"

namespace gb300 {

namespace {

constexpr int kRows = 128;   // query rows per CTA (MMA M)
constexpr int kKeys = 128;   // keys per KV tile (MMA N of Q K^T)
constexpr int kThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr int kRegionBytes = 128 * 128;  // 128 rows x 128 bytes (64 bf16)
constexpr int kPairsPerPass = 16;        // RoPE table pass width
constexpr float kRescaleThreshold = 8.f; // log2 units: rescale O only past a 256x growth

struct TcPar {
  const int32_t* cu_seqlens;
  const int64_t* slot_base;
  const int32_t* cache_lens;
  const int32_t* slot_capacity;
  int64_t num_slots;
  int32_t* status;
  uint16_t* out;
  const uint16_t* q_norm_w;
  RopeFreqs freqs;
  float eps;
  float scale_log2;  // log2(e) / sqrt(D)
  int32_t Hq, log2G, N;
};

template <int D>
struct TcLayout {
  static constexpr int kRegions = D / 64;
  static constexpr int kTile = kRegions * kRegionBytes;  // Q, K or V tile: 128 rows x D
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;           // 2 stages
  static constexpr int kV = kK + 2 * kTile;       // 2 stages
  static constexpr int kP = kV + 2 * kTile;       // 128 x 128 bf16, 2 regions of 64 keys
  static constexpr int kBar = kP + 2 * kRegionBytes;
  static constexpr int kNumBars = 16;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  // + alignment slack; at least 116 KB so that one CTA runs per SM: each CTA
  // allocates all 512 TMEM columns.
  static constexpr int kSmemRaw = kTmemSlot + 16 + 1024;
  static constexpr int kSmemBytes = kSmemRaw > 116 * 1024 ? kSmemRaw : 116 * 1024;
};

enum Bar {
  kQFull = 0, kQReady, kKFull0, kKFull1, kKEmpty0, kKEmpty1, kVFull0, kVFull1, kVEmpty0,
  kVEmpty1, kSFull0, kSFull1, kPFull, kODone, kMmaDone
};

__device__ __forceinline__ void softmax_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kSoftmaxThreads) : "memory");
}

// mbarrier wait whose outcome is the same for every lane of the warp, so that
// warp-collective tcgen05.ld/st after it are never reached by part of a warp.
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity) {
  const bool w = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, w);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const TcPar p) {
  using Lay = TcLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kTmemSlot);
  const uint32_t sbase = smem_u32(smem);

  // ---------------- work item: (sequence b, KV head kh, query tile)
  const int kh = blockIdx.y, b = blockIdx.z;
  const int tokbase = p.cu_seqlens[b];
  const int n_b = p.cu_seqlens[b + 1] - tokbase;
  if (n_b <= 0) return;
  if (tokbase < 0 || tokbase + n_b > p.N) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) set_status(p.status, ATTN_STATUS_SEQLENS);
    return;
  }
  const ReqInfo r = load_request(p.slot_base + b, p.cache_lens + b, p.slot_capacity + b,
                                 p.num_slots, n_b);
  if (!r.valid) return;  // flagged by kv_append
  const int G = 1 << p.log2G;
  const int BT = kRows >> p.log2G;  // tokens per CTA
  const int ntile_b = (n_b + BT - 1) / BT;
  if (ntile_b > (int)gridDim.x) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) set_status(p.status, ATTN_STATUS_BOUNDS);
    return;
  }
  if ((int)blockIdx.x >= ntile_b) return;
  const int t0 = (ntile_b - 1 - (int)blockIdx.x) * BT;  // heaviest tiles first
  const int t_hi = min(t0 + BT, n_b);
  const int kv_total = r.cached + n_b;
  const int nk = (r.cached + t_hi + kKeys - 1) / kKeys;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bars[kQFull], 1);
    mbar_init(&bars[kQReady], kSoftmaxThreads);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kKFull0 + s], 1);
      mbar_init(&bars[kKEmpty0 + s], 1);
      mbar_init(&bars[kVFull0 + s], 1);
      mbar_init(&bars[kVEmpty0 + s], 1);
      mbar_init(&bars[kSFull0 + s], 1);
    }
    mbar_init(&bars[kPFull], kSoftmaxThreads);
    mbar_init(&bars[kODone], 1);
    mbar_init(&bars[kMmaDone], 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tc::alloc(tmem_slot, kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == kProducerWarp) {
    // ================================================================ TMA producer
    if (lane == 0) {
      prefetch_tmap(&qmap);
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
      mbar_arrive_expect_tx(&bars[kQFull], Lay::kTile);
#pragma unroll
      for (int rg = 0; rg < Lay::kRegions; ++rg)
        tma_load_3d(smem + Lay::kQ + rg * kRegionBytes, &qmap, &bars[kQFull], rg * 64, kh * G,
                    tokbase + t0);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < nk && ok; ++j) {
        const int st = j & 1;
        const uint32_t ph = ((j >> 1) & 1) ^ 1;  // phase of this stage's previous use
        const int slot = (int)(r.slot0 + j * kKeys);
        if (j >= 2 && !mbar_wait(&bars[kKEmpty0 + st], ph)) { ok = false; break; }
        mbar_arrive_expect_tx(&bars[kKFull0 + st], Lay::kTile);
#pragma unroll
        for (int rg = 0; rg < Lay::kRegions; ++rg)
          tma_load_3d(smem + Lay::kK + st * Lay::kTile + rg * kRegionBytes, &kmap,
                      &bars[kKFull0 + st], rg * 64, kh, slot);
        k_issued = j + 1;
        if (j >= 2 && !mbar_wait(&bars[kVEmpty0 + st], ph)) { ok = false; break; }
        mbar_arrive_expect_tx(&bars[kVFull0 + st], Lay::kTile);
#pragma unroll
        for (int rg = 0; rg < Lay::kRegions; ++rg)
          tma_load_3d(smem + Lay::kV + st * Lay::kTile + rg * kRegionBytes, &vmap,
                      &bars[kVFull0 + st], rg * 64, kh, slot);
        v_issued = j + 1;
      }
      // Every load issued has landed before the CTA may exit (immediate on
      // the normal path, where the consumers already waited for them).
      (void)mbar_wait(&bars[kQFull], 0);
      for (int j = max(0, k_issued - 2); j < k_issued; ++j)
        (void)mbar_wait(&bars[kKFull0 + (j & 1)], (j >> 1) & 1);
      for (int j = max(0, v_issued - 2); j < v_issued; ++j)
        (void)mbar_wait(&bars[kVFull0 + (j & 1)], (j >> 1) & 1);
      if (!ok) set_status(p.status, ATTN_STATUS_TIMEOUT);
    }
  } else if (warp == kMmaWarp) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kRows, kKeys, false);
      constexpr uint32_t idesc_o = tc::idesc_bf16_f32(kRows, D, true);
      const uint32_t q_addr = sbase + Lay::kQ;
      const uint32_t p_addr = sbase + Lay::kP;
      const uint32_t o_tmem = tmem + 256;
      ok = mbar_wait(&bars[kQReady], 0);
      tc::fence_after();
      for (int j = 0; j <= nk && ok; ++j) {
        if (j < nk) {
          const int st = j & 1;
          if (!mbar_wait(&bars[kKFull0 + st], (j >> 1) & 1)) { ok = false; break; }
          tc::fence_after();
          const uint32_t k_addr = sbase + Lay::kK + st * Lay::kTile;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (ks >> 2) * kRegionBytes + (ks & 3) * 32;
            tc::mma_f16_ss(tmem + (uint32_t)(j & 1) * 128, tc::sdesc_sw128(q_addr + off, 16, 1024),
                           tc::sdesc_sw128(k_addr + off, 16, 1024), idesc_s, ks > 0);
          }
          tc::commit(&bars[kSFull0 + (j & 1)]);
          tc::commit(&bars[kKEmpty0 + st]);
        }
        if (j >= 1) {
          const int jj = j - 1, st = jj & 1;
          if (!mbar_wait(&bars[kPFull], jj & 1)) { ok = false; break; }
          tc::fence_after();
          if (!mbar_wait(&bars[kVFull0 + st], (jj >> 1) & 1)) { ok = false; break; }
          tc::fence_after();
          const uint32_t v_addr = sbase + Lay::kV + st * Lay::kTile;
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk) {
            const uint64_t a = tc::sdesc_sw128(p_addr + (kk >> 2) * kRegionBytes + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = tc::sdesc_sw128(v_addr + kk * 2048, kRegionBytes, 1024);
            tc::mma_f16_ss(o_tmem, a, bd, idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
          }
          tc::commit(&bars[kODone]);
          tc::commit(&bars[kVEmpty0 + st]);
        }
      }
      // Nothing may still be running on the tensor cores when TMEM is freed.
      tc::commit(&bars[kMmaDone]);
      (void)mbar_wait(&bars[kMmaDone], 0);
      if (!ok) set_status(p.status, ATTN_STATUS_TIMEOUT);
    }
  } else {
    // ================================================================ softmax warpgroup
    const int row = threadIdx.x;                 // 0..127 = TMEM lane
    const int tl = row >> p.log2G;                // token within the tile
    const int g = row & (G - 1);
    const int tok = t0 + tl;
    const int h = kh * G + g;
    const int lim = tok < n_b ? r.cached + tok : kv_total - 1;  // last key this row may see
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const uint32_t q_row = sbase + Lay::kQ;
    float2* table = reinterpret_cast<float2*>(smem + Lay::kP);  // RoPE table, P buffer reused

    // ---- Q: RMSNorm with q_norm_w, then RoPE at this row's position, in place
    ok = wait_warp(&bars[kQFull], 0);
    {
      float x[D];
#pragma unroll
      for (int rg = 0; rg < Lay::kRegions; ++rg)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = lds128(q_row + rg * kRegionBytes + sw128(row, c));
          const uint32_t* u = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            x[rg * 64 + c * 8 + 2 * e] = bf16_lo(u[e]);
            x[rg * 64 + c * 8 + 2 * e + 1] = bf16_hi(u[e]);
          }
        }
      float ss = 0.f;
#pragma unroll
      for (int d = 0; d < D; ++d) ss = fmaf(x[d], x[d], ss);
      const float inv = rsqrtf(ss * (1.0f / D) + p.eps);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 wv = __ldg(reinterpret_cast<const uint4*>(p.q_norm_w + c * 8));
        const uint32_t* u = reinterpret_cast<const uint32_t*>(&wv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          x[c * 8 + 2 * e] = bf16_lo(u[e]) * (x[c * 8 + 2 * e] * inv);
          x[c * 8 + 2 * e + 1] = bf16_hi(u[e]) * (x[c * 8 + 2 * e + 1] * inv);
        }
      }
      // cos/sin of (position, pair) for the tile's tokens, kPairsPerPass pairs at a time
      const float pos0 = (float)(r.cached + t0);
#pragma unroll
      for (int pass = 0; pass < D / 2 / kPairsPerPass; ++pass) {
        for (int e = row; e < BT * kPairsPerPass; e += kSoftmaxThreads) {
          const int et = e / kPairsPerPass, i = pass * kPairsPerPass + e % kPairsPerPass;
          float c, s;
          rope_angle(pos0 + (float)et, p.freqs.hi[i], p.freqs.lo[i], p.freqs, &c, &s);
          table[e] = make_float2(c, s);
        }
        softmax_sync();
#pragma unroll
        for (int k = 0; k < kPairsPerPass; ++k) {
          const int i = pass * kPairsPerPass + k;
          const float2 cs = table[tl * kPairsPerPass + k];
          const float x1 = x[i], x2 = x[i + D / 2];
          x[i] = x1 * cs.x - x2 * cs.y;
          x[i + D / 2] = x2 * cs.x + x1 * cs.y;
        }
        softmax_sync();
      }
#pragma unroll
      for (int rg = 0; rg < Lay::kRegions; ++rg)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float* y = &x[rg * 64 + c * 8];
          sts128(q_row + rg * kRegionBytes + sw128(row, c),
                 make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                            pack_bf16(y[6], y[7])));
        }
    }
    tc::fence_proxy_async();
    mbar_arrive(&bars[kQReady]);

    // ---- main loop over KV tiles
    float m = kNegInf, l = 0.f;
    const int cta_min_lim = r.cached + t0;
    const uint32_t p_row = sbase + Lay::kP;
    for (int j = 0; j < nk && ok; ++j) {
      if (!wait_warp(&bars[kSFull0 + (j & 1)], (j >> 1) & 1)) { ok = false; break; }
      tc::fence_after();
      float s[kKeys];
#pragma unroll
      for (int c = 0; c < kKeys / 32; ++c)
        tc::ld_32x32b_x32(lane_base + (uint32_t)(j & 1) * 128 + c * 32, reinterpret_cast<uint32_t*>(s + c * 32));
      tc::wait_ld();
      const int kv0 = j * kKeys;
      // raw scores; keys past this row's causal limit become -inf (select, so
      // arbitrary bits in keys past the sequence end cannot leak through)
      if (kv0 + kKeys - 1 > cta_min_lim) {
#pragma unroll
        for (int c = 0; c < kKeys; ++c) s[c] = (kv0 + c <= lim) ? s[c] : kNegInf;
      }
      // row max with 8 independent chains (one warp per SM sub-partition:
      // latency is hidden by instruction-level parallelism only)
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = s[e];
#pragma unroll
      for (int c = 8; c < kKeys; ++c) mx[c & 7] = fmaxf(mx[c & 7], s[c]);
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * p.scale_log2;
      // Reference max for the exponentials: moved only when the row max grows
      // by more than 2^8 (P stays <= 256, exact after the final division by l),
      // so O is rescaled in TMEM rarely.  Tile 0 always sets it (key 0 is
      // visible to every row, so mt is finite there).
      const bool grow = (j == 0) || (mt > m + kRescaleThreshold);
      const float m_new = grow ? fmaxf(m, mt) : m;
      const float alpha = fast_exp2(m - m_new);  // 0 on tile 0, 1 when not growing
      const float neg_m = -m_new;
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
      for (int c = 0; c < kKeys; ++c) {
        s[c] = fast_exp2(fmaf(s[c], p.scale_log2, neg_m));  // exp2(-inf) = 0
        acc[c & 7] += s[c];
      }
      const float rs = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
      l = l * alpha + rs;
      m = m_new;
      if (j >= 1) {
        // P.V of the previous tile must be complete before O or P is touched
        if (!wait_warp(&bars[kODone], (j - 1) & 1)) { ok = false; break; }
        tc::fence_after();
        // warp-uniform: lanes whose reference max did not move multiply by 1
        if (__any_sync(0xffffffffu, alpha < 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tc::ld_32x32b_x32(lane_base + 256 + c * 32, o);
            tc::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tc::st_32x32b_x32(lane_base + 256 + c * 32, o);
          }
          tc::wait_st();
        }
      }
      if (kv0 + kKeys > kv_total) {
        // keys past the end of the sequence hold arbitrary bits: zero those V rows
        if (!wait_warp(&bars[kVFull0 + (j & 1)], (j >> 1) & 1)) { ok = false; break; }
        if (kv0 + row >= kv_total) {
          const uint32_t v_addr = sbase + Lay::kV + (j & 1) * Lay::kTile;
#pragma unroll
          for (int rg = 0; rg < Lay::kRegions; ++rg)
#pragma unroll
            for (int c = 0; c < 8; ++c) sts128(v_addr + rg * kRegionBytes + sw128(row, c), make_uint4(0, 0, 0, 0));
        }
      }
#pragma unroll
      for (int rg = 0; rg < 2; ++rg)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float* y = &s[rg * 64 + c * 8];
          sts128(p_row + rg * kRegionBytes + sw128(row, c),
                 make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                            pack_bf16(y[6], y[7])));
        }
      tc::fence_proxy_async();
      tc::fence_before();
      mbar_arrive(&bars[kPFull]);
    }
    // ---- epilogue: O / l -> bf16 rows of out
    if (ok) ok = wait_warp(&bars[kODone], (nk - 1) & 1);
    tc::fence_after();
    if (ok) {  // warp-uniform; only the stores depend on the row
      const float inv_l = 1.f / l;
      const bool store = tok < n_b;
      uint16_t* dst = p.out + (int64_t)(tokbase + (store ? tok : 0)) * p.Hq * D + (int64_t)h * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tc::ld_32x32b_x32(lane_base + 256 + c * 32, o);
        tc::wait_ld();
        if (!store) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 v;
          v.x = pack_bf16(__uint_as_float(o[8 * q + 0]) * inv_l, __uint_as_float(o[8 * q + 1]) * inv_l);
          v.y = pack_bf16(__uint_as_float(o[8 * q + 2]) * inv_l, __uint_as_float(o[8 * q + 3]) * inv_l);
          v.z = pack_bf16(__uint_as_float(o[8 * q + 4]) * inv_l, __uint_as_float(o[8 * q + 5]) * inv_l);
          v.w = pack_bf16(__uint_as_float(o[8 * q + 6]) * inv_l, __uint_as_float(o[8 * q + 7]) * inv_l);
          *reinterpret_cast<uint4*>(dst + c * 32 + q * 8) = v;
        }
      }
    } else {
      set_status(p.status, ATTN_STATUS_TIMEOUT);
    }
  }

  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == kMmaWarp) tc::dealloc(tmem, kTmemCols);
}

template <int D>
int launch_prefill_tc_t(const PrefillArgs& a, cudaStream_t stream) {
  using Lay = TcLayout<D>;
  const int Hq = a.cfg.num_q_heads, Hkv = a.cfg.num_kv_heads;
  const int G = Hq / Hkv;
  const int BT = kRows / G;
  CacheMaps maps;
  if (make_cache_maps(a.kv, Hkv, D, kKeys, &maps) != 0) return ATTN_ELAUNCH;
  CUtensorMap qmap;
  if (make_qkv_map(a.qkv, a.N, Hq + 2 * Hkv, D, G, BT, &qmap) != 0) return ATTN_ELAUNCH;
  TcPar p;
  p.cu_seqlens = a.cu_seqlens;
  p.slot_base = a.kv.slot_base;
  p.cache_lens = a.kv.cache_lens;
  p.slot_capacity = a.kv.slot_capacity;
  p.num_slots = a.kv.num_slots;
  p.status = a.status;
  p.out = static_cast<uint16_t*>(a.out);
  p.q_norm_w = static_cast<const uint16_t*>(a.q_norm_w);
  p.freqs = a.freqs;
  p.eps = a.cfg.rms_eps;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  p.Hq = Hq;
  p.log2G = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
  p.N = a.N;
  if (cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Lay::kSmemBytes) != cudaSuccess)
    return ATTN_ELAUNCH;
  const dim3 grid((a.max_seqlen + BT - 1) / BT, Hkv, a.B);
  prefill_tc_kernel<D><<<grid, kThreads, Lay::kSmemBytes, stream>>>(qmap, maps.k, maps.v, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ELAUNCH;
}

}  // namespace

int launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  if (a.B <= 0 || a.N <= 0 || a.max_seqlen <= 0) return ATTN_OK;
  return a.cfg.head_dim == 128 ? launch_prefill_tc_t<128>(a, stream)
                               : launch_prefill_tc_t<64>(a, stream);
}

}  // namespace gb300
