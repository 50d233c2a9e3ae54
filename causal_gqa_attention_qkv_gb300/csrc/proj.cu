// The projections either side of the attention step, on the tcgen05 tensor
// cores: qkv = hidden . W_qkv^T fused with the step's prologue (Q/K RMSNorm,
// RoPE, K/V cache append, prepared Q), and o = attn_out . W_o^T.
//
// Zero-to-sglang Ch.3 code walkthrough, section 3.3 (AttentionLayer.forward:
// qkv_proj, then the attention, then o_proj) and the transformer-basics page,
// "Attention calculation: part 1" (the q/k/v projections of the hidden states
// [1, 12, 4096] and o_proj after the attention): both projections are plain
// linear layers y = x W^T with the weight stored [out_features, in_features].
//
// One persistent kernel, one CTA per SM, output tiles of 128 rows x 256
// columns handed out round-robin (row-block major, so that CTAs running at
// the same time share the rows of x in L2).  CTAs work in pairs (a cluster
// of two): the pair computes two vertically adjacent tiles with the same 256
// columns, and each CTA loads half of that W tile into both CTAs' shared
// memory by TMA multicast (a third less L2 traffic per CTA); a stage is
// refilled once both CTAs' MMAs have read it.  Roles per CTA:
//   warp 0      one thread issues the TMA loads of x (128 x 64) and of its
//               half of W (128 x 64, multicast) into a 4-stage ring of
//               48 KB stages;
//   warp 1      owns the 512 TMEM columns (two 256-column fp32 accumulators)
//               and one thread issues the MMAs, M128 N256 K16, four per stage;
//   warps 2-5   the epilogue: thread r of the four warps holds row r of the
//               accumulator (TMEM lane r), so a head's D values sit in one
//               thread and the RMSNorm and the rotation need no shuffles.
// The accumulator of tile i + 1 fills while the epilogue reads tile i.
#include "kernels.cuh"
#include "tcgen05.cuh"

namespace gb300 {

namespace {

constexpr int kBM = 128;        // tile rows (tokens)
constexpr int kBN = 256;        // tile columns (output features)
constexpr int kBK = 64;         // reduction elements per stage: one 128-byte row
constexpr int kStages = 4;
constexpr int kATile = kBM * kBK * 2;           // 16 KB
constexpr int kBTile = kBN * kBK * 2;           // 32 KB
constexpr int kStageBytes = kATile + kBTile;    // 48 KB
constexpr int kTmemCols = 2 * kBN;              // two accumulators
constexpr int kThreads = 192;                   // warps 0, 1 and the epilogue warps 2..5

// shared memory: stages | barriers | TMEM slot | norm weights (fp32)
constexpr int kBarOff = kStages * kStageBytes;
enum { kFull = 0, kEmpty = kStages, kAccFull = 2 * kStages, kAccEmpty = 2 * kStages + 2, kNumBars = 2 * kStages + 4 };
constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
constexpr int kNormOff = kBarOff + 256;         // float qw[128], kw[128]
constexpr int kSmemBytes = kNormOff + 2 * 128 * 4 + 1024;  // + alignment slack

enum ProjEpi { kEpiPlain = 0, kEpiQkv = 1 };

struct ProjPar {
  int32_t M, N, K;              // rows, output columns, reduction length
  int32_t tiles_n, tiles;
  int32_t* status;
  // plain epilogue: out [M, N] bf16, row stride N
  uint16_t* out;
  // qkv epilogue
  const uint16_t* q_norm_w;     // [D] bf16
  const uint16_t* k_norm_w;
  uint16_t* q_out;              // [M, Hq, D] bf16 (f16 next to an E4M3 cache)
  void* k_cache;
  void* v_cache;
  float inv_k, inv_v;           // E4M3: fp32(1 / scale)
  KvIndex kv;
  const int32_t* cu_seqlens;    // [B + 1]
  int32_t B, Hq, Hkv;
  float eps;
  RopeFreqs freqs;
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t c0,
                                            int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

#ifndef PROJ_PAIR
#define PROJ_PAIR 1
#endif
// CTA pairs: the two CTAs of a cluster compute vertically adjacent tiles
// (rows m0 and m0 + 128, the same 256 columns) and each loads half of the
// shared W tile into both CTAs' shared memory (TMA multicast).
constexpr int kPair = PROJ_PAIR ? 2 : 1;

__device__ __forceinline__ uint32_t cta_rank_in_cluster() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The box goes to the same shared-memory offset of every CTA in `mask`, and
// its bytes are counted on the mbarrier at the same offset in each of them.
__device__ __forceinline__ void tma_load_2d_multicast(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t c0,
                                                      int32_t c1, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "h"(mask)
      : "memory");
}
// Arrive on the mbarrier at `bar`'s offset in every CTA of `mask` once this
// thread's earlier MMAs have completed.
__device__ __forceinline__ void mma_commit_multicast(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// Tile t of this CTA: row block and column block.  With pairs, pair tile t
// gives both CTAs of the cluster the same column block.
__device__ __forceinline__ void tile_coords(const ProjPar& p, int t, uint32_t rank, int& m0, int& n0) {
  m0 = ((t / p.tiles_n) * kPair + (int)rank) * kBM;
  n0 = (t % p.tiles_n) * kBN;
}

// ---------------------------------------------------------------- producer
__device__ void proj_produce(const ProjPar& p, const CUtensorMap* amap, const CUtensorMap* bmap, uint8_t* smem,
                             uint64_t* bars, bool& ok) {
  const int kb_count = (p.K + kBK - 1) / kBK;
  int st = 0;
  uint32_t ph = 0;
  uint32_t filled = 0;  // bit s: stage s was filled at least once
  uint32_t last_par = 0;  // bit s: parity of the last fill of stage s
  const uint32_t rank = kPair > 1 ? cta_rank_in_cluster() : 0u;
  for (int t = blockIdx.x / kPair; t < p.tiles && ok; t += gridDim.x / kPair) {
    int m0, n0;
    tile_coords(p, t, rank, m0, n0);
    for (int kb = 0; kb < kb_count; ++kb) {
      if (!mbar_wait(&bars[kEmpty + st], ph ^ 1)) { ok = false; break; }
      uint8_t* a = smem + st * kStageBytes;
      mbar_arrive_expect_tx(&bars[kFull + st], kStageBytes);
      tma_load_2d(a, amap, &bars[kFull + st], kb * kBK, m0);
      if (kPair > 1)  // this CTA's half of the W tile, into both CTAs
        tma_load_2d_multicast(a + kATile + rank * (kBTile / 2), bmap, &bars[kFull + st], kb * kBK,
                              n0 + (int)rank * (kBN / 2), 0x3);
      else
        tma_load_2d(a + kATile, bmap, &bars[kFull + st], kb * kBK, n0);
      filled |= 1u << st;
      last_par = (last_par & ~(1u << st)) | (ph << st);
      if (++st == kStages) { st = 0; ph ^= 1; }
    }
  }
  // every copy this thread issued has landed before the CTA may exit
  for (int s = 0; s < kStages; ++s)
    if ((filled >> s) & 1u)
      if (!mbar_wait(&bars[kFull + s], (last_par >> s) & 1u)) ok = false;
}

// ---------------------------------------------------------------- MMA issue
__device__ void proj_mma(const ProjPar& p, uint32_t sbase, uint32_t tmem, uint64_t* bars, bool& ok) {
  constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN, false);
  const int kb_count = (p.K + kBK - 1) / kBK;
  int st = 0;
  uint32_t ph = 0;
  int it = 0;
  for (int t = blockIdx.x / kPair; t < p.tiles && ok; t += gridDim.x / kPair, ++it) {
    const int buf = it & 1;
    const uint32_t use = (uint32_t)(it >> 1);
    if (!mbar_wait(&bars[kAccEmpty + buf], (use & 1u) ^ 1u)) { ok = false; break; }
    tc::fence_after();
    const uint32_t d = tmem + (uint32_t)buf * kBN;
    for (int kb = 0; kb < kb_count; ++kb) {
      if (!mbar_wait(&bars[kFull + st], ph)) { ok = false; break; }
      tc::fence_after();
      const uint32_t a = sbase + st * kStageBytes;
      const uint64_t ad = tc::sdesc_sw128(a, 16, 1024);
      const uint64_t bd = tc::sdesc_sw128(a + kATile, 16, 1024);
#pragma unroll
      for (int k = 0; k < kBK / 16; ++k)  // +32 bytes per K step inside the 128-byte swizzle row
        tc::mma_f16_ss(d, ad + (uint64_t)(k * 2), bd + (uint64_t)(k * 2), idesc, (kb | k) != 0 ? 1u : 0u);
      // the stage is free once these MMAs have read it (with pairs: in both CTAs,
      // whose producers both write into it)
      if (kPair > 1) mma_commit_multicast(&bars[kEmpty + st], 0x3);
      else tc::commit(&bars[kEmpty + st]);
      if (++st == kStages) { st = 0; ph ^= 1; }
    }
    if (!ok) break;
    tc::commit(&bars[kAccFull + buf]);
  }
}

// ---------------------------------------------------------------- epilogues
// y = x W^T rounded to bf16, row by row; columns past N are not written
// (N is a multiple of 8).
__device__ void epi_plain(const ProjPar& p, int row, int n0, uint32_t taddr) {
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
    uint32_t r[32];
    tc::ld_32x32b_x32(taddr + c * 32, r);
    tc::wait_ld();
    const int col = n0 + 32 * c;
    if (row >= p.M || col >= p.N) continue;
    uint16_t* dst = p.out + (int64_t)row * p.N + col;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      if (col + 8 * v + 8 > p.N) break;
      uint4 u;
      u.x = pack_bf16(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
      u.y = pack_bf16(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
      u.z = pack_bf16(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
      u.w = pack_bf16(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
      reinterpret_cast<uint4*>(dst)[v] = u;
    }
  }
}

// Store 32 values of a head vector: bf16 (or f16 for a prepared Q next to an
// E4M3 cache), or E4M3 codes of value * r.
template <bool F16>
__device__ __forceinline__ void store_half32(uint16_t* dst, const float (&y)[32]) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    uint4 u;
    if (F16) {
      u = make_uint4(pack_f16(y[8 * v], y[8 * v + 1]), pack_f16(y[8 * v + 2], y[8 * v + 3]),
                     pack_f16(y[8 * v + 4], y[8 * v + 5]), pack_f16(y[8 * v + 6], y[8 * v + 7]));
    } else {
      u = make_uint4(pack_bf16(y[8 * v], y[8 * v + 1]), pack_bf16(y[8 * v + 2], y[8 * v + 3]),
                     pack_bf16(y[8 * v + 4], y[8 * v + 5]), pack_bf16(y[8 * v + 6], y[8 * v + 7]));
    }
    reinterpret_cast<uint4*>(dst)[v] = u;
  }
}
__device__ __forceinline__ void store_e4m3x32(uint8_t* dst, const float (&y)[32], float r) {
#pragma unroll
  for (int v = 0; v < 2; ++v) {
    uint4 u;
    uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e = 16 * v + 4 * q;
      w[q] = e4m3x2(__fmul_rn(y[e], r), __fmul_rn(y[e + 1], r)) |
             (e4m3x2(__fmul_rn(y[e + 2], r), __fmul_rn(y[e + 3], r)) << 16);
    }
    reinterpret_cast<uint4*>(dst)[v] = u;
  }
}

// The step's prologue on this thread's row of the accumulator: for each head
// (D columns) of the tile, Q and K heads are RMS-normalised with their weight
// and rotated at the token's position (pairs (i, i + D/2)); Q goes to q_out,
// K and V to the cache slot of the token.  The accumulators are used as they
// are (fp32, never rounded to bf16 before the norm).
template <int D, bool F8>
__device__ void epi_qkv(const ProjPar& p, int row, int n0, uint32_t taddr, const float* qw, const float* kw) {
  // token facts: 0 = no row, 1 = Q only (cache region too small), 2 = Q and cache
  int ok = 0;
  int64_t slot = 0;
  float pos = 0.f;
  if (row < p.M) {
    int lo = 0, hi = p.B;  // largest b with cu_seqlens[b] <= row
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.cu_seqlens + mid) <= row) lo = mid; else hi = mid;
    }
    const int c0 = __ldg(p.cu_seqlens + lo);
    const int n = __ldg(p.cu_seqlens + lo + 1) - c0;
    const int j = row - c0;
    if (j >= 0 && j < n) {
      const ReqInfo r = load_request(p.kv, lo, n);
      ok = 1;
      pos = (float)(r.cached + j);
      slot = r.valid ? cache_slot(p.kv, r, r.cached + j) : -1;
      if (slot >= 0) ok = 2;
      else if (n0 == 0) set_status(p.status, ATTN_STATUS_CAPACITY);
    } else if (n0 == 0) {
      set_status(p.status, ATTN_STATUS_SEQLENS);
    }
  }
  const int heads = p.Hq + 2 * p.Hkv;
#pragma unroll 1
  for (int h = 0; h < kBN / D; ++h) {
    const int hd = n0 / D + h;
    if (hd >= heads) break;  // uniform over the CTA
    const uint32_t hcol = taddr + h * D;
    if (hd >= p.Hq + p.Hkv) {  // V: rounded once, into the cache
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tc::ld_32x32b_x32(hcol + 32 * c, r);
        tc::wait_ld();
        if (ok != 2) continue;
        const int64_t e0 = (slot * p.Hkv + (hd - p.Hq - p.Hkv)) * D + 32 * c;
        float y[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(r[i]);
        if (F8) store_e4m3x32(static_cast<uint8_t*>(p.v_cache) + e0, y, p.inv_v);
        else store_half32<false>(static_cast<uint16_t*>(p.v_cache) + e0, y);
      }
      continue;
    }
    const bool is_q = hd < p.Hq;
    const float* w = is_q ? qw : kw;
    // sum of squares over the head: one partial per 32 columns, then summed
    float part[D / 32];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t r[32];
      tc::ld_32x32b_x32(hcol + 32 * c, r);
      tc::wait_ld();
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) s = fmaf(__uint_as_float(r[i]), __uint_as_float(r[i]), s);
      part[c] = s;
    }
    float ss = part[0];
#pragma unroll
    for (int c = 1; c < D / 32; ++c) ss += part[c];
    const float inv = rsqrtf(ss * (1.0f / D) + p.eps);
    // rotation pairs (i, i + D/2), 32 pairs at a time (unrolled: the
    // frequency table is indexed with constants)
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      uint32_t r1[32], r2[32];
      tc::ld_32x32b_x32(hcol + 32 * c, r1);
      tc::ld_32x32b_x32(hcol + D / 2 + 32 * c, r2);
      tc::wait_ld();
      float y1[32], y2[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int pi = 32 * c + i;  // pair index < D/2
        float cs, sn;
        rope_angle(pos, p.freqs.hi[pi], p.freqs.lo[pi], p.freqs, &cs, &sn);
        const float a = w[pi] * (__uint_as_float(r1[i]) * inv);
        const float b = w[pi + D / 2] * (__uint_as_float(r2[i]) * inv);
        y1[i] = fmaf(-b, sn, a * cs);
        y2[i] = fmaf(a, sn, b * cs);
      }
      if (is_q) {
        if (ok == 0) continue;
        uint16_t* dst = p.q_out + ((int64_t)row * p.Hq + hd) * D + 32 * c;
        store_half32<F8>(dst, y1);
        store_half32<F8>(dst + D / 2, y2);
      } else {
        if (ok != 2) continue;
        const int64_t e0 = (slot * p.Hkv + (hd - p.Hq)) * D + 32 * c;
        if (F8) {
          store_e4m3x32(static_cast<uint8_t*>(p.k_cache) + e0, y1, p.inv_k);
          store_e4m3x32(static_cast<uint8_t*>(p.k_cache) + e0 + D / 2, y2, p.inv_k);
        } else {
          store_half32<false>(static_cast<uint16_t*>(p.k_cache) + e0, y1);
          store_half32<false>(static_cast<uint16_t*>(p.k_cache) + e0 + D / 2, y2);
        }
      }
    }
  }
}

template <int Epi, int D, bool F8>
__device__ void proj_epilogue(const ProjPar& p, uint32_t tmem, uint64_t* bars, const float* qw, const float* kw,
                              bool& ok) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lane_grp = warp & 3;  // TMEM lanes [32 lane_grp, 32 lane_grp + 32) of this warp
  const uint32_t rank = kPair > 1 ? cta_rank_in_cluster() : 0u;
  int it = 0;
  for (int t = blockIdx.x / kPair; t < p.tiles && ok; t += gridDim.x / kPair, ++it) {
    const int buf = it & 1;
    const uint32_t use = (uint32_t)(it >> 1);
    if (!mbar_wait(&bars[kAccFull + buf], use & 1u)) { ok = false; break; }
    tc::fence_after();
    int m0, n0;
    tile_coords(p, t, rank, m0, n0);
    const int row = m0 + 32 * lane_grp + lane;
    const uint32_t taddr = tmem + ((uint32_t)(32 * lane_grp) << 16) + (uint32_t)buf * kBN;
    if (Epi == kEpiPlain) epi_plain(p, row, n0, taddr);
    else epi_qkv<D, F8>(p, row, n0, taddr, qw, kw);
    tc::fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[kAccEmpty + buf]);
  }
}

template <int Epi, int D, bool F8>
__global__ void __cluster_dims__(kPair, 1, 1) __launch_bounds__(kThreads, 1)
    proj_gemm_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                     const ProjPar p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kTmemSlotOff);
  float* qw = reinterpret_cast<float*>(smem + kNormOff);
  float* kw = qw + 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[kFull + s], 1);
      mbar_init(&bars[kEmpty + s], kPair);  // one MMA completion per CTA of the pair
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kAccFull + s], 1);
      mbar_init(&bars[kAccEmpty + s], 4);  // one arrival per epilogue warp
    }
    fence_barrier_init();
  }
  if (Epi == kEpiQkv && (int)threadIdx.x < D) {
    qw[threadIdx.x] = __uint_as_float((uint32_t)__ldg(p.q_norm_w + threadIdx.x) << 16);
    kw[threadIdx.x] = __uint_as_float((uint32_t)__ldg(p.k_norm_w + threadIdx.x) << 16);
  }
  if (warp == 1) {
    tc::alloc(tmem_slot, kTmemCols);
    tc::relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&amap);
    prefetch_tmap(&bmap);
  }
  tc::fence_before();
  __syncthreads();
  if (kPair > 1) cluster_barrier();  // both CTAs' barriers exist before either multicasts into the other
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  if (warp == 0) {
    if (lane == 0) proj_produce(p, &amap, &bmap, smem, bars, ok);
  } else if (warp == 1) {
    if (lane == 0) proj_mma(p, smem_u32(smem), tmem, bars, ok);
  } else {
    proj_epilogue<Epi, D, F8>(p, tmem, bars, qw, kw, ok);
  }
  if (!ok) set_status(p.status, ATTN_STATUS_TIMEOUT);
  tc::fence_before();
  __syncthreads();
  // neither CTA leaves while the other may still write into its shared memory
  // or arrive on its barriers
  if (kPair > 1) cluster_barrier();
  tc::fence_after();
  if (warp == 1) tc::dealloc(tmem, kTmemCols);
}

template <int Epi, int D, bool F8>
int launch_proj_t(const ProjPar& p0, const void* a, const void* b, cudaStream_t stream) {
  ProjPar p = p0;
  CUtensorMap amap, bmap;
  if (make_matrix_map(a, p.M, p.K, kBM, &amap) != 0) return ATTN_ELAUNCH;
  if (make_matrix_map(b, p.N, p.K, kBN / kPair, &bmap) != 0) return ATTN_ELAUNCH;
  p.tiles_n = (p.N + kBN - 1) / kBN;
  const int64_t row_blocks = ((int64_t)(p.M + kBM - 1) / kBM + kPair - 1) / kPair;  // pairs of row blocks
  const int64_t tiles = row_blocks * p.tiles_n;
  if (tiles > (int64_t(1) << 30)) return ATTN_EINVAL;
  p.tiles = (int)tiles;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ATTN_ELAUNCH;
  if (cudaFuncSetAttribute(proj_gemm_kernel<Epi, D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes) != cudaSuccess)
    return ATTN_ELAUNCH;
  // as many clusters as can be resident at once (pairs must share a GPC,
  // and not every GPC has an even number of SMs): a persistent cluster that
  // could only start after another one finished would double the run time
  int clusters = sms / kPair;
  if (kPair > 1) {
    cudaLaunchConfig_t qc = {};
    qc.gridDim = dim3(kPair * clusters);
    qc.blockDim = dim3(kThreads);
    qc.dynamicSmemBytes = kSmemBytes;
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, proj_gemm_kernel<Epi, D, F8>, &qc) != cudaSuccess || active <= 0)
      return ATTN_ELAUNCH;
    clusters = std::min(clusters, active);
  }
  const int grid = (int)std::min<int64_t>(clusters, tiles) * kPair;
  proj_gemm_kernel<Epi, D, F8><<<grid, kThreads, kSmemBytes, stream>>>(amap, bmap, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ELAUNCH;
}

}  // namespace

int launch_linear(const void* x, const void* w, void* y, int32_t M, int32_t N, int32_t K, int32_t* status,
                  cudaStream_t stream) {
  if (M <= 0 || N <= 0) return ATTN_OK;
  ProjPar p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.out = static_cast<uint16_t*>(y);
  p.status = status;
  return launch_proj_t<kEpiPlain, 128, false>(p, x, w, stream);
}

int launch_qkv_proj(const QkvProjArgs& a, cudaStream_t stream) {
  if (a.N <= 0) return ATTN_OK;
  const int D = a.cfg.head_dim;
  ProjPar p{};
  p.M = a.N;
  p.N = (a.cfg.num_q_heads + 2 * a.cfg.num_kv_heads) * D;
  p.K = a.C;
  p.status = a.status;
  p.q_norm_w = static_cast<const uint16_t*>(a.q_norm_w);
  p.k_norm_w = static_cast<const uint16_t*>(a.k_norm_w);
  p.q_out = static_cast<uint16_t*>(a.q_out);
  p.k_cache = a.kv.k_cache;
  p.v_cache = a.kv.v_cache;
  const bool f8 = a.kv.kv_dtype == ATTN_KV_E4M3;
  p.inv_k = f8 ? 1.0f / a.kv.k_scale : 1.0f;
  p.inv_v = f8 ? 1.0f / a.kv.v_scale : 1.0f;
  p.kv = kv_index(a.kv);
  p.cu_seqlens = a.cu_seqlens;
  p.B = a.B;
  p.Hq = a.cfg.num_q_heads;
  p.Hkv = a.cfg.num_kv_heads;
  p.eps = a.cfg.rms_eps;
  p.freqs = a.freqs;
  if (D == 128)
    return f8 ? launch_proj_t<kEpiQkv, 128, true>(p, a.hidden, a.w_qkv, stream)
              : launch_proj_t<kEpiQkv, 128, false>(p, a.hidden, a.w_qkv, stream);
  return f8 ? launch_proj_t<kEpiQkv, 64, true>(p, a.hidden, a.w_qkv, stream)
            : launch_proj_t<kEpiQkv, 64, false>(p, a.hidden, a.w_qkv, stream);
}

}  // namespace gb300
