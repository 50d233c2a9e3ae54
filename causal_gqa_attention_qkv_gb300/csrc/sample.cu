// Token sampling from rows of logits: greedy argmax, or temperature + top-k +
// top-p truncation and sampling by the inverse distribution function.
//
// Concept chapter section 3.2 (greedy decoding, temperature, top-k, top-p;
// the temperature formula of section 3.2.2) and the walkthrough's section 4.3
// (a greedy batch takes the argmax, the others go through temperature and
// top-k/top-p).
//
// One cluster of kCluster CTAs per row; CTA r of the cluster owns the
// contiguous slice r of the row.  A step reduces over the slice in the CTA
// and publishes the CTA's partial result in its shared memory; the other CTAs
// read it through distributed shared memory and combine the partials in the
// same order, so that all CTAs hold the same result:
//   1. the maximum and its first index (greedy rows stop here);
//   2. weights w_i = exp((l_i - max) / T) as integers in units of 2^-40
//      (every sum below is exact and independent of order), counted and
//      summed in bins of z_i = (max - l_i) log2(e) / T: 3072 bins 1/64 wide
//      over [0, 48), 1023 bins 1/8 wide over [48, 175.875) (weights there
//      round to 0: counts only) and one bin for the rest and -inf, counted in
//      registers.  Bins are intervals of logits: larger logits, higher bins;
//      they are narrow wherever weights count, so that the tokens of a warp
//      seldom meet in one bin's atomics.  CTA r merges the
//      cluster's counts of the r-th eighth of the bins; every CTA then finds,
//      scanning from the top, the eighth and the bin in it where the count
//      reaches top_k or the mass reaches top_p x total;
//   3. one more pass over the slice: the kept mass per chunk of consecutive
//      tokens from the bins above the crossing bin, and the keys of the
//      crossing bin (order-preserving bit patterns of the logits, with weight
//      and index) copied to shared memory.  CTA 0 gathers the cluster's
//      copies and runs a radix select over them in four 8-bit digits, which
//      gives the smallest kept key lambda exactly (ties kept); the copies at
//      or above lambda add their weights to their chunks.  If a bin holds
//      more keys than the copies can, the four digits run over the slices
//      and one more pass sums the kept mass per chunk;
//   4. the smallest index whose cumulative kept weight exceeds u x kept mass:
//      the chunk masses scanned over the cluster, then one warp walks the
//      chunk that holds u x S.
// The first pass reads the row from memory; the others find it in L2.
#include "kernels.cuh"

namespace gb300 {

namespace {

#ifndef SAMPLE_CLUSTER
#define SAMPLE_CLUSTER 8
#endif
#ifndef SAMPLE_THREADS
#define SAMPLE_THREADS 256
#endif
constexpr int kCluster = SAMPLE_CLUSTER;  // CTAs per row
constexpr int kThreads = SAMPLE_THREADS;
constexpr int kMinBlocks = 1024 / kThreads;  // resident CTAs per SM the registers must allow
constexpr int kWarps = kThreads / 32;
constexpr int kFine = 2048;            // bins 2048 .. 4095: z in [0, 32), 1/64 wide
constexpr int kMid = 1024;             // bins 1024 .. 2047: z in [32, 48), 1/64 wide
constexpr int kFar = 1024;             // bins 1 .. 1023: z in [48, 175.875), 1/8 wide; bin 0: the rest
constexpr int kBins = kFar + kMid + kFine;
constexpr int kRange = kBins / kCluster;  // bins merged by each CTA
constexpr int kDigit = 256;            // bins of one 8-bit key digit
constexpr int kCand = 256;             // keys of the crossing bin copied per CTA
constexpr int kGather = kCluster * kCand;
constexpr int kMaxChunks = 256;        // chunks of the final passes, per CTA
using u64 = unsigned long long;
static_assert(kRange % 32 == 0 && kRange >= kDigit, "merged range");
static_assert(kFar % kRange == 0 && kMid % kRange == 0, "a CTA's eighth lies in one part of the bins");

// Shared memory of one CTA (dynamic).
struct SampleSmem {
  union {
    struct {                           // step 2: this CTA's histogram, read by the cluster's merge
      uint32_t cnt_fine[kFine];
      uint32_t mlo_fine[kFine];        // mass = mhi << 32 | mlo (weights up to 2^40): the low words
      uint32_t mhi_fine[kFine];        // wrap into the high ones, counted by the adding thread
      uint32_t cnt_mid[kMid];
      uint32_t mass_mid[kMid];         // weights up to 2^8 (z >= 32): sums below 2^29 (V <= 2^23)
      uint32_t cnt_far[kFar];          // bin 0 included
    } h;
    struct {                           // step 3 when the copies overflow: digit histograms
      uint32_t wcnt[kWarps][kDigit];   // per warp
      u64 wmass[kWarps][kDigit];
      uint32_t pub_cnt[2][kDigit];     // this CTA's, published; double-buffered by digit parity
      u64 pub_mass[2][kDigit];
    } f;
    struct {                           // step 3 on CTA 0: the cluster's copies
      uint32_t key[kGather];
      u64 w[kGather];
    } g;
  } u;
  uint32_t mcnt[kRange];               // the cluster's counts and masses of this CTA's eighth (published)
  u64 mmass[kRange];
  uint32_t scnt[kRange];               // the crossing eighth, copied; then the digit histograms
  u64 smass[kRange];
  uint32_t cand_key[kCand];            // the crossing bin's keys in this slice (published)
  u64 cand_w[kCand];
  int cand_idx[kCand];
  u64 csum[kMaxChunks];                // kept mass per chunk
  // published scalars
  float pub_mx;
  int pub_arg;
  u64 pub_total;                       // W (step 2), then the kept mass of the slice (step 4)
  uint32_t pub_rcnt;                   // the merged eighth's count and mass
  u64 pub_rmass;
  int pub_cand_n;
  uint32_t pub_lam;
  u64 pub_S;
  // this CTA's
  float red_mx[kWarps];
  int red_arg[kWarps];
  u64 red_sum[kWarps];
  uint32_t red_cnt[kWarps];
  uint32_t rng_cnt[kCluster];
  u64 rng_mass[kCluster];
  int cand_n;
  int s_range;
  u64 s_mass_above, s_bin_mass, s_excl;
  uint32_t s_digit, s_cnt_above;
  int s_chunk;
};

// Larger float -> larger key (finite values and -inf).
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SamplePar {
  const float* logits;
  int64_t ld;
  int32_t V, B;
  const float* temperature;
  const int32_t* top_k;
  const float* top_p;
  const float* uniform;
  int32_t* tokens;
};

// z = (mx - v) log2(e) / T as two correctly rounded operations; -z is
// bit for bit (v - mx) log2(e) / T, the exponent of the weight.
__device__ __forceinline__ float zval(float v, float mx, float log2e_over_t) {
  return __fmul_rn(__fsub_rn(mx, v), log2e_over_t);
}

// exp2(-z) = exp((v - mx) / T) in units of 2^-40, computed the same way in
// every pass.  The weight w <= 1 becomes round(w x 2^40) from two 32-bit
// conversions: w x 2^20 = hi + f exactly (hi its integer part), then
// lo = round(f x 2^20).  (A direct float -> 64-bit integer conversion runs on
// the fp64 pipe, which this part has little of.)  For z >= 48 the weight
// is below 2^-48 (1 + 2^-20) and rounds to 0 in these units, so it is not
// evaluated.
__device__ __forceinline__ u64 weight_of(float z) {
  if (!(z < 48.f)) return 0ull;
  const float s = __fmul_rn(exp2f(-z), 1048576.f);
  const uint32_t hi = __float2uint_rd(s);
  const uint32_t lo = __float2uint_rn(__fmul_rn(__fsub_rn(s, __uint2float_rn(hi)), 1048576.f));
  return ((u64)hi << 20) + lo;
}

// Bin of a logit from its z: 4095 - floor(64 z) for z < 32,
// 2047 - floor(64 (z - 32)) for z < 48, 1023 - floor(8 (z - 48)) for
// z < 175.875, else 0 (also -inf).  The scalings are exact and so are the
// subtractions (z and the constant are multiples of the ulp of z, the
// difference is smaller than z), so bin d holds exactly the z of one
// interval [za, zb) (bin_bounds) and the bins are intervals of logits,
// ordered.
__device__ __forceinline__ uint32_t zbin(float z) {
  if (z < 32.f) return (uint32_t)(kBins - 1) - (uint32_t)__fmul_rn(z, 64.f);
  if (z < 48.f) return (uint32_t)(kFar + kMid - 1) - (uint32_t)__fmul_rn(__fsub_rn(z, 32.f), 64.f);
  if (z < 175.875f) return (uint32_t)(kFar - 1) - (uint32_t)__fmul_rn(__fsub_rn(z, 48.f), 8.f);
  return 0u;
}

// The z interval [za, zb) of bin d (bin 0: z >= za, also +inf; d = -1: no
// bin, every finite z below za).
__device__ __forceinline__ void bin_bounds(int d, float& za, float& zb) {
  const float inf = __builtin_huge_valf();
  if (d < 0) {
    za = inf;
    zb = -inf;
  } else if (d >= kFar + kMid) {
    const int m = kBins - 1 - d;
    za = (float)m * 0.015625f;
    zb = (float)(m + 1) * 0.015625f;
  } else if (d >= kFar) {
    const int m = kFar + kMid - 1 - d;
    za = 32.f + (float)m * 0.015625f;
    zb = 32.f + (float)(m + 1) * 0.015625f;
  } else if (d > 0) {
    const int m = kFar - 1 - d;
    za = 48.f + (float)m * 0.125f;
    zb = 48.f + (float)(m + 1) * 0.125f;
  } else {
    za = 175.875f;
    zb = inf;
  }
}

// ---------------------------------------------------------------- cluster
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives; shared-memory writes
// before it are visible to the cluster's reads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Loads from the shared memory of CTA `rank` at the address `p` has in this
// CTA.  Issued back to back, they are in flight together.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t peer_u32(const void* p, uint32_t rank) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(peer_addr(p, rank)) : "memory");
  return v;
}
__device__ __forceinline__ u64 peer_u64(const void* p, uint32_t rank) {
  u64 v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(peer_addr(p, rank)) : "memory");
  return v;
}

// ---------------------------------------------------------------- slice walk
// Calls f(index, value, active) for this thread's share of [lo, hi), the
// same number of times in every thread of the CTA (inactive calls carry no
// element), so that f may use warp-wide operations.  NV loads (float4 when
// the slice start is 16-byte aligned) are issued before their values are used.
template <int NV, class F>
__device__ __forceinline__ void for_slice(const float* row, int lo, int hi, F&& f) {
  const int n = hi - lo;
  if (n <= 0) return;  // uniform across the CTA
  const int tid = threadIdx.x;
  if ((reinterpret_cast<uintptr_t>(row + lo) & 15) == 0) {
    const int nv = n >> 2;
    const float4* r4 = reinterpret_cast<const float4*>(row + lo);
    for (int base = 0; base < nv; base += NV * kThreads) {
      float4 v[NV];
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int i = base + j * kThreads + tid;
        v[j] = i < nv ? __ldg(r4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int i = base + j * kThreads + tid;
        const bool a = i < nv;
        const int e = lo + 4 * i;
        f(e, v[j].x, a);
        f(e + 1, v[j].y, a);
        f(e + 2, v[j].z, a);
        f(e + 3, v[j].w, a);
      }
    }
    const int t0 = lo + 4 * nv;  // fewer than 4 left
    if (t0 < hi) {
      const int e = t0 + tid;
      const bool a = e < hi;
      f(e, a ? __ldg(row + e) : 0.f, a);
    }
  } else {
    for (int base = 0; base < n; base += 4 * NV * kThreads) {
      float v[4 * NV];
#pragma unroll
      for (int j = 0; j < 4 * NV; ++j) {
        const int e = lo + base + j * kThreads + tid;
        v[j] = e < hi ? __ldg(row + e) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 4 * NV; ++j) {
        const int e = lo + base + j * kThreads + tid;
        f(e, v[j], e < hi);
      }
    }
  }
}

// Step 3 when the copies overflow: this CTA's digit histogram (the per-warp
// ones summed) published in buffer buf, then the cluster's (read back from
// every CTA) in scnt / smass.
__device__ __forceinline__ void publish_and_merge(SampleSmem& sm, int buf) {
  const int tid = threadIdx.x;
  for (int d = tid; d < kDigit; d += kThreads) {
    uint32_t cs = 0;
    u64 ms = 0;
    for (int w = 0; w < kWarps; ++w) {
      cs += sm.u.f.wcnt[w][d];
      ms += sm.u.f.wmass[w][d];
    }
    sm.u.f.pub_cnt[buf][d] = cs;
    sm.u.f.pub_mass[buf][d] = ms;
  }
  cluster_sync();
  for (int d = tid; d < kDigit; d += kThreads) {
    uint32_t cv[kCluster];
    u64 mv[kCluster];
#pragma unroll
    for (int r = 0; r < kCluster; ++r) {
      cv[r] = peer_u32(&sm.u.f.pub_cnt[buf][d], r);
      mv[r] = peer_u64(&sm.u.f.pub_mass[buf][d], r);
    }
    uint32_t cs = 0;
    u64 ms = 0;
#pragma unroll
    for (int r = 0; r < kCluster; ++r) {
      cs += cv[r];
      ms += mv[r];
    }
    sm.scnt[d] = cs;
    sm.smass[d] = ms;
  }
}

__device__ __forceinline__ void zero_warp_hists(SampleSmem& sm) {
  for (int i = threadIdx.x; i < kWarps * kDigit; i += kThreads) {
    (&sm.u.f.wcnt[0][0])[i] = 0;
    (&sm.u.f.wmass[0][0])[i] = 0;
  }
}

// Sum of v over the CTA (every thread gets it); red is kWarps entries.
template <class T>
__device__ __forceinline__ T block_sum(T v, T* red) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();  // earlier readers of red are done
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  T t = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += red[w];
  return t;
}

// Warp 0: the first bin, scanning from the largest, at which the cumulative
// count reaches k_lim or the cumulative mass reaches mass_lim (over the bins'
// keys plus cnt_above / mass_above).  Writes the digit, the count and mass of
// the bins above it and the mass of the bin itself.
__device__ __forceinline__ void find_crossing(const uint32_t* cnt, const u64* mass, int nb,
                                              uint32_t cnt_above, u64 mass_above, uint32_t k_lim,
                                              u64 mass_lim, uint32_t* s_digit, uint32_t* s_cnt,
                                              u64* s_mass, u64* s_bin_mass) {
  const int lane = threadIdx.x & 31;
  const int per = nb / 32;
  const int top = nb - 1 - lane * per;  // lane l: bins [nb - (l+1) per, nb - l per), from the top
  uint32_t lc = 0;
  u64 lm = 0;
  for (int j = 0; j < per; ++j) {
    lc += cnt[top - j];
    lm += mass[top - j];
  }
  uint32_t pc = lc;
  u64 pm = lm;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t tc = __shfl_up_sync(0xffffffffu, pc, off);
    const u64 tm = __shfl_up_sync(0xffffffffu, pm, off);
    if (lane >= off) {
      pc += tc;
      pm += tm;
    }
  }
  uint32_t c0 = cnt_above + pc - lc;
  u64 m0 = mass_above + pm - lm;
  int found = -1;
  for (int j = 0; j < per; ++j) {
    const int d = top - j;
    const uint32_t cd = cnt[d];
    const u64 md = mass[d];
    if (cd && (c0 + cd >= k_lim || m0 + md >= mass_lim)) {
      found = d;
      break;
    }
    c0 += cd;
    m0 += md;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, found >= 0);
  // (a crossing always exists: the total reaches the mass limit)
  const int src = hit ? __ffs(hit) - 1 : 31;
  if (lane == src) {
    if (found < 0) {  // not reached: keep the whole range
      found = 0;
      c0 -= cnt[0];
      m0 -= mass[0];
    }
    *s_digit = (uint32_t)found;
    *s_cnt = c0;
    *s_mass = m0;
    *s_bin_mass = mass[found];
  }
}

// Calls f(e0, stride, nact, v, acc) for every group of four tokens of this
// CTA's chunks of q consecutive tokens: the lane's tokens e0 + j stride hold
// v.x .. v.w and the first nact of them are tokens of the chunk.  Each chunk
// is walked by one warp (the same number of calls in every lane, so that f
// may use warp-wide operations); the warp's sum of acc per chunk goes to
// csum.  Chunks of 128 tokens of an aligned slice take one float4 per lane,
// four chunks of a warp in flight.
template <class F>
__device__ __forceinline__ void for_chunks(const float* row, int lo, int hi, int q, int nchunks, bool vec,
                                           u64* csum, F&& f) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (vec && q == 128) {
    for (int ch0 = warp; ch0 < nchunks; ch0 += 4 * kWarps) {
      float4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int ch = ch0 + j * kWarps;
        const int i = lo + ch * 128 + 4 * lane;
        if (ch < nchunks && i + 3 < hi) {
          v[j] = __ldg(reinterpret_cast<const float4*>(row + i));
        } else {
          const bool c = ch < nchunks;
          v[j].x = c && i < hi ? __ldg(row + i) : 0.f;
          v[j].y = c && i + 1 < hi ? __ldg(row + i + 1) : 0.f;
          v[j].z = c && i + 2 < hi ? __ldg(row + i + 2) : 0.f;
          v[j].w = c && i + 3 < hi ? __ldg(row + i + 3) : 0.f;
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int ch = ch0 + j * kWarps;  // uniform over the warp
        if (ch >= nchunks) break;
        const int i = lo + ch * 128 + 4 * lane;
        u64 acc = 0;
        f(i, 1, max(0, min(4, hi - i)), v[j], acc);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) csum[ch] = acc;
      }
    }
  } else {
    for (int ch = warp; ch < nchunks; ch += kWarps) {
      const int c0 = lo + ch * q, c1 = min(hi, c0 + q);
      u64 acc = 0;
      for (int base = c0; base < c1; base += 128) {
        const int e0 = base + lane;
        float4 v;
        v.x = e0 < c1 ? __ldg(row + e0) : 0.f;
        v.y = e0 + 32 < c1 ? __ldg(row + e0 + 32) : 0.f;
        v.z = e0 + 64 < c1 ? __ldg(row + e0 + 64) : 0.f;
        v.w = e0 + 96 < c1 ? __ldg(row + e0 + 96) : 0.f;
        f(e0, 32, max(0, min(4, (c1 - e0 + 31) / 32)), v, acc);
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane == 0) csum[ch] = acc;
    }
  }
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, kMinBlocks)
    sample_kernel(const SamplePar p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SampleSmem& sm = *reinterpret_cast<SampleSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_rank();
  const int V = p.V;
  // this CTA's slice: a multiple of 4 tokens, so that every slice of an
  // aligned row starts 16-byte aligned
  const int span = ((V + kCluster - 1) / kCluster + 3) & ~3;
  const int lo = min(V, (int)rank * span), hi = min(V, lo + span);
  // chunks of the last passes: q consecutive tokens, q a multiple of 128
  const int n = hi - lo;
  const int q = 128 * max(1, (n + 128 * kMaxChunks - 1) / (128 * kMaxChunks));
  const int nchunks = (n + q - 1) / q;

  for (int b = blockIdx.y; b < p.B; b += gridDim.y) {  // uniform over the cluster
    const float* row = p.logits + (int64_t)b * p.ld;
    const bool vec = (reinterpret_cast<uintptr_t>(row + lo) & 15) == 0;

    // 1. maximum and its first index
    float mx = -__builtin_huge_valf();
    int arg = 0x7fffffff;
    for_slice<8>(row, lo, hi, [&](int i, float v, bool a) {
      if (a && (v > mx || (v == mx && i < arg) || arg == 0x7fffffff)) {
        mx = v;
        arg = i;
      }
    });
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, mx, off);
      const int oa = __shfl_xor_sync(0xffffffffu, arg, off);
      if (om > mx || (om == mx && oa < arg)) {
        mx = om;
        arg = oa;
      }
    }
    if (lane == 0) {
      sm.red_mx[warp] = mx;
      sm.red_arg[warp] = arg;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kWarps; ++w)
        if (sm.red_mx[w] > mx || (sm.red_mx[w] == mx && sm.red_arg[w] < arg)) {
          mx = sm.red_mx[w];
          arg = sm.red_arg[w];
        }
      sm.pub_mx = mx;
      sm.pub_arg = arg;
    }
    cluster_sync();
    {
      float om[kCluster];
      int oa[kCluster];
#pragma unroll
      for (int r = 0; r < kCluster; ++r) {
        om[r] = __uint_as_float(peer_u32(&sm.pub_mx, r));
        oa[r] = (int)peer_u32(&sm.pub_arg, r);
      }
      mx = -__builtin_huge_valf();
      arg = 0x7fffffff;
#pragma unroll
      for (int r = 0; r < kCluster; ++r)
        if (om[r] > mx || (om[r] == mx && oa[r] < arg)) {
          mx = om[r];
          arg = oa[r];
        }
    }
    const float T = p.temperature[b];
    if (!(T > 0.f)) {
      if (rank == 0 && tid == 0) p.tokens[b] = arg;
      cluster_sync();  // every CTA has read the published maxima
      continue;
    }
    const float c = 1.4426950408889634f / T;
    const int k = p.top_k[b];
    const uint32_t k_lim = (k > 0 && k < V) ? (uint32_t)k : 0xffffffffu;
    const float top_p = p.top_p[b];
    // without either limit every token of positive weight is kept (tokens of
    // zero weight add nothing to any cumulative sum below)
    const bool truncate = !(k_lim == 0xffffffffu && top_p >= 1.f);

    // 2. counts and masses per bin of z; the total weight W
    for (int i = tid; i < kFine; i += kThreads) {
      sm.u.h.cnt_fine[i] = 0;
      sm.u.h.mlo_fine[i] = 0;
      sm.u.h.mhi_fine[i] = 0;
    }
    for (int i = tid; i < kMid; i += kThreads) {
      sm.u.h.cnt_mid[i] = 0;
      sm.u.h.mass_mid[i] = 0;
    }
    for (int i = tid; i < kFar; i += kThreads) sm.u.h.cnt_far[i] = 0;
    if (tid == 0) sm.cand_n = 0;
    __syncthreads();
    u64 wsum = 0;
    uint32_t n0 = 0;  // tokens of bin 0 (weight 0)
    for_slice<4>(row, lo, hi, [&](int, float v, bool a) {
      if (!a) return;
      // zbin and weight_of, taken apart so that each part of the bins does
      // only its own work
      const float z = zval(v, mx, c);
      if (z < 48.f) {
        const uint32_t m = (uint32_t)__fmul_rn(z, 64.f);  // bin kBins - 1 - m
        const float s = __fmul_rn(exp2f(-z), 1048576.f);
        const uint32_t hi = __float2uint_rd(s);
        const uint32_t lo = __float2uint_rn(__fmul_rn(__fsub_rn(s, __uint2float_rn(hi)), 1048576.f));
        const u64 w = ((u64)hi << 20) + lo;
        wsum += w;
        if (m < (uint32_t)kFine) {
          // two 32-bit atomics instead of one 64-bit one (which costs more
          // than twice as much): the add that wraps the low word carries
          // into the high one
          const uint32_t bi = kFine - 1 - m;
          atomicAdd(&sm.u.h.cnt_fine[bi], 1u);
          uint32_t up = (uint32_t)(w >> 32);
          const uint32_t wl = (uint32_t)w;
          if (wl) {
            const uint32_t old = atomicAdd(&sm.u.h.mlo_fine[bi], wl);
            up += old + wl < old ? 1u : 0u;
          }
          if (up) atomicAdd(&sm.u.h.mhi_fine[bi], up);
        } else {
          atomicAdd(&sm.u.h.cnt_mid[kFine + kMid - 1 - m], 1u);
          if (w) atomicAdd(&sm.u.h.mass_mid[kFine + kMid - 1 - m], (uint32_t)w);
        }
      } else if (z < 175.875f) {
        atomicAdd(&sm.u.h.cnt_far[kFar - 1 - (uint32_t)__fmul_rn(__fsub_rn(z, 48.f), 8.f)], 1u);
      } else {
        ++n0;
      }
    });
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) n0 += __shfl_xor_sync(0xffffffffu, n0, off);
    if (lane == 0 && n0) atomicAdd(&sm.u.h.cnt_far[0], n0);
    {
      const u64 wc = block_sum(wsum, sm.red_sum);
      if (tid == 0) sm.pub_total = wc;
    }
    cluster_sync();  // the histograms and the slices' weights are complete
    u64 W = 0;
    {
      u64 wv[kCluster];
#pragma unroll
      for (int r = 0; r < kCluster; ++r) wv[r] = peer_u64(&sm.pub_total, r);
#pragma unroll
      for (int r = 0; r < kCluster; ++r) W += wv[r];
    }
    u64 mass_lim;
    if (top_p >= 1.f) mass_lim = W;  // reached once every token of positive weight is in
    else if (!(top_p > 0.f)) mass_lim = 0;
    else mass_lim = (u64)ceil((double)top_p * (double)W);

    int zs = -1;  // the crossing bin; -1: every token is above it
    uint32_t cnt_above0 = 0;
    u64 mass_above0 = 0;
    if (truncate) {
      // the cluster's counts and masses of this CTA's eighth of the bins
      uint32_t rc = 0;
      u64 rm = 0;
      for (int j = tid; j < kRange; j += kThreads) {
        const int d = (int)rank * kRange + j;
        uint32_t cv[kCluster];
        u64 mv[kCluster];
        if (d >= kFar + kMid) {  // uniform over the CTA
#pragma unroll
          for (int r = 0; r < kCluster; ++r) {
            cv[r] = peer_u32(&sm.u.h.cnt_fine[d - (kFar + kMid)], r);
            mv[r] = (u64)peer_u32(&sm.u.h.mhi_fine[d - (kFar + kMid)], r) << 32 |
                    peer_u32(&sm.u.h.mlo_fine[d - (kFar + kMid)], r);
          }
        } else if (d >= kFar) {
#pragma unroll
          for (int r = 0; r < kCluster; ++r) {
            cv[r] = peer_u32(&sm.u.h.cnt_mid[d - kFar], r);
            mv[r] = peer_u32(&sm.u.h.mass_mid[d - kFar], r);
          }
        } else {
#pragma unroll
          for (int r = 0; r < kCluster; ++r) {
            cv[r] = peer_u32(&sm.u.h.cnt_far[d], r);
            mv[r] = 0;
          }
        }
        uint32_t cs = 0;
        u64 ms = 0;
#pragma unroll
        for (int r = 0; r < kCluster; ++r) {
          cs += cv[r];
          ms += mv[r];
        }
        sm.mcnt[j] = cs;
        sm.mmass[j] = ms;
        rc += cs;
        rm += ms;
      }
      rc = block_sum(rc, sm.red_cnt);
      rm = block_sum(rm, sm.red_sum);
      if (tid == 0) {
        sm.pub_rcnt = rc;
        sm.pub_rmass = rm;
      }
      cluster_sync();  // the merged eighths are complete; the histograms are read
      // the eighth where the limits are reached, scanning from the top
      if (tid < kCluster) {
        sm.rng_cnt[tid] = peer_u32(&sm.pub_rcnt, tid);
        sm.rng_mass[tid] = peer_u64(&sm.pub_rmass, tid);
      }
      __syncthreads();
      if (tid == 0) {
        uint32_t ca = 0;
        u64 ma = 0;
        int R = 0;
        for (int r = kCluster - 1; r >= 0; --r) {
          const uint32_t cr = sm.rng_cnt[r];
          const u64 mr = sm.rng_mass[r];
          if (cr && (ca + cr >= k_lim || ma + mr >= mass_lim)) {
            R = r;
            break;
          }
          if (r == 0) break;  // not reached: the lowest eighth (its lowest bin keeps everything)
          ca += cr;
          ma += mr;
        }
        sm.s_range = R;
        sm.s_cnt_above = ca;
        sm.s_mass_above = ma;
      }
      __syncthreads();
      const int R = sm.s_range;
      const uint32_t ca = sm.s_cnt_above;
      const u64 ma = sm.s_mass_above;
      for (int j = tid; j < kRange; j += kThreads) {
        sm.scnt[j] = peer_u32(&sm.mcnt[j], R);
        sm.smass[j] = peer_u64(&sm.mmass[j], R);
      }
      __syncthreads();
      if (warp == 0)
        find_crossing(sm.scnt, sm.smass, kRange, ca, ma, k_lim, mass_lim, &sm.s_digit, &sm.s_cnt_above,
                      &sm.s_mass_above, &sm.s_bin_mass);
      __syncthreads();
      zs = R * kRange + (int)sm.s_digit;
      cnt_above0 = sm.s_cnt_above;
      mass_above0 = sm.s_mass_above;
    }

    // 3. kept mass per chunk from the bins above zs; the keys of bin zs
    float za, zb;
    bin_bounds(zs, za, zb);
    for_chunks(row, lo, hi, q, nchunks, vec, sm.csum, [&](int e0, int stride, int nact, float4 v4, u64& acc) {
      const float v[4] = {v4.x, v4.y, v4.z, v4.w};
      float z[4];
      bool cand[4], any = false;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        z[j] = zval(v[j], mx, c);
        const bool a = j < nact;
        if (a && z[j] < za) acc += weight_of(z[j]);
        cand[j] = a && !(z[j] < za) && (z[j] < zb || zs == 0);
        any |= cand[j];
      }
      if (__any_sync(0xffffffffu, any)) {  // uniform over the warp
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const unsigned keep = __ballot_sync(0xffffffffu, cand[j]);
          if (!keep) continue;
          int slot0 = 0;
          if (lane == 0) slot0 = atomicAdd(&sm.cand_n, __popc(keep));
          slot0 = __shfl_sync(0xffffffffu, slot0, 0);
          const int slot = slot0 + __popc(keep & ((1u << lane) - 1u));
          if (cand[j] && slot < kCand) {
            sm.cand_key[slot] = order_key(v[j]);
            sm.cand_w[slot] = weight_of(z[j]);
            sm.cand_idx[slot] = e0 + j * stride;
          }
        }
      }
    });
    __syncthreads();
    if (tid == 0) sm.pub_cand_n = sm.cand_n;
    cluster_sync();  // the copies are complete; the merged eighths and W are read

    uint32_t lam = 0;
    u64 S = W;
    if (truncate) {
      int cn[kCluster];
#pragma unroll
      for (int r = 0; r < kCluster; ++r) cn[r] = (int)peer_u32(&sm.pub_cand_n, r);
      bool fits = true;
#pragma unroll
      for (int r = 0; r < kCluster; ++r) fits = fits && cn[r] <= kCand;

      uint32_t prefix = 0, cnt_above = cnt_above0;
      u64 mass_above = mass_above0, bin_mass = 0;
      if (fits) {
        if (rank == 0) {  // gather the cluster's keys, select over them
          uint32_t* gk = sm.u.g.key;
          u64* gw = sm.u.g.w;
          int off[kCluster + 1];
          off[0] = 0;
#pragma unroll
          for (int r = 0; r < kCluster; ++r) off[r + 1] = off[r] + cn[r];
          const int ng = off[kCluster];
          // every copy loaded at once: entry i of the gathered list is copy
          // i - off[r] of CTA r
          uint32_t kand = 0xffffffffu, kor = 0;
          u64 tot = 0;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t kk[kGather / kThreads / 2];
            u64 ww[kGather / kThreads / 2];
#pragma unroll
            for (int it = 0; it < kGather / kThreads / 2; ++it) {
              const int i = tid + (half * (kGather / kThreads / 2) + it) * kThreads;
              kk[it] = 0;
              ww[it] = 0;
              if (i < ng) {
                int r = 0;
#pragma unroll
                for (int rr = 1; rr < kCluster; ++rr) r = i >= off[rr] ? rr : r;
                kk[it] = peer_u32(&sm.cand_key[i - off[r]], r);
                ww[it] = peer_u64(&sm.cand_w[i - off[r]], r);
              }
            }
#pragma unroll
            for (int it = 0; it < kGather / kThreads / 2; ++it) {
              const int i = tid + (half * (kGather / kThreads / 2) + it) * kThreads;
              if (i < ng) {
                gk[i] = kk[it];
                gw[i] = ww[it];
                kand &= kk[it];
                kor |= kk[it];
                tot += ww[it];
              }
            }
          }
          // digits shared by every copy need no pass when the copies reach
          // a limit (the crossing is then among them): their digit is the
          // crossing digit and nothing lies above it
          kand = __reduce_and_sync(0xffffffffu, kand);
          kor = __reduce_or_sync(0xffffffffu, kor);
          if (lane == 0) {
            sm.red_cnt[warp] = kand;
            sm.red_arg[warp] = (int)kor;
          }
          tot = block_sum(tot, sm.red_sum);  // (its barriers also publish red_cnt, red_arg)
          for (int w = 0; w < kWarps; ++w) {
            kand &= sm.red_cnt[w];
            kor |= (uint32_t)sm.red_arg[w];
          }
          int lv0 = 0;
          if (ng > 0 && (cnt_above + (uint32_t)ng >= k_lim || mass_above + tot >= mass_lim)) {
            const uint32_t diff = kand ^ kor;
            lv0 = diff ? __clz(diff) / 8 : 4;
            prefix = lv0 == 0 ? 0u : kand & (0xffffffffu << (32 - 8 * lv0));
            bin_mass = tot;  // all equal: the one key's mass
          }
          for (int lv = lv0; lv < 4; ++lv) {
            const int shift = 24 - 8 * lv;
            const uint32_t fixed_mask = lv == 0 ? 0u : 0xffffffffu << (32 - 8 * lv);
            for (int d = tid; d < kDigit; d += kThreads) {
              sm.scnt[d] = 0;
              sm.smass[d] = 0;
            }
            __syncthreads();
            for (int i = tid; i < ng; i += kThreads) {
              const uint32_t key = gk[i];
              if ((key & fixed_mask) != prefix) continue;
              const uint32_t d = (key >> shift) & 0xffu;
              atomicAdd(&sm.scnt[d], 1u);
              if (gw[i]) atomicAdd(&sm.smass[d], gw[i]);
            }
            __syncthreads();
            if (warp == 0)
              find_crossing(sm.scnt, sm.smass, kDigit, cnt_above, mass_above, k_lim, mass_lim, &sm.s_digit,
                            &sm.s_cnt_above, &sm.s_mass_above, &sm.s_bin_mass);
            __syncthreads();
            prefix |= sm.s_digit << shift;
            cnt_above = sm.s_cnt_above;
            mass_above = sm.s_mass_above;
            bin_mass = sm.s_bin_mass;
            __syncthreads();
          }
          if (tid == 0) {
            sm.pub_lam = prefix;
            sm.pub_S = mass_above + bin_mass;
          }
        }
        cluster_sync();
        lam = peer_u32(&sm.pub_lam, 0);
        S = peer_u64(&sm.pub_S, 0);
        // the copies at or above lambda join their chunks
        for (int i = tid; i < sm.cand_n; i += kThreads)
          if (sm.cand_key[i] >= lam) atomicAdd(&sm.csum[(sm.cand_idx[i] - lo) / q], sm.cand_w[i]);
        __syncthreads();
      } else {
        // more keys in the bin than the copies hold: the four digits over the slices
        for (int lv = 0; lv < 4; ++lv) {
          const int shift = 24 - 8 * lv;
          const uint32_t fixed_mask = lv == 0 ? 0u : 0xffffffffu << (32 - 8 * lv);
          zero_warp_hists(sm);
          __syncthreads();
          uint32_t* mc = sm.u.f.wcnt[warp];
          u64* mm = sm.u.f.wmass[warp];
          for_slice<4>(row, lo, hi, [&](int, float v, bool a) {
            if (!a) return;
            const uint32_t key = order_key(v);
            const float z = zval(v, mx, c);
            if ((int)zbin(z) != zs || (key & fixed_mask) != prefix) return;
            const uint32_t d = (key >> shift) & 0xffu;
            const u64 w = weight_of(z);
            atomicAdd(&mc[d], 1u);
            if (w) atomicAdd(&mm[d], w);
          });
          __syncthreads();
          publish_and_merge(sm, (lv + 1) & 1);
          __syncthreads();
          if (warp == 0)
            find_crossing(sm.scnt, sm.smass, kDigit, cnt_above, mass_above, k_lim, mass_lim, &sm.s_digit,
                          &sm.s_cnt_above, &sm.s_mass_above, &sm.s_bin_mass);
          __syncthreads();
          prefix |= sm.s_digit << shift;
          cnt_above = sm.s_cnt_above;
          mass_above = sm.s_mass_above;
          bin_mass = sm.s_bin_mass;
          __syncthreads();
        }
        lam = prefix;
        S = mass_above + bin_mass;
        // the kept mass per chunk, from the start
        for_chunks(row, lo, hi, q, nchunks, vec, sm.csum, [&](int, int, int nact, float4 v4, u64& acc) {
          const float v[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (j < nact && order_key(v[j]) >= lam) acc += weight_of(zval(v[j], mx, c));
        });
        __syncthreads();
      }
    }

    // 4. inverse distribution function in vocabulary order
    u64 t = (u64)((double)p.uniform[b] * (double)S);
    if (t >= S) t = S - 1;
    auto kept_w = [&](float v) -> u64 { return order_key(v) >= lam ? weight_of(zval(v, mx, c)) : 0ull; };
    if (tid == 0) sm.s_chunk = -1;
    __syncthreads();
    // exclusive scan of the chunk masses: thread t owns chunks [t per, (t+1) per)
    const int per = (nchunks + kThreads - 1) / kThreads;
    u64 own = 0;
    for (int j = 0; j < per; ++j) {
      const int ch = tid * per + j;
      if (ch < nchunks) own += sm.csum[ch];
    }
    u64 incl = own;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const u64 o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) sm.red_sum[warp] = incl;
    __syncthreads();
    u64 before = 0, K = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) before += sm.red_sum[w];
      K += sm.red_sum[w];
    }
    if (tid == 0) sm.pub_total = K;
    cluster_sync();
    u64 pre = 0;  // kept mass of the slices before this one
    {
      u64 kv[kCluster];
#pragma unroll
      for (int r = 0; r < kCluster; ++r) kv[r] = (uint32_t)r < rank ? peer_u64(&sm.pub_total, r) : 0ull;
#pragma unroll
      for (int r = 0; r < kCluster; ++r) pre += kv[r];
    }
    if (K > 0 && pre <= t && t < pre + K) {  // uniform over the CTA
      u64 x = pre + before + incl - own;  // kept mass before chunk tid * per
      for (int j = 0; j < per; ++j) {
        const int ch = tid * per + j;
        if (ch >= nchunks) break;
        const u64 m = sm.csum[ch];
        if (m > 0 && x <= t && t < x + m) {
          sm.s_chunk = ch;
          sm.s_excl = x;
        }
        x += m;
      }
      __syncthreads();
      if (warp == 0 && sm.s_chunk >= 0) {
        const int c0 = lo + sm.s_chunk * q, c1 = min(hi, c0 + q);
        u64 acc = sm.s_excl;
        for (int base = c0; base < c1; base += 32) {
          const int i = base + lane;
          const u64 wv = i < c1 ? kept_w(__ldg(row + i)) : 0ull;
          u64 inc = wv;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const u64 o = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += o;
          }
          const unsigned hit = __ballot_sync(0xffffffffu, acc + inc > t);
          if (hit) {
            if (lane == __ffs(hit) - 1) p.tokens[b] = i;
            break;
          }
          acc += __shfl_sync(0xffffffffu, inc, 31);
        }
      }
    }
    cluster_sync();  // every CTA has read the published values before they change
  }
}

}  // namespace

int launch_sample(const float* logits, int32_t B, int32_t V, int64_t ld, const float* temperature,
                  const int32_t* top_k, const float* top_p, const float* uniform, int32_t* tokens,
                  cudaStream_t stream) {
  if (B <= 0) return ATTN_OK;
  SamplePar p;
  p.logits = logits;
  p.ld = ld;
  p.V = V;
  p.B = B;
  p.temperature = temperature;
  p.top_k = top_k;
  p.top_p = top_p;
  p.uniform = uniform;
  p.tokens = tokens;
  const int smem = (int)sizeof(SampleSmem);
  if (cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return ATTN_ELAUNCH;
  const dim3 grid(kCluster, (unsigned)std::min<int32_t>(B, 65535));
  sample_kernel<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ELAUNCH;
}

}  // namespace gb300
