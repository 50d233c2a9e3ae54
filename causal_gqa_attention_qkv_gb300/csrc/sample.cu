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
// and publishes the CTA's partial result in its shared memory; every CTA then
// reads the cluster's partials through distributed shared memory and combines
// them in the same order, so that all CTAs hold the same result:
//   1. the maximum and its first index (greedy rows stop here);
//   2. weights w_i = exp((l_i - max) / T) as integers in units of 2^-40
//      (every sum below is exact and independent of order), counted and
//      summed in 256 bins of z_i = (max - l_i) log2(e) / T, 1/8 wide (bins
//      are intervals of logits: larger logits, higher bins; z >= 31.875 and
//      -inf share the lowest).  Scanning the bins from the top finds the bin
//      where the count reaches top_k or the mass reaches top_p x total;
//   3. the keys of that bin (order-preserving bit patterns of the logits) are
//      copied to shared memory; CTA 0 gathers the cluster's copies and runs a
//      radix select over them in four 8-bit digits, which gives the smallest
//      kept key lambda exactly (ties kept).  If a bin holds more keys than the
//      copies can, the four digits run over the slices instead;
//   4. the smallest index whose cumulative kept weight exceeds u x kept mass:
//      kept mass per CTA slice and per chunk of consecutive tokens, then one
//      warp of the CTA holding u x S walks its chunk.
// The first pass reads the row from memory; the others find it in L2.
#include "kernels.cuh"

namespace gb300 {

namespace {

constexpr int kCluster = 8;            // CTAs per row
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 256;
constexpr int kCand = 256;             // keys of the crossing bin copied per CTA
constexpr int kGather = kCluster * kCand;
constexpr int kMaxChunks = 1024;       // chunks of the final pass, per CTA
using u64 = unsigned long long;

// Shared memory of one CTA (dynamic).
struct SampleSmem {
  // published for the other CTAs of the cluster
  float pub_mx;
  int pub_arg;
  u64 pub_total;                       // W (step 2), then the kept mass (step 4)
  int pub_cand_n;
  uint32_t pub_lam;
  u64 pub_S;
  uint32_t pub_cnt[2][kBins];          // histograms, double-buffered by step parity
  u64 pub_mass[2][kBins];
  uint32_t cand_key[kCand];
  u64 cand_w[kCand];
  // this CTA's own
  uint32_t wcnt[kWarps][kBins];        // per-warp histograms; CTA 0's gathered keys in step 3
  u64 wmass[kWarps][kBins];            // per-warp masses; CTA 0's gathered weights in step 3
  uint32_t gcnt[kBins];                // the cluster's histogram
  u64 gmass[kBins];
  u64 csum[kMaxChunks];
  float red_mx[kWarps];
  int red_arg[kWarps];
  u64 red_sum[kWarps];
  int cand_n;
  u64 s_mass_above, s_bin_mass, s_excl;
  uint32_t s_digit, s_cnt_above;
  int s_chunk;
};
static_assert(sizeof(uint32_t) * kWarps * kBins >= sizeof(uint32_t) * kGather, "gathered keys");
static_assert(sizeof(u64) * kWarps * kBins >= sizeof(u64) * kGather, "gathered weights");

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

// exp((v - mx) / T) in units of 2^-40, computed the same way in every pass.
// The weight w <= 1 becomes round(w x 2^40) from two 32-bit conversions:
// w x 2^20 = hi + f exactly (hi its integer part), then lo = round(f x 2^20).
// (A direct float -> 64-bit integer conversion runs on the fp64 pipe, which
// this part has little of.)
__device__ __forceinline__ u64 fixed_weight(float v, float mx, float log2e_over_t) {
  const float s = __fmul_rn(exp2f(__fmul_rn(__fsub_rn(v, mx), log2e_over_t)), 1048576.f);
  const uint32_t hi = __float2uint_rd(s);
  const uint32_t lo = __float2uint_rn(__fmul_rn(__fsub_rn(s, __uint2float_rn(hi)), 1048576.f));
  return ((u64)hi << 20) + lo;
}

// Bin of a logit: 255 - floor(8 z), z = (mx - v) log2(e) / T, or 0 for
// 8 z >= 255 and for -inf.  Each step is a correctly rounded operation that
// does not decrease with v, so the bins are intervals of logits, ordered.
__device__ __forceinline__ uint32_t zbin(float v, float mx, float log2e_over_t) {
  const float zz = __fmul_rn(__fmul_rn(__fsub_rn(mx, v), log2e_over_t), 8.f);
  return zz < 255.f ? 255u - (uint32_t)zz : 0u;
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
// element), so that f may use warp-wide operations.  Four loads (float4 when
// the slice start is 16-byte aligned) are issued before their values are used.
template <class F>
__device__ __forceinline__ void for_slice(const float* row, int lo, int hi, F&& f) {
  const int n = hi - lo;
  if (n <= 0) return;  // uniform across the CTA
  const int tid = threadIdx.x;
  if ((reinterpret_cast<uintptr_t>(row + lo) & 15) == 0) {
    const int nv = n >> 2;
    const float4* r4 = reinterpret_cast<const float4*>(row + lo);
    for (int base = 0; base < nv; base += 4 * kThreads) {
      float4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = base + j * kThreads + tid;
        v[j] = i < nv ? __ldg(r4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
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
    for (int base = 0; base < n; base += 4 * kThreads) {
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = lo + base + j * kThreads + tid;
        v[j] = e < hi ? __ldg(row + e) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = lo + base + j * kThreads + tid;
        f(e, v[j], e < hi);
      }
    }
  }
}

// This CTA's histogram (the per-warp ones summed) published in buffer buf,
// then the cluster's (read back from every CTA) in gcnt / gmass.
__device__ __forceinline__ void publish_and_merge(SampleSmem& sm, int buf) {
  const int tid = threadIdx.x;
  for (int d = tid; d < kBins; d += kThreads) {
    uint32_t cs = 0;
    u64 ms = 0;
    for (int w = 0; w < kWarps; ++w) {
      cs += sm.wcnt[w][d];
      ms += sm.wmass[w][d];
    }
    sm.pub_cnt[buf][d] = cs;
    sm.pub_mass[buf][d] = ms;
  }
  cluster_sync();
  for (int d = tid; d < kBins; d += kThreads) {
    uint32_t cv[kCluster];
    u64 mv[kCluster];
#pragma unroll
    for (int r = 0; r < kCluster; ++r) {
      cv[r] = peer_u32(&sm.pub_cnt[buf][d], r);
      mv[r] = peer_u64(&sm.pub_mass[buf][d], r);
    }
    uint32_t cs = 0;
    u64 ms = 0;
#pragma unroll
    for (int r = 0; r < kCluster; ++r) {
      cs += cv[r];
      ms += mv[r];
    }
    sm.gcnt[d] = cs;
    sm.gmass[d] = ms;
  }
}

__device__ __forceinline__ void zero_warp_hists(SampleSmem& sm) {
  for (int i = threadIdx.x; i < kWarps * kBins; i += kThreads) {
    (&sm.wcnt[0][0])[i] = 0;
    (&sm.wmass[0][0])[i] = 0;
  }
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

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
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

  for (int b = blockIdx.y; b < p.B; b += gridDim.y) {  // uniform over the cluster
    const float* row = p.logits + (int64_t)b * p.ld;

    // 1. maximum and its first index
    float mx = -__builtin_huge_valf();
    int arg = 0x7fffffff;
    for_slice(row, lo, hi, [&](int i, float v, bool a) {
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

    // 2. counts and masses per bin of z; the total weight W
    zero_warp_hists(sm);
    if (tid == 0) sm.cand_n = 0;
    __syncthreads();
    u64 wsum = 0;
    {
      uint32_t* mc = sm.wcnt[warp];
      u64* mm = sm.wmass[warp];
      for_slice(row, lo, hi, [&](int, float v, bool a) {
        if (!a) return;
        const uint32_t d = zbin(v, mx, c);
        const u64 w = fixed_weight(v, mx, c);
        wsum += w;
        atomicAdd(&mc[d], 1u);
        if (w) atomicAdd(&mm[d], w);
      });
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
    if (lane == 0) sm.red_sum[warp] = wsum;
    __syncthreads();
    if (tid == 0) {
      u64 t = 0;
      for (int w = 0; w < kWarps; ++w) t += sm.red_sum[w];
      sm.pub_total = t;
    }
    publish_and_merge(sm, 0);
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

    uint32_t lam;
    u64 S;
    if (k_lim == 0xffffffffu && top_p >= 1.f) {
      // no truncation: every token of positive weight is kept (the tokens of
      // zero weight add nothing to any cumulative sum below)
      lam = 0;
      S = W;
      cluster_sync();  // the published histograms and W have been read
    } else {
      __syncthreads();
      if (warp == 0)
        find_crossing(sm.gcnt, sm.gmass, kBins, 0u, 0ull, k_lim, mass_lim, &sm.s_digit, &sm.s_cnt_above,
                      &sm.s_mass_above, &sm.s_bin_mass);
      __syncthreads();
      const uint32_t zsel = sm.s_digit;
      const uint32_t cnt_above0 = sm.s_cnt_above;
      const u64 mass_above0 = sm.s_mass_above;

      // 3. the keys of bin zsel
      for_slice(row, lo, hi, [&](int, float v, bool a) {
        a = a && zbin(v, mx, c) == zsel;
        const unsigned keep = __ballot_sync(0xffffffffu, a);
        int slot0 = 0;
        if (lane == 0 && keep) slot0 = atomicAdd(&sm.cand_n, __popc(keep));
        slot0 = __shfl_sync(0xffffffffu, slot0, 0);
        const int slot = slot0 + __popc(keep & ((1u << lane) - 1u));
        if (a && slot < kCand) {
          sm.cand_key[slot] = order_key(v);
          sm.cand_w[slot] = fixed_weight(v, mx, c);
        }
      });
      __syncthreads();
      if (tid == 0) sm.pub_cand_n = sm.cand_n;
      cluster_sync();  // also: every CTA has read the published histograms and W
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
          uint32_t* gk = &sm.wcnt[0][0];
          u64* gw = &sm.wmass[0][0];
          int off = 0;
          for (int r = 0; r < kCluster; ++r) {
            for (int i = tid; i < cn[r]; i += kThreads) {
              gk[off + i] = peer_u32(&sm.cand_key[i], r);
              gw[off + i] = peer_u64(&sm.cand_w[i], r);
            }
            off += cn[r];
          }
          const int ng = off;
          for (int lv = 0; lv < 4; ++lv) {
            const int shift = 24 - 8 * lv;
            const uint32_t fixed_mask = lv == 0 ? 0u : 0xffffffffu << (32 - 8 * lv);
            for (int d = tid; d < kBins; d += kThreads) {
              sm.gcnt[d] = 0;
              sm.gmass[d] = 0;
            }
            __syncthreads();
            for (int i = tid; i < ng; i += kThreads) {
              const uint32_t key = gk[i];
              if ((key & fixed_mask) != prefix) continue;
              const uint32_t d = (key >> shift) & 0xffu;
              atomicAdd(&sm.gcnt[d], 1u);
              if (gw[i]) atomicAdd(&sm.gmass[d], gw[i]);
            }
            __syncthreads();
            if (warp == 0)
              find_crossing(sm.gcnt, sm.gmass, kBins, cnt_above, mass_above, k_lim, mass_lim, &sm.s_digit,
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
      } else {
        // more keys in the bin than the copies hold: the four digits over the slices
        for (int lv = 0; lv < 4; ++lv) {
          const int shift = 24 - 8 * lv;
          const uint32_t fixed_mask = lv == 0 ? 0u : 0xffffffffu << (32 - 8 * lv);
          zero_warp_hists(sm);
          __syncthreads();
          uint32_t* mc = sm.wcnt[warp];
          u64* mm = sm.wmass[warp];
          for_slice(row, lo, hi, [&](int, float v, bool a) {
            if (!a) return;
            const uint32_t key = order_key(v);
            if (zbin(v, mx, c) != zsel || (key & fixed_mask) != prefix) return;
            const uint32_t d = (key >> shift) & 0xffu;
            const u64 w = fixed_weight(v, mx, c);
            atomicAdd(&mc[d], 1u);
            if (w) atomicAdd(&mm[d], w);
          });
          __syncthreads();
          publish_and_merge(sm, (lv + 1) & 1);
          __syncthreads();
          if (warp == 0)
            find_crossing(sm.gcnt, sm.gmass, kBins, cnt_above, mass_above, k_lim, mass_lim, &sm.s_digit,
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
      }
    }

    // 4. inverse distribution function in vocabulary order
    u64 t = (u64)((double)p.uniform[b] * (double)S);
    if (t >= S) t = S - 1;
    const int n = hi - lo;
    const int q = 128 * max(1, (n + 128 * kMaxChunks - 1) / (128 * kMaxChunks));  // chunk length
    const int nchunks = (n + q - 1) / q;
    const bool vec = (reinterpret_cast<uintptr_t>(row + lo) & 15) == 0;
    auto kept_w = [&](float v) -> u64 { return order_key(v) >= lam ? fixed_weight(v, mx, c) : 0ull; };
    if (vec && q == 128) {
      // one float4 per lane and chunk; four chunks of a warp in flight
      for (int ch0 = warp; ch0 < nchunks; ch0 += 4 * kWarps) {
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ch = ch0 + j * kWarps;
          const int i = lo + ch * 128 + 4 * lane;
          v[j] = (ch < nchunks && i + 3 < hi) ? __ldg(reinterpret_cast<const float4*>(row + i))
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ch = ch0 + j * kWarps;
          const int i = lo + ch * 128 + 4 * lane;
          u64 acc = 0;
          if (ch < nchunks) {
            if (i + 3 < hi) {
              acc = kept_w(v[j].x) + kept_w(v[j].y) + kept_w(v[j].z) + kept_w(v[j].w);
            } else {
              for (int e = i; e < hi; ++e) acc += kept_w(__ldg(row + e));
            }
          }
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
          if (lane == 0 && ch < nchunks) sm.csum[ch] = acc;
        }
      }
    } else {
      for (int ch = warp; ch < nchunks; ch += kWarps) {
        const int c0 = lo + ch * q, c1 = min(hi, c0 + q);
        u64 acc = 0;
        for (int i = c0 + lane; i < c1; i += 32) acc += kept_w(__ldg(row + i));
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) sm.csum[ch] = acc;
      }
    }
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
