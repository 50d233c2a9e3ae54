// Token sampling from rows of logits: greedy argmax, or temperature + top-k +
// top-p truncation and sampling by the inverse distribution function.
//
// Concept chapter section 3.2 (greedy decoding, temperature, top-k, top-p;
// the temperature formula of section 3.2.2) and the walkthrough's section 4.3
// (a greedy batch takes the argmax, the others go through temperature and
// top-k/top-p).  One CTA per row of V logits:
//   1. the maximum and its first index (greedy rows stop here);
//   2-4. weights w_i = exp((l_i - max) / T) as integers in units of 2^-40
//      (every sum below is exact and independent of order), and a radix
//      select over the order-preserving bit pattern of the logits in three
//      digits of 8, 12 and 12 bits: per digit, the count and the mass of the
//      candidate keys in each bin; scanning the bins from the largest finds
//      the key at which the count reaches top_k or the mass reaches
//      top_p x total first, i.e. the smallest kept logit (ties kept).  The
//      first digit (sign and exponent) puts a row's logits into few bins, so
//      each warp counts into a histogram of its own, merged afterwards;
//   5. the smallest index whose cumulative kept weight exceeds u x kept mass:
//      kept mass per chunk of consecutive tokens, a block scan to the chunk,
//      one warp's walk through it.
// Each pass reads the row (from L2 after the first) with float4 loads.
#include "kernels.cuh"

namespace gb300 {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins0 = 256;   // first digit: 8 bits
constexpr int kBins = 4096;   // second and third digits: 12 bits
// dynamic shared memory: 32 warp histograms of the first digit (counts, then
// masses), later reused for the block histograms of the other two
constexpr int kSmemBytes = kWarps * kBins0 * (4 + 8);
static_assert(kBins * (4 + 8) <= kSmemBytes, "histograms");
constexpr int kMaxChunks = 2 * kThreads;  // chunks of the final scan (kept masses in shared memory)
static_assert(kMaxChunks * 8 <= kSmemBytes, "chunk sums");
using u64 = unsigned long long;

// Larger float -> larger key (finite values and -inf).
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SamplePar {
  const float* logits;
  int64_t ld;
  int32_t V;
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

// Calls f(index, value) for this thread's share of the row: float4 loads two
// at a time when the row is 16-byte aligned (more bytes in flight per
// thread), then the scalar tail.  Within a thread the indices are not in
// increasing order.
template <class F>
__device__ __forceinline__ void for_row(const float* row, int V, F&& f) {
  int tail = 0;
  if ((reinterpret_cast<uintptr_t>(row) & 15) == 0) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int n4 = V >> 2;
    int i = threadIdx.x;
    for (; i + kThreads < n4; i += 2 * kThreads) {
      const float4 a = __ldg(r4 + i), e = __ldg(r4 + i + kThreads);
      const int j = 4 * (i + kThreads);
      f(4 * i, a.x);
      f(4 * i + 1, a.y);
      f(4 * i + 2, a.z);
      f(4 * i + 3, a.w);
      f(j, e.x);
      f(j + 1, e.y);
      f(j + 2, e.z);
      f(j + 3, e.w);
    }
    if (i < n4) {
      const float4 a = __ldg(r4 + i);
      f(4 * i, a.x);
      f(4 * i + 1, a.y);
      f(4 * i + 2, a.z);
      f(4 * i + 3, a.w);
    }
    tail = 4 * n4;
  }
  for (int j = tail + (int)threadIdx.x; j < V; j += kThreads) f(j, __ldg(row + j));
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

__global__ void __launch_bounds__(kThreads) sample_kernel(const SamplePar p) {
  extern __shared__ __align__(16) uint8_t hist[];
  __shared__ uint32_t cnt0[kBins0];
  __shared__ u64 mass0[kBins0];
  __shared__ float s_mx[kWarps];
  __shared__ int s_arg[kWarps];
  __shared__ u64 s_sum[kWarps];
  __shared__ u64 s_sel_above_mass, s_sel_bin_mass, s_excl;
  __shared__ uint32_t s_sel_digit, s_sel_above_cnt;
  __shared__ int s_warp;  // the chunk holding u x S

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int V = p.V;
  const float* row = p.logits + (int64_t)b * p.ld;

  // 1. maximum and its first index
  float mx = -__builtin_huge_valf();
  int arg = 0x7fffffff;
  for_row(row, V, [&](int i, float v) {
    if (v > mx || (v == mx && i < arg) || arg == 0x7fffffff) {
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
    s_mx[warp] = mx;
    s_arg[warp] = arg;
  }
  __syncthreads();
  mx = s_mx[0];
  arg = s_arg[0];
  for (int w = 1; w < kWarps; ++w)
    if (s_mx[w] > mx || (s_mx[w] == mx && s_arg[w] < arg)) {
      mx = s_mx[w];
      arg = s_arg[w];
    }
  const float T = p.temperature[b];
  if (!(T > 0.f)) {
    if (tid == 0) p.tokens[b] = arg;
    return;  // uniform across the block
  }
  if (tid == 0) p.tokens[b] = arg;  // replaced below
  const float c = 1.4426950408889634f / T;
  const int k = p.top_k[b];
  const uint32_t k_lim = (k > 0 && k < V) ? (uint32_t)k : 0xffffffffu;
  const float top_p = p.top_p[b];

  // 2. first digit (bits 31-24): warp histograms, then merged; the total weight
  uint32_t* wcnt = reinterpret_cast<uint32_t*>(hist);
  u64* wmass = reinterpret_cast<u64*>(hist + kWarps * kBins0 * 4);
  for (int i = tid; i < kWarps * kBins0; i += kThreads) {
    wcnt[i] = 0;
    wmass[i] = 0;
  }
  __syncthreads();
  u64 wsum = 0;
  {
    uint32_t* mc = wcnt + warp * kBins0;
    u64* mm = wmass + warp * kBins0;
    for_row(row, V, [&](int, float v) {
      const uint32_t d = order_key(v) >> 24;
      const u64 w = fixed_weight(v, mx, c);
      wsum += w;
      atomicAdd(&mc[d], 1u);
      if (w) atomicAdd(&mm[d], w);
    });
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
  if (lane == 0) s_sum[warp] = wsum;
  __syncthreads();
  for (int d = tid; d < kBins0; d += kThreads) {
    uint32_t cs = 0;
    u64 ms = 0;
    for (int w = 0; w < kWarps; ++w) {
      cs += wcnt[w * kBins0 + d];
      ms += wmass[w * kBins0 + d];
    }
    cnt0[d] = cs;
    mass0[d] = ms;
  }
  u64 W = 0;
  for (int w = 0; w < kWarps; ++w) W += s_sum[w];
  u64 mass_lim;
  if (top_p >= 1.f) mass_lim = W;  // reached once every token of positive weight is in
  else if (!(top_p > 0.f)) mass_lim = 0;
  else mass_lim = (u64)ceil((double)top_p * (double)W);
  __syncthreads();
  if (warp == 0)
    find_crossing(cnt0, mass0, kBins0, 0u, 0ull, k_lim, mass_lim, &s_sel_digit, &s_sel_above_cnt,
                  &s_sel_above_mass, &s_sel_bin_mass);
  __syncthreads();
  uint32_t prefix = s_sel_digit << 24, cnt_above = s_sel_above_cnt;
  u64 mass_above = s_sel_above_mass, bin_mass = s_sel_bin_mass;

  // 3-4. second (bits 23-12) and third (bits 11-0) digits among the keys
  // that share the digits found so far: block histograms
  uint32_t* cnt = reinterpret_cast<uint32_t*>(hist);
  u64* mass = reinterpret_cast<u64*>(hist + kBins * 4);
  for (int lv = 1; lv < 3; ++lv) {
    const int shift = lv == 1 ? 12 : 0;
    const uint32_t fixed_mask = lv == 1 ? 0xff000000u : 0xfffff000u;
    for (int i = tid; i < kBins; i += kThreads) {
      cnt[i] = 0;
      mass[i] = 0;
    }
    __syncthreads();
    for_row(row, V, [&](int, float v) {
      const uint32_t key = order_key(v);
      if ((key & fixed_mask) != prefix) return;
      const uint32_t d = (key >> shift) & (uint32_t)(kBins - 1);
      atomicAdd(&cnt[d], 1u);
      const u64 w = fixed_weight(v, mx, c);
      if (w) atomicAdd(&mass[d], w);
    });
    __syncthreads();
    if (warp == 0)
      find_crossing(cnt, mass, kBins, cnt_above, mass_above, k_lim, mass_lim, &s_sel_digit,
                    &s_sel_above_cnt, &s_sel_above_mass, &s_sel_bin_mass);
    __syncthreads();
    prefix |= s_sel_digit << shift;
    cnt_above = s_sel_above_cnt;
    mass_above = s_sel_above_mass;
    bin_mass = s_sel_bin_mass;
    __syncthreads();  // the bins are cleared for the next level
  }
  const uint32_t lam = prefix;  // keys >= lam are kept
  const u64 S = mass_above + bin_mass;

  // 5. inverse distribution function in vocabulary order: kept mass per
  // chunk of q consecutive tokens (at most kMaxChunks chunks), a block scan to
  // the chunk holding u x S, then one warp walks that chunk.
  u64 t = (u64)((double)p.uniform[b] * (double)S);
  if (t >= S) t = S - 1;
  const int q = 128 * max(1, (V + 128 * kMaxChunks - 1) / (128 * kMaxChunks));
  const int nchunks = (V + q - 1) / q;
  u64* csum = reinterpret_cast<u64*>(hist);  // the histograms are no longer needed
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
  for (int ch = warp; ch < nchunks; ch += kWarps) {
    const int c0 = ch * q, c1 = min(V, c0 + q);
    u64 acc = 0;
    if (vec) {  // chunk starts are multiples of 128 floats: 16-byte aligned
      for (int i = c0 + 4 * lane; i < c1; i += 128) {
        if (i + 3 < c1) {
          const float4 a = __ldg(reinterpret_cast<const float4*>(row + i));
          const float vv[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (order_key(vv[e]) >= lam) acc += fixed_weight(vv[e], mx, c);
        } else {
          for (int e = i; e < c1; ++e) {
            const float v = __ldg(row + e);
            if (order_key(v) >= lam) acc += fixed_weight(v, mx, c);
          }
        }
      }
    } else {
      for (int i = c0 + lane; i < c1; i += 32) {
        const float v = __ldg(row + i);
        if (order_key(v) >= lam) acc += fixed_weight(v, mx, c);
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) csum[ch] = acc;
  }
  if (tid == 0) s_warp = -1;
  __syncthreads();
  {
    // thread t owns chunks 2t and 2t + 1
    const u64 a = 2 * tid < nchunks ? csum[2 * tid] : 0ull;
    const u64 e = 2 * tid + 1 < nchunks ? csum[2 * tid + 1] : 0ull;
    const u64 own = a + e;
    u64 incl = own;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const u64 o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) s_sum[warp] = incl;
    __syncthreads();
    u64 before = 0;
    for (int w = 0; w < warp; ++w) before += s_sum[w];
    const u64 xa = before + incl - own;  // kept mass before chunk 2t
    if (a > 0 && xa <= t && t < xa + a) {
      s_warp = 2 * tid;
      s_excl = xa;
    }
    if (e > 0 && xa + a <= t && t < xa + a + e) {
      s_warp = 2 * tid + 1;
      s_excl = xa + a;
    }
  }
  __syncthreads();
  if (warp == 0 && s_warp >= 0) {
    const int c0 = s_warp * q, c1 = min(V, c0 + q);
    u64 acc = s_excl;
    for (int base = c0; base < c1; base += 32) {
      const int i = base + lane;
      u64 wv = 0;
      if (i < c1) {
        const float v = __ldg(row + i);
        if (order_key(v) >= lam) wv = fixed_weight(v, mx, c);
      }
      u64 incl = wv;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const u64 o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, acc + incl > t);
      if (hit) {
        if (lane == __ffs(hit) - 1) p.tokens[b] = i;
        break;
      }
      acc += __shfl_sync(0xffffffffu, incl, 31);
    }
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
  p.temperature = temperature;
  p.top_k = top_k;
  p.top_p = top_p;
  p.uniform = uniform;
  p.tokens = tokens;
  if (cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
      cudaSuccess)
    return ATTN_ELAUNCH;
  sample_kernel<<<B, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ELAUNCH;
}

}  // namespace gb300
