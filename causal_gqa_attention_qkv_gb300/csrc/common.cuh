// Device helpers shared by the attention kernels: bf16 packing, mbarriers,
// TMA tile loads, ldmatrix / mma.sync fragments, bounded pipeline waits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/attn.h"

namespace gb300 {

// Layout of the caller's workspace: a 256-byte header (status word first),
// then the per-call scratch areas, each 256-byte aligned.
constexpr size_t kWsHeader = 256;

constexpr float kNegInf = -__builtin_huge_valf();

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------- bf16
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------- f16 and E4M3
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Four E4M3 codes (byte i = element i) -> two f16 pairs: lo = elements 0, 1,
// hi = elements 2, 3 (first element in the low half).  Exact: every E4M3
// value is an f16 value.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// E4M3 codes of two fp32 values, first in the low byte: round to nearest
// even, magnitudes beyond 448 clamped to 448.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Byte permute: result byte i = byte sel_i of the pair (a = bytes 0-3, b = 4-7).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// ---------------------------------------------------------------- dependent launches
// A kernel launched with programmatic stream serialisation may start while
// the kernel before it in the stream is still running; it waits here before
// it touches memory that kernel (or any earlier one) writes.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets such a kernel after this one be scheduled once every CTA of this
// kernel has started (its CTAs then fill SMs as this kernel's CTAs exit).
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- status
__device__ __forceinline__ void set_status(int32_t* status, int32_t bit) {
  if (status) atomicOr(status, bit);
}

// ---------------------------------------------------------------- shared memory addresses
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-suspending check of the same condition (mbarrier.try_wait may suspend
// the thread for a while before it returns false; test_wait never does).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after about
// two seconds (a pipeline that never completes is an internal error): returns
// false and the caller records ATTN_STATUS_TIMEOUT and leaves its loop.  The
// first check is inline; the bounded polling loop is out of line, which keeps
// the common case (the phase is already complete) short.
constexpr uint32_t kWaitSpinLimit = 1u << 22;
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 64) __nanosleep(i < 4096 ? 64 : 512);
  }
  return false;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity);
}

// ---------------------------------------------------------------- TMA
// 3-D tiled load global -> shared, completion counted on `bar` (bytes).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3)
      : "memory");
}

// 3-D tiled store shared -> global, tracked as a bulk group of this thread.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                             int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The shared-memory sources of this thread's bulk groups have been read.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// This thread's bulk groups have completed (writes performed).
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a tile
// written by TMA with CU_TENSOR_MAP_SWIZZLE_128B (rows of 128 bytes; the
// chunk index is XORed with the row index modulo 8; tile base 1024-aligned).
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// ---------------------------------------------------------------- mma.sync fragments
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A * B + D, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A * B + D, m16n8k16, f16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float* d, const uint32_t* a, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- RoPE
// Rotation frequencies theta^(-2i/D) for i < D/2 as float-float pairs
// (hi = nearest float, lo = remainder), and 2*pi as a float-float pair for
// the range reduction.  Computed on the host in double for every call.
struct RopeFreqs {
  float hi[64];
  float lo[64];
  float two_pi_hi, two_pi_lo, inv_two_pi;
};

// cos and sin of pos * f for f = hi + lo: float-float product (pos is an
// exact integer below 2^24, so one fma recovers the rounding error of pos*hi
// exactly), then Cody-Waite additive range reduction modulo 2*pi with 2*pi
// split into two floats, then the hardware sin/cos on |r| <= pi.  The angle
// keeps about 1e-7 rad absolute error at any position; cos/sin about 4e-7.
__device__ __forceinline__ void rope_angle(float pos, float f_hi, float f_lo, const RopeFreqs& fr,
                                           float* c, float* s) {
  const float a_hi = pos * f_hi;
  const float a_err = fmaf(pos, f_hi, -a_hi);
  const float a_lo = fmaf(pos, f_lo, a_err);
  const float k = rintf(a_hi * fr.inv_two_pi);
  float r = fmaf(-k, fr.two_pi_hi, a_hi);
  r = fmaf(-k, fr.two_pi_lo, r);
  r += a_lo;
  __sincosf(r, s, c);  // |r| <= pi + 1e-6: hardware sin/cos, absolute error ~4e-7
}

// ---------------------------------------------------------------- head vectors, pair layout
// A head vector of D bf16 values is held by L = D/16 consecutive lanes: lane
// li of the group takes the 8 values at 8 li and the 8 values at D/2 + 8 li
// (two 16-byte loads), so both members of every rotate-half pair (i, i + D/2)
// sit in one lane.  The prologue kernel and the decode kernel's append both
// use these, so they write the same cache entries bit for bit.

// Eight bf16 values (16 bytes) as fp32, element i from bytes 2i, 2i + 1.
__device__ __forceinline__ void unpack_bf16x8(const uint4& raw, float (&y)[8]) {
  const uint32_t* rw = reinterpret_cast<const uint32_t*>(&raw);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    y[2 * e] = bf16_lo(rw[e]);
    y[2 * e + 1] = bf16_hi(rw[e]);
  }
}

// E4M3 codes of eight fp32 values times an fp32 factor (the product rounded
// to fp32 first, as the cache format states), element i in byte i.
__device__ __forceinline__ uint2 e4m3x8(const float (&y)[8], float r) {
  uint2 v;
  v.x = e4m3x2(__fmul_rn(y[0], r), __fmul_rn(y[1], r)) | (e4m3x2(__fmul_rn(y[2], r), __fmul_rn(y[3], r)) << 16);
  v.y = e4m3x2(__fmul_rn(y[4], r), __fmul_rn(y[5], r)) | (e4m3x2(__fmul_rn(y[6], r), __fmul_rn(y[7], r)) << 16);
  return v;
}

// cos/sin of the rotation pairs 8 li .. 8 li + 7 (li = lane % (D/16)) at
// position pos: each lane computes D/64 of the D/2 angles, the lanes that
// need them read them by shuffle.  All 32 lanes must call this.
template <int D>
__device__ __forceinline__ void pair_angles(float pos, const RopeFreqs& fr, int lane, float (&cs)[8],
                                            float (&sn)[8]) {
  constexpr int PPL = D / 64;
  const int li = lane % (D / 16);
  float c_own[PPL], s_own[PPL];
#pragma unroll
  for (int e = 0; e < PPL; ++e) {
    const int pr = lane * PPL + e;
    rope_angle(pos, fr.hi[pr], fr.lo[pr], fr, &c_own[e], &s_own[e]);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int pr = li * 8 + e;
    cs[e] = __shfl_sync(0xffffffffu, c_own[e % PPL], pr / PPL);
    sn[e] = __shfl_sync(0xffffffffu, s_own[e % PPL], pr / PPL);
  }
}

// RMSNorm and rotate-half of one head vector in the pair layout: raw_a /
// raw_b are this lane's values at 8 li and D/2 + 8 li, w_a / w_b the norm
// weights there (bf16).  Sum of squares: two chains of 8 fused multiply-adds,
// their sum, log2(D/16) shuffle adds over the head's lanes; then
// y = w * (x * rsqrt(ss / D + eps)) and (y_i, y_j) -> (y_i c - y_j s,
// y_j c + y_i s) for j = i + D/2.  All 32 lanes must call this.
template <int D>
__device__ __forceinline__ void norm_rope_pair(const uint4& raw_a, const uint4& raw_b, const uint4& w_a,
                                               const uint4& w_b, const float (&cs)[8], const float (&sn)[8],
                                               float eps, float (&ra)[8], float (&rb)[8]) {
  constexpr int L = D / 16;
  float xa[8], xb[8];
  unpack_bf16x8(raw_a, xa);
  unpack_bf16x8(raw_b, xb);
  float sa = 0.f, sb = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    sa = fmaf(xa[e], xa[e], sa);
    sb = fmaf(xb[e], xb[e], sb);
  }
  float ss = sa + sb;
#pragma unroll
  for (int off = L / 2; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float inv = rsqrtf(ss * (1.0f / D) + eps);
  float wa[8], wb[8];
  unpack_bf16x8(w_a, wa);
  unpack_bf16x8(w_b, wb);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    xa[e] = wa[e] * (xa[e] * inv);
    xb[e] = wb[e] * (xb[e] * inv);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    ra[e] = fmaf(xb[e], -sn[e], xa[e] * cs[e]);
    rb[e] = fmaf(xa[e], sn[e], xb[e] * cs[e]);
  }
}

// One query row (D bf16 values at `row`) normalised and rotated, delivered in
// the m16n8k16 A-fragment distribution: this thread (quad member q = lane & 3)
// holds columns 16ks + 2q + {0,1} in frag[ks][0] and 16ks + 8 + 2q + {0,1} in
// frag[ks][1].  The four threads of a quad hold the whole row, so the RMSNorm
// sum is a quad reduction, and RoPE's partner column c + D/2 sits in the same
// thread at ks + D/32.  All 32 lanes must call this (it shuffles); rows with
// valid == false yield zeros.
template <int D>
__device__ __forceinline__ void q_row_frags(const uint16_t* row, bool valid, const uint16_t* w,
                                            float eps, float pos, const RopeFreqs& fr,
                                            uint32_t (&frag)[D / 16][2]) {
  const int q = threadIdx.x & 3;
  float x[D / 16][4];
  float ss = 0.f;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t a = valid ? __ldg(reinterpret_cast<const uint32_t*>(row + 16 * ks + 2 * q)) : 0u;
    const uint32_t b = valid ? __ldg(reinterpret_cast<const uint32_t*>(row + 16 * ks + 8 + 2 * q)) : 0u;
    x[ks][0] = bf16_lo(a);
    x[ks][1] = bf16_hi(a);
    x[ks][2] = bf16_lo(b);
    x[ks][3] = bf16_hi(b);
#pragma unroll
    for (int j = 0; j < 4; ++j) ss = fmaf(x[ks][j], x[ks][j], ss);
  }
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  const float inv = rsqrtf(ss * (1.0f / D) + eps);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t wa = __ldg(reinterpret_cast<const uint32_t*>(w + 16 * ks + 2 * q));
    const uint32_t wb = __ldg(reinterpret_cast<const uint32_t*>(w + 16 * ks + 8 + 2 * q));
    x[ks][0] = bf16_lo(wa) * (x[ks][0] * inv);
    x[ks][1] = bf16_hi(wa) * (x[ks][1] * inv);
    x[ks][2] = bf16_lo(wb) * (x[ks][2] * inv);
    x[ks][3] = bf16_hi(wb) * (x[ks][3] * inv);
  }
#pragma unroll
  for (int ks = 0; ks < D / 32; ++ks) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = 16 * ks + (j >> 1) * 8 + 2 * q + (j & 1);  // rotation pair index < D/2
      float c, s;
      rope_angle(pos, fr.hi[i], fr.lo[i], fr, &c, &s);
      const float x1 = x[ks][j], x2 = x[ks + D / 32][j];
      x[ks][j] = x1 * c - x2 * s;
      x[ks + D / 32][j] = x2 * c + x1 * s;
    }
  }
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    frag[ks][0] = pack_bf16(x[ks][0], x[ks][1]);
    frag[ks][1] = pack_bf16(x[ks][2], x[ks][3]);
  }
}

// One query row normalised and rotated, as f16 A fragments in the layout
// the E4M3 decode kernel reads keys in: quad member c = lane & 3 holds the
// columns [c D/4, (c+1) D/4), frag[ks][0] = columns c D/4 + 4ks + {0,1} and
// frag[ks][1] = c D/4 + 4ks + {2,3} (the dot product does not depend on
// which k slot a column occupies, as long as query and key agree).  The
// RMSNorm sum is a quad reduction; the RoPE partner column (D/2 away) sits
// in quad member c ^ 2.  All 32 lanes must call this; rows with
// valid == false yield zeros.
template <int D>
__device__ __forceinline__ void q_row_frags_quarters(const uint16_t* row, bool valid,
                                                     const uint16_t* w, float eps, float pos,
                                                     const RopeFreqs& fr,
                                                     uint32_t (&frag)[D / 16][2]) {
  constexpr int Q = D / 4;  // columns per quad member
  const int c = threadIdx.x & 3;
  float x[Q];
  float ss = 0.f;
#pragma unroll
  for (int v = 0; v < Q / 8; ++v) {
    const uint4 u = valid ? __ldg(reinterpret_cast<const uint4*>(row + c * Q + 8 * v)) : make_uint4(0, 0, 0, 0);
    const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[8 * v + 2 * j] = bf16_lo(uw[j]);
      x[8 * v + 2 * j + 1] = bf16_hi(uw[j]);
    }
  }
#pragma unroll
  for (int i = 0; i < Q; ++i) ss = fmaf(x[i], x[i], ss);
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  const float inv = rsqrtf(ss * (1.0f / D) + eps);
#pragma unroll
  for (int v = 0; v < Q / 8; ++v) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(w + c * Q + 8 * v));
    const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[8 * v + 2 * j] = bf16_lo(uw[j]) * (x[8 * v + 2 * j] * inv);
      x[8 * v + 2 * j + 1] = bf16_hi(uw[j]) * (x[8 * v + 2 * j + 1] * inv);
    }
  }
  const bool first_half = c < 2;
#pragma unroll
  for (int e = 0; e < Q; ++e) {
    const int i = (c & 1) * Q + e;  // rotation pair index < D/2
    float cs, sn;
    rope_angle(pos, fr.hi[i], fr.lo[i], fr, &cs, &sn);
    const float other = __shfl_xor_sync(0xffffffffu, x[e], 2);
    // first half: x_i c - x_{i+D/2} s; second half: x_{i+D/2} c + x_i s
    x[e] = first_half ? x[e] * cs - other * sn : x[e] * cs + other * sn;
  }
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    frag[ks][0] = pack_f16(x[4 * ks], x[4 * ks + 1]);
    frag[ks][1] = pack_f16(x[4 * ks + 2], x[4 * ks + 3]);
  }
}

// ---------------------------------------------------------------- requests
// How kernels find cache entries (the attn_kv_t indexing fields).
struct KvIndex {
  const int64_t* slot_base;      // contiguous layout
  const int32_t* cache_lens;
  const int32_t* slot_capacity;
  const int32_t* page_table;     // nullptr: contiguous layout
  int64_t num_slots;
  int32_t log2_page;             // log2(page_size) (paged layout)
  int32_t pages_per_req;
};

// Per-request facts every kernel derives the same way from the arguments.
struct ReqInfo {
  int64_t slot0;         // contiguous layout: slot of position 0
  const int32_t* pages;  // paged layout: the request's page-table row, else nullptr
  int32_t cached;        // c_b
  int32_t n_new;         // n_b
  bool valid;            // the request can hold c_b + n_b entries and cu_seqlens is sane
};

__device__ __forceinline__ ReqInfo load_request(const KvIndex& kv, int b, int32_t n_new) {
  ReqInfo r;
  r.cached = kv.cache_lens[b];
  r.n_new = n_new;
  const int64_t end = (int64_t)r.cached + (int64_t)n_new;
  const bool sizes = n_new >= 0 && r.cached >= 0 && end <= (int64_t)kv.slot_capacity[b] && end <= (1 << 24);
  if (kv.page_table) {
    r.pages = kv.page_table + (int64_t)b * kv.pages_per_req;
    r.slot0 = 0;
    r.valid = sizes && end <= ((int64_t)kv.pages_per_req << kv.log2_page);
  } else {
    r.pages = nullptr;
    r.slot0 = kv.slot_base[b];
    r.valid = sizes && r.slot0 >= 0 && r.slot0 + end <= kv.num_slots;
  }
  return r;
}

// Slot of the entry at position pos of a request, or -1 when its page number
// is outside the cache (paged layout; pos < pages_per_req * page_size).
__device__ __forceinline__ int64_t cache_slot(const KvIndex& kv, const ReqInfo& r, int pos) {
  if (!r.pages) return r.slot0 + pos;
  const int64_t pg = __ldg(r.pages + (pos >> kv.log2_page));
  const int64_t slot = (pg << kv.log2_page) + (pos & ((1 << kv.log2_page) - 1));
  return (pg >= 0 && slot < kv.num_slots) ? slot : -1;
}

}  // namespace gb300
