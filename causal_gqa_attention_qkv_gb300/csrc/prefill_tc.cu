// Prefill attention on the 5th-generation tensor cores (tcgen05 + TMEM),
// persistent: one CTA per SM walks a list of work items.
//
// Code walkthrough section 3.3 teaching snippet and transformer-basics
// "Attention calculation: part 1": scores q.k / sqrt(D) against KV head
// h / (Hq/Hkv), future positions masked, softmax in fp32, P rounded to the
// input type, P times V; concept chapter section 2.6: computed the I/O-aware
// way (flash attention), never materialising the score matrix.
//
// Q arrives normed and rotated (prologue kernel).  Work item = (sequence b,
// KV head kh, block of 2 x 128 query rows).  A 128-row Q tile is 128/G tokens
// x the G heads of the group, so every K/V tile loaded serves the whole GQA
// group; the item's two Q tiles (A: its first 128/G tokens, B: the next
// 128/G) share every K/V tile.  Items are numbered round-major: round r holds
// block r counted from the end of every sequence (the heaviest blocks come
// first, the last ones claimed are light), and are handed out dynamically: a
// CTA's Q producer claims the next number from a counter in the workspace and
// publishes it to the CTA's other roles through a ring in shared memory.
//
// Roles (384 threads, three warpgroups):
//   warps 0-3   softmax of Q tile A, warps 4-7 softmax of Q tile B: thread r
//               of a warpgroup owns row r = TMEM lane r of its tile.  Per KV
//               tile: read S from TMEM, mask, online softmax in fp32 (exp2
//               domain), P (bf16; f16 with F8) written over S in TMEM, O rescaled in TMEM
//               when the reference max moves; per item: O / l -> out.
//   warp 8      TMA: K tiles (2-stage ring of 128 keys, across items); with
//               F8 the whole warp also converts each tile to f16.
//   warp 9      MMA issuer (one thread) and TMEM owner.
//   warp 10     TMA: V tiles (2-stage ring; converted the same way with F8).
//   warp 11     claims items; TMA: the item's two Q tiles (one buffer each).
// Each producer runs in a warp of its own: a thread waiting for a free stage
// may be suspended, and diverged lanes of one warp do not run independently.
//
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256,256+D),
// O_B [384,384+D).  Issue order per KV tile j:
//   P.V_A(j), S_A(j+1) = Q_A K(j+1)^T, P.V_B(j), S_B(j+1)
// so the tensor cores compute tile B's products while the softmax of tile A
// runs and the other way round.  Because the tensor-core operations of one
// thread complete in issue order, S_X(j+1) being complete means P.V_X(j) is
// complete: the softmax may rescale O_X as soon as it sees S_X(j+1).
//
// E4M3 caches (F8): the K and V warps copy each 128-key tile of codes into
// the last 128 x D bytes of its stage and convert it there, all 32 lanes, to
// the f16 tile layout the bf16 path gets from TMA (every E4M3 value is an
// f16 value); Q arrives in f16, P is packed to f16, the products run as
// kind::f16 with f16 operands, and the cache scales multiply the scores
// (k_scale) and the output (v_scale).
#include "kernels.cuh"
#include "tcgen05.cuh"

namespace gb300 {

namespace {

constexpr int kTileRows = 128;  // query rows per Q tile (MMA M)
constexpr int kKeys = 128;      // keys per KV tile (MMA N of Q K^T)
constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 128;  // per Q tile
constexpr int kKWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kVWarp = 10;
constexpr int kQWarp = 11;
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kMaxSeqSmem = 32;  // sequences whose facts are cached in shared memory
constexpr int kRing = 4;         // claimed items published ahead of their use
// readers of each ring slot: K, V and MMA threads, one per softmax warp
constexpr int kRingReaders = 3 + 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;  // O_A at 256, O_B at 384; S_A at 0, S_B at 128
constexpr int kRegionBytes = 128 * 128;   // 128 rows x 128 bytes (64 bf16)
constexpr float kRescaleThreshold = 8.f;  // log2 units: move the reference max past 256x growth

struct TcPar {
  const int32_t* cu_seqlens;
  KvIndex kv;
  int32_t half_boxes;  // paged cache with 64-slot pages: a K/V tile is two 64-row boxes
  int32_t* status;
  int32_t* work;  // [0]: next item to claim, [1]: CTAs finished
  uint16_t* out;
  float scale_log2;  // log2(e) / sqrt(D), times k_scale for an E4M3 cache
  float v_scale;     // 1, or v_scale for an E4M3 cache
  int32_t Hq, Hkv, log2G, log2BT, N, B, max_seqlen;
  int32_t num_vitems;  // rounds x B x Hkv, rounds = ceil(max_seqlen / (2 x 128/G))
};

template <int D>
struct TcLayout {
  static constexpr int kRegions = D / 64;
  static constexpr int kTile = kRegions * kRegionBytes;  // Q, K or V tile: 128 rows x D
  static constexpr int kQ = 0;                       // Q tiles A, B
  static constexpr int kK = kQ + 2 * kTile;          // kKStages
  static constexpr int kV = kK + kKStages * kTile;   // kVStages
  // output staging for TMA stores: 4 KB (32 rows x 64 columns bf16) per softmax warp
  static constexpr int kStg = kV + kVStages * kTile;
  static constexpr int kBar = kStg + 8 * 4096;
  static constexpr int kNumBars = 32;
  static constexpr int kSeq = kBar + kNumBars * 8;  // SeqInfo[kMaxSeqSmem]
  static constexpr int kRingOff = kSeq + kMaxSeqSmem * 24;  // int[kRing]
  static constexpr int kTmemSlot = kRingOff + kRing * 4;
  // + alignment slack; at least 116 KB so that one CTA runs per SM (each CTA
  // allocates all 512 TMEM columns).
  static constexpr int kSmemRaw = kTmemSlot + 16 + 1024;
  static constexpr int kSmemBytes = kSmemRaw > 116 * 1024 ? kSmemRaw : 116 * 1024;
  static_assert(kSmemRaw <= 227 * 1024, "shared memory");
};

enum Bar {
  // Every barrier advances one phase per use of its buffer, so no waiter can
  // fall two phases behind.
  kQFullA = 0, kQFullB, kQEmptyA, kQEmptyB,   // Q tiles (empty: the item's last S_X done)
  kKFull0, kKEmpty0 = kKFull0 + kKStages,     // K stages (empty: S_A and S_B of the tile done)
  kVFull0 = kKEmpty0 + kKStages, kVEmpty0 = kVFull0 + kVStages,  // V stages (empty: both P.V done)
  kSFullA = kVEmpty0 + kVStages, kSFullB,     // S_X of a tile complete (and every earlier MMA)
  kPFullA, kPFullB,                           // P_X of a tile in TMEM (128 arrivals)
  kODoneA, kODoneB,                           // the item's last P.V_X complete
  kMmaDone,
  kItemFull0, kItemFree0 = kItemFull0 + kRing,  // item ring: slot written / read by every role
  kKLand0 = kItemFree0 + kRing,               // E4M3: a stage's codes have landed
  kVLand0 = kKLand0 + kKStages,
  kBarCount = kVLand0 + kVStages
};
static_assert(kBarCount <= TcLayout<64>::kNumBars, "barriers");

// ---------------------------------------------------------------- work items
// Item number vi = (r * B + b) * Hkv + kh: block r counted from the end of
// sequence b (an empty slot when sequence b has r blocks or fewer), KV head kh.
struct Item {
  int b, kh, t0, n_b, tokbase, cached, nk, kv_total;
  int64_t slot0;
};

// Per-sequence facts the item numbering needs, kept in shared memory for
// batches of up to kMaxSeqSmem sequences (read from global memory otherwise)
// so that moving to the next item costs no global-memory round trips.
struct SeqInfo {
  int64_t slot0;
  int tokbase, n_b, cached, usable;  // usable: the request's items are computed
};

__device__ __forceinline__ SeqInfo seq_info(const TcPar& p, int b) {
  SeqInfo q;
  q.tokbase = p.cu_seqlens[b];
  q.n_b = p.cu_seqlens[b + 1] - q.tokbase;
  const ReqInfo r = load_request(p.kv, b, q.n_b);
  q.slot0 = r.slot0;
  q.cached = r.cached;
  // sequences with no tokens, outside [0, N), longer than the host bound or
  // with a region too small are skipped (flagged by the prologue / below)
  q.usable = q.n_b > 0 && q.tokbase >= 0 && q.tokbase + q.n_b <= p.N && q.n_b <= p.max_seqlen &&
             r.valid;
  return q;
}

__device__ __forceinline__ bool item_at(const TcPar& p, const SeqInfo* tab, int vi, Item& it) {
  const int rb = vi / p.Hkv;
  it.kh = vi - rb * p.Hkv;
  const int r = rb / p.B;
  const int b = rb - r * p.B;
  const SeqInfo q = tab ? tab[b] : seq_info(p, b);
  if (!q.usable) return false;
  const int log2IT = p.log2BT + 1;
  const int IT = 1 << log2IT;
  const int nblk = (q.n_b + IT - 1) >> log2IT;
  if (r >= nblk) return false;
  it.b = b;
  it.t0 = (nblk - 1 - r) * IT;
  it.n_b = q.n_b;
  it.tokbase = q.tokbase;
  it.cached = q.cached;
  it.slot0 = q.slot0;
  it.kv_total = q.cached + q.n_b;
  it.nk = (q.cached + min(it.t0 + IT, q.n_b) + kKeys - 1) / kKeys;
  return true;
}

// Reads this CTA's items from the ring in order.  A number < 0 ends the walk.
// Single-thread roles acknowledge each slot themselves; in a softmax warp all
// lanes read it and lane 0 acknowledges.
struct ItemWalk {
  const SeqInfo* tab;  // shared-memory sequence table or nullptr
  const int* ring;
  uint64_t* bars;
  int k;               // items read so far
  bool warp_wide;
  bool valid;
  Item it;

  __device__ __forceinline__ void start(const TcPar& p, const SeqInfo* table, const int* ring_,
                                        uint64_t* bars_, bool warp_wide_, bool& ok) {
    tab = table;
    ring = ring_;
    bars = bars_;
    k = 0;
    warp_wide = warp_wide_;
    next(p, ok);
  }
  __device__ __forceinline__ void next(const TcPar& p, bool& ok) {
    const int slot = k % kRing;
    uint64_t* full = &bars[kItemFull0 + slot];
    const uint32_t par = (k / kRing) & 1;
    bool got = mbar_wait(full, par);
    if (warp_wide) got = __all_sync(0xffffffffu, got);
    if (!got) {
      ok = false;
      valid = false;
      return;
    }
    const int vi = *reinterpret_cast<const volatile int*>(&ring[slot]);
    if (warp_wide) __syncwarp();
    if (!warp_wide || (threadIdx.x & 31) == 0) mbar_arrive(&bars[kItemFree0 + slot]);
    ++k;
    valid = vi >= 0 && item_at(p, tab, vi, it);
  }
};

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity) {
  const bool w = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, w);
}

// Packed pairs of fp32 values (the low half is the first element) and the
// paired fp32 operations of this architecture.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2_lo(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo;
}
__device__ __forceinline__ float f2_hi(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return hi;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}


// ---------------------------------------------------------------- roles
// One TMA producer ring (K or V tiles): tile g of the CTA's tile sequence goes
// to stage g % stages once the stage's previous tile has been consumed.
// First cache row of the rows [pos, pos + rows) of item it's sequence (rows
// within one page in the paged layout).  A page outside the cache sets
// ATTN_STATUS_CAPACITY and is read from row 0 instead (its keys are wrong,
// nothing is out of bounds).
__device__ __forceinline__ int kv_row(const TcPar& p, const Item& it, int pos) {
  if (!p.kv.page_table) return (int)(it.slot0 + pos);
  ReqInfo r;
  r.slot0 = 0;
  r.pages = p.kv.page_table + (int64_t)it.b * p.kv.pages_per_req;
  const int64_t s = cache_slot(p.kv, r, pos);
  if (s < 0) {
    set_status(p.status, ATTN_STATUS_CAPACITY);
    return 0;
  }
  return (int)s;
}

template <int D>
__device__ void produce_kv(const TcPar& p, const SeqInfo* seq_tab, const int* ring,
                           const CUtensorMap* map, uint8_t* smem, uint64_t* bars, int base,
                           int full0, int empty0, int stages, bool& ok) {
  using Lay = TcLayout<D>;
  prefetch_tmap(map);
  ItemWalk w;
  w.start(p, seq_tab, ring, bars, false, ok);
  int g = 0;
  while (w.valid && ok) {
    for (int j = 0; j < w.it.nk; ++j, ++g) {
      const int st = g % stages;
      if (g >= stages && !mbar_wait(&bars[empty0 + st], (g / stages - 1) & 1)) { ok = false; break; }
      mbar_arrive_expect_tx(&bars[full0 + st], Lay::kTile);
      uint8_t* dst = smem + base + st * Lay::kTile;
      if (!p.half_boxes) {
        const int row = kv_row(p, w.it, j * kKeys);
#pragma unroll
        for (int rg = 0; rg < Lay::kRegions; ++rg)
          tma_load_3d(dst + rg * kRegionBytes, map, &bars[full0 + st], rg * 64, w.it.kh, row);
      } else {
        // two 64-key pages; a second half past the sequence end re-reads the
        // last page (those keys are masked and their V rows zeroed)
        const int pos1 = min(j * kKeys + 64, ((w.it.kv_total - 1) >> 6) << 6);
        const int row0 = kv_row(p, w.it, j * kKeys), row1 = kv_row(p, w.it, pos1);
#pragma unroll
        for (int rg = 0; rg < Lay::kRegions; ++rg) {
          tma_load_3d(dst + rg * kRegionBytes, map, &bars[full0 + st], rg * 64, w.it.kh, row0);
          tma_load_3d(dst + rg * kRegionBytes + 64 * 128, map, &bars[full0 + st], rg * 64, w.it.kh, row1);
        }
      }
    }
    if (!ok) break;
    w.next(p, ok);
  }
  // Every load issued has landed before the CTA may exit (immediate on the
  // normal path, where the consumers already waited for them).
  for (int t = max(0, g - stages); t < g; ++t) (void)mbar_wait(&bars[full0 + t % stages], (t / stages) & 1);
}

// The same ring for an E4M3 cache, run by the whole warp: lane 0 copies each
// tile of codes (128 keys x D bytes) into the last 128 x D bytes of its stage;
// then every lane converts key rows to the f16 tile layout and lane 0
// releases the stage to the tensor cores.
template <int D>
__device__ void produce_kv_f8(const TcPar& p, const SeqInfo* seq_tab, const int* ring,
                              const CUtensorMap* map, uint8_t* smem, uint64_t* bars, int base,
                              int full0, int empty0, int land0, int stages, bool& ok) {
  using Lay = TcLayout<D>;
  const int lane = threadIdx.x & 31;
  constexpr int kCodeBytes = kKeys * D;
  if (lane == 0) prefetch_tmap(map);
  ItemWalk w;
  w.start(p, seq_tab, ring, bars, true, ok);
  int g = 0, issued = 0;
  while (w.valid && ok) {
    for (int j = 0; j < w.it.nk; ++j, ++g) {
      const int st = g % stages;
      if (!__all_sync(0xffffffffu, g < stages || mbar_wait(&bars[empty0 + st], (g / stages - 1) & 1))) {
        ok = false;
        break;
      }
      uint8_t* dst = smem + base + st * Lay::kTile;
      uint8_t* land = dst + Lay::kTile - kCodeBytes;  // 1024-aligned
      uint64_t* bar = &bars[land0 + st];
      if (lane == 0) {
        mbar_arrive_expect_tx(bar, kCodeBytes);
        if (!p.half_boxes) {
          tma_load_3d(land, map, bar, 0, w.it.kh, kv_row(p, w.it, j * kKeys));
        } else {
          const int pos1 = min(j * kKeys + 64, ((w.it.kv_total - 1) >> 6) << 6);
          tma_load_3d(land, map, bar, 0, w.it.kh, kv_row(p, w.it, j * kKeys));
          tma_load_3d(land + kCodeBytes / 2, map, bar, 0, w.it.kh, kv_row(p, w.it, pos1));
        }
      }
      ++issued;
      if (!__all_sync(0xffffffffu, mbar_wait(bar, (g / stages) & 1))) { ok = false; break; }
      // Lane l converts key rows l, l + 32, l + 64, l + 96: codes of row r
      // (D bytes, 128-byte swizzled when D = 128) -> f16 row r of each
      // 64-column region.  Each row is read whole before any lane writes:
      // for D = 64 later f16 rows cover other lanes' code rows.
      const uint32_t tile = smem_u32(dst), codes = smem_u32(land);
#pragma unroll 1
      for (int i = 0; i < kKeys / 32; ++i) {
        const uint32_t r = (uint32_t)(lane + 32 * i);
        uint4 c[D / 16];
#pragma unroll
        for (int ch = 0; ch < D / 16; ++ch)
          c[ch] = lds128(codes + (D == 128 ? sw128(r, ch) : r * (uint32_t)D + ch * 16));
        __syncwarp();
#pragma unroll
        for (int ch = 0; ch < D / 16; ++ch) {
          uint4 lo, hi;  // codes 16ch .. 16ch + 7 and 16ch + 8 .. 16ch + 15 as f16
          e4m3x4_to_f16(c[ch].x, lo.x, lo.y);
          e4m3x4_to_f16(c[ch].y, lo.z, lo.w);
          e4m3x4_to_f16(c[ch].z, hi.x, hi.y);
          e4m3x4_to_f16(c[ch].w, hi.z, hi.w);
          const uint32_t region = tile + (uint32_t)((2 * ch) >> 3) * kRegionBytes;
          sts128(region + sw128(r, (2 * ch) & 7), lo);
          sts128(region + sw128(r, (2 * ch + 1) & 7), hi);
        }
        __syncwarp();
      }
      tc::fence_proxy_async();  // the f16 tile is visible to the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[full0 + st]);
    }
    if (!ok) break;
    w.next(p, ok);
  }
  // Every copy issued has landed before the CTA may exit.
  if (lane == 0)
    for (int t = max(0, issued - stages); t < issued; ++t)
      (void)mbar_wait(&bars[land0 + t % stages], (t / stages) & 1);
}

// Claims items from the counter in the workspace, publishes each to the
// ring and loads its two Q tiles.  The last slot written holds -1.
template <int D>
__device__ void produce_q(const TcPar& p, const SeqInfo* seq_tab, int* ring,
                          const CUtensorMap* qmap, uint8_t* smem, uint64_t* bars, bool& ok) {
  using Lay = TcLayout<D>;
  prefetch_tmap(qmap);
  const int G = 1 << p.log2G, BT = 1 << p.log2BT;
  int k = 0;
  while (ok) {
    int vi;
    Item it;
    bool have = false;
    while ((vi = atomicAdd(p.work, 1)) < p.num_vitems)
      if (item_at(p, seq_tab, vi, it)) {
        have = true;
        break;
      }
    const int slot = k % kRing;
    if (k >= kRing && !mbar_wait(&bars[kItemFree0 + slot], (k / kRing - 1) & 1)) { ok = false; break; }
    ring[slot] = have ? vi : -1;
    mbar_arrive(&bars[kItemFull0 + slot]);  // release: the slot's value is visible to its readers
    if (!have) break;
    for (int x = 0; x < 2; ++x) {
      if (k >= 1 && !mbar_wait(&bars[kQEmptyA + x], (k - 1) & 1)) { ok = false; break; }
      mbar_arrive_expect_tx(&bars[kQFullA + x], Lay::kTile);
#pragma unroll
      for (int rg = 0; rg < Lay::kRegions; ++rg)
        tma_load_3d(smem + Lay::kQ + x * Lay::kTile + rg * kRegionBytes, qmap, &bars[kQFullA + x],
                    rg * 64, it.kh * G, it.tokbase + it.t0 + x * BT);
    }
    ++k;
  }
  if (k >= 1)
    for (int x = 0; x < 2; ++x) (void)mbar_wait(&bars[kQFullA + x], (k - 1) & 1);
}

template <int D, bool F8>
__device__ void issue_mma(const TcPar& p, const SeqInfo* seq_tab, const int* ring, uint32_t sbase,
                          uint32_t tmem, uint64_t* bars, bool& ok) {
  using Lay = TcLayout<D>;
  constexpr uint32_t idesc_s = F8 ? tc::idesc_f16_f32(kTileRows, kKeys, false)
                                  : tc::idesc_bf16_f32(kTileRows, kKeys, false);
  constexpr uint32_t idesc_o = F8 ? tc::idesc_f16_f32(kTileRows, D, true)
                                  : tc::idesc_bf16_f32(kTileRows, D, true);
  // S_X = Q_X K(st)^T into TMEM columns 128 x
  auto qk = [&](int x, int st) {
    const uint64_t qd = tc::sdesc_sw128(sbase + Lay::kQ + x * Lay::kTile, 16, 1024);
    const uint64_t kd = tc::sdesc_sw128(sbase + Lay::kK + st * Lay::kTile, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint64_t off = (uint64_t)(((ks >> 2) * kRegionBytes + (ks & 3) * 32) >> 4);
      tc::mma_f16_ss(tmem + (uint32_t)x * 128, qd + off, kd + off, idesc_s, ks > 0);
    }
  };
  // O_X (+)= P_X V(sv), P_X (bf16) read from the first 64 columns of S_X
  auto pv = [&](int x, int sv, bool acc) {
    const uint64_t vd = tc::sdesc_sw128(sbase + Lay::kV + sv * Lay::kTile, kRegionBytes, 1024);
#pragma unroll
    for (int kk = 0; kk < kKeys / 16; ++kk)
      tc::mma_f16_ts(tmem + kTmemO + (uint32_t)x * 128, tmem + (uint32_t)x * 128 + kk * 8,
                     vd + (uint64_t)((kk * 2048) >> 4), idesc_o, (acc || kk > 0) ? 1u : 0u);
  };
  ItemWalk w;
  w.start(p, seq_tab, ring, bars, false, ok);
  int g = 0;  // KV tiles of this CTA so far
  int k = 0;  // items so far
  // S_X of an item's first KV tile: issued as soon as Q_X and the K tile have
  // landed and (from the second item on) the previous item's last P.V_X is
  // issued, so the softmax finds it ready after its epilogue.
  auto first_s = [&](int x, int kk, int gg, int nk_) -> bool {
    const int st = gg % kKStages;
    if (!mbar_wait(&bars[kQFullA + x], kk & 1)) return false;
    if (!mbar_wait(&bars[kKFull0 + st], (gg / kKStages) & 1)) return false;
    tc::fence_after();
    qk(x, st);
    tc::commit(&bars[kSFullA + x]);
    if (x == 1) tc::commit(&bars[kKEmpty0 + st]);
    if (nk_ == 1) tc::commit(&bars[kQEmptyA + x]);
    return true;
  };
  if (w.valid && ok && !(first_s(0, 0, 0, w.it.nk) && first_s(1, 0, 0, w.it.nk))) ok = false;
  while (w.valid && ok) {
    const int nk = w.it.nk;
    bool next_valid = false;
    int next_nk = 0;
    for (int j = 0; j < nk; ++j) {
      const int gj = g + j;
      const int sv = gj % kVStages;
      const bool last = j == nk - 1;
      const int st1 = (gj + 1) % kKStages;  // K stage of tile j + 1
      // ---- tile A: the V tile (and with bf16 the next K tile) is waited
      // for before P, off the softmax -> P.V -> S chain
      if (!F8 && !mbar_wait(&bars[kVFull0 + sv], (gj / kVStages) & 1)) { ok = false; break; }
      if (!F8 && !last && !mbar_wait(&bars[kKFull0 + st1], ((gj + 1) / kKStages) & 1)) { ok = false; break; }
      if (!mbar_wait(&bars[kPFullA], gj & 1)) { ok = false; break; }
      if (F8 && !mbar_wait(&bars[kVFull0 + sv], (gj / kVStages) & 1)) { ok = false; break; }
      tc::fence_after();
      pv(0, sv, j > 0);
      if (last) {
        tc::commit(&bars[kODoneA]);
        if (!F8) {
          w.next(p, ok);  // the next item, whose first S_A can go now
          next_valid = w.valid && ok;
          if (next_valid) {
            next_nk = w.it.nk;
            if (!first_s(0, k + 1, g + nk, next_nk)) { ok = false; break; }
          }
        }
      } else {
        // with E4M3 the K tile is converted on chip; its wait stays after P.V
        if (F8 && !mbar_wait(&bars[kKFull0 + st1], ((gj + 1) / kKStages) & 1)) { ok = false; break; }
        tc::fence_after();
        qk(0, st1);
        tc::commit(&bars[kSFullA]);
        if (j + 1 == nk - 1) tc::commit(&bars[kQEmptyA]);
      }
      // ---- tile B
      if (!mbar_wait(&bars[kPFullB], gj & 1)) { ok = false; break; }
      tc::fence_after();
      pv(1, sv, j > 0);
      tc::commit(&bars[kVEmpty0 + sv]);
      if (last) {
        tc::commit(&bars[kODoneB]);
        if (!F8 && next_valid && !first_s(1, k + 1, g + nk, next_nk)) { ok = false; break; }
      } else {
        qk(1, st1);
        tc::commit(&bars[kSFullB]);
        tc::commit(&bars[kKEmpty0 + st1]);
        if (j + 1 == nk - 1) tc::commit(&bars[kQEmptyB]);
      }
    }
    if (!ok) break;
    g += nk;
    ++k;
    if (F8) {  // converted K tiles land late: the next item's first S after its last P.V_B
      w.next(p, ok);
      if (w.valid && ok && !(first_s(0, k, g, w.it.nk) && first_s(1, k, g, w.it.nk))) ok = false;
    }
  }
  // Nothing may still be running on the tensor cores when TMEM is freed.
  tc::commit(&bars[kMmaDone]);
  (void)mbar_wait(&bars[kMmaDone], 0);
}

// Softmax and epilogue of Q tile x (0: A, 1: B) of every item.
template <int D, bool F8>
__device__ void softmax_tile(const TcPar& p, const SeqInfo* seq_tab, const int* ring, uint32_t sbase,
                             uint32_t tmem, uint64_t* bars, const CUtensorMap* omap, int x, bool& ok) {
  using Lay = TcLayout<D>;
  const int row = threadIdx.x & (kSoftmaxThreads - 1);  // = TMEM lane
  const int warp = threadIdx.x >> 5;
  const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  const uint32_t s_col = (uint32_t)x * 128, o_col = kTmemO + (uint32_t)x * 128;
  const int G = 1 << p.log2G, BT = 1 << p.log2BT;
  ItemWalk w;
  w.start(p, seq_tab, ring, bars, true, ok);
  int g = 0;  // KV tiles processed so far
  int k = 0;  // items processed so far
  while (w.valid && ok) {
    const Item it = w.it;
    w.next(p, ok);  // the next item's bounds load while this item runs
    const int tok = it.t0 + x * BT + (row >> p.log2G);
    const int h = it.kh * G + (row & (G - 1));
    const int lim = tok < it.n_b ? it.cached + tok : it.kv_total - 1;  // last key this row sees
    const int tile_min_lim = it.cached + it.t0 + x * BT;
    float m = kNegInf, l = 0.f;
    for (int j = 0; j < it.nk; ++j, ++g) {
      // S_X(j) complete; so is P.V_X(j - 1) (issued earlier by the same thread)
      if (!wait_warp(&bars[kSFullA + x], g & 1)) { ok = false; break; }
      tc::fence_after();
      const uint32_t s_tmem = lane_base + s_col;
      const int kv0 = j * kKeys;
      // keys past this row's causal limit count as -inf (select, so arbitrary
      // bits in keys past the sequence end cannot leak through)
      const bool masked = kv0 + kKeys - 1 > tile_min_lim;
      const int lim_rel = lim - kv0;  // columns c <= lim_rel are visible
      // pass 1: row max over the visible columns, 32 columns at a time
      float mx[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) mx[e] = kNegInf;
      // The limits of a warp's rows do not decrease with the lane: lane 0 has
      // the lowest, lane 31 the highest.  A 32-column chunk past the highest
      // holds no visible key (skipped, P = 0); one below the lowest needs no
      // selects.
      const int lim_lo = __shfl_sync(0xffffffffu, lim_rel, 0);
      const int lim_hi = __shfl_sync(0xffffffffu, lim_rel, 31);
      if (masked) {
#pragma unroll 1
        for (int c0 = 0; c0 < kKeys && c0 <= lim_hi; c0 += 32) {
          uint32_t sr[32];
          tc::ld_32x32b_x32(s_tmem + c0, sr);
          tc::wait_ld();
          if (c0 + 31 <= lim_lo) {
#pragma unroll
            for (int c = 0; c < 32; c += 2)
              mx[(c >> 1) & 3] = max3f(mx[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
          } else {
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const float v0 = c0 + c <= lim_rel ? __uint_as_float(sr[c]) : kNegInf;
              const float v1 = c0 + c + 1 <= lim_rel ? __uint_as_float(sr[c + 1]) : kNegInf;
              mx[(c >> 1) & 3] = max3f(mx[(c >> 1) & 3], v0, v1);
            }
          }
        }
      } else {
        // the whole row per TMEM wait
        uint32_t sr[kKeys];
#pragma unroll
        for (int c0 = 0; c0 < kKeys; c0 += 32) tc::ld_32x32b_x32(s_tmem + c0, sr + c0);
        tc::wait_ld();
#pragma unroll
        for (int c = 0; c < kKeys; c += 2)
          mx[(c >> 1) & 3] = max3f(mx[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
      }
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * p.scale_log2;
      // Reference max: moved only when the row max grows by more than 2^8
      // (P stays <= 256, exact after the final division by l).  The first
      // tile always sets it (key 0 is visible to every row).
      const bool grow = (j == 0) || (mt > m + kRescaleThreshold);
      const float m_new = grow ? fmaxf(m, mt) : m;
      const float alpha = fast_exp2(m - m_new);  // 0 on the first tile, 1 when not moving
      // pass 2: P = exp2(s * scale - m) as bf16 pairs into the first 64
      // columns of S_X, 32 keys at a time (P of keys [32q, 32q + 32) goes to
      // columns [16q, 16q + 16), which hold keys this pass has already read);
      // pairs of columns go through the packed fp32 unit, row sum in 4 pairs
      // of chains
      const uint64_t scale2 = f2_pack(p.scale_log2, p.scale_log2);
      const uint64_t negm2 = f2_pack(-m_new, -m_new);
      uint64_t acc2[4] = {0, 0, 0, 0};
      auto chunk = [&](int q, bool msk) {
        uint32_t sr[32];
        tc::ld_32x32b_x32(s_tmem + q * 32, sr);
        tc::wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float s0 = __uint_as_float(sr[2 * e]), s1 = __uint_as_float(sr[2 * e + 1]);
          if (msk) {
            s0 = q * 32 + 2 * e <= lim_rel ? s0 : kNegInf;
            s1 = q * 32 + 2 * e + 1 <= lim_rel ? s1 : kNegInf;
          }
          const uint64_t t = f2_fma(f2_pack(s0, s1), scale2, negm2);
          const float p0 = fast_exp2(f2_lo(t));  // exp2(-inf) = 0
          const float p1 = fast_exp2(f2_hi(t));
          acc2[e & 3] = f2_add(acc2[e & 3], f2_pack(p0, p1));
          pk[e] = F8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);  // P <= 256: exact range in f16
        }
        tc::st_32x32b_x16(s_tmem + q * 16, pk);
      };
      if (masked) {
#pragma unroll 1
        for (int q = 0; q < kKeys / 32; ++q) {
          if (q * 32 > lim_hi) {  // no visible key in this chunk for any row of the warp
            uint32_t z[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) z[e] = 0u;
            tc::st_32x32b_x16(s_tmem + q * 16, z);
          } else {
            chunk(q, q * 32 + 31 > lim_lo);
          }
        }
      } else {
#pragma unroll 2
        for (int q = 0; q < kKeys / 32; ++q) chunk(q, false);
      }
      const uint64_t a01 = f2_add(acc2[0], acc2[1]), a23 = f2_add(acc2[2], acc2[3]);
      const uint64_t a4 = f2_add(a01, a23);
      const float rs = f2_lo(a4) + f2_hi(a4);
      l = l * alpha + rs;
      m = m_new;
      if (j >= 1 && __any_sync(0xffffffffu, alpha < 1.f)) {  // warp-uniform
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tc::ld_32x32b_x32(lane_base + o_col + c * 32, o);
          tc::wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tc::st_32x32b_x32(lane_base + o_col + c * 32, o);
        }
      }
      tc::wait_st();
      if (x == 0 && kv0 + kKeys > it.kv_total) {
        // keys past the end of the sequence hold arbitrary bits: zero those V
        // rows (before P.V_A, which the tile's P.V_B follows)
        if (!wait_warp(&bars[kVFull0 + g % kVStages], (g / kVStages) & 1)) { ok = false; break; }
        if (kv0 + row >= it.kv_total) {
          const uint32_t v_addr = sbase + Lay::kV + (g % kVStages) * Lay::kTile;
#pragma unroll
          for (int rg = 0; rg < Lay::kRegions; ++rg)
#pragma unroll
            for (int c = 0; c < 8; ++c) sts128(v_addr + rg * kRegionBytes + sw128(row, c), make_uint4(0, 0, 0, 0));
        }
        tc::fence_proxy_async();
      }
      tc::fence_before();
      mbar_arrive(&bars[kPFullA + x]);
    }
    if (!ok) break;
    // ---- item epilogue: O / l -> bf16 rows of out (the item's last P.V_X done)
    if (!wait_warp(&bars[kODoneA + x], k & 1)) { ok = false; break; }
    tc::fence_after();
    {
      const float inv_l = F8 ? p.v_scale / l : 1.f / l;
      // This warp's 32 rows are 32/G whole tokens.  When all of them belong to
      // the sequence they leave through this warp's staging slot (128-byte
      // swizzled, the layout of a 64 d x G heads x 32/G tokens box) by TMA
      // stores, 64 columns at a time; otherwise row by row (rows inside the
      // sequence only).
      const int tpw = 32 >> p.log2G;
      const int wtok0 = it.t0 + x * BT + (warp & 3) * tpw;
      const bool full = wtok0 + tpw <= it.n_b;  // warp-uniform
      const uint32_t slot = sbase + Lay::kStg + warp * 4096;
      const int lane = threadIdx.x & 31;
      const bool store = tok < it.n_b;
      uint16_t* dst = p.out + (int64_t)(it.tokbase + (store ? tok : 0)) * p.Hq * D + (int64_t)h * D;
#pragma unroll 1
      for (int half = 0; half < D / 64; ++half) {
        uint32_t o[64];
        tc::ld_32x32b_x32(lane_base + o_col + half * 64, o);
        tc::ld_32x32b_x32(lane_base + o_col + half * 64 + 32, o + 32);
        tc::wait_ld();
        if (full) {
          // the slot's previous contents have been read by their TMA store
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(o[8 * c + 0]) * inv_l, __uint_as_float(o[8 * c + 1]) * inv_l);
            v.y = pack_bf16(__uint_as_float(o[8 * c + 2]) * inv_l, __uint_as_float(o[8 * c + 3]) * inv_l);
            v.z = pack_bf16(__uint_as_float(o[8 * c + 4]) * inv_l, __uint_as_float(o[8 * c + 5]) * inv_l);
            v.w = pack_bf16(__uint_as_float(o[8 * c + 6]) * inv_l, __uint_as_float(o[8 * c + 7]) * inv_l);
            sts128(slot + sw128(lane, c), v);
          }
          tc::fence_proxy_async();  // the rows are visible to the TMA engine
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(omap, slot, half * 64, it.kh * G, it.tokbase + wtok0);
            bulk_commit_group();
          }
        } else if (store) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(o[8 * c + 0]) * inv_l, __uint_as_float(o[8 * c + 1]) * inv_l);
            v.y = pack_bf16(__uint_as_float(o[8 * c + 2]) * inv_l, __uint_as_float(o[8 * c + 3]) * inv_l);
            v.z = pack_bf16(__uint_as_float(o[8 * c + 4]) * inv_l, __uint_as_float(o[8 * c + 5]) * inv_l);
            v.w = pack_bf16(__uint_as_float(o[8 * c + 6]) * inv_l, __uint_as_float(o[8 * c + 7]) * inv_l);
            *reinterpret_cast<uint4*>(dst + half * 64 + c * 8) = v;
          }
        }
      }
      // the O reads above are complete before the next item's first P.V_X overwrites O_X
      tc::fence_before();
    }
    ++k;
  }
  if ((threadIdx.x & 31) == 0) bulk_wait_all();  // every output store has completed
}

template <int D, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap omap, const TcPar p) {
  using Lay = TcLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kTmemSlot);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Sequences longer than the host bound are left unwritten: flag them once.
  if (blockIdx.x == 0)
    for (int b = threadIdx.x; b < p.B; b += kThreads)
      if (p.cu_seqlens[b + 1] - p.cu_seqlens[b] > p.max_seqlen) set_status(p.status, ATTN_STATUS_BOUNDS);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kQFullA + s], 1);
      mbar_init(&bars[kQEmptyA + s], 1);
      mbar_init(&bars[kSFullA + s], 1);
      mbar_init(&bars[kPFullA + s], kSoftmaxThreads);
      mbar_init(&bars[kODoneA + s], 1);
    }
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&bars[kKFull0 + s], 1);
      mbar_init(&bars[kKEmpty0 + s], 1);
      mbar_init(&bars[kKLand0 + s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bars[kVFull0 + s], 1);
      mbar_init(&bars[kVEmpty0 + s], 1);
      mbar_init(&bars[kVLand0 + s], 1);
    }
    mbar_init(&bars[kMmaDone], 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&bars[kItemFull0 + s], 1);
      mbar_init(&bars[kItemFree0 + s], kRingReaders);
    }
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tc::alloc(tmem_slot, kTmemCols);
    tc::relinquish();
  }
  if (p.B <= kMaxSeqSmem && (int)threadIdx.x < p.B)
    reinterpret_cast<SeqInfo*>(smem + Lay::kSeq)[threadIdx.x] = seq_info(p, threadIdx.x);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  const SeqInfo* seq_tab = p.B <= kMaxSeqSmem ? reinterpret_cast<const SeqInfo*>(smem + Lay::kSeq) : nullptr;
  int* ring = reinterpret_cast<int*>(smem + Lay::kRingOff);
  bool ok = true;
  // Everything above reads only what the caller wrote; the prepared Q and the
  // cache entries come from the kernel before this one.
  grid_dependency_wait();

  if (warp < 8) {
    softmax_tile<D, F8>(p, seq_tab, ring, sbase, tmem, bars, &omap, warp >> 2, ok);
  } else if (F8 && warp == kKWarp) {  // the whole warp converts the tiles
    produce_kv_f8<D>(p, seq_tab, ring, &kmap, smem, bars, Lay::kK, kKFull0, kKEmpty0, kKLand0, kKStages, ok);
  } else if (F8 && warp == kVWarp) {
    produce_kv_f8<D>(p, seq_tab, ring, &vmap, smem, bars, Lay::kV, kVFull0, kVEmpty0, kVLand0, kVStages, ok);
  } else {
    if (lane == 0) {
      if (warp == kKWarp)
        produce_kv<D>(p, seq_tab, ring, &kmap, smem, bars, Lay::kK, kKFull0, kKEmpty0, kKStages, ok);
      else if (warp == kVWarp)
        produce_kv<D>(p, seq_tab, ring, &vmap, smem, bars, Lay::kV, kVFull0, kVEmpty0, kVStages, ok);
      else if (warp == kQWarp)
        produce_q<D>(p, seq_tab, ring, &qmap, smem, bars, ok);
      else
        issue_mma<D, F8>(p, seq_tab, ring, sbase, tmem, bars, ok);
    }
  }
  if (!ok) set_status(p.status, ATTN_STATUS_TIMEOUT);

  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == kMmaWarp) tc::dealloc(tmem, kTmemCols);
  // The last CTA to finish leaves the counters at zero for the next launch
  // (every CTA has stopped claiming by now).
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.work + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(p.work, 0);
      atomicExch(p.work + 1, 0);
    }
  }
}

template <int D, bool F8>
int launch_prefill_tc_t(const PrefillArgs& a, cudaStream_t stream) {
  using Lay = TcLayout<D>;
  const int Hq = a.cfg.num_q_heads, Hkv = a.cfg.num_kv_heads;
  const int G = Hq / Hkv;
  const int log2G = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
  const int BT = kTileRows / G;
  const KvIndex kvi = kv_index(a.kv);
  const bool half_boxes = kvi.page_table != nullptr && kvi.log2_page < 7;
  CacheMaps maps;
  if (make_cache_maps(a.kv, Hkv, D, half_boxes ? 64 : kKeys, &maps) != 0) return ATTN_ELAUNCH;
  CUtensorMap qmap;  // prepared Q viewed as [N, Hq, D]
  if (make_qkv_map(a.q, a.N, Hq, D, G, BT, &qmap) != 0) return ATTN_ELAUNCH;
  CUtensorMap omap;  // out viewed as [N, Hq, D]; one softmax warp's 32 rows per box
  if (make_qkv_map(a.out, a.N, Hq, D, G, 32 / G, &omap) != 0) return ATTN_ELAUNCH;
  TcPar p;
  p.cu_seqlens = a.cu_seqlens;
  p.kv = kvi;
  p.half_boxes = half_boxes ? 1 : 0;
  p.status = a.status;
  p.work = a.work;
  p.out = static_cast<uint16_t*>(a.out);
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)D) * (F8 ? a.kv.k_scale : 1.0f);
  p.v_scale = F8 ? a.kv.v_scale : 1.0f;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.log2G = log2G;
  p.log2BT = 7 - log2G;
  p.N = a.N;
  p.B = a.B;
  p.max_seqlen = a.max_seqlen;
  const int64_t rounds = ((int64_t)a.max_seqlen + (2 * BT) - 1) / (2 * BT);
  const int64_t nv = rounds * a.B * Hkv;
  if (nv > (int64_t(1) << 30)) return ATTN_EINVAL;
  p.num_vitems = (int)nv;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ATTN_ELAUNCH;
  if (cudaFuncSetAttribute(prefill_tc_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Lay::kSmemBytes) != cudaSuccess)
    return ATTN_ELAUNCH;
  const int grid = (int)std::min<int64_t>(sms, nv);
  return launch_dependent(prefill_tc_kernel<D, F8>, dim3(grid), dim3(kThreads), Lay::kSmemBytes, stream, qmap,
                          maps.k, maps.v, omap, p) == cudaSuccess
             ? ATTN_OK
             : ATTN_ELAUNCH;
}

}  // namespace

int launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  if (a.B <= 0 || a.N <= 0 || a.max_seqlen <= 0) return ATTN_OK;
  const bool f8 = a.kv.kv_dtype == ATTN_KV_E4M3;
  if (a.cfg.head_dim == 128)
    return f8 ? launch_prefill_tc_t<128, true>(a, stream) : launch_prefill_tc_t<128, false>(a, stream);
  return f8 ? launch_prefill_tc_t<64, true>(a, stream) : launch_prefill_tc_t<64, false>(a, stream);
}

}  // namespace gb300
