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
// KV head kh, 128-row query tile).  The tile's rows
// are 128/G tokens x G heads of the group, so every K/V tile loaded serves the
// whole GQA group.  Items are numbered sequence by sequence, heaviest tile of
// a sequence first; CTA c takes items c, c + gridDim.x, ...  Roles (224 threads):
//   warps 0-3  softmax: thread r owns row r = TMEM lane r.  Per KV tile: read
//              S from TMEM, mask, online softmax in fp32 (exp2 domain), write P
//              (bf16) to TMEM, rescale O in TMEM when the reference max moves;
//              per item: O / l -> bf16 rows of out.
//   warp 4     TMA producer (one thread): Q (two buffers: the current item
//              and the next) and K (3-stage ring of 128-key tiles running
//              across items).
//   warp 6     TMA producer (one thread): V (2-stage ring).  A warp of its
//              own, so that waiting for a free V stage never holds up the K
//              loads (a waiting thread may be suspended, and diverged lanes
//              of one warp do not run independently of that).
//   warp 5     MMA issuer (one thread) and TMEM owner: S = Q K^T into one of
//              three TMEM buffers and O += P V.  It keeps the S of up to two
//              tiles ahead queued (as their K and Q arrive) and issues P.V of
//              tile g as soon as its P is in TMEM (also across item boundaries).
// TMEM: three S buffers (fp32) in columns [0,384), O in [384, 384+D).  P
// (bf16 pairs, A operand of P.V read from TMEM) overwrites the first 64
// columns of its tile's S buffer once the softmax holds S in registers.
#include "kernels.cuh"
#include "tcgen05.cuh"

namespace gb300 {

namespace {

constexpr int kRows = 128;  // query rows per item (MMA M)
constexpr int kKeys = 128;  // keys per KV tile (MMA N of Q K^T)
constexpr int kThreads = 224;
constexpr int kSoftmaxThreads = 128;
constexpr int kProducerWarp = 4;  // Q and K loads
constexpr int kMmaWarp = 5;
constexpr int kVWarp = 6;         // V loads
constexpr int kQBufs = 2;  // Q tiles in flight: the current item and the next
constexpr int kSBufs = 3;  // S buffers in TMEM = K stages in shared memory
#ifndef PREFILL_LOOKAHEAD
#define PREFILL_LOOKAHEAD 1
#endif
// S = Q K^T tiles issued ahead of the P.V that is waiting for its P.  The
// tensor pipe runs in issue order and tcgen05.mma issue stalls while the pipe
// is full, so every S queued ahead delays that P.V (and the softmax waiting on
// it) by one Q K^T.
constexpr int kLookahead = PREFILL_LOOKAHEAD;
static_assert(kLookahead >= 1 && kLookahead <= kSBufs - 1, "lookahead");

constexpr int kMaxSeqSmem = 32;  // sequences whose facts are cached in shared memory
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 384;  // O columns; [0, 384) hold three S buffers
constexpr int kRegionBytes = 128 * 128;   // 128 rows x 128 bytes (64 bf16)
constexpr float kRescaleThreshold = 8.f;  // log2 units: move the reference max past 256x growth

struct TcPar {
  const int32_t* cu_seqlens;
  const int64_t* slot_base;
  const int32_t* cache_lens;
  const int32_t* slot_capacity;
  int64_t num_slots;
  int32_t* status;
  uint16_t* out;
  float scale_log2;  // log2(e) / sqrt(D)
  int32_t Hq, Hkv, log2G, log2BT, N, B, max_seqlen;
  int32_t num_vitems;  // ((N >> log2BT) + B) * Hkv: size of the item numbering
};

template <int D>
struct TcLayout {
  static constexpr int kRegions = D / 64;
  static constexpr int kTile = kRegions * kRegionBytes;  // Q, K or V tile: 128 rows x D
  static constexpr int kQ = 0;                // kQBufs buffers
  static constexpr int kK = kQ + kQBufs * kTile;  // kSBufs stages
  static constexpr int kV = kK + kSBufs * kTile;  // 2 stages
  static constexpr int kBar = kV + 2 * kTile;
  static constexpr int kNumBars = 24;
  static constexpr int kSeq = kBar + kNumBars * 8;  // SeqInfo[kMaxSeqSmem]
  static constexpr int kTmemSlot = kSeq + kMaxSeqSmem * 24;
  // + alignment slack; at least 116 KB so that one CTA runs per SM (each CTA
  // allocates all 512 TMEM columns).
  static constexpr int kSmemRaw = kTmemSlot + 16 + 1024;
  static constexpr int kSmemBytes = kSmemRaw > 116 * 1024 ? kSmemRaw : 116 * 1024;
};

enum Bar {
  kQFull0 = 0, kQEmpty0 = kQFull0 + kQBufs,
  kKFull0 = kQEmpty0 + kQBufs, kVFull0 = kKFull0 + kSBufs, kVFull1,
  // kSFull + b: S of a tile in S buffer b (K stage b) is complete, which also
  // frees that K stage; kPvDone + st: P.V of a tile using V stage st is
  // complete (O updated, V stage st free).  Each advances one phase per use of
  // its stage, so no waiter can fall two phases behind.
  kSFull0, kPvDone0 = kSFull0 + kSBufs, kPvDone1, kPFull, kMmaDone
};

// ---------------------------------------------------------------- work items
// Item numbering without a table: sequence b owns the "virtual tiles"
// [vstart(b), vstart(b) + ntiles(b)) with vstart(b) = cu_seqlens[b] / BT + b
// (these ranges never overlap; each sequence leaves at most one slot empty).
// Virtual item i = (virtual tile i / Hkv, KV head i % Hkv).
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
  const ReqInfo r = load_request(p.slot_base + b, p.cache_lens + b, p.slot_capacity + b,
                                 p.num_slots, q.n_b);
  q.slot0 = r.slot0;
  q.cached = r.cached;
  // sequences with no tokens, outside [0, N), longer than the host bound or
  // with a region too small are skipped (flagged by the prologue / below)
  q.usable = q.n_b > 0 && q.tokbase >= 0 && q.tokbase + q.n_b <= p.N && q.n_b <= p.max_seqlen &&
             r.valid;
  return q;
}

__device__ __forceinline__ bool item_at(const TcPar& p, const SeqInfo* tab, int vi, Item& it) {
  const int v = vi / p.Hkv;
  it.kh = vi - v * p.Hkv;
  int lo = 0, hi = p.B;  // largest b with vstart(b) <= v
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    const int cu = tab ? tab[mid].tokbase : p.cu_seqlens[mid];
    if ((cu >> p.log2BT) + mid <= v) lo = mid; else hi = mid;
  }
  const int b = lo;
  const SeqInfo q = tab ? tab[b] : seq_info(p, b);
  if (!q.usable) return false;
  const int BT = 1 << p.log2BT;
  const int ntile = (q.n_b + BT - 1) >> p.log2BT;
  const int tfe = v - ((q.tokbase >> p.log2BT) + b);  // tile index counted from the end
  if (tfe < 0 || tfe >= ntile) return false;
  it.b = b;
  it.t0 = (ntile - 1 - tfe) * BT;  // heaviest tile first
  it.n_b = q.n_b;
  it.tokbase = q.tokbase;
  it.cached = q.cached;
  it.slot0 = q.slot0;
  it.kv_total = q.cached + q.n_b;
  it.nk = (q.cached + min(it.t0 + BT, q.n_b) + kKeys - 1) / kKeys;
  return true;
}

// Walks this CTA's items and their KV tiles in order.
struct TileWalk {
  const SeqInfo* tab;  // shared-memory sequence table or nullptr
  int vi;     // current virtual item
  int k;      // ordinal of the current item within this CTA
  int j;      // KV tile within the item
  bool valid;
  Item it;

  __device__ __forceinline__ void start(const TcPar& p, const SeqInfo* table) {
    tab = table;
    vi = blockIdx.x - (int)gridDim.x;
    k = -1;
    next_item(p);
  }
  __device__ __forceinline__ void next_item(const TcPar& p) {
    j = 0;
    for (vi += gridDim.x; vi < p.num_vitems; vi += gridDim.x)
      if (item_at(p, tab, vi, it)) {
        ++k;
        valid = true;
        return;
      }
    valid = false;
  }
  __device__ __forceinline__ void next_tile(const TcPar& p) {
    if (++j >= it.nk) next_item(p);
  }
};

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity) {
  const bool w = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, w);
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
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = 1 << p.log2G;

  // Sequences longer than the host bound are left unwritten: flag them once.
  if (blockIdx.x == 0)
    for (int b = threadIdx.x; b < p.B; b += kThreads)
      if (p.cu_seqlens[b + 1] - p.cu_seqlens[b] > p.max_seqlen) set_status(p.status, ATTN_STATUS_BOUNDS);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQBufs; ++s) {
      mbar_init(&bars[kQFull0 + s], 1);
      mbar_init(&bars[kQEmpty0 + s], 1);
    }
    for (int s = 0; s < kSBufs; ++s) {
      mbar_init(&bars[kKFull0 + s], 1);
      mbar_init(&bars[kSFull0 + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kVFull0 + s], 1);
      mbar_init(&bars[kPvDone0 + s], 1);
    }
    mbar_init(&bars[kPFull], kSoftmaxThreads);
    mbar_init(&bars[kMmaDone], 1);
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
  bool ok = true;

  if (warp == kProducerWarp || warp == kVWarp) {
    // ================================================================ TMA producers
    if (lane == 0) {
      const bool kstream = warp == kProducerWarp;
      if (kstream) {
        prefetch_tmap(&qmap);
        prefetch_tmap(&kmap);
      } else {
        prefetch_tmap(&vmap);
      }
      TileWalk w, qw;  // K or V tiles; items whose Q tile is loaded next
      w.start(p, seq_tab);
      qw.start(p, seq_tab);
      int g = 0;  // tiles issued so far
      int q_issued = 0, issued = 0;
      // Q tile of item qw.k into buffer qw.k % kQBufs (free once the last
      // Q K^T of item qw.k - kQBufs has completed)
      auto q_free = [&]() -> bool {
        return qw.k < kQBufs || mbar_test_wait(&bars[kQEmpty0 + qw.k % kQBufs], (qw.k / kQBufs - 1) & 1);
      };
      auto issue_q = [&]() -> bool {
        const int qs = qw.k % kQBufs;
        if (qw.k >= kQBufs && !mbar_wait(&bars[kQEmpty0 + qs], (qw.k / kQBufs - 1) & 1)) return false;
        mbar_arrive_expect_tx(&bars[kQFull0 + qs], Lay::kTile);
#pragma unroll
        for (int rg = 0; rg < Lay::kRegions; ++rg)
          tma_load_3d(smem + Lay::kQ + qs * Lay::kTile + rg * kRegionBytes, &qmap,
                      &bars[kQFull0 + qs], rg * 64, qw.it.kh * G, qw.it.tokbase + qw.it.t0);
        q_issued = qw.k + 1;
        qw.next_item(p);
        return true;
      };
      const int full0 = kstream ? kKFull0 : kVFull0, empty0 = kstream ? kSFull0 : kPvDone0;
      const int nst = kstream ? kSBufs : 2;  // ring stages
      const int base = kstream ? Lay::kK : Lay::kV;
      const CUtensorMap* map = kstream ? &kmap : &vmap;
      while (w.valid && ok) {
        if (kstream) {
          while (qw.valid && qw.k <= w.k && ok) ok = issue_q();  // this item's Q
          if (!ok) break;
        }
        const int st = g % nst;
        if (g >= nst && !mbar_wait(&bars[empty0 + st], (g / nst - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(&bars[full0 + st], Lay::kTile);
#pragma unroll
        for (int rg = 0; rg < Lay::kRegions; ++rg)
          tma_load_3d(smem + base + st * Lay::kTile + rg * kRegionBytes, map, &bars[full0 + st],
                      rg * 64, w.it.kh, (int)(w.it.slot0 + w.j * kKeys));
        issued = g + 1;
        // prefetch the next two items' Q tiles, without waiting for a buffer
        while (kstream && ok && qw.valid && qw.k <= w.k + kQBufs - 1 && q_free()) ok = issue_q();
        if (!ok) break;
        ++g;
        w.next_tile(p);
      }
      // Every load issued has landed before the CTA may exit (immediate on
      // the normal path, where the consumers already waited for them).
      for (int k = max(0, q_issued - kQBufs); k < q_issued; ++k)
        (void)mbar_wait(&bars[kQFull0 + k % kQBufs], (k / kQBufs) & 1);
      for (int t = max(0, issued - nst); t < issued; ++t)
        (void)mbar_wait(&bars[full0 + t % nst], (t / nst) & 1);
      if (!ok) set_status(p.status, ATTN_STATUS_TIMEOUT);
    }
  } else if (warp == kMmaWarp) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kRows, kKeys, false);
      constexpr uint32_t idesc_o = tc::idesc_bf16_f32(kRows, D, true);
      const uint32_t o_tmem = tmem + kTmemO;
      TileWalk qk, pv;
      qk.start(p, seq_tab);
      pv.start(p, seq_tab);
      int gq = 0, gp = 0;  // next tile for S = Q K^T, next tile for P.V
      // S of tile gq goes to S buffer gq % 3, K stage gq % 3.  It may be issued
      // once P.V of tile gq - 3 (which reads its P from that buffer) has been
      // issued: tensor-core operations run in issue order.  With block ==
      // false issue_qk returns false, issuing nothing, when the tile's K (or,
      // on an item's first tile, its Q) is not in shared memory yet.
      auto issue_qk = [&](bool block) -> bool {
        const int sb = gq % kSBufs, qs = qk.k % kQBufs;
        if (qk.j == 0) {
          uint64_t* qb = &bars[kQFull0 + qs];
          const uint32_t qpar = (qk.k / kQBufs) & 1;
          if (block ? !mbar_wait(qb, qpar) : !mbar_test_wait(qb, qpar)) {
            if (block) ok = false;
            return false;
          }
        }
        uint64_t* kb = &bars[kKFull0 + sb];
        const uint32_t kpar = (gq / kSBufs) & 1;
        if (block ? !mbar_wait(kb, kpar) : !mbar_test_wait(kb, kpar)) {
          if (block) ok = false;
          return false;
        }
        tc::fence_after();
        const uint64_t qd = tc::sdesc_sw128(sbase + Lay::kQ + qs * Lay::kTile, 16, 1024);
        const uint64_t kd = tc::sdesc_sw128(sbase + Lay::kK + sb * Lay::kTile, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t off = (uint64_t)(((ks >> 2) * kRegionBytes + (ks & 3) * 32) >> 4);
          tc::mma_f16_ss(tmem + (uint32_t)sb * 128, qd + off, kd + off, idesc_s, ks > 0);
        }
        tc::commit(&bars[kSFull0 + sb]);  // S ready, K stage sb free
        if (qk.j == qk.it.nk - 1) tc::commit(&bars[kQEmpty0 + qs]);  // last use of this Q tile
        ++gq;
        qk.next_tile(p);
        return true;
      };
      while (pv.valid && ok) {
        // the S that P.V of tile gp consumes must be under way (blocking) ...
        while (ok && qk.valid && gq <= gp) issue_qk(true);
        if (!ok) break;
        // ... and S of up to kLookahead more tiles, as far as they are loaded
        while (ok && qk.valid && gq <= gp + kLookahead && issue_qk(false)) {
        }
        if (!mbar_wait(&bars[kPFull], gp & 1)) { ok = false; break; }
        const int st = gp & 1;
        if (!mbar_wait(&bars[kVFull0 + st], (gp >> 1) & 1)) { ok = false; break; }
        tc::fence_after();
        const uint32_t p_tmem = tmem + (uint32_t)(gp % kSBufs) * 128;  // P in its S buffer
        const uint64_t vd = tc::sdesc_sw128(sbase + Lay::kV + st * Lay::kTile, kRegionBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          tc::mma_f16_ts(o_tmem, p_tmem + kk * 8, vd + (uint64_t)((kk * 2048) >> 4), idesc_o,
                         (pv.j > 0 || kk > 0) ? 1u : 0u);
        tc::commit(&bars[kPvDone0 + st]);  // O updated, V stage st free
        ++gp;
        pv.next_tile(p);
      }
      // Nothing may still be running on the tensor cores when TMEM is freed.
      tc::commit(&bars[kMmaDone]);
      (void)mbar_wait(&bars[kMmaDone], 0);
      if (!ok) set_status(p.status, ATTN_STATUS_TIMEOUT);
    }
  } else {
    // ================================================================ softmax warpgroup
    const int row = threadIdx.x;  // 0..127 = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    TileWalk w;
    w.start(p, seq_tab);
    int g = 0;  // KV tiles processed so far
    while (w.valid && ok) {
      const Item it = w.it;
      w.next_item(p);  // the next item's bounds load while this item runs
      const int tl = row >> p.log2G;
      const int tok = it.t0 + tl;
      const int h = it.kh * G + (row & (G - 1));
      const int lim = tok < it.n_b ? it.cached + tok : it.kv_total - 1;  // last key this row sees
      const int cta_min_lim = it.cached + it.t0;
      float m = kNegInf, l = 0.f;
      for (int j = 0; j < it.nk; ++j, ++g) {
        if (!wait_warp(&bars[kSFull0 + g % kSBufs], (g / kSBufs) & 1)) { ok = false; break; }
        tc::fence_after();
        const uint32_t s_tmem = lane_base + (uint32_t)(g % kSBufs) * 128;
        const int kv0 = j * kKeys;
        // keys past this row's causal limit count as -inf (select, so arbitrary
        // bits in keys past the sequence end cannot leak through)
        const bool masked = kv0 + kKeys - 1 > cta_min_lim;
        const int lim_rel = lim - kv0;  // columns c <= lim_rel are visible
        uint32_t sr[kKeys];
#pragma unroll
        for (int c = 0; c < kKeys / 32; ++c) tc::ld_32x32b_x32(s_tmem + c * 32, sr + c * 32);
        tc::wait_ld();
        if (masked) {
#pragma unroll
          for (int c = 0; c < kKeys; ++c) sr[c] = c <= lim_rel ? sr[c] : __float_as_uint(kNegInf);
        }
        // row max, 8 independent chains (instruction-level parallelism)
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = __uint_as_float(sr[e]);
#pragma unroll
        for (int c = 8; c < kKeys; ++c) mx[c & 7] = fmaxf(mx[c & 7], __uint_as_float(sr[c]));
        const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * p.scale_log2;
        // Reference max: moved only when the row max grows by more than 2^8
        // (P stays <= 256, exact after the final division by l).  The first
        // tile always sets it (key 0 is visible to every row).
        const bool grow = (j == 0) || (mt > m + kRescaleThreshold);
        const float m_new = grow ? fmaxf(m, mt) : m;
        const float alpha = fast_exp2(m - m_new);  // 0 on the first tile, 1 when not moving
        const float neg_m = -m_new;
        // P = exp2(s * scale - m) as bf16 pairs into the first 64 columns of
        // this tile's S buffer (S is in registers now), row sum in 8 chains
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        const uint32_t p_tmem = s_tmem;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int c = h * 64 + 2 * e;
            const float p0 = fast_exp2(fmaf(__uint_as_float(sr[c]), p.scale_log2, neg_m));  // exp2(-inf) = 0
            const float p1 = fast_exp2(fmaf(__uint_as_float(sr[c + 1]), p.scale_log2, neg_m));
            acc[(2 * e) & 7] += p0;
            acc[(2 * e + 1) & 7] += p1;
            pk[e] = pack_bf16(p0, p1);
          }
          tc::st_32x32b_x32(p_tmem + h * 32, pk);
        }
        const float rs = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        l = l * alpha + rs;
        m = m_new;
        if (j >= 1) {
          // O may only be rescaled once the previous tile's P.V is complete
          if (!wait_warp(&bars[kPvDone0 + ((g - 1) & 1)], ((g - 1) >> 1) & 1)) { ok = false; break; }
          tc::fence_after();
          if (__any_sync(0xffffffffu, alpha < 1.f)) {  // warp-uniform
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tc::ld_32x32b_x32(lane_base + kTmemO + c * 32, o);
              tc::wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tc::st_32x32b_x32(lane_base + kTmemO + c * 32, o);
            }
          }
        }
        tc::wait_st();
        if (kv0 + kKeys > it.kv_total) {
          // keys past the end of the sequence hold arbitrary bits: zero those V rows
          if (!wait_warp(&bars[kVFull0 + (g & 1)], (g >> 1) & 1)) { ok = false; break; }
          if (kv0 + row >= it.kv_total) {
            const uint32_t v_addr = sbase + Lay::kV + (g & 1) * Lay::kTile;
#pragma unroll
            for (int rg = 0; rg < Lay::kRegions; ++rg)
#pragma unroll
              for (int c = 0; c < 8; ++c) sts128(v_addr + rg * kRegionBytes + sw128(row, c), make_uint4(0, 0, 0, 0));
          }
          tc::fence_proxy_async();
        }
        tc::fence_before();
        mbar_arrive(&bars[kPFull]);
      }
      if (!ok) break;
      // ---- item epilogue: O / l -> bf16 rows of out (P.V of its last tile done)
      if (!wait_warp(&bars[kPvDone0 + ((g - 1) & 1)], ((g - 1) >> 1) & 1)) { ok = false; break; }
      tc::fence_after();
      {
        const float inv_l = 1.f / l;
        const bool store = tok < it.n_b;
        uint16_t* dst = p.out + (int64_t)(it.tokbase + (store ? tok : 0)) * p.Hq * D + (int64_t)h * D;
        // 32 columns at a time in a rolled loop: this code runs once per item,
        // so it is kept short (it competes for instruction cache with the tile loop)
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tc::ld_32x32b_x32(lane_base + kTmemO + c * 32, o);
          tc::wait_ld();
          if (store) {
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
        }
        // the O reads above are complete before the next item's first P.V overwrites O
        tc::fence_before();
      }
    }
    if (!ok) set_status(p.status, ATTN_STATUS_TIMEOUT);
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
  const int log2G = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
  const int BT = kRows / G;
  CacheMaps maps;
  if (make_cache_maps(a.kv, Hkv, D, kKeys, &maps) != 0) return ATTN_ELAUNCH;
  CUtensorMap qmap;  // prepared Q viewed as [N, Hq, D]
  if (make_qkv_map(a.q, a.N, Hq, D, G, BT, &qmap) != 0) return ATTN_ELAUNCH;
  TcPar p;
  p.cu_seqlens = a.cu_seqlens;
  p.slot_base = a.kv.slot_base;
  p.cache_lens = a.kv.cache_lens;
  p.slot_capacity = a.kv.slot_capacity;
  p.num_slots = a.kv.num_slots;
  p.status = a.status;
  p.out = static_cast<uint16_t*>(a.out);
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.log2G = log2G;
  p.log2BT = 7 - log2G;
  p.N = a.N;
  p.B = a.B;
  p.max_seqlen = a.max_seqlen;
  const int64_t nv = ((int64_t)(a.N >> p.log2BT) + a.B) * Hkv;
  if (nv > (int64_t(1) << 30)) return ATTN_EINVAL;
  p.num_vitems = (int)nv;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ATTN_ELAUNCH;
  if (cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Lay::kSmemBytes) != cudaSuccess)
    return ATTN_ELAUNCH;
  const int grid = (int)std::min<int64_t>(sms, nv);
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
