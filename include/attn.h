/*
 * attn.h -- C ABI of the GB300 (sm_103a) causal grouped-query attention step.
 *
 * The step is the attention part of one decoder layer of a Qwen3-style model,
 * as the zero-to-sglang Ch.3 code walkthrough (section 3.3, "QKV, RoPE, and
 * causal attention": AttentionLayer.forward) and the transformer-basics page
 * ("Attention calculation: part 1", "Prefill vs Decode") describe it:
 *
 *   qkv [N, (Hq + 2*Hkv) * D]  --split-->  Q [N, Hq, D], K [N, Hkv, D], V [N, Hkv, D]
 *   Q, K  <- w * x / sqrt(mean(x^2) + eps)          (per head, over D)
 *   Q, K  <- RoPE at each token's position           (V is not rotated)
 *   cache <- append K, V                             (KV cache update)
 *   out[t, h*D:(h+1)*D] = softmax(q . K^T / sqrt(D)) V over the keys at
 *       positions 0 .. p(t) of the same request, KV head h / (Hq / Hkv)
 *
 * Conventions used by every entry point:
 *
 * Data types.  qkv, the norm weights, the caches and the output are bf16
 *   (IEEE bfloat16 bits, round-to-nearest-even on every store).  All
 *   arithmetic is fp32 (norm, rotation, scores, softmax, accumulation); Q and
 *   the softmax probabilities enter the tensor-core products rounded to bf16.
 * Positions.  Request b has cache_lens[b] = c_b entries already cached and
 *   n_b new tokens; new token j sits at position c_b + j and is written to
 *   slot slot_base[b] + c_b + j.  The query at position p attends to the keys
 *   at positions 0 .. p (its own key included).
 * RMSNorm.  y = w * x / sqrt(mean(x^2) + eps) over each head's D values, one
 *   weight vector [D] for all Q heads and one for all K heads.
 * RoPE.  Rotate-half pairing: for i in [0, D/2), the pair (x_i, x_{i+D/2}) is
 *   rotated by the angle p * theta^(-2i/D):
 *   (x_i, x_{i+D/2}) <- (x_i cos a - x_{i+D/2} sin a, x_{i+D/2} cos a + x_i sin a).
 *   The zero-to-sglang chapters name RoPE and cite RoFormer without printing
 *   a formula; this is the RoFormer rotation with the rotate-half pairing of
 *   the Qwen3 model family.  The norm comes first (q_norm(q_proj(x).view)).
 * Memory.  Every pointer argument is a device pointer unless stated
 *   otherwise.  The library allocates nothing, keeps no state between calls
 *   and never synchronises the stream except in attn_get_status.  All
 *   buffers, the stream and the workspace belong to the caller.  Calls are
 *   asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 *   stream).
 * Graphs.  Every call except attn_get_status may be recorded by stream
 *   capture into a CUDA graph (it allocates nothing, waits for nothing and
 *   reads no device data on the host); replaying the graph repeats the
 *   calls with the same results.  attn_decode_static_scratch wants its first
 *   call before any capture (see there).
 * Sizes.  D in {64, 128}; Hq / Hkv in {1, 2, 4, 8}; Hq <= 128; the cache pool
 *   holds fewer than 2^31 slots; cache_lens[b] + n_b <= 2^24.
 * Errors.  A host-side check failure returns a negative ATTN_E* code and
 *   launches nothing.  Problems only visible on the device (a request whose
 *   region cannot hold c_b + n_b entries, cu_seqlens that are not
 *   non-decreasing or do not end at N, a host bound max_seqlen or
 *   max_cache_len below the device data) set bits of the status word in the
 *   workspace (ATTN_STATUS_*).  A request whose region is too small writes
 *   nothing to the cache; a request past max_seqlen / max_cache_len leaves
 *   its output rows unwritten (its new K/V are still appended).  Nothing
 *   traps.
 */
#ifndef GB300_ATTN_H
#define GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Per-layer shape and constants (host struct, passed by pointer). */
typedef struct attn_config {
  int32_t num_q_heads;  /* Hq */
  int32_t num_kv_heads; /* Hkv; Hq % Hkv == 0 (grouped-query attention) */
  int32_t head_dim;     /* D: 64 or 128 */
  float rms_eps;        /* eps of the Q/K RMSNorm (Qwen3: 1e-6) */
  float rope_theta;     /* RoPE base (Qwen3: 1e6) */
} attn_config_t;

/* The KV cache of one layer (host struct holding device pointers).
 * k_cache, v_cache: [num_slots, Hkv, D] entries (bf16, or E4M3 codes: see
 * kv_dtype below), contiguous, row = one slot.
 * The entry at position p of request b lives in one slot:
 *   contiguous (page_table == NULL): slot slot_base[b] + p; request b owns
 *     slots [slot_base[b], slot_base[b] + slot_capacity[b]);
 *   paged (page_table != NULL): slot page_table[b * pages_per_req + p / page_size]
 *     * page_size + p % page_size, i.e. the cache is num_slots / page_size
 *     pages of page_size slots and page_table row b lists request b's pages in
 *     position order; slot_base is unused (may be NULL).  page_size is a power
 *     of two >= 64 (every 64-key tile of a request lies in one page).  A page
 *     number outside [0, num_slots / page_size) sets ATTN_STATUS_CAPACITY: the
 *     entry is not written and reads of it return zeros.
 * In both layouts c_b + n_b <= slot_capacity[b] (paged: also
 * <= pages_per_req * page_size), else the request is skipped
 * (ATTN_STATUS_CAPACITY).  cache_lens[b] is read, never written: the caller
 * advances it after the call (the transformer-basics "Prefill vs Decode"
 * cache goes 0 -> 12 -> 13).
 *
 * Element type (kv_dtype):
 *   ATTN_KV_BF16 (0): bf16 entries; k_scale and v_scale are ignored.
 *   ATTN_KV_E4M3 (1): one byte per entry, OCP FP8 E4M3 (bias 7, largest
 *     finite 448, no infinity), each cache 1-byte [num_slots, Hkv, D].  The
 *     stored byte of a value x is e4m3(x * r) with r = 1 / scale rounded to
 *     fp32 on the host and x * r an fp32 product: round to nearest even,
 *     magnitudes above 448 clamped to 448.  x is the fp32 normed and rotated K
 *     (the value the bf16 cache rounds to bf16) or the bf16 V input.  Readers
 *     take byte * scale.  k_scale and v_scale are finite and > 0.  This
 *     element type halves the bytes a decode step reads (concept chapter
 *     section 4.3: decode is bound by memory bandwidth; its section 2.6 lists
 *     KV-cache reduction among the modern variants).  Every call takes it;
 *     next to an E4M3 cache the prepared Q of attn_prefill_prepare /
 *     attn_prefill_attend is f16 instead of bf16. */
typedef struct attn_kv {
  void* k_cache;
  void* v_cache;
  int64_t num_slots;
  const int64_t* slot_base;     /* [B] (contiguous layout) */
  const int32_t* cache_lens;    /* [B] */
  const int32_t* slot_capacity; /* [B] */
  const int32_t* page_table;    /* NULL, or [B, pages_per_req] page numbers (paged layout) */
  int32_t page_size;            /* slots per page (paged layout) */
  int32_t pages_per_req;        /* row length of page_table (paged layout) */
  int32_t kv_dtype;             /* ATTN_KV_BF16 or ATTN_KV_E4M3 */
  float k_scale;                /* E4M3: K entry = byte * k_scale */
  float v_scale;                /* E4M3: V entry = byte * v_scale */
} attn_kv_t;

enum { ATTN_KV_BF16 = 0, ATTN_KV_E4M3 = 1 };

enum {
  ATTN_OK = 0,
  ATTN_EINVAL = -1,       /* NULL pointer, negative size, unsupported D or Hq */
  ATTN_EGQA = -2,         /* Hq % Hkv != 0 or Hq / Hkv not in {1, 2, 4, 8} */
  ATTN_EWORKSPACE = -3,   /* workspace NULL, misaligned or smaller than required */
  ATTN_ELAUNCH = -4,      /* a CUDA launch or driver call failed */
  ATTN_EDEVICE = -5,      /* the current device is not sm_103 */
  ATTN_ESCRATCH = -6      /* attn_decode_static_scratch: request exceeds the static scratch */
};

/* Bits of the device status word (see attn_get_status). */
enum {
  ATTN_STATUS_CAPACITY = 1, /* a request's region cannot hold c_b + n_b entries */
  ATTN_STATUS_SEQLENS = 2,  /* cu_seqlens decreasing or cu_seqlens[B] != N */
  ATTN_STATUS_TIMEOUT = 4,  /* a pipeline wait gave up (internal error) */
  ATTN_STATUS_BOUNDS = 8    /* max_seqlen / max_cache_len below a request's length:
                               that request's output rows are left unwritten */
};

/* Workspace bytes needed by any call with at most `max_tokens` new tokens,
 * `max_batch` requests and `max_kv_len` keys per request (c_b + n_b).  The
 * workspace is a caller-owned device buffer, 256-byte aligned: a 256-byte
 * header holding the status word and the prefill work-item counters (the
 * prefill attention kernel hands its work items out through them and leaves
 * them at zero), then the prepared Q of attn_prefill (N * Hq * D bf16) or the
 * split-KV partial results of attn_decode.  Calls that share a workspace must
 * be ordered on one stream.  Returns 0 for invalid arguments. */
ATTN_API size_t attn_workspace_size(const attn_config_t* cfg, int32_t max_tokens, int32_t max_batch,
                           int32_t max_kv_len);

/* Zero the workspace header: the status word and the work-item counters
 * (asynchronous).  Call once after allocating a workspace; attn_get_status
 * clears the status word again. */
ATTN_API int attn_workspace_init(void* workspace, size_t ws_bytes, void* stream);

/* KV append only: split, K RMSNorm + RoPE, write K and V of the N new tokens
 * to the cache (no attention).  qkv: bf16 [N, (Hq+2Hkv)*D]; k_norm_w: bf16 [D];
 * cu_seqlens: int32 [B+1] on the device.  q_norm_w is unused and may be NULL.
 * transformer-basics "Prefill vs Decode": past_key_values.update. */
ATTN_API int attn_kv_append(const attn_config_t* cfg, const void* qkv, const void* q_norm_w,
                   const void* k_norm_w, const int32_t* cu_seqlens, int32_t B, int32_t N,
                   const attn_kv_t* kv, void* workspace, size_t ws_bytes, void* stream);

/* First half of attn_prefill: split qkv, RMSNorm + RoPE on Q and K, append
 * K and V to the cache, and write the prepared (normed, rotated) Q to q_out
 * [N, Hq, D] (device, caller-owned, 16-byte aligned): bf16, or f16 next to
 * an E4M3 cache.  cu_seqlens,
 * B, N and kv as for attn_prefill.  Code walkthrough section 3.3; basics
 * "Attention calculation: part 1" (q_norm / k_norm after .view) and "Prefill
 * vs Decode" (past_key_values.update). */
ATTN_API int attn_prefill_prepare(const attn_config_t* cfg, const void* qkv, const void* q_norm_w,
                                  const void* k_norm_w, const int32_t* cu_seqlens, int32_t B,
                                  int32_t N, const attn_kv_t* kv, void* q_out, void* workspace,
                                  size_t ws_bytes, void* stream);

/* Second half of attn_prefill: causal GQA over the prepared Q [N, Hq, D]
 * (from attn_prefill_prepare) and the cache, which must already hold this
 * call's K/V.  Writes out [N, Hq*D].  The workspace needs only its 256-byte
 * header here.  attn_prefill == attn_prefill_prepare (q_out in the workspace)
 * followed by attn_prefill_attend. */
ATTN_API int attn_prefill_attend(const attn_config_t* cfg, const void* q, const int32_t* cu_seqlens,
                                 int32_t B, int32_t N, int32_t max_seqlen, const attn_kv_t* kv,
                                 void* out, void* workspace, size_t ws_bytes, void* stream);

/* Prefill over ragged packed sequences: the whole step for the N new tokens
 * of B requests (request b's tokens are rows cu_seqlens[b] .. cu_seqlens[b+1]-1
 * of qkv), appending their K/V after the c_b cached entries and attending
 * over c_b + n_b keys.  max_seqlen >= every n_b (host value; bounds the grid).
 * out: bf16 [N, Hq*D].  Concept chapter section 4.1 "Prefill"; code
 * walkthrough section 3.1 (packed [N, C] layout) and section 3.3. */
ATTN_API int attn_prefill(const attn_config_t* cfg, const void* qkv, const void* q_norm_w,
                 const void* k_norm_w, const int32_t* cu_seqlens, int32_t B, int32_t N,
                 int32_t max_seqlen, const attn_kv_t* kv, void* out, void* workspace,
                 size_t ws_bytes, void* stream);

/* Decode: one new token per request (row b of qkv is request b's token at
 * position c_b), appended and attended over c_b + 1 keys with split-KV and a
 * log-sum-exp merge.  max_cache_len >= every c_b (host value).  One kernel
 * launch (two when a request spans several splits): the split that holds
 * position c_b writes the new K/V before it reads its keys, with the same
 * arithmetic as attn_kv_append.
 * out: bf16 [B, Hq*D].  Concept chapter section 4.2 "Decode";
 * transformer-basics "Prefill vs Decode" (one more row of the lower triangle). */
ATTN_API int attn_decode(const attn_config_t* cfg, const void* qkv, const void* q_norm_w,
                const void* k_norm_w, int32_t B, int32_t max_cache_len, const attn_kv_t* kv,
                void* out, void* workspace, size_t ws_bytes, void* stream);

/* The merged Q/K/V projection fused with the first half of attn_prefill.
 * Code walkthrough section 3.3 (AttentionLayer.forward: qkv_proj of the
 * hidden states, then the split, the Q/K norms and RoPE) and transformer
 * basics "Attention calculation: part 1" (the q/k/v projections of the hidden
 * states, a linear layer y = x W^T).
 *   qkv = hidden [N, C] . w_qkv^T, w_qkv [(Hq + 2 Hkv) * D, C] (the linear
 *   layer's weight, row = output feature), bf16 in, fp32 accumulation on the
 *   tensor cores.  The fp32 qkv is never stored or rounded: each Q and K head
 *   is RMS-normalised and rotated from the accumulators, V rounded once, and
 *   then exactly as attn_prefill_prepare: K and V appended to the cache (bf16
 *   or E4M3 codes), the prepared Q written to q_out [N, Hq, D] (bf16, f16 next
 *   to an E4M3 cache; 16-byte aligned), ready for attn_prefill_attend.
 * hidden, w_qkv: bf16, row-major, 16-byte aligned; C = hidden_size, a
 * multiple of 8.  cu_seqlens, B, N and kv as for attn_prefill; decode rows
 * are requests with n_b = 1.  The workspace needs only its 256-byte header
 * (status word). */
ATTN_API int attn_qkv_proj_prepare(const attn_config_t* cfg, const void* hidden, int32_t hidden_size,
                                   const void* w_qkv, const void* q_norm_w, const void* k_norm_w,
                                   const int32_t* cu_seqlens, int32_t B, int32_t N, const attn_kv_t* kv,
                                   void* q_out, void* workspace, size_t ws_bytes, void* stream);

/* The output projection after the attention (code walkthrough section 3.3:
 * o_proj; transformer basics "Attention calculation: part 1"):
 *   out [N, C] = attn_out [N, Hq * D] . w_o^T, w_o [C, Hq * D] (row = output
 *   feature), bf16 in and out, fp32 accumulation on the tensor cores.
 * attn_out is the output of attn_prefill / attn_decode; C = hidden_size, a
 * multiple of 8; all pointers 16-byte aligned.  The workspace needs only its
 * 256-byte header (status word). */
ATTN_API int attn_o_proj(const attn_config_t* cfg, const void* attn_out, int32_t N, const void* w_o,
                         int32_t hidden_size, void* out, void* workspace, size_t ws_bytes, void* stream);

/* Number of KV splits attn_decode (and attn_decode_attend,
 * attn_decode_static_scratch) uses for the longest request of a call with B
 * requests and host bound max_cache_len: the split length is chosen so that
 * about 2048 CTAs run when every request is at its longest, with at least 256
 * keys and at most 16 splits per request.  1 means every output row is
 * written by the split kernel directly (no partials, no merge launch).
 * Returns ATTN_EINVAL (< 0) for invalid arguments.  Host-only. */
ATTN_API int32_t attn_decode_splits(const attn_config_t* cfg, int32_t B, int32_t max_cache_len);

/* Attention half of attn_decode (the cache must already hold the new
 * token's K/V at slot slot_base[b] + c_b).  attn_decode gives bit for bit the
 * output and cache of attn_kv_append (cu_seqlens = 0, 1, ..., B) followed by
 * attn_decode_attend, in fewer launches. */
ATTN_API int attn_decode_attend(const attn_config_t* cfg, const void* qkv, const void* q_norm_w,
                                int32_t B, int32_t max_cache_len, const attn_kv_t* kv, void* out,
                                void* workspace, size_t ws_bytes, void* stream);

/* Decode without any caller-provided scratch, for callers that cannot
 * allocate device memory where they run decode (a plugin inside a host
 * framework that owns all device allocations; a serving loop that cannot
 * afford cudaMalloc's implicit synchronisation).  Same arguments and result
 * as attn_decode, except that the split-KV partial results live in a
 * library-owned static device array of 16 MiB per GPU (held by every GPU that
 * loads the library until the process exits) instead of a workspace.
 *   - With splits = attn_decode_splits(cfg, B, max_cache_len) > 1 the
 *     partials take B * Hq * splits * (D + 2) * 4 bytes (each of the two
 *     arrays rounded up to 256 bytes); requests needing more than the array
 *     return ATTN_ESCRATCH and launch nothing.  With splits == 1 every output
 *     row is written directly and the call needs no scratch at any B.
 *   - device_status: optional caller-owned device int32 (NULL: not recorded)
 *     that receives the ATTN_STATUS_* bits; the caller zeroes it.
 *   - The first call on a device looks up the array's device address on the
 *     current device (cudaGetSymbolAddress) and keeps it for the process;
 *     make that first call before any stream capture, and after any
 *     cudaDeviceReset of that device (a reset after it leaves the kept
 *     address stale: do not reset a device that has used this call).
 *   - All calls share the array: calls that overlap on the GPU race.
 *   - Allocates nothing (no cudaMalloc, no cudaFree, no allocating library
 *     call).
 * Not part of the attention method: the zero-to-sglang and transformer-basics
 * pages this library follows have no counterpart to it. */
ATTN_API int attn_decode_static_scratch(const attn_config_t* cfg, const void* qkv,
                                        const void* q_norm_w, const void* k_norm_w, int32_t B,
                                        int32_t max_cache_len, const attn_kv_t* kv, void* out,
                                        int32_t* device_status, void* stream);

/* Read the status word into *status (host pointer) and clear it, both
 * ordered on `stream`, then synchronise that stream (only that stream).
 * Returns ATTN_OK or ATTN_ELAUNCH. */
ATTN_API int attn_get_status(void* workspace, void* stream, int32_t* status);

/* Static string for an ATTN_E* code. */
ATTN_API const char* attn_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* GB300_ATTN_H */
