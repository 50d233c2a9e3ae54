// C ABI of the attention step (declared in include/attn.h): argument checks,
// workspace carving, tensor-map encoding and kernel launches.  No allocation,
// no state between calls, no stream synchronisation except attn_get_status.
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "../../include/sample.h"
#include "kernels.cuh"

namespace gb300 {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// bf16 cache: boxes of 64 (d) x 1 (head) x box_rows, 128-byte swizzled.
// E4M3 cache (one byte per entry): boxes of D x 1 x box_rows, 128-byte
// swizzled for D = 128, unswizzled 64-byte rows for D = 64.
int encode_cache_map(void* base, int64_t num_slots, int Hkv, int D, int box_rows, bool f8,
                     CUtensorMap* m) {
  auto enc = encoder();
  if (!enc) return -1;
  const cuuint64_t es = f8 ? 1 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)num_slots};
  cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)Hkv * D * es};
  cuuint32_t box[3] = {f8 ? (cuuint32_t)D : 64u, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw =
      (!f8 || D == 128) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = enc(m, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base,
                   dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

bool is_pow2_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

int check_config(const attn_config_t* cfg) {
  if (!cfg) return ATTN_EINVAL;
  if (cfg->head_dim != 64 && cfg->head_dim != 128) return ATTN_EINVAL;
  if (cfg->num_q_heads <= 0 || cfg->num_kv_heads <= 0 || cfg->num_q_heads > 128) return ATTN_EINVAL;
  if (!(cfg->rms_eps >= 0.f) || !(cfg->rope_theta > 1.f)) return ATTN_EINVAL;
  if (cfg->num_q_heads % cfg->num_kv_heads != 0) return ATTN_EGQA;
  if (!is_pow2_group(cfg->num_q_heads / cfg->num_kv_heads)) return ATTN_EGQA;
  return ATTN_OK;
}

int check_kv(const attn_kv_t* kv) {
  if (!kv || !kv->k_cache || !kv->v_cache || !kv->cache_lens || !kv->slot_capacity)
    return ATTN_EINVAL;
  if (kv->page_table) {
    const int ps = kv->page_size;
    if (ps < 64 || ps > (1 << 20) || (ps & (ps - 1)) != 0 || kv->pages_per_req <= 0)
      return ATTN_EINVAL;
  } else if (!kv->slot_base) {
    return ATTN_EINVAL;
  }
  if (kv->num_slots <= 0 || kv->num_slots >= (int64_t(1) << 31)) return ATTN_EINVAL;
  if (kv->kv_dtype == ATTN_KV_E4M3) {
    if (!(kv->k_scale > 0.f) || !(kv->v_scale > 0.f) || std::isinf(kv->k_scale) ||
        std::isinf(kv->v_scale))
      return ATTN_EINVAL;
  } else if (kv->kv_dtype != ATTN_KV_BF16) {
    return ATTN_EINVAL;
  }
  if ((reinterpret_cast<uintptr_t>(kv->k_cache) | reinterpret_cast<uintptr_t>(kv->v_cache)) & 15)
    return ATTN_EINVAL;
  return ATTN_OK;
}

int check_device() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ELAUNCH;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return ATTN_ELAUNCH;
  return (major == 10 && minor == 3) ? ATTN_OK : ATTN_EDEVICE;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Split-KV partials of a decode call.  With one split per request the split
// kernel writes the output directly and the partials are never touched.
size_t partial_bytes(const attn_config_t& c, int64_t B, int max_splits) {
  if (max_splits <= 1) return 0;
  size_t rows = (size_t)B * c.num_q_heads * max_splits;
  return align_up(rows * c.head_dim * 4, 256) + align_up(rows * 2 * 4, 256);
}

int32_t* status_of(void* ws) { return static_cast<int32_t*>(ws); }
// prefill work-item counters: 64 bytes into the header
int32_t* work_of(void* ws) { return static_cast<int32_t*>(ws) + 16; }

}  // namespace

void make_rope_freqs(float theta, int head_dim, RopeFreqs* out) {
  const int half = head_dim / 2;
  for (int i = 0; i < 64; ++i) {
    double f = i < half ? std::pow((double)theta, -2.0 * i / head_dim) : 0.0;
    float hi = (float)f;
    out->hi[i] = hi;
    out->lo[i] = (float)(f - (double)hi);
  }
  const double two_pi = 6.283185307179586476925286766559;
  out->two_pi_hi = (float)two_pi;
  out->two_pi_lo = (float)(two_pi - (double)out->two_pi_hi);
  out->inv_two_pi = (float)(1.0 / two_pi);
}

int abi_check_config(const attn_config_t* cfg) { return check_config(cfg); }
int abi_check_kv(const attn_kv_t* kv) { return check_kv(kv); }
int abi_check_device() { return check_device(); }

int make_qkv_map(const void* qkv, int N, int Htot, int D, int G, int BT, CUtensorMap* m) {
  auto enc = encoder();
  if (!enc) return -1;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Htot, (cuuint64_t)N};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Htot * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)BT};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(qkv), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

int make_matrix_map(const void* base, int64_t rows, int64_t cols, int box_rows, CUtensorMap* m) {
  auto enc = encoder();
  if (!enc) return -1;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

int make_cache_maps(const attn_kv_t& kv, int Hkv, int D, int box_rows, CacheMaps* maps) {
  const bool f8 = kv.kv_dtype == ATTN_KV_E4M3;
  if (encode_cache_map(kv.k_cache, kv.num_slots, Hkv, D, box_rows, f8, &maps->k) != 0) return -1;
  if (encode_cache_map(kv.v_cache, kv.num_slots, Hkv, D, box_rows, f8, &maps->v) != 0) return -1;
  return 0;
}

namespace {

// Checks shared by the entry points that read qkv and write out.
int check_common(const attn_config_t* cfg, const attn_kv_t* kv, const void* qkv,
                 const void* w, const void* out) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if ((rc = check_kv(kv))) return rc;
  if (!qkv || !w || !out) return ATTN_EINVAL;
  if (!aligned16(qkv) || !aligned16(w) || !aligned16(out)) return ATTN_EINVAL;
  return ATTN_OK;
}

bool ws_ok(const void* ws, size_t bytes, size_t need) {
  return ws && (reinterpret_cast<uintptr_t>(ws) & 255) == 0 && bytes >= need;
}

// Prologue kernel: K (and, with q_out, Q) norm + RoPE, K/V cache append.
int append(const attn_config_t* cfg, const void* qkv, const void* q_norm_w, const void* k_norm_w,
           const int32_t* cu_seqlens, int32_t B, int32_t N, const attn_kv_t* kv, void* q_out,
           void* workspace, cudaStream_t s) {
  PrologueArgs a;
  a.cfg = *cfg;
  a.qkv = qkv;
  a.q_norm_w = q_norm_w;
  a.k_norm_w = k_norm_w;
  a.q_out = q_out;
  a.cu_seqlens = cu_seqlens;
  a.B = B;
  a.N = N;
  a.kv = *kv;
  a.status = status_of(workspace);
  make_rope_freqs(cfg->rope_theta, cfg->head_dim, &a.freqs);
  return launch_prologue(a, s) == cudaSuccess ? ATTN_OK : ATTN_ELAUNCH;
}

int prefill_attend(const attn_config_t* cfg, const void* q, const int32_t* cu_seqlens, int32_t B,
                   int32_t N, int32_t max_seqlen, const attn_kv_t* kv, void* out, void* workspace,
                   cudaStream_t s) {
  PrefillArgs pa;
  pa.cfg = *cfg;
  pa.B = B;
  pa.N = N;
  pa.max_seqlen = max_seqlen;
  pa.cu_seqlens = cu_seqlens;
  pa.kv = *kv;
  pa.q = q;
  pa.out = out;
  pa.status = status_of(workspace);
  pa.work = work_of(workspace);
  return launch_prefill(pa, s);
}

size_t q_stage_bytes(const attn_config_t* cfg, int64_t N) {
  return align_up((size_t)N * cfg->num_q_heads * cfg->head_dim * 2, 256);
}

size_t decode_ws_need(const attn_config_t* cfg, int32_t B, int32_t max_cache_len, int* split_len,
                      int* max_splits) {
  *split_len = decode_split_len(std::max(B, 1), cfg->num_kv_heads, max_cache_len + 1, max_splits);
  return kWsHeader + partial_bytes(*cfg, B, *max_splits);
}

// Split-KV decode (and merge); with k_norm_w, the new tokens' K/V are
// appended inside the split kernel first.
int decode_attend(const attn_config_t* cfg, const void* qkv, const void* q_norm_w, const void* k_norm_w,
                  int32_t B, int32_t max_cache_len, const attn_kv_t* kv, void* out, void* workspace,
                  cudaStream_t s) {
  int split_len = 0, max_splits = 1;
  decode_ws_need(cfg, B, max_cache_len, &split_len, &max_splits);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t rows = (size_t)B * cfg->num_q_heads * max_splits;
  DecodeArgs d;
  d.cfg = *cfg;
  d.B = B;
  d.kv = *kv;
  d.qkv = qkv;
  d.q_norm_w = q_norm_w;
  d.k_norm_w = k_norm_w;
  make_rope_freqs(cfg->rope_theta, cfg->head_dim, &d.freqs);
  d.out = out;
  d.part_o = reinterpret_cast<float*>(ws + kWsHeader);
  d.part_ml = reinterpret_cast<float*>(ws + kWsHeader + align_up(rows * cfg->head_dim * 4, 256));
  d.split_len = split_len;
  d.max_splits = max_splits;
  d.status = status_of(workspace);
  return launch_decode(d, s);
}

}  // namespace
}  // namespace gb300

using namespace gb300;

extern "C" {

size_t attn_workspace_size(const attn_config_t* cfg, int32_t max_tokens, int32_t max_batch,
                           int32_t max_kv_len) {
  if (check_config(cfg) != ATTN_OK || max_tokens < 0 || max_batch < 0 || max_kv_len < 0) return 0;
  int split_len = 0, max_splits = 1;
  const size_t decode = decode_ws_need(cfg, max_batch, std::max(max_kv_len, 1) - 1, &split_len, &max_splits);
  const size_t prefill = kWsHeader + q_stage_bytes(cfg, max_tokens);
  return std::max(prefill, decode);
}

int32_t attn_decode_splits(const attn_config_t* cfg, int32_t B, int32_t max_cache_len) {
  if (check_config(cfg) != ATTN_OK || B < 0 || max_cache_len < 0) return ATTN_EINVAL;
  int max_splits = 1;
  decode_split_len(std::max(B, 1), cfg->num_kv_heads, max_cache_len + 1, &max_splits);
  return max_splits;
}

int attn_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
  if (!ws_ok(workspace, ws_bytes, kWsHeader)) return ATTN_EWORKSPACE;
  return cudaMemsetAsync(workspace, 0, kWsHeader, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? ATTN_OK
             : ATTN_ELAUNCH;
}

int attn_kv_append(const attn_config_t* cfg, const void* qkv, const void* q_norm_w,
                   const void* k_norm_w, const int32_t* cu_seqlens, int32_t B, int32_t N,
                   const attn_kv_t* kv, void* workspace, size_t ws_bytes, void* stream) {
  (void)q_norm_w;
  int rc = check_common(cfg, kv, qkv, k_norm_w, k_norm_w);
  if (rc) return rc;
  if (!cu_seqlens || B < 0 || N < 0) return ATTN_EINVAL;
  if (!ws_ok(workspace, ws_bytes, kWsHeader)) return ATTN_EWORKSPACE;
  if ((rc = check_device())) return rc;
  if (N == 0 || B == 0) return ATTN_OK;
  return append(cfg, qkv, nullptr, k_norm_w, cu_seqlens, B, N, kv, nullptr, workspace,
                static_cast<cudaStream_t>(stream));
}

int attn_prefill_prepare(const attn_config_t* cfg, const void* qkv, const void* q_norm_w,
                         const void* k_norm_w, const int32_t* cu_seqlens, int32_t B, int32_t N,
                         const attn_kv_t* kv, void* q_out, void* workspace, size_t ws_bytes,
                         void* stream) {
  int rc = check_common(cfg, kv, qkv, q_norm_w, q_out);
  if (rc) return rc;
  if (!k_norm_w || !aligned16(k_norm_w)) return ATTN_EINVAL;
  if (!cu_seqlens || B < 0 || N < 0) return ATTN_EINVAL;
  if (!ws_ok(workspace, ws_bytes, kWsHeader)) return ATTN_EWORKSPACE;
  if ((rc = check_device())) return rc;
  if (N == 0 || B == 0) return ATTN_OK;
  return append(cfg, qkv, q_norm_w, k_norm_w, cu_seqlens, B, N, kv, q_out, workspace,
                static_cast<cudaStream_t>(stream));
}

int attn_prefill_attend(const attn_config_t* cfg, const void* q, const int32_t* cu_seqlens,
                        int32_t B, int32_t N, int32_t max_seqlen, const attn_kv_t* kv, void* out,
                        void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_common(cfg, kv, q, q, out);
  if (rc) return rc;
  if (!cu_seqlens || B < 0 || N < 0 || max_seqlen < 0) return ATTN_EINVAL;
  if (!ws_ok(workspace, ws_bytes, kWsHeader)) return ATTN_EWORKSPACE;
  if ((rc = check_device())) return rc;
  if (N == 0 || B == 0) return ATTN_OK;
  return prefill_attend(cfg, q, cu_seqlens, B, N, max_seqlen, kv, out, workspace,
                        static_cast<cudaStream_t>(stream));
}

int attn_prefill(const attn_config_t* cfg, const void* qkv, const void* q_norm_w,
                 const void* k_norm_w, const int32_t* cu_seqlens, int32_t B, int32_t N,
                 int32_t max_seqlen, const attn_kv_t* kv, void* out, void* workspace,
                 size_t ws_bytes, void* stream) {
  int rc = check_common(cfg, kv, qkv, q_norm_w, out);
  if (rc) return rc;
  if (!k_norm_w || !aligned16(k_norm_w)) return ATTN_EINVAL;
  if (!cu_seqlens || B < 0 || N < 0 || max_seqlen < 0) return ATTN_EINVAL;
  if (!ws_ok(workspace, ws_bytes, kWsHeader + q_stage_bytes(cfg, N))) return ATTN_EWORKSPACE;
  if ((rc = check_device())) return rc;
  if (N == 0 || B == 0) return ATTN_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* q_stage = static_cast<uint8_t*>(workspace) + kWsHeader;
  if ((rc = append(cfg, qkv, q_norm_w, k_norm_w, cu_seqlens, B, N, kv, q_stage, workspace, s)))
    return rc;
  return prefill_attend(cfg, q_stage, cu_seqlens, B, N, max_seqlen, kv, out, workspace, s);
}

int attn_decode_attend(const attn_config_t* cfg, const void* qkv, const void* q_norm_w, int32_t B,
                       int32_t max_cache_len, const attn_kv_t* kv, void* out, void* workspace,
                       size_t ws_bytes, void* stream) {
  int rc = check_common(cfg, kv, qkv, q_norm_w, out);
  if (rc) return rc;
  if (B < 0 || max_cache_len < 0) return ATTN_EINVAL;
  int split_len = 0, max_splits = 1;
  if (!ws_ok(workspace, ws_bytes, decode_ws_need(cfg, B, max_cache_len, &split_len, &max_splits)))
    return ATTN_EWORKSPACE;
  if ((rc = check_device())) return rc;
  if (B == 0) return ATTN_OK;
  return decode_attend(cfg, qkv, q_norm_w, nullptr, B, max_cache_len, kv, out, workspace,
                       static_cast<cudaStream_t>(stream));
}

int attn_decode(const attn_config_t* cfg, const void* qkv, const void* q_norm_w,
                const void* k_norm_w, int32_t B, int32_t max_cache_len, const attn_kv_t* kv,
                void* out, void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_common(cfg, kv, qkv, q_norm_w, out);
  if (rc) return rc;
  if (!k_norm_w || !aligned16(k_norm_w)) return ATTN_EINVAL;
  if (B < 0 || max_cache_len < 0) return ATTN_EINVAL;
  int split_len = 0, max_splits = 1;
  if (!ws_ok(workspace, ws_bytes, decode_ws_need(cfg, B, max_cache_len, &split_len, &max_splits)))
    return ATTN_EWORKSPACE;
  if ((rc = check_device())) return rc;
  if (B == 0) return ATTN_OK;
  return decode_attend(cfg, qkv, q_norm_w, k_norm_w, B, max_cache_len, kv, out, workspace,
                       static_cast<cudaStream_t>(stream));
}

int attn_qkv_proj_prepare(const attn_config_t* cfg, const void* hidden, int32_t hidden_size, const void* w_qkv,
                          const void* q_norm_w, const void* k_norm_w, const int32_t* cu_seqlens, int32_t B,
                          int32_t N, const attn_kv_t* kv, void* q_out, void* workspace, size_t ws_bytes,
                          void* stream) {
  int rc = check_common(cfg, kv, hidden, q_norm_w, q_out);
  if (rc) return rc;
  if (!w_qkv || !aligned16(w_qkv) || !k_norm_w || !aligned16(k_norm_w)) return ATTN_EINVAL;
  if (!cu_seqlens || B < 0 || N < 0 || hidden_size <= 0 || hidden_size % 8 != 0) return ATTN_EINVAL;
  if (!ws_ok(workspace, ws_bytes, kWsHeader)) return ATTN_EWORKSPACE;
  if ((rc = check_device())) return rc;
  if (N == 0 || B == 0) return ATTN_OK;
  QkvProjArgs a;
  a.cfg = *cfg;
  a.hidden = hidden;
  a.C = hidden_size;
  a.w_qkv = w_qkv;
  a.q_norm_w = q_norm_w;
  a.k_norm_w = k_norm_w;
  a.cu_seqlens = cu_seqlens;
  a.B = B;
  a.N = N;
  a.kv = *kv;
  a.q_out = q_out;
  a.status = status_of(workspace);
  make_rope_freqs(cfg->rope_theta, cfg->head_dim, &a.freqs);
  return launch_qkv_proj(a, static_cast<cudaStream_t>(stream));
}

int attn_o_proj(const attn_config_t* cfg, const void* attn_out, int32_t N, const void* w_o, int32_t hidden_size,
                void* out, void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!attn_out || !w_o || !out || !aligned16(attn_out) || !aligned16(w_o) || !aligned16(out)) return ATTN_EINVAL;
  if (N < 0 || hidden_size <= 0 || hidden_size % 8 != 0) return ATTN_EINVAL;
  if (!ws_ok(workspace, ws_bytes, kWsHeader)) return ATTN_EWORKSPACE;
  if ((rc = check_device())) return rc;
  if (N == 0) return ATTN_OK;
  return launch_linear(attn_out, w_o, out, N, hidden_size, cfg->num_q_heads * cfg->head_dim, status_of(workspace),
                       static_cast<cudaStream_t>(stream));
}

int attn_get_status(void* workspace, void* stream, int32_t* status) {
  if (!workspace || !status) return ATTN_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // ordered on the caller's stream only (a plain cudaMemcpy would also wait
  // for every blocking stream through the legacy default stream)
  int32_t word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return ATTN_ELAUNCH;
  if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), s) != cudaSuccess) return ATTN_ELAUNCH;
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ELAUNCH;
  *status = word;
  return ATTN_OK;
}

int attn_sample_tokens(const float* logits, int32_t B, int32_t V, int64_t ld, const float* temperature,
                       const int32_t* top_k, const float* top_p, const float* uniform, int32_t* tokens,
                       void* stream) {
  if (!logits || !temperature || !top_k || !top_p || !uniform || !tokens) return ATTN_EINVAL;
  if (B < 0 || V < 1 || V > (1 << 23) || ld < V) return ATTN_EINVAL;  // sums of 2^-40 units fit 64 bits
  int rc = check_device();
  if (rc) return rc;
  return launch_sample(logits, B, V, ld, temperature, top_k, top_p, uniform, tokens,
                       static_cast<cudaStream_t>(stream));
}

const char* attn_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "ok";
    case ATTN_EINVAL: return "invalid argument (NULL pointer, negative size, unsupported shape or misaligned buffer)";
    case ATTN_EGQA: return "Hq must be a multiple of Hkv with Hq/Hkv in {1, 2, 4, 8}";
    case ATTN_EWORKSPACE: return "workspace missing, not 256-byte aligned or too small";
    case ATTN_ELAUNCH: return "CUDA launch or driver call failed";
    case ATTN_EDEVICE: return "the current CUDA device is not sm_103 (GB300)";
    case ATTN_ESCRATCH: return "request needs more split-KV scratch than the library's static 16 MiB buffer (use attn_decode with a workspace)";
    default: return "unknown error";
  }
}

}  // extern "C"
