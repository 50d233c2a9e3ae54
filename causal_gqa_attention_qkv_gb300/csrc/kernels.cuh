// Launch interfaces between the C ABI (attn_abi.cu) and the kernels.
#pragma once

#include "common.cuh"

namespace gb300 {

void make_rope_freqs(float theta, int head_dim, RopeFreqs* out);

// The indexing fields of a (checked) attn_kv_t, as the kernels use them.
inline KvIndex kv_index(const attn_kv_t& kv) {
  KvIndex x;
  x.slot_base = kv.slot_base;
  x.cache_lens = kv.cache_lens;
  x.slot_capacity = kv.slot_capacity;
  x.page_table = kv.page_table;
  x.num_slots = kv.num_slots;
  x.log2_page = 0;
  if (kv.page_table)
    while ((1 << x.log2_page) < kv.page_size) ++x.log2_page;
  x.pages_per_req = kv.pages_per_req;
  return x;
}

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the one before it in the stream finishes.  It must call
// grid_dependency_wait() before touching memory an earlier kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Host-side argument checks of the C ABI (ATTN_OK or an ATTN_E* code).
int abi_check_config(const attn_config_t* cfg);
int abi_check_kv(const attn_kv_t* kv);
int abi_check_device();

// K RMSNorm + RoPE and the K/V append of N new tokens; with q_out, also Q
// RMSNorm + RoPE into q_out [N, Hq, D] bf16.
struct PrologueArgs {
  attn_config_t cfg;
  const void* qkv;
  const void* q_norm_w;  // used when q_out != NULL
  const void* k_norm_w;
  void* q_out;           // NULL: K/V only
  const int32_t* cu_seqlens;  // NULL in decode mode (token b = request b)
  int32_t B, N;
  attn_kv_t kv;
  int32_t* status;
  RopeFreqs freqs;
};
cudaError_t launch_prologue(const PrologueArgs& a, cudaStream_t stream);

// Tensor maps over the K and V cache pools, [num_slots, Hkv, D] bf16, 128-byte
// swizzled boxes of 64 (d) x 1 (head) x box_rows (slots).
struct CacheMaps {
  CUtensorMap k;
  CUtensorMap v;
};
int make_cache_maps(const attn_kv_t& kv, int Hkv, int D, int box_rows, CacheMaps* maps);

// Tensor map over qkv viewed as [N, Htot, D] bf16 (Htot = Hq + 2*Hkv), 128-byte
// swizzled boxes of 64 (d) x G (heads) x BT (tokens): one box is the half
// (64 of D columns) of a 128-row Q tile of packed (token, group head) rows.
int make_qkv_map(const void* qkv, int N, int Htot, int D, int G, int BT, CUtensorMap* map);

// The attention kernels read Q straight from qkv and normalise and rotate
// it themselves.
struct DecodeArgs {
  attn_config_t cfg;
  int32_t B;
  attn_kv_t kv;
  const void* qkv;       // [B, W] bf16
  const void* q_norm_w;  // [D] bf16
  const void* k_norm_w;  // [D] bf16: append the new K/V inside the kernel; NULL: already in the cache
  RopeFreqs freqs;
  void* out;      // [B, Hq*D] bf16
  float* part_o;  // [B, Hq, max_splits, D] fp32
  float* part_ml; // [B, Hq, max_splits, 2] fp32 (running max in log2 units, sum)
  int32_t split_len, max_splits;
  int32_t* status;
};
int decode_split_len(int B, int Hkv, int max_kv_len, int* max_splits);
int launch_decode(const DecodeArgs& a, cudaStream_t stream);

struct PrefillArgs {
  attn_config_t cfg;
  int32_t B, N, max_seqlen;
  const int32_t* cu_seqlens;
  attn_kv_t kv;
  const void* q;  // [N, Hq, D] bf16, normed and rotated
  void* out;      // [N, Hq*D] bf16
  int32_t* status;
  // two int32 in the workspace header: next work item, CTAs finished; zero
  // before the launch, left zero by it
  int32_t* work;
};
int launch_prefill(const PrefillArgs& a, cudaStream_t stream);

// Row-major bf16 matrix [rows, cols] as a 2-D tensor map with 128-byte
// swizzled boxes of 64 columns x box_rows rows (cols % 8 == 0).
int make_matrix_map(const void* base, int64_t rows, int64_t cols, int box_rows, CUtensorMap* map);

// y [M, N] = x [M, K] . w[N, K]^T, bf16 in and out, fp32 accumulation on the
// tensor cores (N % 8 == 0, K % 8 == 0, 16-byte aligned pointers).
int launch_linear(const void* x, const void* w, void* y, int32_t M, int32_t N, int32_t K, int32_t* status,
                  cudaStream_t stream);

// qkv = hidden [N, C] . w_qkv[(Hq+2Hkv)D, C]^T kept in fp32 and handed to the
// prologue: Q/K RMSNorm + RoPE, K/V append, prepared Q into q_out [N, Hq, D].
struct QkvProjArgs {
  attn_config_t cfg;
  const void* hidden;
  int32_t C;
  const void* w_qkv;
  const void* q_norm_w;
  const void* k_norm_w;
  const int32_t* cu_seqlens;
  int32_t B, N;
  attn_kv_t kv;
  void* q_out;
  int32_t* status;
  RopeFreqs freqs;
};
int launch_qkv_proj(const QkvProjArgs& a, cudaStream_t stream);

// One token per row of logits (include/sample.h); arguments checked by the caller.
int launch_sample(const float* logits, int32_t B, int32_t V, int64_t ld, const float* temperature,
                  const int32_t* top_k, const float* top_p, const float* uniform, int32_t* tokens,
                  cudaStream_t stream);

}  // namespace gb300
