// attn_decode_static_scratch: the decode step with its split-KV scratch in a
// fixed, library-owned device buffer instead of a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run
// decode: a plugin inside a host framework that owns every device
// allocation, or a latency-critical serving loop where cudaMalloc's implicit
// device synchronisation is not acceptable.  This entry point lets them run
// the decode step with nothing but their input and output buffers.
//
// The scratch is the file-scope array below (kStaticScratchBytes per GPU,
// held by every GPU that loads the library until the process exits).  Host
// code must not pass the array's name to a kernel: in host code it is only a
// stand-in symbol.  The device address is obtained once per device, with that
// device current, by cudaGetSymbolAddress, on the first call of this entry
// point on that device.  Calls share the array and it keeps the last call's
// contents; nothing in it has to start at zero (every partial result a call
// reads was written earlier in the same call).  Calls that overlap on the GPU
// (different streams, or different host threads without ordering) race on it.
#include <mutex>

#include "kernels.cuh"

namespace gb300 {

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB per device
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (set-up on first use).
int static_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ELAUNCH;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return ATTN_ELAUNCH;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

}  // namespace gb300

using namespace gb300;

extern "C" int attn_decode_static_scratch(const attn_config_t* cfg, const void* qkv,
                                          const void* q_norm_w, const void* k_norm_w, int32_t B,
                                          int32_t max_cache_len, const attn_kv_t* kv, void* out,
                                          int32_t* device_status, void* stream) {
  int rc = abi_check_config(cfg);
  if (rc) return rc;
  if ((rc = abi_check_kv(kv))) return rc;
  if (!qkv || !q_norm_w || !k_norm_w || !out || B < 0 || max_cache_len < 0) return ATTN_EINVAL;
  if (((reinterpret_cast<uintptr_t>(qkv) | reinterpret_cast<uintptr_t>(q_norm_w) |
        reinterpret_cast<uintptr_t>(k_norm_w) | reinterpret_cast<uintptr_t>(out)) & 15) != 0)
    return ATTN_EINVAL;
  int max_splits = 1;
  const int split_len =
      decode_split_len(std::max(B, 1), cfg->num_kv_heads, max_cache_len + 1, &max_splits);
  // With one split per request the split kernel writes `out` directly and no
  // partial result is stored: such calls need no scratch at all.
  const size_t rows = (size_t)B * cfg->num_q_heads * max_splits;
  const size_t o_bytes = align_up(rows * cfg->head_dim * 4, 256);
  const size_t need = max_splits > 1 ? o_bytes + align_up(rows * 2 * 4, 256) : 0;
  if (need > kStaticScratchBytes) return ATTN_ESCRATCH;
  if ((rc = abi_check_device())) return rc;
  if (B == 0) return ATTN_OK;
  void* scratch = nullptr;
  if ((rc = static_scratch(&scratch))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);


  DecodeArgs d;
  d.cfg = *cfg;
  d.B = B;
  d.kv = *kv;
  d.qkv = qkv;
  d.q_norm_w = q_norm_w;
  d.k_norm_w = k_norm_w;  // the new K/V are appended inside the split kernel
  make_rope_freqs(cfg->rope_theta, cfg->head_dim, &d.freqs);
  d.out = out;
  d.part_o = static_cast<float*>(scratch);
  d.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + o_bytes);
  d.split_len = split_len;
  d.max_splits = max_splits;
  d.status = device_status;
  return launch_decode(d, s);
}
