"""ctypes binding of libattn.so (include/attn.h).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels.  PyTorch provides device memory and the current
stream.  If the library has not been built (or cannot be loaded) every call
raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn.so")

ATTN_STATUS_CAPACITY = 1
ATTN_STATUS_SEQLENS = 2
ATTN_STATUS_TIMEOUT = 4
ATTN_STATUS_BOUNDS = 8


class AttnConfig(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("rms_eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float)]


class AttnKV(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("num_slots", ctypes.c_int64), ("slot_base", ctypes.c_void_p),
                ("cache_lens", ctypes.c_void_p), ("slot_capacity", ctypes.c_void_p),
                ("page_table", ctypes.c_void_p), ("page_size", ctypes.c_int32),
                ("pages_per_req", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


ATTN_KV_BF16 = 0
ATTN_KV_E4M3 = 1


class AttnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"attn error {code}: {msg}")
        self.code = code


_lib = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t
_CFG = ctypes.POINTER(AttnConfig)
_KV = ctypes.POINTER(AttnKV)

EXPORTS = {
    "attn_workspace_size": (_SZ, [_CFG, _I32, _I32, _I32]),
    "attn_workspace_init": (ctypes.c_int, [_P, _SZ, _P]),
    "attn_kv_append": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _I32, _I32, _KV, _P, _SZ, _P]),
    "attn_prefill": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _I32, _I32, _I32, _KV, _P, _P, _SZ, _P]),
    "attn_decode": (ctypes.c_int, [_CFG, _P, _P, _P, _I32, _I32, _KV, _P, _P, _SZ, _P]),
    "attn_prefill_prepare": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _I32, _I32, _KV, _P, _P, _SZ, _P]),
    "attn_prefill_attend": (ctypes.c_int, [_CFG, _P, _P, _I32, _I32, _I32, _KV, _P, _P, _SZ, _P]),
    "attn_decode_attend": (ctypes.c_int, [_CFG, _P, _P, _I32, _I32, _KV, _P, _P, _SZ, _P]),
    "attn_decode_static_scratch": (ctypes.c_int, [_CFG, _P, _P, _P, _I32, _I32, _KV, _P, _P, _P]),
    "attn_decode_splits": (_I32, [_CFG, _I32, _I32]),
    "attn_qkv_proj_prepare": (ctypes.c_int, [_CFG, _P, _I32, _P, _P, _P, _P, _I32, _I32, _KV, _P, _P, _SZ, _P]),
    "attn_o_proj": (ctypes.c_int, [_CFG, _P, _I32, _P, _I32, _P, _P, _SZ, _P]),
    "attn_get_status": (ctypes.c_int, [_P, _P, ctypes.POINTER(ctypes.c_int32)]),
    "attn_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "attn_sample_tokens": (ctypes.c_int, [_P, _I32, _I32, ctypes.c_int64, _P, _P, _P, _P, _P, _P]),
}


def load(path: str = LIB_PATH):
    """Load libattn.so and declare its exports (raises if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built: run causal_gqa_attention_qkv_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(rc: int) -> None:
    if rc != 0:
        raise AttnError(rc, load().attn_strerror(rc).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# The current stream's handle without building a torch Stream object per call
# (a few microseconds on every launch); torch.cuda.current_stream() otherwise.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream=None):
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    if _raw_stream is not None:
        return ctypes.c_void_p(_raw_stream(torch.cuda.current_device()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def config(num_q_heads: int, num_kv_heads: int, head_dim: int, rms_eps: float = 1e-6,
           rope_theta: float = 1e6) -> AttnConfig:
    return AttnConfig(num_q_heads, num_kv_heads, head_dim, rms_eps, rope_theta)


@dataclasses.dataclass
class KVCache:
    """Device tensors of one layer's KV cache (see attn_kv_t)."""

    k_cache: torch.Tensor       # bf16, or uint8 E4M3 codes, [num_slots, Hkv, D]
    v_cache: torch.Tensor       # same type and shape as k_cache
    slot_base: torch.Tensor     # int64 [B] (contiguous layout)
    cache_lens: torch.Tensor    # int32 [B]
    slot_capacity: torch.Tensor  # int32 [B]
    page_table: torch.Tensor | None = None  # int32 [B, pages_per_req] (paged layout)
    page_size: int = 0
    k_scale: float = 1.0        # E4M3 caches: entry = code * scale
    v_scale: float = 1.0

    # The C struct is built (and the tensors checked) once and rebuilt when a
    # field is assigned; tensors changed in place (resize_, set_) are not seen.
    def __setattr__(self, name, value):
        object.__setattr__(self, name, value)
        if name != "_built":
            object.__setattr__(self, "_built", None)

    def struct(self) -> AttnKV:
        built = self.__dict__.get("_built")
        if built is None:
            built = self._make_struct()
            object.__setattr__(self, "_built", built)
        return built

    def _make_struct(self) -> AttnKV:
        fp8 = self.k_cache.dtype == torch.uint8
        for name in ("k_cache", "v_cache"):
            t = getattr(self, name)
            assert t.dtype == (torch.uint8 if fp8 else torch.bfloat16), name
            assert t.is_contiguous() and t.is_cuda, name
        assert self.slot_base.dtype == torch.int64 and self.slot_base.is_contiguous()
        assert self.cache_lens.dtype == torch.int32 and self.cache_lens.is_contiguous()
        assert self.slot_capacity.dtype == torch.int32 and self.slot_capacity.is_contiguous()
        pt, ps, ppr = None, 0, 0
        if self.page_table is not None:
            assert self.page_table.dtype == torch.int32 and self.page_table.is_contiguous()
            assert self.page_table.dim() == 2
            pt, ps, ppr = self.page_table.data_ptr(), int(self.page_size), int(self.page_table.shape[1])
        return AttnKV(self.k_cache.data_ptr(), self.v_cache.data_ptr(), self.k_cache.shape[0],
                      self.slot_base.data_ptr(), self.cache_lens.data_ptr(),
                      self.slot_capacity.data_ptr(), pt, ps, ppr,
                      ATTN_KV_E4M3 if fp8 else ATTN_KV_BF16, float(self.k_scale), float(self.v_scale))


def decode_splits(cfg: AttnConfig, B: int, max_cache_len: int) -> int:
    """Number of KV splits attn_decode uses for its longest request (the
    library's own policy, attn_decode_splits)."""
    n = load().attn_decode_splits(ctypes.byref(cfg), int(B), int(max_cache_len))
    if n < 0:
        raise AttnError(int(n), load().attn_strerror(int(n)).decode())
    return int(n)


def workspace_size(cfg: AttnConfig, max_tokens: int, max_batch: int, max_kv_len: int) -> int:
    n = load().attn_workspace_size(ctypes.byref(cfg), max_tokens, max_batch, max_kv_len)
    if n == 0:
        raise AttnError(-1, "invalid workspace query")
    return int(n)


def new_workspace(cfg: AttnConfig, max_tokens: int, max_batch: int, max_kv_len: int,
                  device="cuda") -> torch.Tensor:
    """Allocate (with torch) and initialise a workspace."""
    n = workspace_size(cfg, max_tokens, max_batch, max_kv_len)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    _check(load().attn_workspace_init(_ptr(ws), n, _stream()))
    return ws


def _bf16(t, name):
    assert t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous(), name
    return _ptr(t)


def kv_append(cfg: AttnConfig, qkv, k_norm_w, cu_seqlens, kv: KVCache, workspace, stream=None):
    B = cu_seqlens.numel() - 1
    s = kv.struct()
    _check(load().attn_kv_append(ctypes.byref(cfg), _bf16(qkv, "qkv"), None, _bf16(k_norm_w, "k_norm_w"),
                                 _ptr(cu_seqlens), B, qkv.shape[0], ctypes.byref(s), _ptr(workspace),
                                 workspace.numel(), _stream(stream)))


def prefill(cfg: AttnConfig, qkv, q_norm_w, k_norm_w, cu_seqlens, max_seqlen: int, kv: KVCache,
            out, workspace, stream=None):
    assert cu_seqlens.dtype == torch.int32 and cu_seqlens.is_cuda
    B = cu_seqlens.numel() - 1
    s = kv.struct()
    _check(load().attn_prefill(ctypes.byref(cfg), _bf16(qkv, "qkv"), _bf16(q_norm_w, "q_norm_w"),
                               _bf16(k_norm_w, "k_norm_w"), _ptr(cu_seqlens), B, qkv.shape[0],
                               int(max_seqlen), ctypes.byref(s), _bf16(out, "out"), _ptr(workspace),
                               workspace.numel(), _stream(stream)))


def decode(cfg: AttnConfig, qkv, q_norm_w, k_norm_w, max_cache_len: int, kv: KVCache, out,
           workspace, stream=None):
    B = qkv.shape[0]
    s = kv.struct()
    _check(load().attn_decode(ctypes.byref(cfg), _bf16(qkv, "qkv"), _bf16(q_norm_w, "q_norm_w"),
                              _bf16(k_norm_w, "k_norm_w"), B, int(max_cache_len), ctypes.byref(s),
                              _bf16(out, "out"), _ptr(workspace), workspace.numel(), _stream(stream)))


def prefill_prepare(cfg: AttnConfig, qkv, q_norm_w, k_norm_w, cu_seqlens, kv: KVCache, q_out,
                    workspace, stream=None):
    """First half of ``prefill``: K/V appended to the cache, prepared Q
    (normed, rotated, bf16 [N, Hq, D]) written to ``q_out``."""
    B = cu_seqlens.numel() - 1
    s = kv.struct()
    _check(load().attn_prefill_prepare(ctypes.byref(cfg), _bf16(qkv, "qkv"), _bf16(q_norm_w, "q_norm_w"),
                                       _bf16(k_norm_w, "k_norm_w"), _ptr(cu_seqlens), B, qkv.shape[0],
                                       ctypes.byref(s), _bf16(q_out, "q_out"), _ptr(workspace),
                                       workspace.numel(), _stream(stream)))


def prefill_attend(cfg: AttnConfig, q, cu_seqlens, max_seqlen: int, kv: KVCache, out, workspace,
                   stream=None):
    """Second half of ``prefill``: attention over the prepared Q ``q``
    [N, Hq, D] (the cache already holds the new K/V)."""
    B = cu_seqlens.numel() - 1
    s = kv.struct()
    _check(load().attn_prefill_attend(ctypes.byref(cfg), _bf16(q, "q"), _ptr(cu_seqlens), B, q.shape[0],
                                      int(max_seqlen), ctypes.byref(s), _bf16(out, "out"), _ptr(workspace),
                                      workspace.numel(), _stream(stream)))


def decode_attend(cfg: AttnConfig, qkv, q_norm_w, max_cache_len: int, kv: KVCache, out, workspace,
                  stream=None):
    """Attention half of ``decode`` (the cache already holds the new K/V)."""
    s = kv.struct()
    _check(load().attn_decode_attend(ctypes.byref(cfg), _bf16(qkv, "qkv"), _bf16(q_norm_w, "q_norm_w"),
                                     qkv.shape[0], int(max_cache_len), ctypes.byref(s), _bf16(out, "out"),
                                     _ptr(workspace), workspace.numel(), _stream(stream)))


def decode_static_scratch(cfg: AttnConfig, qkv, q_norm_w, k_norm_w, max_cache_len: int, kv: KVCache,
                          out, device_status=None, stream=None):
    """``decode`` with the split-KV scratch in the library's static device
    buffer (no workspace; for callers that cannot allocate)."""
    s = kv.struct()
    _check(load().attn_decode_static_scratch(
        ctypes.byref(cfg), _bf16(qkv, "qkv"), _bf16(q_norm_w, "q_norm_w"), _bf16(k_norm_w, "k_norm_w"),
        qkv.shape[0], int(max_cache_len), ctypes.byref(s), _bf16(out, "out"), _ptr(device_status),
        _stream(stream)))


def qkv_proj_prepare(cfg: AttnConfig, hidden, w_qkv, q_norm_w, k_norm_w, cu_seqlens, kv: KVCache, q_out,
                     workspace, stream=None):
    """The merged Q/K/V projection fused with ``prefill_prepare``: qkv =
    hidden [N, C] . w_qkv^T in fp32, then Q/K norm + RoPE, K/V appended,
    prepared Q written to ``q_out`` [N, Hq, D]."""
    assert hidden.dim() == 2 and w_qkv.dim() == 2 and w_qkv.shape[1] == hidden.shape[1]
    B = cu_seqlens.numel() - 1
    s = kv.struct()
    _check(load().attn_qkv_proj_prepare(ctypes.byref(cfg), _bf16(hidden, "hidden"), hidden.shape[1],
                                        _bf16(w_qkv, "w_qkv"), _bf16(q_norm_w, "q_norm_w"),
                                        _bf16(k_norm_w, "k_norm_w"), _ptr(cu_seqlens), B, hidden.shape[0],
                                        ctypes.byref(s), _ptr(q_out), _ptr(workspace), workspace.numel(),
                                        _stream(stream)))


def o_proj(cfg: AttnConfig, attn_out, w_o, out, workspace, stream=None):
    """out [N, C] = attn_out [N, Hq*D] . w_o^T (w_o [C, Hq*D])."""
    assert w_o.dim() == 2 and out.shape == (attn_out.shape[0], w_o.shape[0])
    _check(load().attn_o_proj(ctypes.byref(cfg), _bf16(attn_out, "attn_out"), attn_out.shape[0],
                              _bf16(w_o, "w_o"), w_o.shape[0], _bf16(out, "out"), _ptr(workspace),
                              workspace.numel(), _stream(stream)))


def get_status(workspace, stream=None) -> int:
    st = ctypes.c_int32(0)
    _check(load().attn_get_status(_ptr(workspace), _stream(stream), ctypes.byref(st)))
    return int(st.value)


def sample_tokens(logits, temperature, top_k, top_p, uniform, tokens=None, stream=None):
    """One token per row of fp32 logits [B, V] (include/sample.h): greedy where
    temperature <= 0, else temperature + top-k + top-p, sampled with the row's
    uniform number.  Returns the int32 [B] device tensor of tokens."""
    assert logits.dtype == torch.float32 and logits.is_cuda and logits.dim() == 2 and logits.stride(1) == 1
    B, V = logits.shape
    for t, dt in ((temperature, torch.float32), (top_k, torch.int32), (top_p, torch.float32),
                  (uniform, torch.float32)):
        assert t.dtype == dt and t.is_cuda and t.is_contiguous() and t.numel() == B
    if tokens is None:
        tokens = torch.empty(B, dtype=torch.int32, device=logits.device)
    _check(load().attn_sample_tokens(_ptr(logits), B, V, logits.stride(0), _ptr(temperature), _ptr(top_k),
                                     _ptr(top_p), _ptr(uniform), _ptr(tokens), _stream(stream)))
    return tokens
