"""CPU fp64 oracle of the causal GQA attention step (qkv split, Q/K RMSNorm,
RoPE, KV append, causal grouped-query attention).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
product path never imports it and shares no code with it; the arithmetic
lives in ``oracle.c`` (plain C, fp64, OpenMP over rows) and is described, with
the passages it follows, in that file's header.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force from the teaching snippet, closed forms, torch's ``rms_norm``,
the complex form of RoPE, invariants; the E4M3 codec against torch's
``float8_e4m3fn`` for every code and for ties; sampling against closed-form
distributions, scipy's softmax and its limits).  The RoPE pairing convention
itself (rotate-half) is a reading the pages leave open: parity unpinned for
that choice, pinned for everything given it.  So is the one-byte cache
format (E4M3, one scale per cache, code of fp32(x) * fp32(1/scale)): the
pages name no format; pinned given that reading.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_D = ctypes.c_double
_F = ctypes.c_float


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (IEEE fp64, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call([
            "gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
            "-shared", "-fPIC", "-o", tmp, _SRC, "-lm",
        ])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.oracle_bf16_round.restype = ctypes.c_uint16
        lib.oracle_bf16_round.argtypes = [_D]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [_D]
        lib.oracle_e4m3_decode.restype = _D
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_rmsnorm.restype = None
        lib.oracle_rmsnorm.argtypes = [_P, _P, ctypes.c_int, _D, _P]
        lib.oracle_rope.restype = None
        lib.oracle_rope.argtypes = [_P, ctypes.c_int, _D, _D]
        lib.oracle_prologue.restype = ctypes.c_int
        lib.oracle_prologue.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, _D, _D,
            _P, _I64, _P, _P, ctypes.c_int, _P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_int,
            _I64, _P, _P, ctypes.c_int, _F, _F, _I64, _P, _P, _P]
        lib.oracle_prologue_projected.restype = ctypes.c_int
        lib.oracle_prologue_projected.argtypes = lib.oracle_prologue.argtypes
        lib.oracle_linear.restype = None
        lib.oracle_linear.argtypes = [_I64, _I64, _I64, _P, _P, _P]
        lib.oracle_attention.restype = None
        lib.oracle_attention.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, ctypes.c_int, _F, _F, ctypes.c_int, _P,
            _P, _P, _P, ctypes.c_int, ctypes.c_int, _I64, _P, _P, _P, _P]
        lib.oracle_sample.restype = _I64
        lib.oracle_sample.argtypes = [_I64, _P, _D, _I64, _D, _D, ctypes.POINTER(_D)]
        lib.oracle_sample_bracket.restype = ctypes.c_int
        lib.oracle_sample_bracket.argtypes = [_I64, _P, _D, _I64, _D, _I64, ctypes.POINTER(_D),
                                              ctypes.POINTER(_D)]
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    return _load().oracle_num_threads()


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_P)


def _bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> contiguous uint16 array of its bits (a copy)."""
    assert t.dtype == torch.bfloat16
    return np.array(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16), copy=True)


def _bits_view(t: torch.Tensor) -> np.ndarray:
    """bf16 CPU tensor -> uint16 array sharing its memory (read-only use)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def _cache_copy(t: torch.Tensor) -> np.ndarray:
    """A cache tensor's entries as a new array: uint16 bf16 bits, or the
    uint8 E4M3 bytes of a one-byte cache."""
    if t.dtype == torch.uint8:
        return np.array(t.detach().cpu().contiguous().numpy(), copy=True)
    return _bits(t)


def _cache_view(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.uint8:
        return t.detach().cpu().contiguous().numpy()
    return _bits_view(t)


def _cache_tensor(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(a) if a.dtype == np.uint8 else bits_to_bf16(a)


def _kv_format(inputs: dict):
    """(kv_fp8, k_scale, v_scale) of the inputs' cache."""
    if inputs.get("kv_dtype", "bf16") == "e4m3":
        return 1, float(inputs["k_scale"]), float(inputs["v_scale"])
    return 0, 1.0, 1.0


def e4m3_encode(x: float) -> int:
    """The E4M3 code nearest to ``x`` (ties to even, magnitudes beyond 448
    clamped to 448)."""
    return int(_load().oracle_e4m3_encode(float(x)))


def e4m3_decode(b: int) -> float:
    return float(_load().oracle_e4m3_decode(int(b)))


def bf16_round(x: float) -> int:
    """Bits of the bf16 nearest to ``x`` (ties to even)."""
    return int(_load().oracle_bf16_round(float(x)))


def rmsnorm(x, w, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    y = np.empty_like(x)
    _load().oracle_rmsnorm(_ptr(x), _ptr(w), x.shape[-1], float(eps), _ptr(y))
    return y


def rope(x, pos: float, theta: float) -> np.ndarray:
    y = np.array(x, dtype=np.float64, copy=True)
    _load().oracle_rope(_ptr(y), y.shape[-1], float(pos), float(theta))
    return y


def _pages(inputs: dict):
    """(page table int32 [B, P] flattened, page size, P) of a paged cache, or a
    dummy table and page size 0 for the contiguous layout."""
    pt = inputs.get("page_table")
    if pt is None:
        return np.zeros(1, dtype=np.int32), 0, 0
    pt = np.ascontiguousarray(pt.numpy().astype(np.int32))
    return pt.reshape(-1), int(inputs["page_size"]), int(pt.shape[1])


def linear(x, w) -> np.ndarray:
    """y = x w^T in fp64: x ``[N, C]`` (bf16 tensor or float array), w bf16
    ``[O, C]`` (the linear layer's weight layout).  Returns fp64 ``[N, O]``."""
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().double().numpy()
    x = np.ascontiguousarray(x, dtype=np.float64)
    wb = _bits(w)
    N, C = x.shape
    O = wb.shape[0]
    assert wb.shape[1] == C
    y = np.zeros((N, O), dtype=np.float64)
    _load().oracle_linear(N, C, O, _ptr(x), _ptr(wb), _ptr(y))
    return y


def prologue(cfg: dict, inputs: dict, q_rows=None, qkv64=None):
    """Steps 1-4.  Returns (k_cache, v_cache, q, bad) where the caches are new
    tensors of the input caches' type (bf16, or uint8 E4M3 codes; the inputs
    are not modified), q is fp64 ``[N, Hq, D]`` (or
    ``[R, D]`` for the (token, head) pairs in ``q_rows``), and ``bad`` counts
    requests whose cache region is too small (they write nothing).

    ``qkv64`` (fp64 ``[N, (Hq+2Hkv)*D]``, e.g. from ``linear``) replaces the
    bf16 qkv: the projection's output enters the norm, the rotation and the
    cache without a bf16 rounding of its own."""
    lib = _load()
    Hq, Hkv, D = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    assert D <= 256 and D % 2 == 0 and Hq % Hkv == 0
    if qkv64 is not None:
        qkv = np.ascontiguousarray(qkv64, dtype=np.float64)
        fn = lib.oracle_prologue_projected
    else:
        qkv = _bits_view(inputs["qkv"])
        fn = lib.oracle_prologue
    N = qkv.shape[0]
    kc = _cache_copy(inputs["k_cache"])
    vc = _cache_copy(inputs["v_cache"])
    fp8, ks, vs = _kv_format(inputs)
    qw, kw = _bits(inputs["q_norm_w"]), _bits(inputs["k_norm_w"])
    cu = np.ascontiguousarray(inputs["cu_seqlens"].numpy().astype(np.int32))
    cl = np.ascontiguousarray(inputs["cache_lens"].numpy().astype(np.int32))
    sb = np.ascontiguousarray(inputs["slot_base"].numpy().astype(np.int64))
    cap = np.ascontiguousarray(inputs["slot_capacity"].numpy().astype(np.int32))
    pt, ps, ppr = _pages(inputs)
    B = cl.shape[0]
    if q_rows is None:
        nq = -1
        q = np.zeros((N, Hq, D), dtype=np.float64)
        qt = qh = np.zeros(1, dtype=np.int32)
    else:
        rows = np.ascontiguousarray(np.asarray(q_rows, dtype=np.int32).reshape(-1, 2))
        nq = rows.shape[0]
        qt = np.ascontiguousarray(rows[:, 0])
        qh = np.ascontiguousarray(rows[:, 1])
        q = np.zeros((nq, D), dtype=np.float64)
    bad = fn(Hq, Hkv, D, float(cfg["rms_eps"]), float(cfg["rope_theta"]),
                              _ptr(qkv), N, _ptr(qw), _ptr(kw), B, _ptr(cu), _ptr(cl), _ptr(sb),
                              _ptr(cap), _ptr(pt), ps, ppr, kc.shape[0], _ptr(kc), _ptr(vc), fp8, ks,
                              vs, nq, _ptr(qt), _ptr(qh), _ptr(q))
    return _cache_tensor(kc), _cache_tensor(vc), q, bad


def attention(cfg: dict, k_cache: torch.Tensor, v_cache: torch.Tensor, inputs: dict,
              rows, q: np.ndarray) -> np.ndarray:
    """Step 5 for the (token, head) pairs ``rows`` ([R, 2]) with their fp64
    queries ``q`` ([R, D]).  Returns fp64 ``[R, D]``."""
    lib = _load()
    Hq, Hkv, D = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
    R = rows.shape[0]
    tok = np.ascontiguousarray(rows[:, 0])
    head = np.ascontiguousarray(rows[:, 1])
    q = np.ascontiguousarray(q, dtype=np.float64).reshape(R, D)
    kc, vc = _cache_view(k_cache), _cache_view(v_cache)
    fp8, ks, vs = _kv_format(inputs)
    cu = np.ascontiguousarray(inputs["cu_seqlens"].numpy().astype(np.int32))
    cl = np.ascontiguousarray(inputs["cache_lens"].numpy().astype(np.int32))
    sb = np.ascontiguousarray(inputs["slot_base"].numpy().astype(np.int64))
    pt, ps, ppr = _pages(inputs)
    out = np.zeros((R, D), dtype=np.float64)
    lib.oracle_attention(Hq, Hkv, D, _ptr(kc), _ptr(vc), fp8, ks, vs, cl.shape[0], _ptr(cu), _ptr(cl),
                         _ptr(sb),
                         _ptr(pt), ps, ppr, R, _ptr(tok), _ptr(head), _ptr(q), _ptr(out))
    return out


def sample(logits, temperature, top_k, top_p, uniform):
    """Tokens chosen from rows of fp32 logits ``[B, V]`` (greedy for
    temperature <= 0; else temperature, top-k, top-p, inverse-CDF sampling in
    vocabulary order with ``uniform``).  Returns (tokens int64 [B], margins
    float64 [B]): a margin is the relative distance of the row's real-valued
    decisions from a boundary (inf for greedy rows)."""
    lib = _load()
    x = np.ascontiguousarray(np.asarray(logits, dtype=np.float32))
    B, V = x.shape
    toks = np.zeros(B, dtype=np.int64)
    margins = np.zeros(B, dtype=np.float64)
    m = _D()
    for b in range(B):
        toks[b] = lib.oracle_sample(V, x[b].ctypes.data_as(_P), float(temperature[b]), int(top_k[b]),
                                    float(top_p[b]), float(uniform[b]), ctypes.byref(m))
        margins[b] = m.value
    return toks, margins


def sample_bracket(logits_row, temperature, top_k, top_p, token):
    """(kept, lo, hi) for a non-greedy row: whether ``token`` survives the
    truncation and the range [lo, hi) of u that selects it."""
    x = np.ascontiguousarray(np.asarray(logits_row, dtype=np.float32))
    lo, hi = _D(), _D()
    kept = _load().oracle_sample_bracket(x.shape[0], x.ctypes.data_as(_P), float(temperature), int(top_k),
                                         float(top_p), int(token), ctypes.byref(lo), ctypes.byref(hi))
    return bool(kept), lo.value, hi.value


def all_rows(num_tokens: int, num_q_heads: int) -> np.ndarray:
    t = np.repeat(np.arange(num_tokens, dtype=np.int32), num_q_heads)
    h = np.tile(np.arange(num_q_heads, dtype=np.int32), num_tokens)
    return np.stack([t, h], axis=1)


def step(cfg: dict, inputs: dict, rows=None):
    """The whole step: prologue then attention for ``rows`` (default: every
    (token, head) pair, in [N, Hq] order).  Returns a dict with the updated
    caches, the rows and the fp64 outputs ``[R, D]``."""
    N = inputs["qkv"].shape[0]
    if rows is None:
        rows = all_rows(N, cfg["num_q_heads"])
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
    kc, vc, q, bad = prologue(cfg, inputs, q_rows=rows)
    out = attention(cfg, kc, vc, inputs, rows, q)
    return {"k_cache": kc, "v_cache": vc, "rows": rows, "out": out, "q": q, "bad": bad}


def projected_step(cfg: dict, inputs: dict, hidden, w_qkv, w_o):
    """The step with the projections either side of it: qkv = hidden w_qkv^T
    (fp64, not rounded), the step on every (token, head) row, then
    o = attention_out w_o^T.  hidden bf16 ``[N, C]``, w_qkv bf16
    ``[(Hq+2Hkv)*D, C]``, w_o bf16 ``[C, Hq*D]``.  Returns the step's dict
    plus ``qkv64`` and ``o`` (fp64 ``[N, C]``)."""
    N = hidden.shape[0]
    qkv64 = linear(hidden, w_qkv)
    rows = all_rows(N, cfg["num_q_heads"])
    kc, vc, q, bad = prologue(cfg, inputs, q_rows=rows, qkv64=qkv64)
    att = attention(cfg, kc, vc, inputs, rows, q)
    o = linear(att.reshape(N, -1), w_o)
    return {"k_cache": kc, "v_cache": vc, "rows": rows, "out": att, "q": q, "bad": bad, "qkv64": qkv64,
            "o": o}


def cfg_of(w) -> dict:
    """The per-call configuration of a workload (plain dict)."""
    return {"num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "rms_eps": w.rms_eps, "rope_theta": w.rope_theta}
