"""Seeded synthetic inputs for the attention step.

This module only draws random numbers and lays them out; it holds none of the
step's arithmetic (no norm, no rotation, no attention).  The CUDA path and the
CPU oracle are both fed from the host tensors it returns, so that the two see
bit-identical inputs.

Layouts (all row-major, host tensors on the CPU):

* ``qkv``            bf16 ``[N, (Hq + 2*Hkv) * D]`` -- the packed output of the
  merged Q/K/V projection for the N tokens of one call (zero-to-sglang Ch.3
  code walkthrough, section 3.1 "packed [N, C]" and section 3.3 ``qkv_proj``).
  Columns ``[0, Hq*D)`` are Q, then ``Hkv*D`` columns of K, then of V; each
  head's D values are contiguous.
* ``q_norm_w``/``k_norm_w`` bf16 ``[D]`` -- the learned RMSNorm weights shared by
  all Q (resp. K) heads, drawn as ``1 + 0.1 * N(0, 1)``.
* ``cu_seqlens`` int32 ``[B + 1]`` -- prefix sums of the new-token counts.
* ``cache_lens`` int32 ``[B]`` -- entries already cached per request.
* ``slot_base`` int64 ``[B]``, ``slot_capacity`` int32 ``[B]`` -- each request owns
  the contiguous slots ``[slot_base, slot_base + slot_capacity)`` of one pool.
* ``k_cache``/``v_cache`` bf16 ``[num_slots, Hkv, D]`` -- the pool.  The first
  ``cache_lens[b]`` slots of request b hold N(0, 1) values (taken as already
  normed and rotated keys); every other slot (the rest of each region and the
  guard slots between regions) holds ``unused_fill`` so that a stray read or
  write is visible.
* With ``kv_dtype="e4m3"`` the pool is uint8 ``[num_slots, Hkv, D]`` of E4M3
  codes with one scale per cache (``k_scale``, ``v_scale``): the cached
  entries are N(0, 1) values divided by the scale and cast with torch's own
  ``float8_e4m3fn`` conversion; the unused fill is the E4M3 NaN code or a
  finite sentinel code.
"""
from __future__ import annotations

import dataclasses
from typing import Sequence

import torch

# bf16 bit patterns used to fill slots that no valid read may touch.
BF16_QNAN_BITS = 0x7FC0
BF16_SENTINEL_BITS = 0x4B3D  # a finite, distinctive value (12.3125 * 2**10)

GUARD_SLOTS = 3  # slots between two requests' regions, never written

# E4M3 codes for the same purpose, and the default scales of a one-byte cache
# (normed keys and N(0, 1) values stay well inside +-448 * scale).
E4M3_NAN_BITS = 0x7F
E4M3_SENTINEL_BITS = 0x5B  # a finite, distinctive code (22.0)
E4M3_K_SCALE = 0.04
E4M3_V_SCALE = 0.02


@dataclasses.dataclass(frozen=True)
class Workload:
    """One packed call (or a prefill call followed by a decode call).

    Requests ``[0, decode_from)`` go through ``attn_prefill`` and requests
    ``[decode_from, B)`` (each with exactly one new token) through
    ``attn_decode``.
    """

    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    new_lens: tuple
    cache_lens: tuple
    seed: int
    decode_from: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6

    @property
    def batch(self) -> int:
        return len(self.new_lens)

    @property
    def num_tokens(self) -> int:
        return int(sum(self.new_lens))

    @property
    def qkv_width(self) -> int:
        return (self.num_q_heads + 2 * self.num_kv_heads) * self.head_dim

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def attended_pairs(self, lo: int = 0, hi: int | None = None) -> int:
        """Unmasked (query, key) pairs of requests [lo, hi), diagonal included."""
        hi = self.batch if hi is None else hi
        total = 0
        for n, c in zip(self.new_lens[lo:hi], self.cache_lens[lo:hi]):
            # query j (0-based) at position c + j sees c + j + 1 keys
            total += n * c + n * (n + 1) // 2
        return total


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def tiny() -> Workload:
    """T=12 prompt, Hq=4, Hkv=2, D=64, empty cache; a decode step follows."""
    return Workload("tiny_T12_hq4_hkv2_d64", 4, 2, 64, (12,), (0,), seed=0, decode_from=1)


def qwen3_4b_prefill() -> Workload:
    """8 packed sequences with lengths U[256, 2048], Hq=32, Hkv=8, D=128."""
    g = _gen(1)
    lens = torch.randint(256, 2049, (8,), generator=g).tolist()
    return Workload("qwen3_4b_prefill_8seq_U256_2048", 32, 8, 128, tuple(lens), (0,) * 8, seed=1,
                    decode_from=8)


def decode_batch() -> Workload:
    """64 requests with one new token each, cached lengths U[512, 8192]."""
    g = _gen(2)
    cl = torch.randint(512, 8193, (64,), generator=g).tolist()
    return Workload("decode_b64_cache_U512_8192", 32, 8, 128, (1,) * 64, tuple(cl), seed=2,
                    decode_from=0)


def long_prefill() -> Workload:
    """One 32768-token sequence, Hq=64, Hkv=8 (group 8), D=128."""
    return Workload("long_prefill_T32768_hq64_hkv8", 64, 8, 128, (32768,), (0,), seed=3,
                    decode_from=1)


def mixed_step() -> Workload:
    """4 chunks of 1024 tokens with prior cache U[0, 4096] plus 256 decode
    rows with cached lengths U[1024, 16384], all packed in one qkv."""
    g = _gen(4)
    chunk_c = torch.randint(0, 4097, (4,), generator=g).tolist()
    dec_c = torch.randint(1024, 16385, (256,), generator=g).tolist()
    return Workload("mixed_4x1024chunks_256decode", 32, 8, 128, (1024,) * 4 + (1,) * 256,
                    tuple(chunk_c + dec_c), seed=4, decode_from=4)


def custom(name: str, hq: int, hkv: int, d: int, new_lens: Sequence[int],
           cache_lens: Sequence[int], seed: int, decode_from: int | None = None) -> Workload:
    """A workload of arbitrary shape (tests: ragged tails, edge cases)."""
    new_lens = tuple(int(x) for x in new_lens)
    cache_lens = tuple(int(x) for x in cache_lens)
    if decode_from is None:
        decode_from = len(new_lens)
    return Workload(name, hq, hkv, d, new_lens, cache_lens, seed=seed, decode_from=decode_from)


ALL = {w.name: w for w in (tiny(), qwen3_4b_prefill(), decode_batch(), long_prefill(), mixed_step())}


def _bf16_normal(g: torch.Generator, shape, scale: float = 1.0, shift: float = 0.0) -> torch.Tensor:
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    if shift != 0.0:
        x.add_(shift)
    return x.to(torch.bfloat16)


def _fill_bits(t: torch.Tensor, bits: int) -> None:
    t.view(torch.int16).fill_(bits if bits < 0x8000 else bits - 0x10000)


def _e4m3_codes(x: torch.Tensor, scale: float) -> torch.Tensor:
    """uint8 E4M3 codes of x / scale (torch's conversion; inputs clamped to +-448)."""
    return (x / scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def make_inputs(w: Workload, extra_capacity: Sequence[int] | None = None,
                unused_fill: str = "nan", page_size: int = 0, kv_dtype: str = "bf16",
                k_scale: float = E4M3_K_SCALE, v_scale: float = E4M3_V_SCALE) -> dict:
    """Draw all inputs of one call of workload ``w`` (host tensors).

    ``extra_capacity[b]`` is the number of free slots left after request b's
    new tokens (default: one, so that one decode step can follow).
    ``unused_fill`` is ``"nan"`` (quiet-NaN bits) or ``"sentinel"``.
    ``page_size`` > 0 lays the cache out in pages of that many slots: request b
    gets ceil(capacity_b / page_size) pages drawn from a seeded random
    permutation of the pool (plus three pages no request owns), listed in
    ``page_table`` (int32 [B, max pages]; unused entries -1).  The logical
    contents (qkv, weights, prior cache entries by position) are the same as
    with the contiguous layout for the same workload.
    ``kv_dtype="e4m3"`` makes a one-byte cache (codes, ``k_scale``, ``v_scale``).
    """
    assert kv_dtype in ("bf16", "e4m3")
    fp8 = kv_dtype == "e4m3"
    g = _gen(1000 + w.seed)
    B, H, Hkv, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    N = w.num_tokens
    qkv = _bf16_normal(g, (N, w.qkv_width))
    q_w = _bf16_normal(g, (D,), 0.1, 1.0)
    k_w = _bf16_normal(g, (D,), 0.1, 1.0)
    if extra_capacity is None:
        extra_capacity = [1] * B
    cap = [w.cache_lens[b] + w.new_lens[b] + int(extra_capacity[b]) for b in range(B)]
    base, s = [], GUARD_SLOTS
    for b in range(B):
        base.append(s)
        s += cap[b] + GUARD_SLOTS
    num_slots = s
    page_table = None
    if page_size:
        npg = [(c + page_size - 1) // page_size for c in cap]
        total = sum(npg) + 3
        perm = torch.randperm(total, generator=_gen(5000 + w.seed)).tolist()
        page_table = torch.full((B, max(npg + [1])), -1, dtype=torch.int32)
        k = 0
        for b in range(B):
            page_table[b, :npg[b]] = torch.tensor(perm[k:k + npg[b]], dtype=torch.int32)
            k += npg[b]
        num_slots = total * page_size
        base = [0] * B
    if fp8:
        k_cache = torch.full((num_slots, Hkv, D), E4M3_NAN_BITS if unused_fill == "nan" else E4M3_SENTINEL_BITS,
                             dtype=torch.uint8)
        v_cache = k_cache.clone()
    else:
        k_cache = torch.empty((num_slots, Hkv, D), dtype=torch.bfloat16)
        v_cache = torch.empty((num_slots, Hkv, D), dtype=torch.bfloat16)
        bits = BF16_QNAN_BITS if unused_fill == "nan" else BF16_SENTINEL_BITS
        _fill_bits(k_cache, bits)
        _fill_bits(v_cache, bits)
    for b in range(B):
        c = w.cache_lens[b]
        if c:
            kp, vp = _bf16_normal(g, (c, Hkv, D)), _bf16_normal(g, (c, Hkv, D))
            if fp8:
                kp, vp = _e4m3_codes(kp.float(), k_scale), _e4m3_codes(vp.float(), v_scale)
            if page_table is None:
                k_cache[base[b]:base[b] + c] = kp
                v_cache[base[b]:base[b] + c] = vp
            else:
                pos = torch.arange(c)
                slots = page_table[b, pos // page_size].long() * page_size + pos % page_size
                k_cache[slots] = kp
                v_cache[slots] = vp
    cu = [0]
    for n in w.new_lens:
        cu.append(cu[-1] + n)
    return {
        "qkv": qkv,
        "q_norm_w": q_w,
        "k_norm_w": k_w,
        "cu_seqlens": torch.tensor(cu, dtype=torch.int32),
        "cache_lens": torch.tensor(w.cache_lens, dtype=torch.int32),
        "slot_base": torch.tensor(base, dtype=torch.int64),
        "slot_capacity": torch.tensor(cap, dtype=torch.int32),
        "k_cache": k_cache,
        "v_cache": v_cache,
        "num_slots": num_slots,
        "page_table": page_table,
        "page_size": page_size,
        "kv_dtype": kv_dtype,
        "k_scale": float(k_scale),
        "v_scale": float(v_scale),
    }


def make_followup_decode_qkv(w: Workload) -> torch.Tensor:
    """qkv rows (one per request) of the decode step that follows a call of ``w``."""
    g = _gen(2000 + w.seed)
    return _bf16_normal(g, (w.batch, w.qkv_width))


def sample_rows(w: Workload, count: int, tail: int, seed: int) -> torch.Tensor:
    """(token, head) pairs to check at full size: every head of the last
    ``tail`` tokens of each request, plus ``count`` seeded random pairs.
    Returns int32 ``[R, 2]`` (unique, sorted)."""
    g = _gen(3000 + seed)
    rows = set()
    start = 0
    for n in w.new_lens:
        for t in range(max(start, start + n - tail), start + n):
            for h in range(w.num_q_heads):
                rows.add((t, h))
        start += n
    if count and w.num_tokens:
        toks = torch.randint(0, w.num_tokens, (count,), generator=g).tolist()
        heads = torch.randint(0, w.num_q_heads, (count,), generator=g).tolist()
        rows.update(zip(toks, heads))
    return torch.tensor(sorted(rows), dtype=torch.int32).reshape(-1, 2)


QWEN3_VOCAB = 151936


def make_sampling_inputs(B: int, V: int = QWEN3_VOCAB, seed: int = 0, greedy_share: float = 0.1) -> dict:
    """Seeded logits and per-row sampling parameters (host tensors).

    Logits are fp32 ``[B, V]``: N(0, 1) * 2 for every token plus, per row, 1-8
    candidate tokens raised by U[4, 12] (the peaked shape of a language-model
    head's output; no trained weights).  Per row: temperature from {0.3, 0.7,
    1.0, 1.5} (0 = greedy for about ``greedy_share`` of the rows), top_k from
    {0 (none), 1, 20, 50, 2000}, top_p from {1.0 (none), 0.95, 0.9, 0.5},
    uniform in [0, 1).
    """
    g = _gen(7000 + seed)
    logits = torch.randn((B, V), generator=g, dtype=torch.float32) * 2.0
    for b in range(B):
        n = int(torch.randint(1, 9, (1,), generator=g))
        idx = torch.randint(0, V, (n,), generator=g)
        logits[b, idx] += 4.0 + 8.0 * torch.rand(n, generator=g)
    pick = lambda vals: torch.tensor(vals)[torch.randint(0, len(vals), (B,), generator=g)]
    temperature = pick([0.3, 0.7, 1.0, 1.5]).float()
    temperature[torch.rand(B, generator=g) < greedy_share] = 0.0
    return {
        "logits": logits,
        "temperature": temperature,
        "top_k": pick([0, 1, 20, 50, 2000]).to(torch.int32),
        "top_p": pick([1.0, 0.95, 0.9, 0.5]).float(),
        "uniform": torch.rand(B, generator=g, dtype=torch.float32),
    }


QWEN3_4B_HIDDEN = 2560


def make_projection_inputs(w: Workload, hidden: int = QWEN3_4B_HIDDEN, seed: int = 0) -> dict:
    """Seeded hidden states and random projection weights around the step
    (host bf16 tensors; no trained weights): ``hidden`` ``[N, C]`` N(0, 1),
    ``w_qkv`` ``[(Hq+2Hkv)*D, C]`` and ``w_o`` ``[C, Hq*D]`` N(0, 1/fan_in), so
    that the projected qkv has about unit variance like the step's own qkv."""
    g = _gen(8000 + seed)
    N, C = w.num_tokens, hidden
    return {
        "hidden": _bf16_normal(g, (N, C)),
        "w_qkv": _bf16_normal(g, (w.qkv_width, C), C ** -0.5),
        "w_o": _bf16_normal(g, (C, w.num_q_heads * w.head_dim), (w.num_q_heads * w.head_dim) ** -0.5),
    }
