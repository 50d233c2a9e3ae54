"""Helpers shared by the GPU parity tests: run a workload through the C ABI
and compare outputs and caches with the CPU oracle."""
import numpy as np
import torch

import oracle

# Floating-point tolerance on bf16 outputs against the fp64 oracle: max-abs
# error and relative Frobenius error (fp32 accumulation, bf16 operands).
MAX_ABS = 2e-2
REL_FRO = 1e-2


def ordered_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 bits mapped to integers that are monotone in the value (so that
    adjacent representable values differ by one)."""
    u = t.contiguous().view(torch.int16).numpy().astype(np.int32) & 0xFFFF
    return np.where(u < 0x8000, u, 0x8000 - u)


def written_slots(host: dict, lo: int = 0, hi: int | None = None) -> np.ndarray:
    """Slots of the new tokens of requests lo..hi-1 (contiguous or paged layout)."""
    cl = host["cache_lens"].numpy()
    cu = host["cu_seqlens"].numpy()
    sb = host["slot_base"].numpy()
    pt = host.get("page_table")
    ps = int(host.get("page_size", 0))
    hi = len(cl) if hi is None else hi
    out = []
    for b in range(lo, hi):
        n = cu[b + 1] - cu[b]
        for pos in range(cl[b], cl[b] + n):
            out.append(sb[b] + pos if pt is None else int(pt[b, pos // ps]) * ps + pos % ps)
    return np.asarray(out, dtype=np.int64)


# K is computed in fp32 on the device and in fp64 by the oracle, then rounded
# to bf16 by both.  The device's fp32 error on an element of a rotation pair
# (y_i, y_j), j = i +- D/2, is at most K_FP32_REL * |(y_i, y_j)| (the pair's
# Euclidean norm, which the rotation preserves), from its operations with unit
# roundoff u = 2^-24:
#   sum of squares: two chains of 8 fused multiply-adds per lane, their sum,
#     then log2(D/16) shuffle adds: at most 12 roundings on any term, all
#     terms >= 0, so relative error <= 12u;
#   (ss / D + eps) one rounding, rsqrtf <= 2 ulp (4u) as CUDA documents it:
#     the inverse norm within 12u / 2 + u / 2 + 4u = 10.5u;
#   x * inv, then * w: two roundings, so y within 12.5u relative;
#   rotation fma(y_j, +-sin, y_i * cos): two roundings, and cos / sin with
#     absolute error <= 9.2e-7 (angle: three fp32 roundings of a reduced
#     angle |r| <= pi, 3 * pi * u = 5.6e-7; __sincosf on [-pi, pi]: 2^-21.41
#     = 3.6e-7 as CUDA documents it).
# Total <= (14.5u + 9.2e-7) * (|y_i| + |y_j|) <= 1.78e-6 * sqrt(2) * |pair|
# = 21.2 * 2^-23 * |pair|; the constant is taken as 22 * 2^-23.  The pair norm
# is estimated from the oracle's bf16 values, which are within 2^-8 of the
# exact ones (covered by the rounding up from 21.2 to 22).  So a written K
# element may differ from the oracle's by half a bf16 step of each side plus
# that error: one step where the exact value sits next to a rounding tie, more
# only where the pair is much larger than the element itself.
K_FP32_REL = 22 * 2.0 ** -23
K_MAX_MISMATCH_FRACTION = 1e-2


def bf16_step(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (normal range)."""
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 7)


def e4m3_order(codes: np.ndarray) -> np.ndarray:
    """E4M3 codes (sign-magnitude) mapped to integers monotone in the value:
    neighbouring codes differ by one, +0 and -0 both map to 0."""
    c = codes.astype(np.int32)
    return np.where(c < 0x80, c, -(c & 0x7F))


def check_caches_e4m3(host: dict, ref: dict, k_gpu: torch.Tensor, v_gpu: torch.Tensor) -> None:
    """One-byte caches: V codes bit-exact everywhere (both sides code the same
    fp32 product); K codes at most one code apart on the written slots (the
    device's fp32 K differs from the correctly rounded one by a few fp32 ulps,
    which moves a value across a rounding boundary only when it sits next to
    one) and unchanged everywhere else."""
    kg, vg = k_gpu.cpu().numpy(), v_gpu.cpu().numpy()
    kr, vr = ref["k_cache"].numpy(), ref["v_cache"].numpy()
    assert np.array_equal(vg, vr), "V cache differs"
    slots = written_slots(host)
    mask = np.zeros(kg.shape[0], dtype=bool)
    mask[slots] = True
    assert np.array_equal(kg[~mask], kr[~mask]), "K cache changed outside the appended slots"
    if slots.size:
        d = np.abs(e4m3_order(kg[slots]) - e4m3_order(kr[slots]))
        assert d.max() <= 1, f"K codes {int(d.max())} apart"
        frac = float((d != 0).mean())
        assert frac <= K_MAX_MISMATCH_FRACTION, f"{frac:.3%} of K codes differ"


def check_caches(host: dict, ref: dict, k_gpu: torch.Tensor, v_gpu: torch.Tensor) -> None:
    """V bit-exact everywhere; K within the derived fp32 bound (half a bf16
    step of each side + K_FP32_REL * pair norm) on the written slots and
    bit-exact (unchanged) everywhere else."""
    if k_gpu.dtype == torch.uint8:
        return check_caches_e4m3(host, ref, k_gpu, v_gpu)
    k_gpu, v_gpu = k_gpu.cpu(), v_gpu.cpu()
    assert torch.equal(v_gpu.view(torch.int16), ref["v_cache"].view(torch.int16)), "V cache differs"
    slots = written_slots(host)
    mask = np.zeros(k_gpu.shape[0], dtype=bool)
    mask[slots] = True
    kg = k_gpu.view(torch.int16).numpy()
    kr = ref["k_cache"].view(torch.int16).numpy()
    assert np.array_equal(kg[~mask], kr[~mask]), "K cache changed outside the appended slots"
    if slots.size:
        idx = torch.from_numpy(slots)
        g = k_gpu[idx].float().numpy().astype(np.float64)
        r = ref["k_cache"][idx].float().numpy().astype(np.float64)
        err = np.abs(g - r)
        D = r.shape[-1]
        pair = np.hypot(r, np.roll(r, D // 2, axis=-1))  # element i with i +- D/2
        bound = 0.5 * bf16_step(g) + 0.5 * bf16_step(r) + K_FP32_REL * pair
        assert (err <= bound).all(), f"K off by {float((err / bound).max()):.2f} x the fp32 bound"
        frac = float((g != r).mean())
        assert frac <= K_MAX_MISMATCH_FRACTION, f"{frac:.3%} of K elements differ"


def check_out(out_rows: torch.Tensor, ref_out: np.ndarray, what: str = "") -> dict:
    got = out_rows.double().cpu().numpy()
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    diff = got - ref_out
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref_out), 1e-30)) if diff.size else 0.0
    assert max_abs <= MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {MAX_ABS}"
    assert rel <= REL_FRO, f"{what}: rel-Frobenius {rel:.3e} > {REL_FRO}"
    return {"max_abs": max_abs, "rel_fro": rel}


def gather_rows(out: torch.Tensor, w, rows: np.ndarray) -> torch.Tensor:
    o = out.view(w.num_tokens, w.num_q_heads, w.head_dim)
    t = torch.from_numpy(np.ascontiguousarray(rows[:, 0])).long().to(out.device)
    h = torch.from_numpy(np.ascontiguousarray(rows[:, 1])).long().to(out.device)
    return o[t, h]


def run_and_compare(w, host: dict, rows=None, check_cache: bool = True) -> dict:
    """Run workload w on the GPU through the C ABI and compare with the oracle
    on ``rows`` ((token, head) pairs; default every row)."""
    from causal_gqa_attention_qkv_gb300 import step

    ds = step.upload(w, host)
    ds.run()
    torch.cuda.synchronize()
    status = ds.status()
    assert status == 0, f"device status {status}"
    cfg = oracle.cfg_of(w)
    if rows is None:
        rows = oracle.all_rows(w.num_tokens, w.num_q_heads)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
    ref = oracle.step(cfg, host, rows=rows)
    stats = check_out(gather_rows(ds.out, w, rows), ref["out"], w.name)
    if check_cache:
        check_caches(host, ref, ds.k_cache, ds.v_cache)
    stats["rows"] = int(rows.shape[0])
    return {"stats": stats, "ds": ds, "ref": ref}
