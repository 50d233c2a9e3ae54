"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs.  Outputs: max-abs <= 2e-2 and relative Frobenius <= 1e-2
(bf16 outputs, fp32 accumulation); caches: V bit-exact, K within half a bf16
step of each side plus the derived fp32 error of the norm and rotation, every
slot outside the appended ones unchanged.  Full-size prefill workloads are
checked on every head of the last 256 positions of each sequence plus 2048
seeded random (token, head) rows."""
import numpy as np
import pytest
import torch

import oracle
from causal_gqa_attention_qkv_gb300 import inputs as gen
from parity_util import check_caches, check_out, gather_rows, run_and_compare, written_slots

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_gqa_attention_qkv_gb300 import build
    build.build()


def test_tiny_prefill_then_decode_cache_0_12_13():
    w = gen.tiny()
    host = gen.make_inputs(w)
    res = run_and_compare(w, host)
    ds = res["ds"]
    # decode step against the 12-entry cache the prefill left behind
    dw = gen.custom("tiny_decode", w.num_q_heads, w.num_kv_heads, w.head_dim, [1], [12], seed=0,
                    decode_from=0)
    dhost = dict(host, qkv=gen.make_followup_decode_qkv(w), cu_seqlens=torch.tensor([0, 1], dtype=torch.int32),
                 cache_lens=torch.tensor([12], dtype=torch.int32), k_cache=ds.k_cache.cpu(),
                 v_cache=ds.v_cache.cpu())
    r2 = run_and_compare(dw, dhost)
    base = int(host["slot_base"][0])
    # exactly slot base+12 changed in the decode step
    before = ds.k_cache.cpu().view(torch.int16)
    after = r2["ds"].k_cache.cpu().view(torch.int16)
    changed = (before != after).flatten(1).any(1).nonzero().flatten().tolist()
    assert changed == [base + 12]


RAGGED = [
    # (Hq, Hkv, D, new lens, cached lens)
    (8, 2, 128, [1, 17, 64, 100, 200], [0, 5, 0, 130, 37]),
    (8, 8, 64, [33, 2, 70], [0, 64, 1]),
    (16, 2, 64, [9, 130, 1], [3, 0, 200]),
    (8, 1, 128, [40, 65], [0, 300]),
    (32, 8, 128, [257, 31], [0, 100]),
]


@pytest.mark.parametrize("hq,hkv,d,lens,cache", RAGGED)
def test_ragged_prefill_all_rows(hq, hkv, d, lens, cache):
    w = gen.custom(f"ragged_{hq}_{hkv}_{d}", hq, hkv, d, lens, cache, seed=sum(lens) + hq)
    run_and_compare(w, gen.make_inputs(w))


DECODE = [
    (32, 8, 128, [0, 1, 63, 64, 65, 255, 256, 257, 1000, 3000]),
    (4, 2, 64, [0, 5, 511, 2047]),
    (16, 2, 128, [7, 129, 4000]),
    (8, 8, 64, [12, 300]),
]


@pytest.mark.parametrize("hq,hkv,d,cache", DECODE)
def test_decode_all_rows(hq, hkv, d, cache):
    w = gen.custom(f"decode_{hq}_{hkv}_{d}", hq, hkv, d, [1] * len(cache), cache, seed=len(cache) + d,
                   decode_from=0)
    run_and_compare(w, gen.make_inputs(w))


# Paged KV cache: the cache is pages of page_size slots listed per request in a
# page table (a seeded random permutation of the pool).  The same logical
# inputs must give the oracle's result and the same bits as the contiguous
# layout (the kernels' arithmetic does not depend on where an entry lives).
PAGED = [
    # (page size, Hq, Hkv, D, new lens, cached lens, decode_from)
    (64, 32, 8, 128, [300, 77, 513, 129], [0, 200, 64, 1000], 4),
    (128, 32, 8, 128, [300, 77, 513, 129], [0, 200, 64, 1000], 4),
    (256, 16, 2, 64, [130, 1, 65], [3, 0, 700], 3),
    (64, 32, 8, 128, [1] * 8, [0, 1, 63, 64, 65, 700, 3000, 5000], 0),
    (128, 8, 8, 64, [1] * 4, [12, 127, 128, 2047], 0),
    (64, 32, 8, 128, [100, 64, 1, 1, 1], [50, 0, 10, 700, 0], 2),
]


@pytest.mark.parametrize("ps,hq,hkv,d,lens,cache,df", PAGED)
def test_paged_cache_all_rows_and_same_bits_as_contiguous(ps, hq, hkv, d, lens, cache, df):
    w = gen.custom(f"paged_{ps}_{hq}_{d}_{df}", hq, hkv, d, lens, cache, seed=ps + sum(lens), decode_from=df)
    paged = run_and_compare(w, gen.make_inputs(w, page_size=ps))["ds"]
    from causal_gqa_attention_qkv_gb300 import step
    contiguous = step.upload(w, gen.make_inputs(w))
    contiguous.run()
    torch.cuda.synchronize()
    assert torch.equal(paged.out.view(torch.int16), contiguous.out.view(torch.int16))


# One-byte (E4M3) caches: the append codes K and V, decode reads the codes.
# Scales: the generator's defaults, a power of two, and one small enough that
# some K and V products pass 448 and are clamped.
E4M3_DECODE = [
    # (Hq, Hkv, D, cached lens, page size, k_scale, v_scale)
    (32, 8, 128, [0, 1, 63, 64, 65, 255, 256, 257, 1000, 3000], 0, 0.04, 0.02),
    (4, 2, 64, [0, 5, 511, 2047], 0, 0.04, 0.02),
    (16, 2, 128, [7, 129, 4000], 64, 2.0 ** -5, 2.0 ** -6),
    (8, 8, 64, [12, 300, 64], 128, 0.04, 0.02),
    (32, 8, 128, [33, 900], 0, 0.003, 0.004),
]


@pytest.mark.parametrize("hq,hkv,d,cache,ps,ks,vs", E4M3_DECODE)
def test_e4m3_cache_decode_all_rows(hq, hkv, d, cache, ps, ks, vs):
    w = gen.custom(f"e4m3_{hq}_{hkv}_{d}_{ps}", hq, hkv, d, [1] * len(cache), cache, seed=len(cache) + d + ps,
                   decode_from=0)
    host = gen.make_inputs(w, page_size=ps, kv_dtype="e4m3", k_scale=ks, v_scale=vs)
    res = run_and_compare(w, host)
    if ks == 0.003:  # some products passed 448 and were clamped (on both sides: the caches match)
        slots = written_slots(host)
        for name in ("k_cache", "v_cache"):
            assert ((res["ref"][name].numpy()[slots] & 0x7F) == 0x7E).any(), name


E4M3_PREFILL = [
    # (Hq, Hkv, D, new lens, cached lens, page size, decode_from)
    (32, 8, 128, [300, 77, 513, 129, 1], [0, 200, 64, 1000, 5], 0, 5),
    (16, 2, 64, [130, 1, 65, 257], [3, 0, 700, 128], 0, 4),
    (32, 8, 128, [300, 77, 513, 129], [0, 200, 64, 1000], 64, 4),
    (8, 8, 64, [200, 31], [64, 0], 128, 2),
    (16, 2, 64, [130, 1, 65], [3, 0, 700], 64, 3),    # D 64 over 64-slot pages: two 64-row boxes
    (32, 8, 128, [100, 64, 1, 1, 1], [50, 0, 10, 700, 0], 0, 2),
]


@pytest.mark.parametrize("hq,hkv,d,lens,cache,ps,df", E4M3_PREFILL)
def test_e4m3_cache_prefill_and_mixed_all_rows(hq, hkv, d, lens, cache, ps, df):
    """Prefill (and the decode rows of a mixed step) over a one-byte cache:
    the tiles are converted to f16 in shared memory; every row and both
    caches against the oracle."""
    w = gen.custom(f"e4m3p_{hq}_{hkv}_{d}_{ps}_{df}", hq, hkv, d, lens, cache, seed=sum(lens) + d + ps,
                   decode_from=df)
    run_and_compare(w, gen.make_inputs(w, page_size=ps, kv_dtype="e4m3"))


def test_e4m3_full_qwen3_4b_prefill_sampled():
    w = gen.qwen3_4b_prefill()
    run_and_compare(w, gen.make_inputs(w, kv_dtype="e4m3"), rows=_sampled(w, tail=64, count=4096, seed=5))


def test_e4m3_decode_static_scratch_matches_workspace_decode():
    from causal_gqa_attention_qkv_gb300 import attn, step
    w = gen.custom("e4m3_static", 32, 8, 128, [1] * 6, [5, 70, 700, 2000, 64, 4095], seed=91, decode_from=0)
    host = gen.make_inputs(w, kv_dtype="e4m3")
    a = step.upload(w, host)
    a.run()
    b = step.upload(w, host)
    attn.decode_static_scratch(b.cfg, b.qkv, b.q_norm_w, b.k_norm_w, b.max_cache_len, b.kv_decode, b.out)
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert torch.equal(a.k_cache, b.k_cache) and torch.equal(a.v_cache, b.v_cache)


@pytest.mark.parametrize("hq,hkv,d,cache,ps,kvd", [
    (32, 8, 128, [0, 5, 63, 64, 700, 3000, 9000], 0, "bf16"),   # several splits per request
    (4, 2, 64, [12, 300], 0, "bf16"),                          # one split: no merge
    (16, 2, 128, [7, 129, 4000], 64, "bf16"),                  # paged
    (32, 8, 128, [0, 5, 700, 3000, 9000], 0, "e4m3"),
    (8, 8, 64, [12, 300, 5000], 128, "e4m3"),
])
def test_decode_append_inside_equals_append_then_attend(hq, hkv, d, cache, ps, kvd):
    """attn_decode appends the new tokens' K/V inside the split kernel; the
    result must equal attn_kv_append followed by attn_decode_attend bit for
    bit (output and both caches), and match the oracle."""
    from causal_gqa_attention_qkv_gb300 import attn, step
    w = gen.custom(f"fused_{hq}_{hkv}_{d}_{ps}_{kvd}", hq, hkv, d, [1] * len(cache), cache,
                   seed=len(cache) * 7 + d + ps, decode_from=0)
    host = gen.make_inputs(w, page_size=ps, kv_dtype=kvd)
    a = step.upload(w, host)
    attn.decode(a.cfg, a.qkv, a.q_norm_w, a.k_norm_w, a.max_cache_len, a.kv_decode, a.out, a.workspace)
    b = step.upload(w, host)
    cu = torch.arange(len(cache) + 1, dtype=torch.int32, device=b.out.device)
    attn.kv_append(b.cfg, b.qkv, b.k_norm_w, cu, b.kv_decode, b.workspace)
    attn.decode_attend(b.cfg, b.qkv, b.q_norm_w, b.max_cache_len, b.kv_decode, b.out, b.workspace)
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    for x, y in ((a.k_cache, b.k_cache), (a.v_cache, b.v_cache)):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    ref = oracle.step(oracle.cfg_of(w), host)
    check_out(gather_rows(a.out, w, ref["rows"]), ref["out"], w.name)
    check_caches(host, ref, a.k_cache, a.v_cache)


def test_e4m3_full_decode_batch_all_rows():
    w = gen.decode_batch()
    run_and_compare(w, gen.make_inputs(w, kv_dtype="e4m3"))


def test_empty_calls_are_no_ops():
    """N = 0 and B = 0 calls return OK, write nothing and set no status.  The
    ABI wants valid pointers even then (a torch view with no elements reports
    address 0), so the library is called with the real buffers and zero sizes."""
    import ctypes
    from causal_gqa_attention_qkv_gb300 import attn, step
    w = gen.custom("empty_base", 8, 2, 128, [5], [3], seed=40)
    ds = step.upload(w, gen.make_inputs(w))
    k0, v0, o0 = ds.k_cache.clone(), ds.v_cache.clone(), ds.out.clone()
    lib, P, st = attn.load(), attn._ptr, attn._stream()
    cu = torch.zeros(2, dtype=torch.int32, device=ds.out.device)  # one request with no tokens
    ws, nws = P(ds.workspace), ds.workspace.numel()
    for kv in (ds.kv_prefill,):
        s = kv.struct()
        for B in (0, 1):
            assert lib.attn_prefill(ctypes.byref(ds.cfg), P(ds.qkv), P(ds.q_norm_w), P(ds.k_norm_w), P(cu), B, 0,
                                    0, ctypes.byref(s), P(ds.out), ws, nws, st) == 0
            assert lib.attn_kv_append(ctypes.byref(ds.cfg), P(ds.qkv), None, P(ds.k_norm_w), P(cu), B, 0,
                                      ctypes.byref(s), ws, nws, st) == 0
        assert lib.attn_decode(ctypes.byref(ds.cfg), P(ds.qkv), P(ds.q_norm_w), P(ds.k_norm_w), 0, 0,
                               ctypes.byref(s), P(ds.out), ws, nws, st) == 0
    torch.cuda.synchronize()
    assert ds.status() == 0
    assert torch.equal(k0.view(torch.int16), ds.k_cache.view(torch.int16))
    assert torch.equal(v0.view(torch.int16), ds.v_cache.view(torch.int16))
    assert torch.equal(o0.view(torch.int16), ds.out.view(torch.int16))


def test_zero_length_sequences_in_a_packed_batch():
    """Requests with no new tokens (cu_seqlens repeats a value) are skipped;
    the others are computed as usual."""
    w = gen.custom("zero_len", 32, 8, 128, [0, 37, 0, 1, 130, 0], [5, 0, 0, 200, 64, 9], seed=41)
    run_and_compare(w, gen.make_inputs(w))


@pytest.mark.parametrize("hq,hkv,d,lens,cache", [
    (128, 16, 128, [70, 130], [0, 40]),   # the most heads the ABI takes, group 8
    (128, 128, 64, [33, 65], [7, 0]),     # multi-head (group 1) at the head limit
])
def test_largest_head_counts(hq, hkv, d, lens, cache):
    w = gen.custom(f"heads_{hq}_{hkv}_{d}", hq, hkv, d, lens, cache, seed=hq + hkv + d)
    run_and_compare(w, gen.make_inputs(w))


@pytest.mark.parametrize("hq,hkv,d,lens,cache,kvd", [
    (8, 1, 64, [3000, 1999, 1], [0, 100, 7], "bf16"),    # 2 steps of 8 heads, the second K + V
    (6, 3, 128, [2500, 500], [0, 33], "bf16"),           # 3 steps of 4 heads, two of them mixed
    (6, 3, 128, [2500, 500], [0, 33], "e4m3"),
])
def test_prologue_runs_cut_across_tokens(hq, hkv, d, lens, cache, kvd):
    """Enough (token, step) units that the prologue's per-warp runs are cut
    across token boundaries (steps per token not dividing the run length),
    with steps that mix Q, K and V heads: every row and the caches."""
    w = gen.custom(f"runs_{hq}_{hkv}_{d}_{kvd}", hq, hkv, d, lens, cache, seed=sum(lens) + d)
    run_and_compare(w, gen.make_inputs(w, kv_dtype=kvd))


def test_mixed_prefill_and_decode_small():
    w = gen.custom("mixed_small", 32, 8, 128, [100, 64, 1, 1, 1], [50, 0, 10, 700, 0], seed=77,
                   decode_from=2)
    run_and_compare(w, gen.make_inputs(w))


def test_prefill_one_token_rows_equal_decode():
    # attn_prefill with n_b = 1 gives the decode result (same definition)
    cache = [5, 300, 1000]
    wp = gen.custom("p1", 16, 4, 128, [1, 1, 1], cache, seed=91, decode_from=3)
    wd = gen.custom("d1", 16, 4, 128, [1, 1, 1], cache, seed=91, decode_from=0)
    host = gen.make_inputs(wp)
    a = run_and_compare(wp, host)["ds"].out.cpu()
    b = run_and_compare(wd, host)["ds"].out.cpu()
    torch.testing.assert_close(a.float(), b.float(), rtol=0, atol=1.6e-2)


def test_deterministic_and_idempotent():
    w = gen.custom("det", 8, 2, 128, [150, 40], [20, 0], seed=5)
    host = gen.make_inputs(w)
    from causal_gqa_attention_qkv_gb300 import step
    ds = step.upload(w, host)
    ds.run()
    first = ds.out.clone()
    k1 = ds.k_cache.clone()
    ds.run()  # cache_lens not advanced: writes the same slots again
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), ds.out.view(torch.int16))
    assert torch.equal(k1.view(torch.int16), ds.k_cache.view(torch.int16))


def test_prefill_output_only_16_byte_aligned():
    """An output that starts 16 bytes past a 32-byte boundary (allowed by the
    ABI) gets the same bits as a 32-byte-aligned one."""
    from causal_gqa_attention_qkv_gb300 import attn, step
    w = gen.custom("align16", 32, 8, 128, [200, 33, 96], [0, 70, 0], seed=6)
    host = gen.make_inputs(w)
    ds = step.upload(w, host)
    ds.run()
    torch.cuda.synchronize()
    ref = ds.out.clone()
    n, width = ds.out.shape
    buf = torch.full((n * width + 16,), float("nan"), dtype=torch.bfloat16, device=ds.out.device)
    out = buf[8:8 + n * width].view(n, width)  # 16 bytes past the allocation start
    assert out.data_ptr() % 32 == 16
    attn.prefill(ds.cfg, ds.qkv, ds.q_norm_w, ds.k_norm_w, ds.cu_seqlens, ds.max_seqlen, ds.kv_prefill,
                 out, ds.workspace)
    torch.cuda.synchronize()
    assert ds.status() == 0
    assert torch.equal(ref.view(torch.int16), out.view(torch.int16))


def test_prefill_leaves_work_counters_zero():
    """The prefill attention kernel hands out work items through two counters
    in the workspace header (bytes 64..71) and must leave them at zero, so the
    next call on the same workspace starts from item 0."""
    w = gen.custom("counters", 16, 4, 128, [300, 77, 513], [0, 40, 0], seed=8)
    from causal_gqa_attention_qkv_gb300 import step
    ds = step.upload(w, gen.make_inputs(w))
    for _ in range(3):
        ds.run()
        torch.cuda.synchronize()
        header = ds.workspace[:256].view(torch.int32).cpu()
        assert int(header[16]) == 0 and int(header[17]) == 0, header[16:18].tolist()
    assert ds.status() == 0


def test_status_capacity_and_seqlens():
    from causal_gqa_attention_qkv_gb300 import attn, step
    w = gen.custom("cap", 8, 2, 64, [10, 6], [0, 4], seed=8)
    host = gen.make_inputs(w)
    host["slot_capacity"][1] = 9  # needs 4 + 6
    ds = step.upload(w, host)
    ds.run()
    assert ds.status() & attn.ATTN_STATUS_CAPACITY
    assert ds.status() == 0  # read-and-clear
    # request 1 wrote nothing; request 0 is intact
    ref = oracle.step(oracle.cfg_of(w), host)
    assert ref["bad"] == 1
    kc = ds.k_cache.cpu().view(torch.int16)
    b1 = int(host["slot_base"][1])
    assert torch.equal(kc[b1 + 4:b1 + 10], host["k_cache"][b1 + 4:b1 + 10].view(torch.int16))
    rows = oracle.all_rows(10, w.num_q_heads)
    check_out(gather_rows(ds.out, w, rows), ref["out"][:rows.shape[0]], "valid request")
    # cu_seqlens that do not end at N
    ds2 = step.upload(w, gen.make_inputs(w))
    ds2.cu_seqlens[-1] = 15
    ds2.run()
    assert ds2.status() & attn.ATTN_STATUS_SEQLENS


def test_abi_rejects_bad_arguments_on_device():
    from causal_gqa_attention_qkv_gb300 import attn, step
    w = gen.custom("args", 8, 2, 64, [4], [0], seed=9)
    ds = step.upload(w, gen.make_inputs(w))
    small_ws = ds.workspace[:128]
    with pytest.raises(attn.AttnError) as e:
        attn.prefill(ds.cfg, ds.qkv, ds.q_norm_w, ds.k_norm_w, ds.cu_seqlens, 4, ds.kv_prefill, ds.out,
                     small_ws)
    assert e.value.code == -3
    bad = attn.config(8, 3, 64)
    with pytest.raises(attn.AttnError) as e:
        attn.prefill(bad, ds.qkv, ds.q_norm_w, ds.k_norm_w, ds.cu_seqlens, 4, ds.kv_prefill, ds.out,
                     ds.workspace)
    assert e.value.code == -2


# ------------------------------------------------------------------ full sizes
def _sampled(w, tail, count, seed):
    return gen.sample_rows(w, count=count, tail=tail, seed=seed).numpy()


def test_full_tiny_config():
    w = gen.tiny()
    run_and_compare(w, gen.make_inputs(w))


def test_full_qwen3_4b_prefill():
    w = gen.qwen3_4b_prefill()
    run_and_compare(w, gen.make_inputs(w), rows=_sampled(w, tail=64, count=4096, seed=1))


def test_full_decode_batch_all_rows():
    w = gen.decode_batch()
    run_and_compare(w, gen.make_inputs(w))


def test_full_long_prefill_sampled():
    w = gen.long_prefill()
    run_and_compare(w, gen.make_inputs(w), rows=_sampled(w, tail=256, count=2048, seed=3))


def test_full_mixed_step_sampled():
    w = gen.mixed_step()
    host = gen.make_inputs(w)
    rows = _sampled(w, tail=256, count=2048, seed=4)
    run_and_compare(w, host, rows=rows)


def test_status_bounds_when_host_bounds_too_small():
    from causal_gqa_attention_qkv_gb300 import attn, step
    w = gen.custom("bounds", 8, 2, 64, [100], [0], seed=10)
    ds = step.upload(w, gen.make_inputs(w))
    ds.max_seqlen = 10
    ds.run()
    assert ds.status() & attn.ATTN_STATUS_BOUNDS
    wd = gen.custom("bounds_d", 8, 2, 64, [1, 1], [5000, 10], seed=11, decode_from=0)
    host = gen.make_inputs(wd)
    dd = step.upload(wd, host)
    dd.max_cache_len = 100
    dd.run()
    assert dd.status() & attn.ATTN_STATUS_BOUNDS
    # the short request is still computed correctly
    ref = oracle.step(oracle.cfg_of(wd), host, rows=oracle.all_rows(2, 8)[8:])
    check_out(gather_rows(dd.out, wd, ref["rows"]), ref["out"], "short request")
