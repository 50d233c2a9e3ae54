"""GPU parity of the projections either side of the step (code walkthrough
section 3.3: qkv_proj, the attention, o_proj): the tcgen05 projection kernel
through the C ABI against the oracle's fp64 linear layer and projected step.

Tolerances.  Outputs, prepared Q and the appended cache entries are bf16
results of fp32 accumulation: max-abs <= 2e-2 and relative Frobenius <= 1e-2
against the fp64 oracle, as for the step itself; one-byte (E4M3) cache codes
at most one code apart, in at most 1 % of the entries.  The plain linear layer is
also held to the worst-case bound of its arithmetic: the bf16 products are
exact and each of the K - 1 fp32 additions errs by at most one fp32 ulp of
its partial sum (2^-23 relative, any order, rounding or truncating), so
|y - y_exact| <= (K - 1) 2^-23 sum_c |x_c w_c| before the final bf16
rounding, which adds at most half a bf16 step of the result.  Slots outside
the appended ones stay bit-identical."""
import numpy as np
import pytest
import torch

import oracle
from causal_gqa_attention_qkv_gb300 import inputs as gen
from parity_util import K_MAX_MISMATCH_FRACTION, check_out, e4m3_order, written_slots

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_gqa_attention_qkv_gb300 import build
    build.build()


def _bf16_step(x):
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 7)


@pytest.mark.parametrize("M,N,K,hq,d", [(1, 8, 64, 1, 64), (12, 64, 256, 4, 64), (130, 264, 192, 3, 64),
                                        (300, 2560, 4096, 32, 128), (257, 6144, 2560, 20, 128)])
def test_o_proj_matches_oracle(M, N, K, hq, d):
    """Ragged row counts, output widths that are not a multiple of the
    256-column tile, reductions of 1 to 64 stages."""
    from causal_gqa_attention_qkv_gb300 import attn
    assert K == hq * d
    g = torch.Generator().manual_seed(M * 7 + N + K)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) * K ** -0.5).to(torch.bfloat16)
    cfg = attn.config(hq, hq, d)  # o_proj reads only Hq * D
    ws = attn.new_workspace(cfg, 1, 1, 1)
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    attn.o_proj(cfg, x.cuda(), w.cuda(), y, ws)
    torch.cuda.synchronize()
    assert attn.get_status(ws) == 0
    ref = oracle.linear(x, w)
    got = y.double().cpu().numpy()
    check_out(y, ref, f"o_proj {M}x{N}x{K}")
    absdot = np.abs(x.double().numpy()) @ np.abs(w.double().numpy()).T
    bound = 0.5 * _bf16_step(got) + (K - 1) * 2.0 ** -23 * absdot
    err = np.abs(got - ref)
    assert (err <= bound).all(), f"o_proj off by {float((err / bound).max()):.2f} x its bound"


def _projected(w, C, seed, page_size=0, kv_dtype="bf16"):
    """Run qkv projection + prepare, prefill attention and o_proj on the GPU;
    the same through the oracle.  Returns both sides."""
    from causal_gqa_attention_qkv_gb300 import attn, step
    host = gen.make_inputs(w, page_size=page_size, kv_dtype=kv_dtype)
    pr = gen.make_projection_inputs(w, hidden=C, seed=seed)
    ds = step.upload(w, host)
    # every request (one-token rows included) goes through the prefill path here
    B = w.batch
    cu = torch.tensor(host["cu_seqlens"][:B + 1].tolist(), dtype=torch.int32, device="cuda")
    cap = torch.tensor(host["slot_capacity"].tolist(), dtype=torch.int32, device="cuda")
    sb = torch.tensor(host["slot_base"].tolist(), dtype=torch.int64, device="cuda")
    pt = host.get("page_table")
    kv = attn.KVCache(ds.k_cache, ds.v_cache, sb, ds.cache_lens, cap,
                      None if pt is None else pt.cuda(), int(host.get("page_size", 0)),
                      float(host.get("k_scale", 1.0)), float(host.get("v_scale", 1.0)))
    N = w.num_tokens
    hid, wq, wo = pr["hidden"].cuda(), pr["w_qkv"].cuda(), pr["w_o"].cuda()
    qdt = torch.float16 if kv_dtype == "e4m3" else torch.bfloat16
    q = torch.full((N, w.num_q_heads, w.head_dim), float("nan"), dtype=qdt, device="cuda")
    att = torch.full((N, w.num_q_heads * w.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = torch.full((N, C), float("nan"), dtype=torch.bfloat16, device="cuda")
    attn.qkv_proj_prepare(ds.cfg, hid, wq, ds.q_norm_w, ds.k_norm_w, cu, kv, q.view(torch.bfloat16), ds.workspace)
    attn.prefill_attend(ds.cfg, q.view(torch.bfloat16), cu, max(w.new_lens), kv, att, ds.workspace)
    attn.o_proj(ds.cfg, att, wo, o, ds.workspace)
    torch.cuda.synchronize()
    assert ds.status() == 0
    ref = oracle.projected_step(oracle.cfg_of(w), host, pr["hidden"], pr["w_qkv"], pr["w_o"])
    return {"host": host, "ds": ds, "q": q, "att": att, "o": o, "ref": ref}


def _check_projected(w, r):
    host, ref = r["host"], r["ref"]
    Hq, D = w.num_q_heads, w.head_dim
    check_out(r["q"].view(-1, D).float(), ref["q"].reshape(-1, D), f"{w.name}: prepared Q")
    check_out(r["att"].view(-1, D), ref["out"], f"{w.name}: attention")
    check_out(r["o"], ref["o"], f"{w.name}: o_proj")
    slots = written_slots(host)
    kg, vg = r["ds"].k_cache.cpu(), r["ds"].v_cache.cpu()
    mask = np.zeros(kg.shape[0], dtype=bool)
    mask[slots] = True
    for name, gpu in (("k_cache", kg), ("v_cache", vg)):
        refc = ref[name]
        if gpu.dtype == torch.uint8:
            gi, ri = gpu.numpy(), refc.numpy()
            assert np.array_equal(gi[~mask], ri[~mask]), f"{name} changed outside the appended slots"
            # both sides code the same value up to the fp32 error of the
            # projection: neighbouring codes where it sits next to a rounding
            # boundary, in at most 1 % of the entries
            d = np.abs(e4m3_order(gi[slots]) - e4m3_order(ri[slots]))
            assert d.max() <= 1, f"{w.name}: {name} codes {int(d.max())} apart"
            assert float((d != 0).mean()) <= K_MAX_MISMATCH_FRACTION, f"{w.name}: {name} codes differ"
        else:
            gb, rb = gpu.view(torch.int16).numpy(), refc.view(torch.int16).numpy()
            assert np.array_equal(gb[~mask], rb[~mask]), f"{name} changed outside the appended slots"
            check_out(gpu[torch.from_numpy(slots)], refc[torch.from_numpy(slots)].double().numpy(),
                      f"{w.name}: {name}")


PROJ = [
    # (Hq, Hkv, D, new lens, cached lens, hidden size, page size, kv dtype)
    (8, 2, 128, [1, 17, 64, 100, 200], [0, 5, 0, 130, 37], 512, 0, "bf16"),
    (16, 2, 64, [9, 130, 1], [3, 0, 200], 256, 0, "bf16"),
    (32, 8, 128, [300, 77, 1, 1], [0, 200, 64, 1000], 2560, 64, "bf16"),
    (4, 2, 64, [12], [0], 320, 0, "bf16"),                     # the tiny shape: 12 tokens, W = 512
    (8, 8, 64, [70, 33], [0, 64], 136, 0, "bf16"),             # hidden size not a multiple of 64
    (32, 8, 128, [130, 1, 65], [3, 0, 700], 512, 0, "e4m3"),
    (16, 4, 128, [40, 65], [0, 300], 1024, 128, "e4m3"),
]


@pytest.mark.parametrize("hq,hkv,d,lens,cache,C,ps,kvd", PROJ)
def test_projected_step_matches_oracle(hq, hkv, d, lens, cache, C, ps, kvd):
    w = gen.custom(f"proj_{hq}_{hkv}_{d}_{C}_{ps}_{kvd}", hq, hkv, d, lens, cache, seed=sum(lens) + C)
    _check_projected(w, _projected(w, C, seed=C + d, page_size=ps, kv_dtype=kvd))


def test_projected_qwen3_4b_prefill():
    """The Qwen3-4B shape: hidden size 2560, 8 packed sequences, 9942 tokens."""
    w = gen.qwen3_4b_prefill()
    _check_projected(w, _projected(w, gen.QWEN3_4B_HIDDEN, seed=1))
