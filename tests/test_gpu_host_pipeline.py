"""GPU tests of the chunked, stream-pipelined prefill from host buffers
(step.HostPrefill): the output and the caches must be bit-identical to one
unchunked prefill call on the same inputs (every output row walks the same
key tiles through the same kernels), and sampled rows must match the oracle."""
import numpy as np
import pytest
import torch

import oracle
from causal_gqa_attention_qkv_gb300 import inputs as gen
from parity_util import check_out, gather_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_gqa_attention_qkv_gb300 import build
    build.build()


def _pipelined(w, host, chunk_tokens):
    from causal_gqa_attention_qkv_gb300 import step
    ds = step.upload(w, host)
    N = w.num_tokens
    q_stage = torch.empty((N, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=ds.out.device)
    out_dev = torch.full_like(ds.out, float("nan"))
    hp = step.HostPrefill(ds.cfg, ds.q_norm_w, ds.k_norm_w, ds.kv_prefill, ds.workspace, torch.empty_like(ds.qkv),
                          q_stage, out_dev, chunk_tokens=chunk_tokens)
    plan = hp.plan(host["cu_seqlens"].tolist(), host["cache_lens"].tolist())
    qkv_h = host["qkv"].pin_memory()
    out_h = torch.full((N, w.num_q_heads * w.head_dim), float("nan"), dtype=torch.bfloat16).pin_memory()
    hp.run(plan, qkv_h, out_h)
    torch.cuda.synchronize()
    assert ds.status() == 0 and hp.status() == 0
    return ds, out_h, plan


CASES = [
    # (name, Hq, Hkv, D, new lens, cached lens, chunk tokens, page size, kv dtype)
    ("one_long", 32, 8, 128, [10000], [0], 4096, 0, "bf16"),
    ("ragged_cut", 16, 2, 128, [3000, 0, 6000, 1, 513], [5, 0, 7, 100, 64], 4096, 0, "bf16"),
    ("small_chunks", 8, 2, 64, [300, 77, 513], [0, 200, 64], 128, 0, "bf16"),
    ("paged", 32, 8, 128, [2000, 1500], [64, 0], 1024, 64, "bf16"),
    ("e4m3", 32, 8, 128, [2500, 700], [0, 300], 1024, 0, "e4m3"),
]


@pytest.mark.parametrize("name,hq,hkv,d,lens,cache,chunk,ps,kvd", CASES)
def test_pipelined_prefill_equals_one_call(name, hq, hkv, d, lens, cache, chunk, ps, kvd):
    from causal_gqa_attention_qkv_gb300 import step
    w = gen.custom(f"pipe_{name}", hq, hkv, d, lens, cache, seed=sum(lens) + hq + chunk)
    host = gen.make_inputs(w, page_size=ps, kv_dtype=kvd)
    ds, out_h, plan = _pipelined(w, host, chunk)
    assert len(plan.chunks) == -(-w.num_tokens // chunk)
    ref = step.upload(w, host)
    ref.run()
    torch.cuda.synchronize()
    assert ref.status() == 0
    assert torch.equal(out_h.view(torch.int16), ref.out.cpu().view(torch.int16))
    for a, b in ((ds.k_cache, ref.k_cache), (ds.v_cache, ref.v_cache)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    rows = gen.sample_rows(w, count=512, tail=8, seed=len(lens)).numpy()
    expect = oracle.step(oracle.cfg_of(w), host, rows=rows)["out"]
    check_out(gather_rows(out_h, w, rows), expect, f"{name}: pipelined vs oracle")


def test_pipelined_long_prefill_full_size_sampled():
    """The 32 768-token long prefill in 4 096-token chunks, as the benchmark
    runs it end to end: bit-identical to one call, sampled rows vs the oracle."""
    from causal_gqa_attention_qkv_gb300 import step
    w = gen.long_prefill()
    host = gen.make_inputs(w)
    ds, out_h, plan = _pipelined(w, host, 4096)
    assert len(plan.chunks) == 8
    ref = step.upload(w, host)
    ref.run()
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.int16), ref.out.cpu().view(torch.int16))
    assert torch.equal(ds.k_cache.view(torch.int16), ref.k_cache.view(torch.int16))
    rows = gen.sample_rows(w, count=256, tail=4, seed=11).numpy()
    expect = oracle.step(oracle.cfg_of(w), host, rows=rows)["out"]
    check_out(gather_rows(out_h, w, rows), expect, "long prefill pipelined vs oracle")
