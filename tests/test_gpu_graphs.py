"""GPU tests of stream capture: a whole step (prefill part and decode part,
the decode rows appending their K/V inside the split kernel) recorded into a
CUDA graph and replayed must give the eager step's output and caches bit for
bit (the calls allocate nothing and wait for nothing, and the prefill
kernel leaves its work counters at zero for the next replay)."""
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


CASES = [
    # (Hq, Hkv, D, new lens, cached lens, decode_from, page size, kv dtype)
    (32, 8, 128, [300, 64, 1, 1, 1], [50, 0, 10, 3000, 0], 2, 0, "bf16"),
    (16, 4, 128, [130, 1, 1], [0, 700, 5000], 1, 64, "e4m3"),
    (4, 2, 64, [12], [0], 1, 0, "bf16"),
]


@pytest.mark.parametrize("hq,hkv,d,lens,cache,df,ps,kvd", CASES)
def test_step_replayed_from_a_cuda_graph(hq, hkv, d, lens, cache, df, ps, kvd):
    from causal_gqa_attention_qkv_gb300 import step
    w = gen.custom(f"graph_{hq}_{d}_{kvd}", hq, hkv, d, lens, cache, seed=sum(lens) + hq, decode_from=df)
    host = gen.make_inputs(w, page_size=ps, kv_dtype=kvd)
    eager = step.upload(w, host)
    eager.run()
    torch.cuda.synchronize()
    assert eager.status() == 0

    ds = step.upload(w, host)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # one eager call on the capture stream first
        ds.run()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ds.run()
    for _ in range(3):
        ds.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert ds.status() == 0
        assert torch.equal(ds.out.view(torch.int16), eager.out.view(torch.int16))
        for a, b in ((ds.k_cache, eager.k_cache), (ds.v_cache, eager.v_cache)):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    ref = oracle.step(oracle.cfg_of(w), host)
    check_out(gather_rows(ds.out, w, ref["rows"]), ref["out"], f"{w.name}: replayed")
