"""GPU parity of token sampling (include/sample.h) against the CPU oracle.

A row's token depends on real-valued decisions (the top-p crossing and the
position of u in the cumulative kept probabilities).  Where the oracle's
decisions are more than 1e-5 (relative) from a boundary the token is unique
and must match; closer rows must match the oracle at a perturbed u or top_p
(any of those tokens is a valid answer)."""
import numpy as np
import pytest
import torch

import oracle
from causal_gqa_attention_qkv_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

MARGIN = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_gqa_attention_qkv_gb300 import build
    build.build()


def gpu_tokens(h):
    from causal_gqa_attention_qkv_gb300 import attn
    dev = {k: v.cuda() for k, v in h.items()}
    t = attn.sample_tokens(dev["logits"], dev["temperature"], dev["top_k"], dev["top_p"], dev["uniform"])
    torch.cuda.synchronize()
    return t.cpu().numpy().astype(np.int64)


def check(h, got):
    """Rows far from every boundary: the oracle's token.  The others: a token
    that the truncation keeps (with top_p moved by up to MARGIN) and whose
    range of u lies within MARGIN of the row's u."""
    x = h["logits"].numpy()
    T, k, p, u = (h[n].numpy() for n in ("temperature", "top_k", "top_p", "uniform"))
    want, margin = oracle.sample(x, T, k, p, u)
    unique = margin > MARGIN
    assert np.array_equal(got[unique], want[unique]), np.flatnonzero(got[unique] != want[unique])
    for b in np.flatnonzero(~unique):
        ok = False
        for pp in ((p[b] - MARGIN, p[b], p[b] + MARGIN) if p[b] < 1.0 else (p[b],)):
            kept, lo, hi = oracle.sample_bracket(x[b], T[b], k[b], pp, got[b])
            ok |= kept and lo - MARGIN <= u[b] <= hi + MARGIN
        assert ok, (b, int(got[b]), int(want[b]))
    return int((~unique).sum())


@pytest.mark.parametrize("B,V,seed", [(256, 1000, 1), (96, 32000, 2), (64, gen.QWEN3_VOCAB, 3)])
def test_sampling_matches_oracle(B, V, seed):
    h = gen.make_sampling_inputs(B, V, seed=seed)
    check(h, gpu_tokens(h))


def test_sampling_edge_cases_and_determinism():
    V = 3000
    h = gen.make_sampling_inputs(12, V, seed=4, greedy_share=0.0)
    x = h["logits"]
    x[0] = 0.5                                  # all equal: uniform over the vocabulary
    x[1, 100:] = float("-inf")                  # a masked vocabulary
    x[2, :] = -1e30; x[2, 7] = 3.0; x[2, 9] = 3.0   # two tied leaders far above the rest
    h["top_k"][3] = V                           # top-k = V: no limit
    h["top_p"][4] = 0.0                         # top-p <= 0: the largest logit only
    h["temperature"][5] = 1e-6                  # tiny temperature
    h["uniform"][6] = float(np.nextafter(np.float32(1.0), np.float32(0.0)))   # u just below 1
    h["uniform"][7] = 0.0
    h["top_k"][8] = 1
    a = gpu_tokens(h)
    check(h, a)
    assert np.array_equal(a, gpu_tokens(h))     # same inputs, same tokens
    assert a[1] < 100 and a[2] in (7, 9) and a[8] == int(np.argmax(x[8].numpy()))


def test_sampling_single_token_vocabulary():
    h = gen.make_sampling_inputs(5, 1, seed=5)
    assert (gpu_tokens(h) == 0).all()


def test_sampling_crossing_in_each_bin_range():
    """Rows whose truncation ends in each part of the kernel's bins of
    z = (max - l) log2(e) / T: the fine bins (z < 32), the coarse bins
    (32 <= z < 159.875, tiny weights), the last bin (weight 0), and crossing
    bins holding more tokens than the kernel copies (its slower path), plus
    ties at the crossing."""
    V = 32000
    h = gen.make_sampling_inputs(8, V, seed=8, greedy_share=0.0)
    g = torch.Generator().manual_seed(81)
    x = torch.randn((8, V), generator=g) * 2.0
    x[0] = 0.25                                           # one bin holds every token
    x[1, 5] = 40.0                                        # the rest far below: weight 0
    x[7] = torch.round(x[7] * 2.0) / 2.0                  # many ties
    h["logits"] = x
    rows = [  # (temperature, top_k, top_p)
        (1.0, 50, 1.0),                                   # count crossing among 32000 equal keys
        (0.3, 2000, 1.0),                                 # count crossing in the weight-0 bin
        (0.05, 20, 1.0),                                  # count crossing in the coarse bins
        (0.3, 0, float(np.nextafter(np.float32(1.0), np.float32(0.0)))),  # mass crossing in the coarse bins
        (1.5, 0, 0.9),                                    # mass crossing in dense fine bins
        (1.5, 0, 0.5),
        (1.0, 2000, 0.95),
        (1.0, 100, 1.0),                                  # ties at the crossing are kept
    ]
    for b, (t, k, p) in enumerate(rows):
        h["temperature"][b], h["top_k"][b], h["top_p"][b] = t, k, p
    a = gpu_tokens(h)
    check(h, a)
    assert np.array_equal(a, gpu_tokens(h))
