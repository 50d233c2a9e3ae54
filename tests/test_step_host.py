"""Host logic of the step module (no GPU): the token chunks of the
pipelined prefill from host buffers.  Every chunk must be a valid packed
prefill call whose requests, token counts and cached lengths reproduce the
original call token for token."""
import random

import pytest

from causal_gqa_attention_qkv_gb300 import step


def _check(cu, cl, chunk):
    chunks, meta = step.plan_chunks(cu, cl, chunk)
    N = cu[-1]
    covered = []
    for c in chunks:
        assert 0 < c.t1 - c.t0 <= chunk
        ccu = meta[c.cu[0]:c.cu[1]]
        ccl = meta[c.cl[0]:c.cl[1]]
        assert len(ccu) == c.b1 - c.b0 + 1 and len(ccl) == c.b1 - c.b0
        assert ccu[0] == 0 and ccu[-1] == c.t1 - c.t0
        assert c.max_seqlen == max(b - a for a, b in zip(ccu, ccu[1:]))
        for j, b in enumerate(range(c.b0, c.b1)):
            n = ccu[j + 1] - ccu[j]
            for k in range(n):
                # token k of request b in this chunk is packed token t, at position p
                t = c.t0 + ccu[j] + k
                assert cu[b] <= t < cu[b + 1]
                p = ccl[j] + k
                assert p == cl[b] + (t - cu[b])
                covered.append(t)
    assert covered == list(range(N))


@pytest.mark.parametrize("lens,cache,chunk", [
    ([32768], [0], 4096),
    ([3000, 0, 6000, 1, 513], [5, 0, 7, 100, 64], 4096),
    ([300, 77, 513], [0, 200, 64], 128),
    ([1] * 10, list(range(10)), 3),
    ([5], [0], 100),
    ([0, 0, 7, 0], [1, 2, 3, 4], 2),
])
def test_plan_chunks_reproduces_every_token(lens, cache, chunk):
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    _check(cu, cache, chunk)


def test_plan_chunks_random():
    rng = random.Random(7)
    for _ in range(200):
        B = rng.randint(1, 12)
        lens = [rng.choice([0, 1, rng.randint(1, 300)]) for _ in range(B)]
        if sum(lens) == 0:
            lens[0] = 1
        cache = [rng.randint(0, 500) for _ in range(B)]
        cu = [0]
        for n in lens:
            cu.append(cu[-1] + n)
        _check(cu, cache, rng.randint(1, 400))


def test_plan_chunks_empty_batch():
    chunks, meta = step.plan_chunks([0, 0], [3], 16)
    assert chunks == [] and meta == []
