"""attn_decode_static_scratch: decode for callers that cannot allocate device
memory where they run decode (e.g. a plugin inside a framework that owns all
device allocations, or a serving loop that cannot take cudaMalloc's implicit
device synchronisation).  Its split-KV scratch is the library's static device
buffer, which keeps whatever the previous call left in it.

The output must match attn_decode (with a caller workspace) and the CPU
oracle within the parity tolerance on two calls in a row, after an earlier
call of a different shape has filled the buffer with other, non-zero
partials.  A call whose requests are not split needs no scratch at any batch
size; a call whose partials really exceed the buffer is refused.

This file is collected last on purpose, and it passes both alone in a fresh
process and after every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from causal_gqa_attention_qkv_gb300 import inputs as gen
from parity_util import MAX_ABS, REL_FRO, check_out, gather_rows

pytestmark = pytest.mark.gpu

ATTN_ESCRATCH = -6


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_gqa_attention_qkv_gb300 import attn, build
    build.build()
    return attn.load()


def _static_call(lib, ds, w, out, status, B=None, max_cache_len=None):
    kv = ds.kv_decode.struct()
    return lib.attn_decode_static_scratch(
        ctypes.byref(ds.cfg), ctypes.c_void_p(ds.qkv.data_ptr()), ctypes.c_void_p(ds.q_norm_w.data_ptr()),
        ctypes.c_void_p(ds.k_norm_w.data_ptr()), w.batch if B is None else B,
        ds.max_cache_len if max_cache_len is None else max_cache_len, ctypes.byref(kv),
        ctypes.c_void_p(out.data_ptr()), None if status is None else ctypes.c_void_p(status.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _workspace_result(w, host):
    from causal_gqa_attention_qkv_gb300 import step
    ds = step.upload(w, host)
    ds.run()  # attn_decode with a torch-allocated workspace
    torch.cuda.synchronize()
    assert ds.status() == 0
    return ds


def test_static_scratch_decode_matches_workspace_decode_and_oracle(lib):
    from causal_gqa_attention_qkv_gb300 import attn, step
    # A different workload first (group 1, other lengths, more splits), so
    # that the buffer holds its partials when the target workload runs.
    w0 = gen.custom("no_alloc_filler", 16, 16, 128, [1] * 5, [8000, 6000, 300, 12000, 4500], seed=29,
                    decode_from=0)
    ds0 = step.upload(w0, gen.make_inputs(w0))
    assert attn.decode_splits(ds0.cfg, w0.batch, ds0.max_cache_len) > 2
    st0 = torch.zeros(1, dtype=torch.int32, device=ds0.out.device)
    assert _static_call(lib, ds0, w0, ds0.out, st0) == 0
    torch.cuda.synchronize()
    assert int(st0.item()) == 0

    # target: several requests long enough to be split
    w = gen.custom("no_alloc_decode", 32, 8, 128, [1] * 6, [0, 700, 3000, 5000, 257, 9000], seed=31,
                   decode_from=0)
    host = gen.make_inputs(w)
    ds = _workspace_result(w, host)
    assert attn.decode_splits(ds.cfg, w.batch, ds.max_cache_len) > 1
    ref = ds.out.clone()
    rows = oracle.all_rows(w.num_tokens, w.num_q_heads)
    expect = oracle.step(oracle.cfg_of(w), host, rows=rows)["out"]

    status = torch.zeros(1, dtype=torch.int32, device=ds.out.device)
    out = torch.empty_like(ds.out)
    for call in range(2):
        out.fill_(float("nan"))
        rc = _static_call(lib, ds, w, out, status)
        assert rc == 0, lib.attn_strerror(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        stats = check_out(out, ref.double().cpu().numpy(), f"static-scratch call {call} vs attn_decode")
        assert stats["max_abs"] <= MAX_ABS and stats["rel_fro"] <= REL_FRO
        check_out(gather_rows(out, w, rows), expect, f"static-scratch call {call} vs oracle")


def test_static_scratch_unsplit_batch_needs_no_scratch(lib):
    """1024 short requests: one split each, so the output rows are written
    directly and the call succeeds although B * Hq * (D + 2) * 4 bytes would
    exceed the buffer."""
    from causal_gqa_attention_qkv_gb300 import attn
    g = np.random.default_rng(33)
    cache = g.integers(1, 300, size=1024).tolist()
    w = gen.custom("no_alloc_wide", 32, 8, 128, [1] * 1024, cache, seed=33, decode_from=0)
    host = gen.make_inputs(w)
    ds = _workspace_result(w, host)
    assert attn.decode_splits(ds.cfg, w.batch, ds.max_cache_len) == 1
    assert 1024 * 32 * 130 * 4 > (16 << 20)
    status = torch.zeros(1, dtype=torch.int32, device=ds.out.device)
    out = torch.full_like(ds.out, float("nan"))
    rc = _static_call(lib, ds, w, out, status)
    assert rc == 0, lib.attn_strerror(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_out(out, ds.out.double().cpu().numpy(), "unsplit static-scratch vs attn_decode")
    rows = gen.sample_rows(w, count=512, tail=0, seed=33).numpy()
    check_out(gather_rows(out, w, rows), oracle.step(oracle.cfg_of(w), host, rows=rows)["out"],
              "unsplit static-scratch vs oracle")


def test_static_scratch_rejects_requests_beyond_its_size(lib):
    from causal_gqa_attention_qkv_gb300 import attn, step
    # 127 requests of up to 65536 keys with 128 query heads split in two:
    # 127 * 128 * 2 * (128 + 2) * 4 bytes is about 16.9 MB, past the 16 MiB
    # buffer.  The size check comes before any pointer is used or anything is
    # launched, so the small workload's buffers stand in for the real ones.
    w = gen.custom("no_alloc_small", 128, 16, 128, [1], [10], seed=32, decode_from=0)
    ds = step.upload(w, gen.make_inputs(w))
    assert attn.decode_splits(ds.cfg, 127, 65535) == 2
    rc = _static_call(lib, ds, w, ds.out, None, B=127, max_cache_len=65535)
    assert rc == ATTN_ESCRATCH
    assert b"static" in lib.attn_strerror(rc)
