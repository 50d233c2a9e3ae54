"""attn_decode_static_scratch: decode for callers that cannot allocate device
memory (e.g. a plugin inside a framework that owns all device allocations).
Its split-KV scratch is the library's static device buffer; its output must
match attn_decode (with a caller workspace) within the parity tolerance, on two
calls in a row (the buffer keeps the previous call's contents).

This file is collected last on purpose, and it passes both alone in a fresh
process and after every other test."""
import ctypes

import pytest
import torch

from causal_gqa_attention_qkv_gb300 import inputs as gen
from parity_util import MAX_ABS, REL_FRO, check_out

pytestmark = pytest.mark.gpu

ATTN_ESCRATCH = -6


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_gqa_attention_qkv_gb300 import attn, build
    build.build()
    return attn.load()


def test_static_scratch_decode_matches_workspace_decode(lib):
    from causal_gqa_attention_qkv_gb300 import attn, step
    # several requests long enough to be split (so the partial buffers are used)
    w = gen.custom("no_alloc_decode", 32, 8, 128, [1] * 6, [0, 700, 3000, 5000, 257, 9000], seed=31,
                   decode_from=0)
    host = gen.make_inputs(w)
    ds = step.upload(w, host)
    assert attn.decode_max_splits(w.batch, w.num_kv_heads, max(w.cache_lens) + 1) > 1
    ds.run()  # attn_decode with a torch-allocated workspace
    torch.cuda.synchronize()
    assert ds.status() == 0
    ref = ds.out.clone()

    kv = ds.kv_decode.struct()
    status = torch.zeros(1, dtype=torch.int32, device=ds.out.device)
    out = torch.empty_like(ds.out)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out.fill_(float("nan"))
        rc = lib.attn_decode_static_scratch(
            ctypes.byref(ds.cfg), ctypes.c_void_p(ds.qkv.data_ptr()), ctypes.c_void_p(ds.q_norm_w.data_ptr()),
            ctypes.c_void_p(ds.k_norm_w.data_ptr()), w.batch, ds.max_cache_len, ctypes.byref(kv),
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(status.data_ptr()), stream)
        assert rc == 0, lib.attn_strerror(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        stats = check_out(out, ref.double().cpu().numpy(), f"static-scratch call {call}")
        assert stats["max_abs"] <= MAX_ABS and stats["rel_fro"] <= REL_FRO


def test_static_scratch_rejects_requests_beyond_its_size(lib):
    from causal_gqa_attention_qkv_gb300 import step
    w = gen.custom("no_alloc_small", 32, 8, 128, [1], [10], seed=32, decode_from=0)
    ds = step.upload(w, gen.make_inputs(w))
    kv = ds.kv_decode.struct()
    # 4096 requests of up to 65536 keys need far more than 16 MiB of partials;
    # the size check comes before any pointer is used or anything is launched.
    rc = lib.attn_decode_static_scratch(
        ctypes.byref(ds.cfg), ctypes.c_void_p(ds.qkv.data_ptr()), ctypes.c_void_p(ds.q_norm_w.data_ptr()),
        ctypes.c_void_p(ds.k_norm_w.data_ptr()), 4096, 65535, ctypes.byref(kv),
        ctypes.c_void_p(ds.out.data_ptr()), None, None)
    assert rc == ATTN_ESCRATCH
    assert b"static" in lib.attn_strerror(rc)
