"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point the headers under include/ declare, and rejects bad arguments before
touching a pointer or the device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from causal_gqa_attention_qkv_gb300 import attn, build
    build.build()
    return attn.load()


def declared_functions():
    """Every ATTN_API function of every header under include/."""
    names = set()
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names.update(re.findall(r"ATTN_API\s+[\w\s\*]*?\b(attn_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ("attn_prefill", "attn_decode", "attn_kv_append", "attn_workspace_size",
              "attn_prefill_prepare", "attn_prefill_attend", "attn_decode_attend",
              "attn_get_status", "attn_strerror", "attn_workspace_init", "attn_sample_tokens"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    from causal_gqa_attention_qkv_gb300 import attn
    nm = subprocess.run(["nm", "-D", "--defined-only", attn.LIB_PATH], capture_output=True, text=True,
                        check=True).stdout
    exported = set(re.findall(r"\sT\s+(attn_\w+)", nm))
    for n in declared_functions():
        assert n in exported, n
        assert getattr(lib, n) is not None


def test_strerror(lib):
    for code in (0, -1, -2, -3, -4, -5, -99):
        assert isinstance(lib.attn_strerror(code), bytes)
    assert b"multiple" in lib.attn_strerror(-2)


def test_workspace_size(lib):
    from causal_gqa_attention_qkv_gb300 import attn
    cfg = attn.config(32, 8, 128)
    # prefill: 256-byte status header + the prepared Q; decode: header + split partials
    assert attn.workspace_size(cfg, 4096, 0, 4096) == 256 + 4096 * 32 * 128 * 2
    c = attn.workspace_size(cfg, 16, 64, 16384)
    d = attn.workspace_size(cfg, 16, 8, 4096)
    assert 256 < d < c
    assert c >= 256 + 64 * 32 * 128 * 4
    assert lib.attn_workspace_size(ctypes.byref(attn.config(32, 5, 128)), 16, 1, 16) == 0
    assert lib.attn_workspace_size(ctypes.byref(attn.config(32, 8, 96)), 16, 1, 16) == 0


def _kv(attn):
    fake = 1 << 20  # never dereferenced: every call below fails its checks first
    return attn.AttnKV(fake, fake, 100, fake, fake, fake)


@pytest.mark.parametrize("hq,hkv,d,code", [(32, 5, 128, -2), (24, 8, 128, -2), (32, 8, 96, -1),
                                            (0, 1, 64, -1), (256, 32, 64, -1)])
def test_bad_config_rejected(lib, hq, hkv, d, code):
    from causal_gqa_attention_qkv_gb300 import attn
    cfg = attn.config(hq, hkv, d)
    fake = ctypes.c_void_p(1 << 20)
    kv = _kv(attn)
    rc = lib.attn_prefill(ctypes.byref(cfg), fake, fake, fake, fake, 1, 4, 4, ctypes.byref(kv), fake,
                          fake, 1 << 20, None)
    assert rc == code
    rc = lib.attn_decode(ctypes.byref(cfg), fake, fake, fake, 1, 4, ctypes.byref(kv), fake, fake,
                         1 << 20, None)
    assert rc == code


def test_null_and_alignment_rejected(lib):
    from causal_gqa_attention_qkv_gb300 import attn
    cfg = attn.config(8, 2, 64)
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 2)
    kv = _kv(attn)
    call = lambda qkv, ws, wsb, n=4, kvp=ctypes.byref(kv): lib.attn_prefill(
        ctypes.byref(cfg), qkv, fake, fake, fake, 1, n, 4, kvp, fake, ws, wsb, None)
    assert call(None, fake, 1 << 20) == -1          # NULL qkv
    assert call(odd, fake, 1 << 20) == -1           # misaligned qkv
    assert call(fake, fake, 1 << 20, n=-1) == -1    # negative N
    assert call(fake, None, 1 << 20) == -3          # no workspace
    assert call(fake, fake, 100) == -3              # workspace too small
    assert call(fake, fake, 256 + 4 * 8 * 64 * 2 - 16) == -3  # no room for the prepared Q
    assert call(fake, ctypes.c_void_p((1 << 20) + 16), 1 << 20) == -3  # not 256-aligned
    assert call(fake, fake, 1 << 20, kvp=None) == -1  # no cache
    bad_kv = attn.AttnKV(1 << 20, 1 << 20, 0, 1 << 20, 1 << 20, 1 << 20)
    assert call(fake, fake, 1 << 20, kvp=ctypes.byref(bad_kv)) == -1  # empty pool
    assert lib.attn_get_status(None, None, None) == -1


@pytest.mark.parametrize("B,max_cache", [(1, 12), (5, 3000), (64, 8192), (256, 16384), (8, 299),
                                         (1024, 300), (127, 65535), (4096, 65535)])
def test_decode_splits_and_workspace_size(lib, B, max_cache):
    """attn_decode_splits follows its documented policy (at most 16 splits,
    at least 256 keys per split when a request is split, about 2048 CTAs at
    the longest length), and the workspace holds the partials only when a
    request is split."""
    from causal_gqa_attention_qkv_gb300 import attn
    cfg = attn.config(32, 8, 128)
    ms = attn.decode_splits(cfg, B, max_cache)
    max_kv = max_cache + 1
    assert 1 <= ms <= 16
    assert (ms - 1) * 256 < max_kv  # every split but the last holds at least 256 keys
    if B * 8 * 2 <= 2048 // 2 and max_kv >= 16 * 256:
        assert ms > 1  # few CTAs and long requests: the keys are split
    al = lambda x: (x + 255) // 256 * 256
    partials = al(B * 32 * ms * 128 * 4) + al(B * 32 * ms * 2 * 4) if ms > 1 else 0
    assert attn.workspace_size(cfg, 1, B, max_kv) == 256 + max(partials, al(32 * 128 * 2))
    assert lib.attn_decode_splits(ctypes.byref(cfg), -1, 5) < 0
    assert lib.attn_decode_splits(None, 1, 5) < 0


@pytest.mark.parametrize("page_size,ppr", [(48, 4), (32, 4), (96, 4), (128, 0), (0, 4)])
def test_bad_page_layout_rejected(lib, page_size, ppr):
    """A paged cache needs a power-of-two page size >= 64 and a positive page-table
    row length; the check comes before any pointer is used or anything launched."""
    from causal_gqa_attention_qkv_gb300 import attn
    cfg = attn.config(32, 8, 128)
    fake = 1 << 20
    kv = attn.AttnKV(fake, fake, 1024, None, fake, fake, fake, page_size, ppr)
    f = ctypes.c_void_p(fake)
    rc = lib.attn_kv_append(ctypes.byref(cfg), f, f, f, f, 1, 4, ctypes.byref(kv), f, 1 << 20, None)
    assert rc == -1
    rc = lib.attn_decode(ctypes.byref(cfg), f, f, f, 1, 4, ctypes.byref(kv), f, f, 1 << 20, None)
    assert rc == -1


def test_contiguous_layout_needs_slot_base(lib):
    from causal_gqa_attention_qkv_gb300 import attn
    cfg = attn.config(32, 8, 128)
    fake = 1 << 20
    kv = attn.AttnKV(fake, fake, 1024, None, fake, fake, None, 0, 0)
    f = ctypes.c_void_p(fake)
    assert lib.attn_kv_append(ctypes.byref(cfg), f, f, f, f, 1, 4, ctypes.byref(kv), f, 1 << 20, None) == -1


@pytest.mark.parametrize("dtype,ks,vs,ok", [
    (1, 0.04, 0.02, True), (1, 0.0, 0.02, False), (1, 0.04, -1.0, False), (1, float("inf"), 0.02, False),
    (1, 0.04, float("nan"), False), (2, 1.0, 1.0, False), (-1, 1.0, 1.0, False), (0, 0.0, 0.0, True)])
def test_cache_element_type_checked(lib, dtype, ks, vs, ok):
    """kv_dtype is bf16 (scales ignored) or E4M3 with finite positive scales,
    checked by every call before any pointer is used: without a GPU the calls
    that pass the checks stop at the device query (-4 or -5)."""
    from causal_gqa_attention_qkv_gb300 import attn
    cfg = attn.config(32, 8, 128)
    fake = 1 << 20
    kv = attn.AttnKV(fake, fake, 1024, fake, fake, fake, None, 0, 0, dtype, ks, vs)
    f = ctypes.c_void_p(fake)
    k = ctypes.byref(kv)
    past_checks = (-4, -5)
    rc = lib.attn_decode(ctypes.byref(cfg), f, f, f, 1, 4, k, f, f, 1 << 20, None)
    assert (rc in past_checks) if ok else rc == -1
    rc = lib.attn_kv_append(ctypes.byref(cfg), f, f, f, f, 1, 4, k, f, 1 << 20, None)
    assert (rc in past_checks) if ok else rc == -1
    rc = lib.attn_prefill(ctypes.byref(cfg), f, f, f, f, 1, 4, 4, k, f, f, 1 << 20, None)
    assert (rc in past_checks) if ok else rc == -1
    rc = lib.attn_prefill_prepare(ctypes.byref(cfg), f, f, f, f, 1, 4, k, f, f, 1 << 20, None)
    assert (rc in past_checks) if ok else rc == -1
    rc = lib.attn_prefill_attend(ctypes.byref(cfg), f, f, 1, 4, 4, k, f, f, 1 << 20, None)
    assert (rc in past_checks) if ok else rc == -1


def test_sample_arguments_checked(lib):
    f = ctypes.c_void_p(1 << 20)
    call = lambda lg=f, B=4, V=100, ld=100, tok=f: lib.attn_sample_tokens(lg, B, V, ld, f, f, f, f, tok, None)
    assert call(lg=None) == -1
    assert call(tok=None) == -1
    assert call(B=-1) == -1
    assert call(V=0) == -1
    assert call(V=(1 << 23) + 1, ld=(1 << 23) + 1) == -1
    assert call(ld=99) == -1
    assert call() in (-4, -5)  # past the checks: no GPU here


def test_projection_arguments_checked(lib):
    """attn_qkv_proj_prepare and attn_o_proj check their pointers, alignment,
    the hidden size (positive, a multiple of 8), the cache and the workspace
    before touching anything; calls that pass the checks stop at the device
    query without a GPU (-4 or -5)."""
    from causal_gqa_attention_qkv_gb300 import attn
    cfg = attn.config(32, 8, 128)
    fake = 1 << 20
    f = ctypes.c_void_p(fake)
    odd = ctypes.c_void_p(fake + 8)
    kv = attn.AttnKV(fake, fake, 1024, fake, fake, fake)
    k = ctypes.byref(kv)
    past_checks = (-4, -5)

    def qkv(hidden=f, C=2560, w=f, q=f, kvp=k, ws=f, wsb=1 << 20, B=1, N=4):
        return lib.attn_qkv_proj_prepare(ctypes.byref(cfg), hidden, C, w, f, f, f, B, N, kvp, q, ws, wsb, None)

    assert qkv() in past_checks
    assert qkv(hidden=None) == -1
    assert qkv(hidden=odd) == -1
    assert qkv(w=None) == -1
    assert qkv(w=odd) == -1
    assert qkv(q=None) == -1
    assert qkv(C=0) == -1
    assert qkv(C=100) == -1          # not a multiple of 8
    assert qkv(N=-1) == -1
    assert qkv(kvp=None) == -1
    assert qkv(ws=None) == -3
    assert qkv(wsb=100) == -3

    def oproj(x=f, N=4, w=f, C=2560, out=f, ws=f, wsb=1 << 20, c=cfg):
        return lib.attn_o_proj(ctypes.byref(c), x, N, w, C, out, ws, wsb, None)

    assert oproj() in past_checks
    assert oproj(x=None) == -1
    assert oproj(w=odd) == -1
    assert oproj(out=None) == -1
    assert oproj(C=12) == -1
    assert oproj(N=-1) == -1
    assert oproj(ws=None) == -3
    assert oproj(c=attn.config(32, 5, 128)) == -2
