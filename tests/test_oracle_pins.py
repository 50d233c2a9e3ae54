"""Pins of the CPU oracle to things other than itself.

Each test checks one part of the oracle against what the pages or the
mathematics fix: a literal brute force of the teaching snippet (code
walkthrough section 3.3), torch's own ``rms_norm``, the complex form of RoPE
from the RoFormer paper the concept chapter cites, closed forms, and the
invariants the pages state (causality, rows of softmax summing to one, decode
as one more row of the lower triangle, cache lengths 0 -> 12 -> 13).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from causal_gqa_attention_qkv_gb300 import inputs as gen

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def bits_of(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- bf16 rounding
def test_bf16_round_matches_torch_on_float32_values():
    g = torch.Generator().manual_seed(11)
    x = torch.cat([torch.randn(20000, generator=g) * 10 ** torch.randint(-30, 30, (20000,), generator=g),
                   torch.tensor([0.0, -0.0, 1.0, -2.5, 3.0e38, 1e-40, -1e-42])])
    ref = bits_of(x.to(torch.bfloat16))
    got = np.array([oracle.bf16_round(float(v)) for v in x.tolist()], dtype=np.uint16)
    assert np.array_equal(ref, got)


def test_bf16_round_ties_and_no_double_rounding():
    # quantum at 1.0 is 2**-7: exact midpoints go to the even neighbour
    assert oracle.bf16_round(1.0 + 2 ** -8) == 0x3F80
    assert oracle.bf16_round(1.0 + 3 * 2 ** -8) == 0x3F82
    # just above a midpoint rounds up even though float32 would land on the tie
    assert oracle.bf16_round(1.0 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert oracle.bf16_round(-(1.0 + 2 ** -8 + 2 ** -40)) == 0xBF81


# ---------------------------------------------------------------- RMSNorm
@pytest.mark.parametrize("D", [8, 64, 128])
def test_rmsnorm_matches_torch_rms_norm(D):
    g = torch.Generator().manual_seed(D)
    x = torch.randn(16, D, generator=g, dtype=torch.float64) * 3
    w = 1 + 0.1 * torch.randn(D, generator=g, dtype=torch.float64)
    ref = torch.nn.functional.rms_norm(x, (D,), weight=w, eps=1e-6).numpy()
    got = np.stack([oracle.rmsnorm(x[i].numpy(), w.numpy(), 1e-6) for i in range(16)])
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_rmsnorm_constant_vector_closed_form():
    D, eps = 64, 1e-6
    w = np.linspace(0.5, 1.5, D)
    for c in (2.0, -0.003, 1e-3):
        y = oracle.rmsnorm(np.full(D, c), w, eps)
        np.testing.assert_allclose(y, w * c / math.sqrt(c * c + eps), rtol=1e-14)


# ---------------------------------------------------------------- RoPE
def rope_complex(x, pos, theta):
    """RoFormer's complex form: pair (x_i, x_{i+D/2}) as x_i + j x_{i+D/2},
    multiplied by exp(j * pos * theta_i), theta_i a geometric sequence from 1
    with ratio theta^(-2/D)."""
    D = x.shape[-1]
    half = D // 2
    ratio = theta ** (-2.0 / D)
    freqs = ratio ** np.arange(half, dtype=np.float64)
    z = (x[:half] + 1j * x[half:]) * np.exp(1j * pos * freqs)
    return np.concatenate([z.real, z.imag])


@pytest.mark.parametrize("D,pos", [(2, 0.7), (8, 3.0), (64, 11.0), (128, 4097.0), (128, 40000.0)])
def test_rope_matches_complex_form(D, pos):
    x = np.random.default_rng(D).standard_normal(D)
    np.testing.assert_allclose(oracle.rope(x, pos, 1e6), rope_complex(x, pos, 1e6), rtol=0,
                               atol=1e-9 * max(1.0, pos / 1000))


def test_rope_pair0_rotates_by_position_counterclockwise():
    x = np.zeros(8)
    x[0] = 1.0
    y = oracle.rope(x, 0.5, 1e6)
    np.testing.assert_allclose([y[0], y[4]], [math.cos(0.5), math.sin(0.5)], atol=1e-15)
    np.testing.assert_allclose(np.delete(y, [0, 4]), 0, atol=0)


def test_rope_invariants():
    rng = np.random.default_rng(5)
    D, theta = 128, 1e6
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    # p = 0 is the identity
    np.testing.assert_array_equal(oracle.rope(q, 0.0, theta), q)
    # a rotation keeps the norm
    for p in (1.0, 17.0, 3000.0):
        assert abs(np.linalg.norm(oracle.rope(q, p, theta)) - np.linalg.norm(q)) < 1e-12
    # q.k depends only on the position difference
    for m, n, s in ((5, 2, 100), (0, 9, 31), (1000, 1000, 7)):
        d1 = oracle.rope(q, m, theta) @ oracle.rope(k, n, theta)
        d2 = oracle.rope(q, m + s, theta) @ oracle.rope(k, n + s, theta)
        assert abs(d1 - d2) < 1e-10


# ---------------------------------------------------------------- attention
def brute_force(q, k, v, cache_len=0):
    """The code walkthrough's section 3.3 teaching snippet, in fp64, with the
    lower triangle shifted by the cached length (a query at position c + j sees
    keys 0 .. c + j).  q [B,Hq,T,D]; k, v [B,Hkv,c+T,D]."""
    groups = q.shape[1] // k.shape[1]
    k = k.repeat_interleave(groups, dim=1)
    v = v.repeat_interleave(groups, dim=1)
    scores = q @ k.transpose(-1, -2) / q.shape[-1] ** 0.5
    T, S = q.shape[-2], k.shape[-2]
    allowed = torch.ones(T, S, dtype=torch.bool).tril(diagonal=cache_len)
    scores = scores.masked_fill(~allowed, float("-inf"))
    weights = scores.softmax(dim=-1)
    return weights @ v


def run_oracle_attention(q, k, v, cache_len=0, Hq=None):
    """Put K/V (bf16 values) of one request in a slot pool and ask the oracle
    for every (token, head) row.  q [Hq,T,D] fp64, k/v [Hkv,c+T,D] bf16."""
    Hq, T, D = q.shape
    Hkv, S, _ = k.shape
    base = 5
    kc = torch.full((base + S + 2, Hkv, D), float("nan"), dtype=torch.bfloat16)
    vc = kc.clone()
    kc[base:base + S] = k.transpose(0, 1)
    vc[base:base + S] = v.transpose(0, 1)
    inp = {"cu_seqlens": torch.tensor([0, T], dtype=torch.int32),
           "cache_lens": torch.tensor([cache_len], dtype=torch.int32),
           "slot_base": torch.tensor([base], dtype=torch.int64)}
    cfg = {"num_q_heads": Hq, "num_kv_heads": Hkv, "head_dim": D}
    rows = oracle.all_rows(T, Hq)
    qr = q.transpose(0, 1).reshape(T * Hq, D).numpy()
    out = oracle.attention(cfg, kc, vc, inp, rows, qr)
    return torch.from_numpy(out.reshape(T, Hq, D)).transpose(0, 1)


@pytest.mark.parametrize("Hq,Hkv,T,D,c", [
    (4, 2, 3, 8, 0),     # the walkthrough's section 5 shape walk
    (4, 4, 5, 8, 0),     # Hkv = Hq: plain multi-head attention
    (4, 1, 6, 16, 0),    # Hkv = 1: multi-query attention
    (8, 2, 7, 16, 4),    # with a cached prefix
    (6, 3, 1, 8, 9),     # one decode row
])
def test_attention_matches_teaching_snippet(Hq, Hkv, T, D, c):
    g = torch.Generator().manual_seed(Hq * 100 + T)
    q = torch.randn(Hq, T, D, generator=g, dtype=torch.float64)
    k = torch.randn(Hkv, c + T, D, generator=g).to(torch.bfloat16)
    v = torch.randn(Hkv, c + T, D, generator=g).to(torch.bfloat16)
    ref = brute_force(q[None], k.double()[None], v.double()[None], c)[0]
    got = run_oracle_attention(q, k, v, c)
    torch.testing.assert_close(got, ref, rtol=1e-12, atol=1e-12)


def test_gqa_maps_heads_by_repeat_interleave_not_modulo():
    # Hq=4, Hkv=2: heads 0,1 -> kv 0 and heads 2,3 -> kv 1; one key so out = V
    q = torch.randn(4, 1, 8, dtype=torch.float64)
    k = torch.randn(2, 1, 8).to(torch.bfloat16)
    v = torch.stack([torch.full((1, 8), 1.0), torch.full((1, 8), 2.0)]).to(torch.bfloat16)
    got = run_oracle_attention(q, k, v)
    assert got[:, 0, 0].tolist() == [1.0, 1.0, 2.0, 2.0]


def test_first_row_is_first_value_exactly():
    g = torch.Generator().manual_seed(3)
    q = torch.randn(4, 6, 8, generator=g, dtype=torch.float64)
    k = torch.randn(2, 6, 8, generator=g).to(torch.bfloat16)
    v = torch.randn(2, 6, 8, generator=g).to(torch.bfloat16)
    got = run_oracle_attention(q, k, v)
    for h in range(4):
        assert torch.equal(got[h, 0], v[h // 2, 0].double())


def test_softmax_rows_nonnegative_sum_to_one_and_causal():
    # V[u] = e_u turns the output into the softmax row itself
    T, D = 9, 16
    g = torch.Generator().manual_seed(4)
    q = torch.randn(2, T, D, generator=g, dtype=torch.float64) * 2
    k = torch.randn(1, T, D, generator=g).to(torch.bfloat16)
    v = torch.eye(D)[:T][None].to(torch.bfloat16)
    P = run_oracle_attention(q, k, v)[..., :T]
    assert (P >= 0).all()
    torch.testing.assert_close(P.sum(-1), torch.ones(2, T, dtype=torch.float64), rtol=0, atol=1e-14)
    assert (P.triu(diagonal=1) == 0).all()
    assert (P[:, torch.ones(T, T, dtype=torch.bool).tril()] > 0).all()


def test_equal_keys_give_prefix_mean_of_values():
    T, D = 7, 8
    g = torch.Generator().manual_seed(6)
    q = torch.randn(2, T, D, generator=g, dtype=torch.float64)
    k = torch.randn(1, 1, D, generator=g).to(torch.bfloat16).expand(1, T, D).contiguous()
    v = torch.randn(1, T, D, generator=g).to(torch.bfloat16)
    got = run_oracle_attention(q, k, v)
    vd = v[0].double()
    ref = torch.cumsum(vd, 0) / torch.arange(1, T + 1, dtype=torch.float64)[:, None]
    torch.testing.assert_close(got[0], ref, rtol=1e-13, atol=1e-14)
    torch.testing.assert_close(got[1], ref, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- whole step
def torch_pipeline(w, inp):
    """The transformer-basics "Attention calculation: part 1" order in fp64:
    split + view, q_norm / k_norm (torch rms_norm), RoPE (complex form), then
    the K that goes to the cache rounded to bf16.  One request, empty cache."""
    N = w.num_tokens
    Hq, Hkv, D = w.num_q_heads, w.num_kv_heads, w.head_dim
    x = inp["qkv"].double()
    q = x[:, :Hq * D].view(N, Hq, D)
    k = x[:, Hq * D:(Hq + Hkv) * D].view(N, Hkv, D)
    v = inp["qkv"][:, (Hq + Hkv) * D:].view(N, Hkv, D)
    q = torch.nn.functional.rms_norm(q, (D,), weight=inp["q_norm_w"].double(), eps=w.rms_eps)
    k = torch.nn.functional.rms_norm(k, (D,), weight=inp["k_norm_w"].double(), eps=w.rms_eps)
    qr = torch.stack([torch.stack([torch.from_numpy(rope_complex(q[t, h].numpy(), t, w.rope_theta))
                                   for h in range(Hq)]) for t in range(N)])
    kr = torch.stack([torch.stack([torch.from_numpy(rope_complex(k[t, h].numpy(), t, w.rope_theta))
                                   for h in range(Hkv)]) for t in range(N)])
    return qr, kr, v


def test_whole_step_tiny_matches_torch_pipeline_and_brute_force():
    w = gen.tiny()
    inp = gen.make_inputs(w)
    cfg = oracle.cfg_of(w)
    res = oracle.step(cfg, inp)
    qr, kr, v = torch_pipeline(w, inp)
    N, Hq, Hkv, D = w.num_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim
    np.testing.assert_allclose(res["q"].reshape(N, Hq, D), qr.numpy(), rtol=0, atol=1e-12)
    base = int(inp["slot_base"][0])
    kc = res["k_cache"][base:base + N]
    ulp = (bits_of(kc).astype(np.int32) - bits_of(kr.float().to(torch.bfloat16)).astype(np.int32))
    assert np.abs(ulp).max() <= 1
    assert torch.equal(res["v_cache"][base:base + N].view(torch.int16), v.view(torch.int16))
    ref = brute_force(qr.transpose(0, 1)[None], kc.double().transpose(0, 1)[None],
                      v.double().transpose(0, 1)[None])[0].transpose(0, 1)
    np.testing.assert_allclose(res["out"].reshape(N, Hq, D), ref.numpy(), rtol=0, atol=1e-12)


def test_cache_bookkeeping_0_12_13_and_untouched_slots():
    w = gen.tiny()
    inp = gen.make_inputs(w, unused_fill="sentinel")
    cfg = oracle.cfg_of(w)
    base = int(inp["slot_base"][0])
    before = bits_of(inp["k_cache"]).copy()
    res = oracle.step(cfg, inp)
    after = bits_of(res["k_cache"])
    changed = np.nonzero((after != before).any(axis=(1, 2)))[0]
    assert changed.tolist() == list(range(base, base + 12))
    # decode: cache length 12 -> 13, exactly one more slot
    dinp = dict(inp, qkv=gen.make_followup_decode_qkv(w), cu_seqlens=torch.tensor([0, 1], dtype=torch.int32),
                cache_lens=torch.tensor([12], dtype=torch.int32), k_cache=res["k_cache"],
                v_cache=res["v_cache"])
    res2 = oracle.step(cfg, dinp)
    changed2 = np.nonzero((bits_of(res2["k_cache"]) != after).any(axis=(1, 2)))[0]
    assert changed2.tolist() == [base + 12]


def test_decode_is_one_more_row_of_prefill():
    # prefill over L+1 tokens vs prefill over L then decode of token L
    L = 10
    w = gen.custom("pin", 8, 2, 32, [L + 1], [0], seed=21)
    inp = gen.make_inputs(w)
    cfg = oracle.cfg_of(w)
    full = oracle.step(cfg, inp)
    first = dict(inp, qkv=inp["qkv"][:L].clone(), cu_seqlens=torch.tensor([0, L], dtype=torch.int32))
    r1 = oracle.step(cfg, first)
    dec = dict(inp, qkv=inp["qkv"][L:].clone(), cu_seqlens=torch.tensor([0, 1], dtype=torch.int32),
               cache_lens=torch.tensor([L], dtype=torch.int32), k_cache=r1["k_cache"],
               v_cache=r1["v_cache"])
    r2 = oracle.step(cfg, dec)
    np.testing.assert_array_equal(r2["out"], full["out"][-w.num_q_heads:])
    assert torch.equal(r2["k_cache"].view(torch.int16), full["k_cache"].view(torch.int16))


def test_changing_future_tokens_leaves_earlier_outputs_unchanged():
    w = gen.custom("pin", 4, 2, 16, [9, 6], [3, 0], seed=22)
    inp = gen.make_inputs(w)
    cfg = oracle.cfg_of(w)
    a = oracle.step(cfg, inp)
    qkv = inp["qkv"].clone()
    qkv[5:9] = torch.randn(4, qkv.shape[1]).to(torch.bfloat16)   # tokens 5..8 of request 0
    qkv[12:15] = torch.randn(3, qkv.shape[1]).to(torch.bfloat16)  # tokens 3..5 of request 1
    b = oracle.step(cfg, dict(inp, qkv=qkv))
    Hq = w.num_q_heads
    keep = [t for t in range(w.num_tokens) if t < 5 or 9 <= t < 12]
    for t in keep:
        np.testing.assert_array_equal(a["out"][t * Hq:(t + 1) * Hq], b["out"][t * Hq:(t + 1) * Hq])
    assert not np.array_equal(a["out"][8 * Hq:9 * Hq], b["out"][8 * Hq:9 * Hq])


def test_ragged_batch_positions_restart_per_request():
    # the second request's first token sits at position c_1, whatever came before it
    w = gen.custom("pin", 4, 2, 16, [5, 3], [0, 7], seed=23)
    inp = gen.make_inputs(w)
    cfg = oracle.cfg_of(w)
    res = oracle.step(cfg, inp)
    alone = gen.custom("pin", 4, 2, 16, [3], [7], seed=23)
    inp1 = dict(inp, qkv=inp["qkv"][5:].clone(), cu_seqlens=torch.tensor([0, 3], dtype=torch.int32),
                cache_lens=inp["cache_lens"][1:].clone(), slot_base=inp["slot_base"][1:].clone(),
                slot_capacity=inp["slot_capacity"][1:].clone())
    res1 = oracle.step(oracle.cfg_of(alone), inp1)
    np.testing.assert_array_equal(res1["out"], res["out"][5 * 4:])


def test_region_too_small_writes_nothing():
    w = gen.custom("pin", 4, 2, 16, [4, 4], [0, 2], seed=24)
    inp = gen.make_inputs(w)
    inp["slot_capacity"][1] = 5  # needs 2 + 4
    kc, vc, _, bad = oracle.prologue(oracle.cfg_of(w), inp)
    assert bad == 1
    b1 = int(inp["slot_base"][1])
    assert torch.equal(kc[b1 + 2:b1 + 6].view(torch.int16), inp["k_cache"][b1 + 2:b1 + 6].view(torch.int16))
    b0 = int(inp["slot_base"][0])
    assert not torch.equal(kc[b0:b0 + 4].view(torch.int16), inp["k_cache"][b0:b0 + 4].view(torch.int16))


@pytest.mark.parametrize("page_size", [64, 128])
def test_paged_cache_gives_the_contiguous_result(page_size):
    """The paged layout only moves where an entry lives: for the same logical
    inputs the outputs are bit-identical to the contiguous layout, each
    position's K/V lands in slot page_table[b, p // page_size] * page_size +
    p % page_size, and no other slot changes."""
    w = gen.custom("paged_pin", 4, 2, 64, [50, 130, 1, 7], [100, 0, 70, 129], seed=21)
    cfg = oracle.cfg_of(w)
    hc = gen.make_inputs(w)
    hp = gen.make_inputs(w, page_size=page_size)
    rc, rp = oracle.step(cfg, hc), oracle.step(cfg, hp)
    assert rc["bad"] == 0 and rp["bad"] == 0
    assert np.array_equal(rc["out"], rp["out"])
    kc, vc = rc["k_cache"].view(torch.int16), rc["v_cache"].view(torch.int16)
    kp, vp = rp["k_cache"].view(torch.int16), rp["v_cache"].view(torch.int16)
    touched = torch.zeros(kp.shape[0], dtype=torch.bool)
    pt = hp["page_table"]
    for b in range(w.batch):
        end = w.cache_lens[b] + w.new_lens[b]
        pos = torch.arange(end)
        sp = pt[b, pos // page_size].long() * page_size + pos % page_size
        sc = hc["slot_base"][b] + pos
        assert torch.equal(kp[sp], kc[sc]) and torch.equal(vp[sp], vc[sc])
        touched[sp] = True
    k0, v0 = hp["k_cache"].view(torch.int16), hp["v_cache"].view(torch.int16)
    assert torch.equal(kp[~touched], k0[~touched]) and torch.equal(vp[~touched], v0[~touched])


# ---------------------------------------------------------------- E4M3 cache entries
def _torch_e4m3_values(codes):
    return torch.as_tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def test_e4m3_decode_matches_torch_for_every_code():
    """Every one of the 256 codes decodes as torch's float8_e4m3fn reads it;
    0x7F and 0xFF are the only NaNs and 448 is the largest finite value."""
    got = np.array([oracle.e4m3_decode(b) for b in range(256)])
    ref = _torch_e4m3_values(np.arange(256))
    nan = np.isnan(ref)
    assert np.flatnonzero(nan).tolist() == [0x7F, 0xFF] and np.isnan(got[nan]).all()
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[~nan].max() == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_e4m3_encode_matches_torch_in_range_and_rounds_ties_to_even():
    g = np.random.default_rng(5)
    x = np.concatenate([g.normal(size=20000) * 40, g.normal(size=20000) * 1e-2,
                        g.uniform(-447.9, 447.9, 20000), [0.0, -0.0, 2.0 ** -10, -(2.0 ** -10)]])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)
    # every midpoint between neighbouring positive codes goes to the even code
    vals = [(oracle.e4m3_decode(b), b) for b in range(0x7F)]
    for (va, a), (vb, b) in zip(vals, vals[1:]):
        mid = (va + vb) / 2
        assert oracle.e4m3_encode(mid) == (a if a % 2 == 0 else b)
        assert oracle.e4m3_encode(np.nextafter(mid, 0.0)) == a
        assert oracle.e4m3_encode(np.nextafter(mid, 1e9)) == b


def test_e4m3_encode_saturates_beyond_448():
    for x in (448.0, 448.1, 463.9, 464.0, 500.0, 1e30, math.inf):
        assert oracle.e4m3_encode(x) == 0x7E
        assert oracle.e4m3_encode(-x) == 0xFE


def test_e4m3_cache_store_rule_and_reads():
    """A one-byte cache holds e4m3(fp32(x) * fp32(1 / scale)) per entry:
    V codes equal torch's own cast of that fp32 product; K codes read back
    within half a code step (plus half a bf16 step) of the bf16 cache's K;
    and attention over the codes equals attention over a bf16 cache holding
    the decoded values when those are exact in bf16 (scale a power of two)."""
    w = gen.custom("e4m3_pin", 8, 2, 64, [11, 5], [6, 0], seed=31)
    cfg = oracle.cfg_of(w)
    for ks, vs in ((0.04, 0.02), (2.0 ** -4, 2.0 ** -5)):
        h8 = gen.make_inputs(w, kv_dtype="e4m3", k_scale=ks, v_scale=vs)
        r8 = oracle.step(cfg, h8)
        hb = gen.make_inputs(w)
        rb = oracle.step(cfg, hb)
        k8, v8 = r8["k_cache"].numpy(), r8["v_cache"].numpy()
        kb = rb["k_cache"].double().numpy()
        Hq, Hkv, D = w.num_q_heads, w.num_kv_heads, w.head_dim
        for b in range(w.batch):
            for j in range(w.new_lens[b]):
                t = int(h8["cu_seqlens"][b]) + j
                slot = int(h8["slot_base"][b]) + w.cache_lens[b] + j
                v_in = h8["qkv"][t, (Hq + Hkv) * D:].float().reshape(Hkv, D)
                want = (v_in * torch.tensor(1.0 / np.float32(vs), dtype=torch.float32)) \
                    .to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                assert np.array_equal(v8[slot], want)
                kr = _torch_e4m3_values(k8[slot]) * np.float32(ks)
                # code step at |x| / scale, in units of x
                step = ks * 2.0 ** (np.floor(np.log2(np.maximum(np.abs(kb[slot]) / ks, 2.0 ** -6))) - 3)
                assert (np.abs(kr - kb[slot]) <= 0.5 * step + 2.0 ** -8 * np.abs(kb[slot]) + 1e-12).all()
        if ks == 2.0 ** -4:
            # the same codes, decoded into a bf16 cache: identical attention in fp64
            hbf = dict(h8, kv_dtype="bf16",
                       k_cache=(torch.from_numpy(k8).view(torch.float8_e4m3fn).double() * ks).to(torch.bfloat16),
                       v_cache=(torch.from_numpy(v8).view(torch.float8_e4m3fn).double() * vs).to(torch.bfloat16))
            rows = oracle.all_rows(w.num_tokens, Hq)
            a8 = oracle.attention(cfg, r8["k_cache"], r8["v_cache"], h8, rows, r8["q"])
            ab = oracle.attention(cfg, hbf["k_cache"], hbf["v_cache"], hbf, rows, r8["q"])
            assert np.array_equal(a8, ab)


# ---------------------------------------------------------------- sampling
def _grid(n):
    return (np.arange(n) + 0.5) / n


def _freq(logits, T, k, p, n=20000):
    """Token frequencies of the oracle over a uniform grid of n values of u."""
    L = np.repeat(np.asarray(logits, dtype=np.float32)[None], n, 0)
    toks, _ = oracle.sample(L, [T] * n, [k] * n, [p] * n, _grid(n))
    return np.bincount(toks, minlength=L.shape[1]) / n, toks


def test_sample_greedy_is_the_first_maximum():
    g = np.random.default_rng(1)
    x = g.integers(-5, 5, size=(50, 40)).astype(np.float32)  # many ties
    toks, margins = oracle.sample(x, [0.0] * 50, [0] * 50, [1.0] * 50, g.random(50))
    assert np.array_equal(toks, np.argmax(x, axis=1)) and np.isinf(margins).all()


def test_sample_closed_form_top_p_and_top_k_ties():
    """probabilities 0.5, 0.3, 0.15, 0.05 (the logits are their logs):
    top-p 0.8 keeps the first two (0.5 + 0.3 reaches 0.8), 0.81 the first
    three; top-k 2 with three tied leaders keeps all three (ties enter
    together)."""
    lp = np.log([0.5, 0.3, 0.15, 0.05])
    f, _ = _freq(lp + 0.0, 1.0, 0, 0.79)
    np.testing.assert_allclose(f, [0.625, 0.375, 0, 0], atol=1e-3)
    f, _ = _freq(lp, 1.0, 0, 0.81)
    np.testing.assert_allclose(f, np.array([0.5, 0.3, 0.15, 0]) / 0.95, atol=1e-3)
    f, _ = _freq(lp, 1.0, 0, 1.0)
    np.testing.assert_allclose(f, [0.5, 0.3, 0.15, 0.05], atol=1e-3)
    f, _ = _freq([1.0, 1.0, 0.0, 1.0], 1.0, 2, 1.0)
    np.testing.assert_allclose(f, [1 / 3, 1 / 3, 0, 1 / 3], atol=1e-3)


@pytest.mark.parametrize("T,k,p", [(1.0, 0, 1.0), (0.7, 10, 1.0), (1.3, 0, 0.9), (0.5, 25, 0.6), (2.0, 5, 0.99)])
def test_sample_frequencies_match_truncated_softmax(T, k, p):
    """Over a fine grid of u the oracle's frequencies equal the truncated,
    renormalised softmax(logits / T): scipy's softmax, numpy's sort for the
    k most probable and for the smallest prefix reaching p."""
    from scipy.special import softmax
    g = np.random.default_rng(int(T * 10) + k)
    x = (g.normal(size=60) * 2).astype(np.float32)
    P = softmax(x.astype(np.float64) / T)
    order = np.argsort(-P, kind="stable")
    keep = np.ones(60, dtype=bool)
    if 0 < k < 60:
        keep &= P >= P[order[k - 1]]
    if p < 1:
        c = np.cumsum(P[order])
        n = int(np.searchsorted(c, p * c[-1] * (1 - 1e-12)))
        keep &= P >= P[order[n]]
    want = np.where(keep, P, 0.0)
    want /= want.sum()
    f, _ = _freq(x, T, k, p, n=40000)
    np.testing.assert_allclose(f, want, atol=2e-4)


def test_sample_inverse_cdf_in_vocabulary_order_and_limits():
    g = np.random.default_rng(9)
    x = (g.normal(size=30) * 3).astype(np.float32)
    _, toks = _freq(x, 1.0, 0, 1.0, n=5000)
    assert np.all(np.diff(toks) >= 0)  # u increasing -> token index nondecreasing
    f, _ = _freq(x, 1e4, 0, 1.0, n=30000)  # very high temperature: nearly uniform
    np.testing.assert_allclose(f, np.full(30, 1 / 30), atol=2e-3)
    for T, k, p in ((1e-3, 0, 1.0), (1.0, 1, 1.0), (1.0, 0, 1e-9)):  # limits that reach greedy
        f, _ = _freq(x, T, k, p, n=200)
        assert f[np.argmax(x)] == 1.0


def test_sample_bracket_contains_u_of_the_sampled_token():
    """The bracket helper used to accept near-boundary device tokens agrees with
    the sampler: the sampled token is kept and its range of u contains u, and a
    token below the kept threshold is reported as not kept."""
    g = np.random.default_rng(17)
    for r in range(40):
        x = (g.normal(size=200) * 2).astype(np.float32)
        T, k, p, u = float(g.choice([0.5, 1.0, 2.0])), int(g.choice([0, 5, 50])), float(g.choice([1.0, 0.9, 0.5])), float(g.random())
        tok, _ = oracle.sample(x[None], [T], [k], [p], [u])
        kept, lo, hi = oracle.sample_bracket(x, T, k, p, int(tok[0]))
        assert kept and lo - 1e-12 <= u < hi + 1e-12
        if k == 5:
            low = int(np.argmin(x))
            assert not oracle.sample_bracket(x, T, k, p, low)[0]


@pytest.mark.parametrize("page_size", [64, 128])
def test_paged_e4m3_cache_gives_the_contiguous_result(page_size):
    """With one-byte entries as with bf16 ones, the page table only moves where
    an entry lives: identical outputs, and each position's codes in its page
    slot."""
    w = gen.custom("paged_e4m3_pin", 4, 2, 64, [50, 130, 1], [100, 0, 129], seed=23)
    cfg = oracle.cfg_of(w)
    hc = gen.make_inputs(w, kv_dtype="e4m3")
    hp = gen.make_inputs(w, page_size=page_size, kv_dtype="e4m3")
    rc, rp = oracle.step(cfg, hc), oracle.step(cfg, hp)
    assert rc["bad"] == 0 and rp["bad"] == 0
    assert np.array_equal(rc["out"], rp["out"])
    pt = hp["page_table"]
    for b in range(w.batch):
        pos = torch.arange(w.cache_lens[b] + w.new_lens[b])
        sp = pt[b, pos // page_size].long() * page_size + pos % page_size
        sc = hc["slot_base"][b] + pos
        assert torch.equal(rp["k_cache"][sp], rc["k_cache"][sc]) and torch.equal(rp["v_cache"][sp], rc["v_cache"][sc])


# ---------------------------------------------------------------- projections around the step
def test_linear_matches_torch_fp64_matmul():
    g = torch.Generator().manual_seed(41)
    for N, C, O in ((3, 7, 5), (17, 64, 40), (64, 2560, 96)):
        x = torch.randn(N, C, generator=g).to(torch.bfloat16)
        w = torch.randn(O, C, generator=g).to(torch.bfloat16)
        ref = (x.double() @ w.double().T).numpy()
        np.testing.assert_allclose(oracle.linear(x, w), ref, rtol=1e-12, atol=1e-12)


def test_projected_prologue_with_identity_weights_is_the_plain_prologue():
    """hidden = the step's qkv and w_qkv = I: the projection reproduces the bf16
    qkv exactly, so the projected prologue must give the plain one's caches and
    queries bit for bit (V included: a bf16 value rounds to itself)."""
    w = gen.custom("proj_id", 8, 2, 64, [9, 4], [3, 0], seed=43)
    cfg = oracle.cfg_of(w)
    h = gen.make_inputs(w)
    eye = torch.eye(w.qkv_width, dtype=torch.bfloat16)
    plain = oracle.prologue(cfg, h)
    proj = oracle.prologue(cfg, h, qkv64=oracle.linear(h["qkv"], eye))
    assert torch.equal(plain[0].view(torch.int16), proj[0].view(torch.int16))
    assert torch.equal(plain[1].view(torch.int16), proj[1].view(torch.int16))
    assert np.array_equal(plain[2], proj[2])


def test_projected_step_rounds_v_once_and_applies_the_output_projection():
    w = gen.custom("proj_step", 8, 2, 64, [6, 3], [2, 5], seed=44)
    cfg = oracle.cfg_of(w)
    h = gen.make_inputs(w)
    pr = gen.make_projection_inputs(w, hidden=96, seed=44)
    r = oracle.projected_step(cfg, h, pr["hidden"], pr["w_qkv"], pr["w_o"])
    Hq, Hkv, D = w.num_q_heads, w.num_kv_heads, w.head_dim
    # V entries: the projection's V columns rounded once by torch's own fp64 -> bf16 conversion
    for b in range(w.batch):
        for j in range(w.new_lens[b]):
            t = int(h["cu_seqlens"][b]) + j
            slot = int(h["slot_base"][b]) + w.cache_lens[b] + j
            v64 = torch.from_numpy(r["qkv64"][t, (Hq + Hkv) * D:].reshape(Hkv, D).copy())
            assert torch.equal(r["v_cache"][slot].view(torch.int16), v64.to(torch.bfloat16).view(torch.int16))
    ref_o = torch.from_numpy(r["out"]).reshape(w.num_tokens, Hq * D) @ pr["w_o"].double().T
    np.testing.assert_allclose(r["o"], ref_o.numpy(), rtol=1e-12, atol=1e-12)
