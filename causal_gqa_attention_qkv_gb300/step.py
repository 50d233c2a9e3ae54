"""One packed attention step on the device: upload the inputs of a workload
and issue the C-ABI calls on the current stream.

A packed batch may mix prefill requests (several new tokens, possibly with a
cached prefix) and decode requests (one new token).  As the concept chapter's
section 4 puts it, prefill and decode are two stages of the same loop; here
the requests ``[0, decode_from)`` of a batch go through ``attn_prefill`` and
the requests ``[decode_from, B)`` through ``attn_decode``, writing disjoint
row ranges of one packed output and disjoint cache slots.  When a batch has
both, the decode call runs on a side stream beside the prefill call (with a
workspace of its own): the prefill part is bound by the tensor cores and the
decode part by HBM, so each fills the other's idle units.
"""
from __future__ import annotations

import dataclasses

import torch

from . import attn


@dataclasses.dataclass
class DeviceStep:
    """Device-resident tensors of one packed call plus its workspace."""

    cfg: attn.AttnConfig
    qkv: torch.Tensor
    q_norm_w: torch.Tensor
    k_norm_w: torch.Tensor
    cu_seqlens: torch.Tensor      # int32 [B_prefill + 1] (prefill part, rebased to 0)
    kv_prefill: attn.KVCache | None
    kv_decode: attn.KVCache | None
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    cache_lens: torch.Tensor      # int32 [B] (all requests; the kv views slice it)
    out: torch.Tensor
    workspace: torch.Tensor
    n_prefill_tokens: int
    max_seqlen: int
    max_cache_len: int            # largest cached length among decode requests
    decode_workspace: torch.Tensor | None = None  # the decode part's own, when both parts are present
    side_stream: torch.cuda.Stream | None = None  # where the decode part runs then

    def run(self, stream=None) -> None:
        """Issue the step (asynchronous): the prefill part, and the decode part
        beside it on a side stream when both are present (joined back into
        ``stream`` before this returns), else one after the other."""
        v = self.__dict__.get("_views")
        if v is None:  # the row ranges of the two parts, sliced once
            n = self.n_prefill_tokens
            v = (self.qkv[:n], self.out[:n], self.qkv[n:], self.out[n:])
            self.__dict__["_views"] = v
        side = None
        if self.kv_prefill is not None and self.kv_decode is not None and self.side_stream is not None:
            main = stream if stream is not None else torch.cuda.current_stream(self.out.device)
            side = self.side_stream
            side.wait_stream(main)
        if self.kv_prefill is not None:
            attn.prefill(self.cfg, v[0], self.q_norm_w, self.k_norm_w, self.cu_seqlens, self.max_seqlen,
                         self.kv_prefill, v[1], self.workspace, stream)
        if self.kv_decode is not None:
            ws = self.workspace if side is None else self.decode_workspace
            attn.decode(self.cfg, v[2], self.q_norm_w, self.k_norm_w, self.max_cache_len, self.kv_decode,
                        v[3], ws, stream if side is None else side)
        if side is not None:
            main.wait_stream(side)

    def status(self) -> int:
        st = attn.get_status(self.workspace)
        if self.decode_workspace is not None:
            st |= attn.get_status(self.decode_workspace)
        return st

    def launches(self) -> int:
        """Kernels one run() launches."""
        n = 2 if self.kv_prefill is not None else 0
        if self.kv_decode is not None:
            B = self.qkv.shape[0] - self.n_prefill_tokens
            n += 1 + (1 if attn.decode_splits(self.cfg, B, self.max_cache_len) > 1 else 0)
        return n


def upload(w, host: dict, device="cuda") -> DeviceStep:
    """Copy the host inputs of workload ``w`` (from ``inputs.make_inputs``) to
    the device and allocate the output and the workspace."""
    cfg = attn.config(w.num_q_heads, w.num_kv_heads, w.head_dim, w.rms_eps, w.rope_theta)
    dev = lambda t: t.to(device, non_blocking=False).contiguous()
    k_cache, v_cache = dev(host["k_cache"]), dev(host["v_cache"])
    df = w.decode_from
    n_pre = int(host["cu_seqlens"][df])
    slot_base, cache_lens, cap = dev(host["slot_base"]), dev(host["cache_lens"]), dev(host["slot_capacity"])
    pt = dev(host["page_table"]) if host.get("page_table") is not None else None
    ps = int(host.get("page_size", 0))
    scales = (float(host.get("k_scale", 1.0)), float(host.get("v_scale", 1.0)))
    part = lambda t, lo, hi: None if t is None else t[lo:hi].contiguous()
    kv_p = kv_d = None
    if df > 0:
        kv_p = attn.KVCache(k_cache, v_cache, slot_base[:df], cache_lens[:df], cap[:df],
                            part(pt, 0, df), ps, *scales)
    if df < w.batch:
        assert all(n == 1 for n in w.new_lens[df:]), "decode requests take one token each"
        kv_d = attn.KVCache(k_cache, v_cache, slot_base[df:], cache_lens[df:], cap[df:],
                            part(pt, df, w.batch), ps, *scales)
    N = w.num_tokens
    out = torch.zeros((N, w.num_q_heads * w.head_dim), dtype=torch.bfloat16, device=device)
    max_kv = max([c + n for c, n in zip(w.cache_lens, w.new_lens)] + [1])
    ws = attn.new_workspace(cfg, max(N, 1), max(w.batch, 1), max_kv, device)
    both = 0 < df < w.batch
    ws_dec = attn.new_workspace(cfg, 1, w.batch - df, max_kv, device) if both else None
    side = torch.cuda.Stream(out.device) if both else None
    return DeviceStep(
        cfg=cfg, qkv=dev(host["qkv"]), q_norm_w=dev(host["q_norm_w"]), k_norm_w=dev(host["k_norm_w"]),
        cu_seqlens=dev(host["cu_seqlens"][:df + 1]), kv_prefill=kv_p, kv_decode=kv_d,
        k_cache=k_cache, v_cache=v_cache, cache_lens=cache_lens, out=out, workspace=ws, n_prefill_tokens=n_pre,
        max_seqlen=max(list(w.new_lens[:df]) + [0]),
        max_cache_len=max(list(w.cache_lens[df:]) + [0]), decode_workspace=ws_dec, side_stream=side)


@dataclasses.dataclass
class _Chunk:
    t0: int
    t1: int
    b0: int
    b1: int             # requests [b0, b1) overlap the chunk
    max_seqlen: int
    cu: tuple           # offsets of the chunk's cu_seqlens and cached lengths in the metadata
    cl: tuple


@dataclasses.dataclass
class ChunkPlan:
    """Token chunks of one packed prefill call and their metadata: per chunk
    its cu_seqlens and the cached length of each request it touches (int32,
    in one pinned host buffer copied to the device with the first chunk)."""

    chunks: list
    meta_host: torch.Tensor
    meta_dev: torch.Tensor

    @property
    def h2d_bytes(self) -> int:
        return self.meta_host.numel() * 4


def plan_chunks(cu_seqlens, cache_lens, chunk_tokens):
    """Split a packed prefill call (host cu_seqlens [B + 1], cached lengths
    [B]) into calls of at most chunk_tokens tokens, in token order
    (chunk_tokens: one size, or the sizes of the first chunks, the last one
    repeated).  Chunk c covers tokens [t0, t1) and the requests [b0, b1) with
    tokens there; its own cu_seqlens counts each request's tokens inside the
    chunk, and each request's cached length is advanced by its tokens in
    earlier chunks.  Returns (chunks, metadata): the chunks' cu_seqlens and
    cached lengths are int32 runs of the metadata list at the offsets the
    chunks record."""
    sizes = [int(chunk_tokens)] if isinstance(chunk_tokens, int) else [int(x) for x in chunk_tokens]
    assert sizes and min(sizes) >= 1
    cu = [int(x) for x in cu_seqlens]
    cl = [int(x) for x in cache_lens]
    N = cu[-1]
    chunks, meta = [], []
    t0, b0 = 0, 0
    while t0 < N:
        t1 = min(N, t0 + sizes[min(len(chunks), len(sizes) - 1)])
        while cu[b0 + 1] <= t0:  # first request with a token at or after t0
            b0 += 1
        b1 = b0
        while b1 < len(cu) - 1 and cu[b1] < t1:
            b1 += 1
        ccu, ccl, mx = [0], [], 0
        for b in range(b0, b1):
            lo, hi = max(cu[b], t0), min(cu[b + 1], t1)
            n = max(0, hi - lo)
            ccu.append(ccu[-1] + n)
            ccl.append(cl[b] + max(0, lo - cu[b]))
            mx = max(mx, n)
        o = len(meta)
        meta += ccu + ccl
        chunks.append(_Chunk(t0, t1, b0, b1, mx, (o, o + len(ccu)), (o + len(ccu), o + len(ccu) + len(ccl))))
        t0 = t1
    return chunks, meta


class HostPrefill:
    """Prefill from pinned host buffers in token chunks, pipelined over five
    streams: the qkv rows of each chunk are copied in (one stream), prepared
    (K/V appended, Q normed and rotated; one stream, in chunk order), their
    attention runs on one of two streams in turn, each with a workspace of
    its own, and the output rows are copied out (one stream).  Chunk c + 1's
    attention needs only the cache entries of chunks 0 .. c + 1, so it can
    start on the SMs that chunk c's attention has already left.

    Each chunk is a valid packed prefill call of its own: the part of every
    request that falls in its token range, with that request's cached length
    advanced by the request's tokens in earlier chunks (the concept chapter's
    section 4: a long prompt may be prefilled in chunks over its own cache).
    The chunks run in order on one stream, so chunk c attends over the keys
    the earlier chunks appended; every output row is computed by the same
    kernels over the same key tiles as in one unchunked call.

    Device buffers (qkv, prepared Q, output, the KV cache and its index
    arrays, the workspace) belong to the caller and are reused across calls.
    """

    def __init__(self, cfg: attn.AttnConfig, q_norm_w, k_norm_w, kv: attn.KVCache, workspace, qkv_dev,
                 q_stage, out_dev, chunk_tokens=4096):
        self.cfg, self.q_norm_w, self.k_norm_w, self.kv = cfg, q_norm_w, k_norm_w, kv
        self.ws, self.qkv_dev, self.q_stage, self.out_dev = workspace, qkv_dev, q_stage, out_dev
        # one chunk size, or the sizes of the first chunks (the last repeated)
        self.chunk_tokens = (max(1, int(chunk_tokens)) if isinstance(chunk_tokens, int)
                             else [max(1, int(x)) for x in chunk_tokens])
        dev = qkv_dev.device
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_prep = torch.cuda.Stream(device=dev)
        self.s_att = (torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev))
        self.s_out = torch.cuda.Stream(device=dev)
        # one item counter per attention stream; attention alone needs only the workspace header
        self.ws_att = (workspace, attn.new_workspace(cfg, 0, 1, 1, device=dev))

    def plan(self, cu_seqlens, cache_lens) -> ChunkPlan:
        """Chunks of the packed batch given its host cu_seqlens [B + 1] and
        cached lengths [B]."""
        chunks, meta = plan_chunks(cu_seqlens, cache_lens, self.chunk_tokens)
        meta_host = torch.tensor(meta if meta else [0], dtype=torch.int32).pin_memory()
        meta_dev = torch.empty_like(meta_host, device=self.qkv_dev.device)
        return ChunkPlan(chunks, meta_host, meta_dev)

    def run(self, plan: ChunkPlan, qkv_host, out_host, start_event=None, end_event=None) -> int:
        """Issue the pipelined step (asynchronous; returns the kernel launches).
        qkv_host / out_host: pinned host tensors [N, W] / [N, Hq*D].  Optional
        events are recorded before the first copy and after the last one."""
        dev = self.qkv_dev.device
        cur = torch.cuda.current_stream(dev)
        kv, meta = self.kv, plan.meta_dev
        landed, done = [], []
        self.s_in.wait_stream(cur)
        with torch.cuda.stream(self.s_in):
            if start_event is not None:
                start_event.record(self.s_in)
            meta.copy_(plan.meta_host, non_blocking=True)
            for c in plan.chunks:
                self.qkv_dev[c.t0:c.t1].copy_(qkv_host[c.t0:c.t1], non_blocking=True)
                e = torch.cuda.Event()
                e.record(self.s_in)
                landed.append(e)
        prepped, ckvs = [], []
        with torch.cuda.stream(self.s_prep):
            for c, e in zip(plan.chunks, landed):
                self.s_prep.wait_event(e)
                cu_d = meta[c.cu[0]:c.cu[1]]
                ckv = attn.KVCache(kv.k_cache, kv.v_cache, kv.slot_base[c.b0:c.b1], meta[c.cl[0]:c.cl[1]],
                                   kv.slot_capacity[c.b0:c.b1],
                                   None if kv.page_table is None else kv.page_table[c.b0:c.b1],
                                   kv.page_size, kv.k_scale, kv.v_scale)
                attn.prefill_prepare(self.cfg, self.qkv_dev[c.t0:c.t1], self.q_norm_w, self.k_norm_w, cu_d, ckv,
                                     self.q_stage[c.t0:c.t1], self.ws, self.s_prep)
                e1 = torch.cuda.Event()
                e1.record(self.s_prep)  # also: the chunks before it are prepared
                prepped.append(e1)
                ckvs.append((cu_d, ckv))
        for i, (c, e1, (cu_d, ckv)) in enumerate(zip(plan.chunks, prepped, ckvs)):
            s = self.s_att[i % 2]
            s.wait_stream(cur)
            with torch.cuda.stream(s):
                s.wait_event(e1)
                attn.prefill_attend(self.cfg, self.q_stage[c.t0:c.t1], cu_d, c.max_seqlen, ckv,
                                    self.out_dev[c.t0:c.t1], self.ws_att[i % 2], s)
                e2 = torch.cuda.Event()
                e2.record(s)
                done.append(e2)
        with torch.cuda.stream(self.s_out):
            for c, e in zip(plan.chunks, done):
                self.s_out.wait_event(e)
                out_host[c.t0:c.t1].copy_(self.out_dev[c.t0:c.t1], non_blocking=True)
            if end_event is not None:
                end_event.record(self.s_out)
        cur.wait_stream(self.s_out)
        return 2 * len(plan.chunks)

    def status(self) -> int:
        """The device status words of both workspaces (0: no error)."""
        return max(attn.get_status(w) for w in self.ws_att)
