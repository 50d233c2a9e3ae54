"""One packed attention step on the device: upload the inputs of a workload
and issue the C-ABI calls on the current stream.

A packed batch may mix prefill requests (several new tokens, possibly with a
cached prefix) and decode requests (one new token).  As the concept chapter's
section 4 puts it, prefill and decode are two stages of the same loop; here
the requests ``[0, decode_from)`` of a batch go through ``attn_prefill`` and
the requests ``[decode_from, B)`` through ``attn_decode``, back to back on
one stream, writing disjoint row ranges of one packed output.
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

    def run(self, stream=None) -> None:
        """Issue the step: prefill part then decode part (asynchronous)."""
        if self.kv_prefill is not None:
            attn.prefill(self.cfg, self.qkv[:self.n_prefill_tokens], self.q_norm_w, self.k_norm_w,
                         self.cu_seqlens, self.max_seqlen, self.kv_prefill,
                         self.out[:self.n_prefill_tokens], self.workspace, stream)
        if self.kv_decode is not None:
            attn.decode(self.cfg, self.qkv[self.n_prefill_tokens:], self.q_norm_w, self.k_norm_w,
                        self.max_cache_len, self.kv_decode, self.out[self.n_prefill_tokens:],
                        self.workspace, stream)

    def status(self) -> int:
        return attn.get_status(self.workspace)

    def launches(self) -> int:
        """Kernels one run() launches."""
        n = 2 if self.kv_prefill is not None else 0
        if self.kv_decode is not None:
            B = self.qkv.shape[0] - self.n_prefill_tokens
            n += 2 + (1 if attn.decode_splits(self.cfg, B, self.max_cache_len) > 1 else 0)
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
    return DeviceStep(
        cfg=cfg, qkv=dev(host["qkv"]), q_norm_w=dev(host["q_norm_w"]), k_norm_w=dev(host["k_norm_w"]),
        cu_seqlens=dev(host["cu_seqlens"][:df + 1]), kv_prefill=kv_p, kv_decode=kv_d,
        k_cache=k_cache, v_cache=v_cache, cache_lens=cache_lens, out=out, workspace=ws, n_prefill_tokens=n_pre,
        max_seqlen=max(list(w.new_lens[:df]) + [0]),
        max_cache_len=max(list(w.cache_lens[df:]) + [0]))
