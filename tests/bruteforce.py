"""Dense fp64 attention written with torch library routines, for tiny inputs.

This is the check the oracle is pinned to. It shares nothing with the oracle's
C code: it gathers each request's pages into a dense [L, Hkv, D] tensor with
tensor indexing, dequantises with torch's own float8_e4m3fn conversion, expands
the GQA groups with ``repeat_interleave``, builds an explicit boolean
[rows, L] mask and calls ``torch.softmax`` / ``torch.logsumexp``.

The mask follows "perf(attention): run up to 8 query rows per request in the
triton decode kernel", section "Changes": row i of a request with R rows over
L cached keys sits at position L - R + i and sees keys j <= that position;
with a window W > 0 it also needs j >= position - W + 1.
"""
from __future__ import annotations

import math

import torch


def dequant_cache(wl, which: str) -> torch.Tensor:
    """[num_pages, P, Hkv, D] float64 values of the K or V cache."""
    c = wl.k_pages if which == "k" else wl.v_pages
    s = wl.k_scale if which == "k" else wl.v_scale
    c = c.cpu()
    if wl.layout == "HND":
        c = c.permute(0, 2, 1, 3)
    if wl.scale_mode == 3:
        # MLA record: 512 E4M3 codes x a scale per 128 channels, then 64 bf16
        c = c.contiguous()
        nope = c[..., :512].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
        sc = s.cpu().to(torch.float64).repeat_interleave(128, dim=-1)
        rope = c[..., 512:].contiguous().view(torch.bfloat16).to(torch.float64)
        return torch.cat([nope * sc, rope], dim=-1)
    if wl.kv_e4m3:
        x = c.contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    elif getattr(wl, "kv_int8", False):
        x = c.contiguous().view(torch.int8).to(torch.float64)
    else:
        x = c.to(torch.float64)
    if wl.scale_mode == 1:
        x = x * s.cpu().to(torch.float64)[0]
    elif wl.scale_mode == 2:
        x = x * s.cpu().to(torch.float64)[..., None]
    return x


def dequant_q(wl) -> torch.Tensor:
    q = wl.q.cpu()
    if wl.q_e4m3:
        return q.contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    return q.to(torch.float64)


def visibility_mask(L: int, R: int, window: int) -> torch.Tensor:
    pos = torch.arange(R) + (L - R)
    j = torch.arange(L)
    m = j[None, :] <= pos[:, None]
    if window > 0:
        m &= j[None, :] >= (pos[:, None] - window + 1)
    return m


def dense_attention(wl):
    """(out [rows, Hq, Dv], lse [rows, Hq]) in float64."""
    P, H, Hq = wl.page_size, wl.num_kv_heads, wl.num_qo_heads
    G = Hq // H
    kd, vd = dequant_cache(wl, "k"), dequant_cache(wl, "v")
    qd = dequant_q(wl)
    total = qd.shape[0]
    dv = getattr(wl, "head_dim_v", None) or wl.head_dim  # MLA: V = the first dv channels
    out = torch.full((total, Hq, dv), float("nan"), dtype=torch.float64)
    lse = torch.full((total, Hq), float("nan"), dtype=torch.float64)
    qo = wl.qo_indptr.cpu().tolist()
    kvi = wl.kv_indptr.cpu().tolist()
    lens = wl.kv_len.cpu().tolist()
    table = wl.page_table.cpu().long()
    wins = wl.window.cpu().tolist() if wl.window is not None else [0] * len(lens)
    for b, L in enumerate(lens):
        R = qo[b + 1] - qo[b]
        if R == 0:
            continue
        npg = math.ceil(L / P)
        pages = table[kvi[b]:kvi[b] + npg]
        K = kd[pages].reshape(npg * P, H, -1)[:L].repeat_interleave(G, dim=1)
        V = vd[pages].reshape(npg * P, H, -1)[:L, :, :dv].repeat_interleave(G, dim=1)
        qb = qd[qo[b]:qo[b + 1]]
        s = torch.einsum("rhd,lhd->rhl", qb, K) * wl.sm_scale
        mask = visibility_mask(L, R, wins[b])
        s = s.masked_fill(~mask[:, None, :], float("-inf"))
        out[qo[b]:qo[b + 1]] = torch.einsum("rhl,lhd->rhd", torch.softmax(s, dim=-1), V)
        lse[qo[b]:qo[b + 1]] = torch.logsumexp(s, dim=-1)
    return out, lse
