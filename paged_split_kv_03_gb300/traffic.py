"""Algorithmic bytes and flops of one paged decode call (the roofline's
numerator).

Byte model, per call (GB = 1e9 bytes):
  * K and V: every token a CTA has to stream, i.e. for each request the
    tokens [lo_page * P, L) -- from the first page that holds a visible key of
    any of its rows to its last token -- times Hkv * D * element size, for K
    and for V. Masked keys inside those pages count; pages wholly outside every
    row's window do not, and neither do the per-head re-reads the kernel
    avoids (each kv head's K/V counts once for all of its q heads).
  * per-(token, kv head) scales: 4 bytes per streamed token per kv head, for K
    and for V; per-tensor scales: 8 bytes.
  * Q read, out (bf16) and lse (fp32) written.
  * page-table entries read (one int32 per streamed page per request) and the
    int32 kv_indptr / kv_len / qo_indptr / window arrays.
  * split scratch: for every request with more than one KV split, each split
    writes and stage 2 reads (Dv + 1) fp32 per (row, q head).
  * MLA ("fp8 support", FlashMLA PR #54): one latent cache of D channels is
    both K and V (V its first Dv); it counts once, as the page's MBU does
    (the kernel reads V's channels again, from L2). Out has Dv channels.

With the scratch, lse and index terms left out this is the accounting of
"[Feature Request] Support q_len > 1 for FP8 decode" (hpc-ops issue #4): its
FP8 decode benchmark (bs 128, 64/8 heads, D 128, ctx 2048) reports
3672.1 GB/s at 6800 iter/s, which is (K+V at 1 B + Q at 1 B + O at 2 B) per
iteration; the golden test pins that.

Flops: 4 * D per (row, q head, visible key) -- QK^T and PV, two flops per
multiply-add.
"""
from __future__ import annotations


def _split_range(L, R, W, P, chunk_pages):
    p0 = L - R
    lo = max(0, p0 - W + 1) if W > 0 else 0
    lo_page = lo // P
    npages = -(-L // P)
    span = npages - lo_page
    nsplit = -(-span // chunk_pages) if span > 0 else 0
    return lo, lo_page, npages, nsplit


def call_bytes(wl, chunk_pages: int | None = None, include_scratch: bool = True,
               plan=None) -> dict:
    """Algorithmic bytes of one call on workload ``wl`` (a synth.Workload);
    ``chunk_pages`` is the plan's chunk (None: treat as one split). With a
    ``plan`` (a pda_plan_t), its chunk and its tail requests' shorter chunk
    are used instead."""
    tail_from, tail_chunk = None, None
    if plan is not None:
        chunk_pages, tail_from, tail_chunk = plan.chunk_pages, plan.tail_from, plan.tail_chunk_pages
    P, H, D, Hq = wl.page_size, wl.num_kv_heads, wl.head_dim, wl.num_qo_heads
    Dv = getattr(wl, "head_dim_v", None) or D
    mla = getattr(wl, "v_pages", None) is not None and wl.v_pages is getattr(wl, "k_pages", None)
    kv_terms = 1 if mla else 2
    kv_elt = 1 if (wl.kv_e4m3 or getattr(wl, "kv_int8", False)) else 2
    q_elt = 1 if wl.q_e4m3 else 2
    lens = wl.kv_len.cpu().tolist()
    qo = wl.qo_indptr.cpu().tolist()
    wins = wl.window.cpu().tolist() if wl.window is not None else [0] * len(lens)
    kv = scales = table = scratch = 0
    rows_total = qo[-1]
    for b, L in enumerate(lens):
        R = qo[b + 1] - qo[b]
        if R <= 0 or L < R:
            continue
        cp = tail_chunk if tail_from is not None and b >= tail_from else chunk_pages
        lo, lo_page, npages, nsplit = _split_range(L, R, wins[b], P, cp or 1 << 30)
        tokens = L - lo_page * P
        if wl.scale_mode == 3:  # MLA records: 512 codes + 64 bf16, four block scales
            kv += tokens * H * 640
            scales += tokens * H * 16
        else:
            kv += kv_terms * tokens * H * D * kv_elt
        if wl.scale_mode == 2:
            scales += kv_terms * tokens * H * 4
        table += (npages - lo_page) * 4
        if include_scratch and nsplit > 1:
            scratch += 2 * nsplit * R * Hq * (Dv + 1) * 4
    if wl.scale_mode == 1:
        scales += 4 * kv_terms
    q = rows_total * Hq * D * q_elt
    out = rows_total * Hq * Dv * 2
    lse = rows_total * Hq * 4
    index = 4 * (3 * len(lens) + 2) + (4 * len(lens) if wl.window is not None else 0)
    total = kv + scales + q + out + lse + table + index + scratch
    return dict(kv=kv, scales=scales, q=q, out=out, lse=lse, page_table=table, index=index,
                scratch=scratch, total=total)


def call_flops(wl) -> int:
    """2 * (D + Dv) per (row, q head, visible key): 4 * D unless MLA."""
    D, Hq = wl.head_dim, wl.num_qo_heads
    Dv = getattr(wl, "head_dim_v", None) or D
    lens = wl.kv_len.cpu().tolist()
    qo = wl.qo_indptr.cpu().tolist()
    wins = wl.window.cpu().tolist() if wl.window is not None else [0] * len(lens)
    visible = 0
    for b, L in enumerate(lens):
        R = qo[b + 1] - qo[b]
        for i in range(R):
            pos = L - R + i
            lo = max(0, pos - wins[b] + 1) if wins[b] > 0 else 0
            visible += pos - lo + 1
    return 2 * (D + Dv) * Hq * visible
