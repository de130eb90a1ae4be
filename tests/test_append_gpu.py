"""GPU parity of quantise-on-append (pda_append_kv) against the oracle:
every byte of both caches and every scale must match exactly, for the three
cache kinds (bf16 copy, E4M3 and int8 per tensor and per token and kv head), head
dims 64 / 128 / 256 / 512, both cache layouts, ragged rows per request, and the
status bits of requests the kernel must skip."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_split_kv_03_gb300 import binding as B
from paged_split_kv_03_gb300.synth import SCALE_NONE, SCALE_TENSOR, SCALE_TOKEN_HEAD, make_workload

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)

CASES = {
    "pth_d256_p16": dict(kv_dtype="e4m3", scale_mode=SCALE_TOKEN_HEAD, head_dim=256, page_size=16,
                         rows=[1, 8, 3, 0], kv_lens=[40, 300, 3, 17], num_qo_heads=16,
                         num_kv_heads=2),
    "pth_d128_p64_hnd": dict(kv_dtype="e4m3", scale_mode=SCALE_TOKEN_HEAD, head_dim=128,
                             page_size=64, rows=[2, 5], kv_lens=[2, 700], num_qo_heads=64,
                             num_kv_heads=8, layout="HND"),
    "pth_d64_p8": dict(kv_dtype="e4m3", scale_mode=SCALE_TOKEN_HEAD, head_dim=64, page_size=8,
                       rows=[4, 1, 2], kv_lens=[9, 8, 31], num_qo_heads=6, num_kv_heads=3),
    "tensor_d128_p64": dict(kv_dtype="e4m3", scale_mode=SCALE_TENSOR, head_dim=128, page_size=64,
                            rows=1, kv_lens=[2048, 65, 64, 1, 900], num_qo_heads=64,
                            num_kv_heads=8),
    "bf16_d256_p16": dict(kv_dtype="bf16", scale_mode=SCALE_NONE, head_dim=256, page_size=16,
                          rows=[4, 1], kv_lens=[33, 16], num_qo_heads=16, num_kv_heads=2),
    "pth_d512_p16": dict(kv_dtype="e4m3", scale_mode=SCALE_TOKEN_HEAD, head_dim=512,
                         page_size=16, rows=[2, 8], kv_lens=[40, 300], num_qo_heads=16,
                         num_kv_heads=1),
    "i8pth_d128_p16": dict(kv_dtype="int8", scale_mode=SCALE_TOKEN_HEAD, head_dim=128,
                           page_size=16, rows=[8, 1, 3], kv_lens=[300, 17, 3], num_qo_heads=16,
                           num_kv_heads=2),
    "i8t_d256_p64_hnd": dict(kv_dtype="int8", scale_mode=SCALE_TENSOR, head_dim=256, page_size=64,
                             rows=[2, 5], kv_lens=[2, 700], num_qo_heads=16, num_kv_heads=2,
                             layout="HND"),
    "bf16_d512_p64_hnd": dict(kv_dtype="bf16", scale_mode=SCALE_NONE, head_dim=512,
                              page_size=64, rows=[3], kv_lens=[70], num_qo_heads=4,
                              num_kv_heads=2, layout="HND"),
}


def _mode(wl):
    if getattr(wl, "kv_int8", False):
        return (oracle.APPEND_INT8_TENSOR if wl.scale_mode == SCALE_TENSOR
                else oracle.APPEND_INT8_TOKEN_HEAD)
    if not wl.kv_e4m3:
        return oracle.APPEND_BF16
    return oracle.APPEND_TENSOR if wl.scale_mode == SCALE_TENSOR else oracle.APPEND_TOKEN_HEAD


def _setup(args, seed=0):
    args = dict(args)
    args.setdefault("batch", len(args["kv_lens"]))
    wl = make_workload(name="append", seed=seed + 31, device="cpu", **args)
    rows = wl.total_rows
    g = torch.Generator().manual_seed(seed + 7)
    k_new = (torch.randn(rows, wl.num_kv_heads, wl.head_dim, generator=g) * 2).to(torch.bfloat16)
    v_new = (torch.randn(rows, wl.num_kv_heads, wl.head_dim, generator=g) * 2).to(torch.bfloat16)
    if rows:
        k_new[0, 0] = 0  # a zero row: scale 1, codes 0
        k_new[-1, -1, 0] = 500.0  # a peak far above the rest of its row
    return wl, k_new, v_new


def _run(wl, k_new, v_new):
    dwl = wl.to(DEV)
    dec = B.Decoder(B.params_for(dwl), device=DEV)
    dec.reset_status()
    k_pages, v_pages = dwl.k_pages.clone(), dwl.v_pages.clone()
    ks = None if dwl.k_scale is None else dwl.k_scale.clone()
    vs = None if dwl.v_scale is None else dwl.v_scale.clone()
    B.pda_append_kv(dec.plan, k_new.to(DEV), v_new.to(DEV), dwl.page_table, dwl.kv_indptr,
                    dwl.kv_len, dwl.qo_indptr, max(1, wl.max_q_len), k_pages, v_pages, ks, vs,
                    dec.scratch)
    torch.cuda.synchronize()
    return k_pages.cpu(), v_pages.cpu(), ks, vs, dec.status()


def _oracle(wl, k_new, v_new):
    return oracle.append_kv(k_new=k_new, v_new=v_new, page_table=wl.page_table,
                            kv_indptr=wl.kv_indptr, kv_len=wl.kv_len, qo_indptr=wl.qo_indptr,
                            k_pages=wl.k_pages, v_pages=wl.v_pages, k_scale=wl.k_scale,
                            v_scale=wl.v_scale, num_kv_heads=wl.num_kv_heads,
                            head_dim=wl.head_dim, page_size=wl.page_size, mode=_mode(wl),
                            strides=wl.strides, num_pages=wl.num_pages)


def _bytes(t):
    t = t.contiguous()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy().view(np.uint8).reshape(-1)


@pytest.mark.parametrize("name", sorted(CASES))
def test_append_bit_exact(name):
    wl, k_new, v_new = _setup(CASES[name])
    k_pages, v_pages, ks, vs, status = _run(wl, k_new, v_new)
    assert status == 0
    kc, vc, rks, rvs, rc = _oracle(wl, k_new, v_new)
    assert rc == 0
    assert np.array_equal(_bytes(k_pages), kc.reshape(-1)), "K cache bytes differ"
    assert np.array_equal(_bytes(v_pages), vc.reshape(-1)), "V cache bytes differ"
    if wl.scale_mode == SCALE_TOKEN_HEAD:
        assert np.array_equal(ks.cpu().numpy().reshape(-1).view(np.uint32),
                              rks.reshape(-1).view(np.uint32)), "K scales differ"
        assert np.array_equal(vs.cpu().numpy().reshape(-1).view(np.uint32),
                              rvs.reshape(-1).view(np.uint32)), "V scales differ"


def test_append_then_decode_reads_the_new_tokens():
    """Decode over a cache the kernel appended to matches the oracle over the
    cache the oracle appended to (the same bytes, so this is the decode path
    seeing the appended rows through its own page-table reads)."""
    wl, k_new, v_new = _setup(CASES["pth_d256_p16"], seed=3)
    k_pages, v_pages, ks, vs, status = _run(wl, k_new, v_new)
    assert status == 0
    wl.k_pages, wl.v_pages, wl.k_scale, wl.v_scale = k_pages, v_pages, ks.cpu(), vs.cpu()
    dwl = wl.to(DEV)
    dec = B.Decoder(B.params_for(dwl), device=DEV)
    out = torch.empty(wl.total_rows, wl.num_qo_heads, wl.head_dim, dtype=torch.bfloat16,
                      device=DEV)
    lse = torch.empty(wl.total_rows, wl.num_qo_heads, dtype=torch.float32, device=DEV)
    dec.run(dwl, out, lse)
    torch.cuda.synchronize()
    assert dec.status() == 0
    ref_o, ref_l, rc = oracle.attention_for(wl)
    assert rc == 0
    err = np.abs(out.float().cpu().numpy().reshape(ref_o.shape) - ref_o)
    assert err.max() <= 3e-2 and err.mean() <= 3e-3
    assert np.abs(lse.cpu().numpy().reshape(-1) - ref_l).max() <= 1e-3


def test_append_mla_records_bit_exact_then_decode():
    """MLA records: the new rows' latents -> E4M3 nope codes with a scale per
    128 channels and bf16 rope, byte-exact against the oracle; decode over the
    appended cache then matches the oracle on it."""
    args = dict(batch=3, rows=[2, 1, 1], kv_lens=[300, 65, 2], num_qo_heads=16, num_kv_heads=1,
                head_dim=576, head_dim_v=512, page_size=64, kv_dtype="e4m3", scale_mode=3)
    wl = make_workload(name="append_mla", seed=41, device="cpu", **args)
    g = torch.Generator().manual_seed(42)
    k_new = (torch.randn(wl.total_rows, 1, 576, generator=g) * 2).to(torch.bfloat16)
    k_new[0, 0, 128:256] = 0  # a zero block: scale 0, codes 0
    dwl = wl.to(DEV)
    dec = B.Decoder(B.params_for(dwl), device=DEV)
    dec.reset_status()
    pages, scales = dwl.k_pages.clone(), dwl.k_scale.clone()
    B.pda_append_kv(dec.plan, k_new.to(DEV), None, dwl.page_table, dwl.kv_indptr, dwl.kv_len,
                    dwl.qo_indptr, max(1, wl.max_q_len), pages, None, scales, None, dec.scratch)
    torch.cuda.synchronize()
    assert dec.status() == 0
    kc, _, ks, _, rc = oracle.append_kv(
        k_new=k_new, v_new=None, page_table=wl.page_table, kv_indptr=wl.kv_indptr,
        kv_len=wl.kv_len, qo_indptr=wl.qo_indptr, k_pages=wl.k_pages, v_pages=None,
        k_scale=wl.k_scale, v_scale=None, num_kv_heads=1, head_dim=576, page_size=64,
        mode=oracle.APPEND_MLA_RECORD, strides=wl.strides, num_pages=wl.num_pages)
    assert rc == 0
    assert np.array_equal(_bytes(pages.cpu()), kc.reshape(-1)), "record bytes differ"
    assert np.array_equal(scales.cpu().numpy().reshape(-1).view(np.uint32),
                          ks.reshape(-1).view(np.uint32)), "block scales differ"
    # decode over the appended records
    wl.k_pages = wl.v_pages = pages.cpu()
    wl.k_scale = wl.v_scale = scales.cpu()
    dwl = wl.to(DEV)
    out = torch.empty(wl.total_rows, 16, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(wl.total_rows, 16, dtype=torch.float32, device=DEV)
    dec.run(dwl, out, lse)
    torch.cuda.synchronize()
    assert dec.status() == 0
    ref_o, ref_l, rc = oracle.attention_for(wl)
    assert rc == 0
    err = np.abs(out.float().cpu().numpy().reshape(ref_o.shape) - ref_o)
    assert err.max() <= 3e-2 and err.mean() <= 3e-3
    assert np.abs(lse.cpu().numpy().reshape(-1) - ref_l).max() <= 1e-3


def test_append_status_and_isolation():
    """A request whose page id is out of range, and one with kv_len < rows,
    set their status bits and are skipped; the other requests are written."""
    wl, k_new, v_new = _setup(CASES["pth_d256_p16"], seed=5)
    pt = wl.page_table.clone()
    b_bad = 1  # request 1: its last page id out of range
    last = int(wl.kv_indptr[b_bad]) + (int(wl.kv_len[b_bad]) - 1) // wl.page_size
    pt[last] = wl.num_pages + 5
    wl.page_table = pt
    kl = wl.kv_len.clone()
    kl[2] = 1  # request 2 has 3 rows
    wl.kv_len = kl
    k_pages, v_pages, ks, vs, status = _run(wl, k_new, v_new)
    assert status & B.PDA_STATUS_PAGE_OOB and status & B.PDA_STATUS_KV_LEN_LT_ROWS
    kc, vc, rks, rvs, rc = _oracle(wl, k_new, v_new)
    assert rc != 0
    assert np.array_equal(_bytes(k_pages), kc.reshape(-1))
    assert np.array_equal(_bytes(v_pages), vc.reshape(-1))
