"""pda_decode_static: decode for callers that cannot allocate device memory.

A plugin whose host framework owns every device allocation (and hands it only
input and output pointers), or code that must not call cudaMalloc under its
host's memory budget, cannot supply pda_decode's split_scratch. For them the
library keeps the split scratch in its own fixed device array. These tests
call that entry point through the C ABI twice in a row, on two different
workloads, and check each result against pda_decode with a caller-provided
scratch: the two run the same kernels on the same plan, so their outputs must
agree bit for bit. The status word of the built-in array is read through
pda_get_status with a NULL scratch after every call. This file is named to
be collected last.
"""
import pytest
import torch

from paged_split_kv_03_gb300 import binding as B
from paged_split_kv_03_gb300.synth import SCALE_TOKEN_HEAD, make_workload


def _outputs(wl):
    o = torch.full((wl.total_rows, wl.num_qo_heads, wl.head_dim), float("nan"),
                   dtype=torch.bfloat16, device=wl.q.device)
    l_ = torch.full((wl.total_rows, wl.num_qo_heads), float("nan"), dtype=torch.float32,
                    device=wl.q.device)
    return o, l_


def _static(dec, wl, out, lse):
    B.pda_decode_static(dec.plan, wl.q, wl.k_pages, wl.v_pages, wl.page_table, wl.kv_indptr,
                        wl.kv_len, wl.qo_indptr, wl.max_q_len, wl.window, wl.sm_scale,
                        wl.k_scale, wl.v_scale, out, lse)


@pytest.mark.gpu
def test_static_scratch_matches_caller_scratch_twice_in_a_row():
    dev = "cuda"
    workloads = [
        make_workload(name="noalloc_bf16", batch=3, rows=[4, 1, 8], kv_lens=[3000, 700, 1500],
                      num_qo_heads=16, num_kv_heads=2, head_dim=256, page_size=16,
                      windows=[0, 64, 0], seed=71, device=dev),
        make_workload(name="noalloc_fp8", batch=2, rows=[2, 6], kv_lens=[5000, 999],
                      num_qo_heads=48, num_kv_heads=2, head_dim=128, page_size=32,
                      kv_dtype="e4m3", scale_mode=SCALE_TOKEN_HEAD, seed=72, device=dev),
    ]
    for wl in workloads:  # two calls in a row; the second finds the first's leftovers
        params = B.params_for(wl, chunk_pages=8)
        dec = B.Decoder(params)
        assert dec.plan.max_splits > 1  # the split scratch is really used
        ref_o, ref_l = _outputs(wl)
        dec.run(wl, ref_o, ref_l)
        out, lse = _outputs(wl)
        _static(dec, wl, out, lse)
        torch.cuda.synchronize()
        assert dec.status() == 0
        assert B.pda_get_status(dec.plan, None) == 0  # the built-in array's own status
        assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16)), wl.name
        assert torch.equal(lse, ref_l), wl.name


@pytest.mark.gpu
def test_static_call_reports_device_status():
    """A request with fewer cached tokens than rows is flagged in the built-in
    array's status word (read with a NULL scratch) and left unwritten; the
    next call clears the word first."""
    wl = make_workload(name="noalloc_status", batch=2, rows=[3, 2], kv_lens=[900, 400],
                       num_qo_heads=16, num_kv_heads=2, head_dim=128, page_size=16, seed=73,
                       device="cuda")
    dec = B.Decoder(B.params_for(wl, chunk_pages=4, max_kv_len=1024))
    good_len = wl.kv_len.clone()
    wl.kv_len[0] = 2  # fewer tokens than its 3 rows
    out, lse = _outputs(wl)
    _static(dec, wl, out, lse)
    assert B.pda_get_status(dec.plan, None) & B.PDA_STATUS_KV_LEN_LT_ROWS
    assert torch.isnan(out[:3].float()).all()  # the flagged request is not written
    wl.kv_len.copy_(good_len)
    out2, lse2 = _outputs(wl)
    _static(dec, wl, out2, lse2)
    assert B.pda_get_status(dec.plan, None) == 0
    B.pda_reset_status(dec.plan, None)
    assert B.pda_get_status(dec.plan, None) == 0
    ref_o, ref_l = _outputs(wl)
    dec.run(wl, ref_o, ref_l)
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), ref_o.view(torch.int16))


def test_static_scratch_rejects_plans_larger_than_the_array():
    """A plan whose split scratch exceeds the built-in array is refused with
    PDA_ERR_TOO_LARGE before anything touches a device."""
    p = B.PdaParams()
    for k, v in dict(num_qo_heads=64, num_kv_heads=8, head_dim=256, page_size=16, q_dtype=0,
                     kv_dtype=0, scale_mode=0, max_batch=512, max_q_len=8, max_kv_len=131072,
                     num_pages=1 << 20, kv_stride_page=16 * 8 * 256, kv_stride_token=8 * 256,
                     kv_stride_head=256, device=0, num_sms=152, batch=0, chunk_pages=16,
                     kernel=0).items():
        setattr(p, k, v)
    plan, nbytes, _ = B.pda_plan(p)
    assert nbytes > B.PDA_STATIC_SCRATCH_BYTES
    fake = 1 << 20
    rc = B.pda_decode_static(plan, fake, fake, fake, fake, fake, fake, fake, 8, None, 0.1, None,
                             None, fake, fake, stream=0, check=False)
    assert rc == B.PDA_ERR_TOO_LARGE
    assert "scratch" in B.pda_strerror(rc)
    # the host checks come first: a NULL query is refused as such
    rc = B.pda_decode_static(plan, None, fake, fake, fake, fake, fake, fake, 8, None, 0.1, None,
                             None, fake, fake, stream=0, check=False)
    assert rc == B.PDA_ERR_NULL
