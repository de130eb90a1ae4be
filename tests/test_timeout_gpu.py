"""The bounded pipeline waits of the tcgen05 stage 1 run out without a
device fault.

Every mbarrier wait of the kernel is bounded: when the bound passes, the CTA
records PDA_STATUS_WAIT_TIMEOUT, raises its abort flag, drains what it issued,
frees its tensor memory and returns. To make a wait run out, the host sets
the PDA_INJECT_WITHHOLD_KV hook: the producer warps issue no K/V load at all,
so nothing asynchronous is in flight when the consumers give up, and a short
wait limit keeps the test fast. Nothing faults, traps or spins without a
bound. The next normal call on the same scratch (after pda_reset_status)
must again match the oracle.
"""
import pytest
import torch

from gpu_helpers import TOL_BF16, TOL_FP8, assert_close, dv_of, oracle_ref
from paged_split_kv_03_gb300 import binding as B
from paged_split_kv_03_gb300.synth import (SCALE_MLA_BLOCK, SCALE_TENSOR, SCALE_TOKEN_HEAD,
                                           make_workload)

pytestmark = pytest.mark.gpu

CASES = {
    "bf16_d128": (dict(batch=2, rows=[2, 1], kv_lens=[600, 300], num_qo_heads=16,
                       num_kv_heads=2, head_dim=128, page_size=16), TOL_BF16),
    "fp8pth_d256": (dict(batch=2, rows=[4, 8], kv_lens=[900, 400], num_qo_heads=16,
                         num_kv_heads=2, head_dim=256, page_size=16, kv_dtype="e4m3",
                         scale_mode=SCALE_TOKEN_HEAD), TOL_FP8),
    # the E4M3 MLA latent (V taken from the K unit in the ring) and the
    # mixed-precision records (their own softmax with five running maxima)
    "mla_fp8": (dict(batch=2, rows=[1, 1], kv_lens=[700, 300], num_qo_heads=16,
                     num_kv_heads=1, head_dim=576, head_dim_v=512, page_size=64,
                     kv_dtype="e4m3", q_dtype="e4m3", scale_mode=SCALE_TENSOR), TOL_FP8),
    "mla_records": (dict(batch=2, rows=[1, 2], kv_lens=[700, 300], num_qo_heads=16,
                         num_kv_heads=1, head_dim=576, head_dim_v=512, page_size=64,
                         kv_dtype="e4m3", scale_mode=SCALE_MLA_BLOCK), TOL_FP8),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_withheld_loads_time_out_and_the_next_call_is_correct(name):
    args, tol = CASES[name]
    wl = make_workload(name=name, seed=31, device="cuda", **args)
    # one split per request: no merge runs, so a timed-out CTA leaves its rows unwritten
    chunk = 4096
    bad = B.Decoder(B.params_for(wl, chunk_pages=chunk, kernel=B.PDA_KERNEL_TC,
                                 wait_limit_us=2000, inject=B.PDA_INJECT_WITHHOLD_KV))
    assert bad.plan.max_splits == 1 and bad.plan.wait_limit_us == 2000
    out = torch.full((wl.total_rows, wl.num_qo_heads, dv_of(wl)), float("nan"),
                     dtype=torch.bfloat16, device="cuda")
    lse = torch.full((wl.total_rows, wl.num_qo_heads), float("nan"), device="cuda")
    bad.run(wl, out, lse)
    torch.cuda.synchronize()  # the kernel returned: every wait was bounded
    assert bad.status() == B.PDA_STATUS_WAIT_TIMEOUT
    assert torch.isnan(out.float()).all() and torch.isnan(lse).all()

    good = B.Decoder(B.params_for(wl, chunk_pages=chunk, kernel=B.PDA_KERNEL_TC))
    assert good.plan.scratch_bytes == bad.plan.scratch_bytes
    good.scratch = bad.scratch  # the same scratch as the call that timed out
    good.reset_status()
    good.run(wl, out, lse)
    torch.cuda.synchronize()
    assert good.status() == 0
    ref_o, ref_l = oracle_ref(wl)
    assert_close(out.float().cpu(), lse.cpu(), ref_o, ref_l, tol, what=f"{name} after timeout")
