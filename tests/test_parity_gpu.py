"""GPU parity: the CUDA library (called through its C ABI) against the fp64
oracle on the same seeded inputs, element by element, plus bit-exact
structured cases for the page gather and the masks, the invariants, CUDA-graph
replay and the device status bits.

The semantics are those of "perf(attention): run up to 8 query rows per
request in the triton decode kernel" (FreeToken PR #900), "Changes": rows
limited to their own position and window, per-row merge of the KV split,
q heads per CTA dividing the GQA group (48 query / 2 kv heads included).
"""
import math

import numpy as np
import pytest
import torch

from gpu_helpers import (TOL_BF16, TOL_FP8, assert_close, dv_of, oracle_ref, run_decode,
                         sample_items, tol_for)
from paged_split_kv_03_gb300 import binding as B
from paged_split_kv_03_gb300.synth import (SCALE_NONE, SCALE_TENSOR, SCALE_TOKEN_HEAD,
                                           config_workload, make_workload)

pytestmark = pytest.mark.gpu
DEV = "cuda"

# Small workloads the oracle checks in full. Each spans several tiles, ragged
# tails, forced multi-chunk splits and the degenerate cases (R = 0 requests,
# one-token contexts, windows of 1, page sizes below and above the 64-token
# tile, G = 1 / 3 / 8 / 16 / 24 / 48).
SMALL = {
    "bf16_d128_g8_r1": dict(batch=3, rows=1, kv_lens=[512, 77, 1], num_qo_heads=16,
                            num_kv_heads=2, head_dim=128, page_size=16),
    "bf16_d256_g8_r4_split": dict(batch=2, rows=4, kv_lens=[3000, 1203], num_qo_heads=16,
                                  num_kv_heads=2, head_dim=256, page_size=16, chunk=16),
    "bf16_d128_g24_mixed_win": dict(batch=8, rows=[1, 2, 3, 4, 5, 6, 7, 8],
                                    kv_lens=[700, 2100, 999, 1500, 64, 8, 1025, 1800],
                                    windows=[64, 0, 64, 0, 1, 0, 5, 0], num_qo_heads=48,
                                    num_kv_heads=2, head_dim=128, page_size=32, chunk=8),
    "bf16_d64_g3_hnd": dict(batch=3, rows=8, kv_lens=[9, 100, 1000], num_qo_heads=6,
                            num_kv_heads=2, head_dim=64, page_size=16, layout="HND", chunk=4),
    "fp8t_qfp8_d128_g8": dict(batch=8, rows=1, kv_lens=2048, num_qo_heads=64, num_kv_heads=8,
                              head_dim=128, page_size=64, kv_dtype="e4m3", q_dtype="e4m3",
                              scale_mode=SCALE_TENSOR),
    "fp8pth_d256_g8_outliers": dict(batch=3, rows=[1, 4, 8], kv_lens=[4000, 5000, 33],
                                    num_qo_heads=16, num_kv_heads=2, head_dim=256, page_size=16,
                                    kv_dtype="e4m3", scale_mode=SCALE_TOKEN_HEAD,
                                    k_outlier_frac=0.01, chunk=32),
    "fp8pth_qfp8_d128_g1_p8": dict(batch=2, rows=2, kv_lens=[300, 5], num_qo_heads=8,
                                   num_kv_heads=8, head_dim=128, page_size=8, kv_dtype="e4m3",
                                   q_dtype="e4m3", scale_mode=SCALE_TOKEN_HEAD, windows=[17, 0]),
    "fp8t_d256_g16_p128": dict(batch=2, rows=4, kv_lens=[1500, 130], num_qo_heads=16,
                               num_kv_heads=1, head_dim=256, page_size=128, kv_dtype="e4m3",
                               scale_mode=SCALE_TENSOR, chunk=2),
    "fp8t_d128_g24_r2": dict(batch=2, rows=[2, 1], kv_lens=[1800, 700], num_qo_heads=48,
                             num_kv_heads=2, head_dim=128, page_size=32, kv_dtype="e4m3",
                             scale_mode=SCALE_TENSOR, chunk=16),
    "fp8t_qfp8_d128_g8_r38": dict(batch=2, rows=[3, 8], kv_lens=[1000, 2500], num_qo_heads=16,
                                  num_kv_heads=2, head_dim=128, page_size=16, kv_dtype="e4m3",
                                  q_dtype="e4m3", scale_mode=SCALE_TENSOR),
    "bf16_d128_g48_rows": dict(batch=4, rows=[1, 2, 3, 8], kv_lens=700, num_qo_heads=48,
                               num_kv_heads=1, head_dim=128, page_size=16),
    "bf16_zero_row_requests": dict(batch=4, rows=[0, 3, 0, 1], kv_lens=[50, 260, 7, 1],
                                   num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=16),
    "bf16_p256": dict(batch=2, rows=3, kv_lens=[600, 257], num_qo_heads=4, num_kv_heads=2,
                      head_dim=128, page_size=256, windows=[100, 0]),
    "bf16_p1": dict(batch=2, rows=2, kv_lens=[130, 3], num_qo_heads=4, num_kv_heads=2,
                    head_dim=64, page_size=1, chunk=64),
    # head_dim 512 (tcgen05 path only): one kv head, G = 16 / 8 / 2
    # int8 caches: both scale kinds, windows, HND, head_dim 64-256
    "i8t_d128_g8_win": dict(batch=3, rows=[1, 4, 8], kv_lens=[700, 1500, 33],
                            windows=[0, 64, 0], num_qo_heads=16, num_kv_heads=2, head_dim=128,
                            page_size=16, kv_dtype="int8", scale_mode=SCALE_TENSOR),
    "i8pth_d256_g8_split": dict(batch=2, rows=[8, 2], kv_lens=[2000, 300], num_qo_heads=16,
                                num_kv_heads=2, head_dim=256, page_size=16, kv_dtype="int8",
                                scale_mode=SCALE_TOKEN_HEAD, k_outlier_frac=0.01, chunk=16),
    "i8pth_d64_g3_hnd": dict(batch=3, rows=8, kv_lens=[9, 100, 1000], num_qo_heads=6,
                             num_kv_heads=2, head_dim=64, page_size=16, layout="HND",
                             kv_dtype="int8", scale_mode=SCALE_TOKEN_HEAD, chunk=4),
    "bf16_d512_g16_r148": dict(batch=3, rows=[1, 4, 8], kv_lens=[700, 1500, 33],
                               windows=[0, 64, 0], num_qo_heads=16, num_kv_heads=1,
                               head_dim=512, page_size=16, chunk=4),
    "bf16_d512_g2_p64": dict(batch=2, rows=[8, 2], kv_lens=[900, 130], num_qo_heads=4,
                             num_kv_heads=2, head_dim=512, page_size=64, layout="HND"),
    "fp8pth_d512_g16": dict(batch=2, rows=[8, 3], kv_lens=[1300, 260], num_qo_heads=16,
                            num_kv_heads=1, head_dim=512, page_size=64, kv_dtype="e4m3",
                            scale_mode=SCALE_TOKEN_HEAD, chunk=8),
    "bf16_d512_g16_r2": dict(batch=2, rows=[2, 1], kv_lens=[600, 1300], num_qo_heads=16,
                             num_kv_heads=1, head_dim=512, page_size=32),
    # MLA latents (576 channels, V = the first 512): bf16, E4M3 per tensor / per token
    "mla_bf16_split_win": dict(batch=3, rows=[1, 2, 1], kv_lens=[700, 1300, 65],
                               windows=[0, 0, 32], num_qo_heads=16, num_kv_heads=1,
                               head_dim=576, head_dim_v=512, page_size=64, chunk=4),
    "mla_fp8t_g16": dict(batch=2, rows=[2, 1], kv_lens=[1000, 130], num_qo_heads=16,
                         num_kv_heads=1, head_dim=576, head_dim_v=512, page_size=16,
                         kv_dtype="e4m3", q_dtype="e4m3", scale_mode=SCALE_TENSOR),
    "mla_fp8pth_g8_p32": dict(batch=2, rows=[1, 2], kv_lens=[333, 2100], num_qo_heads=8,
                              num_kv_heads=1, head_dim=576, head_dim_v=512, page_size=32,
                              kv_dtype="e4m3", q_dtype="e4m3", scale_mode=SCALE_TOKEN_HEAD,
                              chunk=8),
    "mla_mix_split_win": dict(batch=3, rows=[1, 2, 1], kv_lens=[700, 1300, 65],
                              windows=[0, 0, 32], num_qo_heads=16, num_kv_heads=1,
                              head_dim=576, head_dim_v=512, page_size=64, kv_dtype="e4m3",
                              scale_mode=3, chunk=4),
    "mla_mix_g8_hnd_p16": dict(batch=2, rows=[2, 1], kv_lens=[1000, 130], num_qo_heads=8,
                               num_kv_heads=1, head_dim=576, head_dim_v=512, page_size=16,
                               kv_dtype="e4m3", scale_mode=3, layout="HND"),
    "fp8t_qfp8_d512_g8": dict(batch=2, rows=[2, 1], kv_lens=[1000, 129], num_qo_heads=8,
                              num_kv_heads=1, head_dim=512, page_size=32, kv_dtype="e4m3",
                              q_dtype="e4m3", scale_mode=SCALE_TENSOR),
}
# peaked stress cases (Q x 4): compared with the bf16 output's half-ulp added;
# the running maxima move often, so the lazy O rescale runs
PEAKED_SMALL = {
    "bf16": dict(batch=2, rows=[4, 8], kv_lens=[2000, 900], num_qo_heads=16, num_kv_heads=2,
                 head_dim=256, page_size=16, q_mult=4.0, chunk=16),
    "fp8pth": dict(batch=2, rows=[4, 8], kv_lens=[2000, 900], num_qo_heads=16, num_kv_heads=2,
                   head_dim=256, page_size=16, q_mult=4.0, chunk=16, kv_dtype="e4m3",
                   scale_mode=SCALE_TOKEN_HEAD),
    "i8pth": dict(batch=2, rows=[4, 8], kv_lens=[2000, 900], num_qo_heads=16, num_kv_heads=2,
                  head_dim=256, page_size=16, q_mult=4.0, chunk=16, kv_dtype="int8",
                  scale_mode=SCALE_TOKEN_HEAD),
    "bf16_d512": dict(batch=2, rows=[4, 8], kv_lens=[2000, 900], num_qo_heads=16,
                      num_kv_heads=1, head_dim=512, page_size=16, q_mult=4.0, chunk=16),
    "fp8pth_d512": dict(batch=2, rows=[4, 8], kv_lens=[2000, 900], num_qo_heads=16,
                        num_kv_heads=1, head_dim=512, page_size=16, q_mult=4.0, chunk=16,
                        kv_dtype="e4m3", scale_mode=SCALE_TOKEN_HEAD),
}


def _make(name, args, seed=0):
    args = dict(args)
    chunk = args.pop("chunk", 0)
    wl = make_workload(name=name, seed=seed + 17, device=DEV, **args)
    return wl, chunk


KERNELS = {"mma": B.PDA_KERNEL_MMA, "tc": B.PDA_KERNEL_TC}


def _tc_ok(wl):
    """Shapes the tcgen05 path is built for (head_dim 128/256/512, pages of >= 8;
    int8 caches up to head_dim 256)."""
    return (wl.head_dim in (128, 256, 512, 576) and wl.page_size >= 8 and
            (not wl.kv_int8 or wl.head_dim <= 256))


def _mma_ok(wl):
    """Shapes the mma.sync path is built for (head_dim up to 256)."""
    return wl.head_dim <= 256


def _refused(wl, chunk, kernel):
    """A shape one path is not built for: its plan is refused up front with
    PDA_ERR_UNSUPPORTED (nothing is launched)."""
    p = B.params_for(wl, chunk_pages=chunk, kernel=KERNELS[kernel])
    assert B.pda_plan(p, check=False)[2] == B.PDA_ERR_UNSUPPORTED


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_full_parity(name, kernel):
    wl, chunk = _make(name, SMALL[name])
    if not (_tc_ok(wl) if kernel == "tc" else _mma_ok(wl)):
        return _refused(wl, chunk, kernel)
    out, lse, status, dec = run_decode(wl, chunk_pages=chunk, kernel=KERNELS[kernel])
    assert status == 0
    ref_o, ref_l = oracle_ref(wl)
    assert_close(out, lse, ref_o, ref_l, tol_for(wl), what=f"{name}/{kernel}")


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("kind", sorted(PEAKED_SMALL))
def test_small_peaked_parity(kind, kernel):
    wl, chunk = _make(f"{kind}_peaked", PEAKED_SMALL[kind])
    if not (_tc_ok(wl) if kernel == "tc" else _mma_ok(wl)):
        return _refused(wl, chunk, kernel)
    out, lse, status, dec = run_decode(wl, chunk_pages=chunk, kernel=KERNELS[kernel])
    assert status == 0
    ref_o, ref_l = oracle_ref(wl)
    assert_close(out, lse, ref_o, ref_l, tol_for(wl), what=f"{kind} peaked", output_rounding=True)


@pytest.mark.parametrize("name", ["mla_mix_split_win", "mla_mix_g8_hnd_p16"])
def test_records_wide_block_scales(name):
    """MLA records whose block scales are shrunk by 2^0 .. 2^-8, independently
    per token and 128-channel block (the codes unchanged, so every block still
    reaches the code 448): the records build weighs each block's P against a
    running maximum of that block's own, so a token whose scale in one block is
    far below the block's largest still gets its share. Compared in full with
    the oracle on the same records."""
    wl, chunk = _make(name, SMALL[name], seed=9)
    g = torch.Generator().manual_seed(23)
    e = torch.randint(-8, 1, tuple(wl.k_scale.shape), generator=g).to(torch.float32)
    wl.k_scale = wl.k_scale * torch.exp2(e).to(wl.k_scale.device)
    wl.v_scale = wl.k_scale
    out, lse, status, dec = run_decode(wl, chunk_pages=chunk)
    assert status == 0 and dec.plan.kernel == B.PDA_KERNEL_TC
    ref_o, ref_l = oracle_ref(wl)
    assert_close(out, lse, ref_o, ref_l, TOL_FP8, what=f"{name} wide block scales")


@pytest.mark.parametrize("chunk", [3, 16, 0])
def test_wide_head_blocks(chunk):
    """bf16 head_dim 128 with a GQA group of 24: the 96-column build holds
    all 24 heads of a request with up to 4 rows (72 or 96 columns) and 12
    heads for 5-8 rows (two head blocks), over one or several splits, with
    windows; every output element against the oracle."""
    wl, _ = _make("wide", dict(batch=6, rows=[1, 3, 4, 5, 7, 8], kv_lens=[700, 3000, 2049, 1500, 4096, 900],
                               num_qo_heads=48, num_kv_heads=2, head_dim=128, page_size=32,
                               windows=[0, 0, 100, 0, 0, 40]))
    out, lse, status, dec = run_decode(wl, chunk_pages=chunk, kernel=B.PDA_KERNEL_TC)
    assert status == 0
    assert dec.plan.rows_per_cta == 96 and dec.plan.heads_per_cta[4] == 24
    assert dec.plan.heads_per_cta[5] == 12 and dec.plan.head_blocks == 2
    ref_o, ref_l = oracle_ref(wl)
    assert_close(out, lse, ref_o, ref_l, TOL_BF16, what=f"96 columns, chunk {chunk}")


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("chunk", [4, 16, 64, 0])
def test_split_count_invariance(chunk, kernel):
    """Different KV chunkings (1..many splits per request) all match the
    oracle, and match one another within the same tolerance."""
    wl, _ = _make("split", dict(batch=2, rows=[3, 8], kv_lens=[4096, 1111], num_qo_heads=16,
                                num_kv_heads=2, head_dim=128, page_size=16, windows=[0, 300]))
    out, lse, status, dec = run_decode(wl, chunk_pages=chunk, kernel=KERNELS[kernel])
    assert status == 0
    ref_o, ref_l = oracle_ref(wl)
    assert_close(out, lse, ref_o, ref_l, TOL_BF16, what=f"chunk {chunk} ({dec.plan.max_splits})")


# ------------------------------------------------------- full-size workloads
# (workload, sizes, sampled items of the normal case, of the peaked case):
# None compares every output element with the oracle. Every shape the
# benchmark times is here; the largest peaked variants are sampled.
CONFIGS = [
    ("tiny", {}, None, None),
    ("fp8_decode", {}, None, None),
    ("fp8_decode", dict(layout="HND"), None, None),
    ("mtp_verify_bf16", dict(bs=1, R=1), None, None),
    ("mtp_verify_bf16", dict(bs=1, R=4), None, None),
    ("mtp_verify_bf16", dict(bs=1, R=8), None, None),
    ("mtp_verify_bf16", dict(bs=16, R=1), None, None),
    ("mtp_verify_bf16", dict(bs=16, R=4), None, 96),
    ("mtp_verify_bf16", dict(bs=16, R=8), None, 96),
    ("longctx_fp8_pth", dict(bs=1, R=1), None, None),
    ("longctx_fp8_pth", dict(bs=1, R=4), None, None),
    ("longctx_fp8_pth", dict(bs=1, R=8), None, None),
    ("longctx_fp8_pth", dict(bs=16, R=1), None, 96),
    ("longctx_fp8_pth", dict(bs=16, R=4), None, 96),
    ("longctx_fp8_pth", dict(bs=16, R=8), 256, 64),
    ("mixed", {}, None, 160),
    ("longctx_int8_pth", dict(bs=1, R=8), None, 64),
    ("longctx_int8_pth", dict(bs=16, R=1), 256, 64),
    ("longctx_int8_pth", dict(bs=16, R=8), None, 64),
    ("mla_fp8", {}, None, None),
    ("mla_fp8", dict(R=2), None, 96),
    ("mla_bf16", {}, None, 96),
    ("mla_bf16", dict(R=2), 96, 96),
    ("mla_fp8_mixed", {}, None, None),
    ("mla_fp8_mixed", dict(R=2), 96, 96),
    ("d512_mtp_bf16", dict(bs=1, R=1), None, None),
    ("d512_mtp_bf16", dict(bs=1, R=4), None, None),
    ("d512_mtp_bf16", dict(bs=1, R=8, kv_lens=131072), 48, 48),
    ("d512_mtp_fp8", dict(bs=1, R=1), None, None),
    ("d512_mtp_fp8", dict(bs=1, R=8), None, None),
    ("d512_mtp_fp8", dict(bs=1, R=4, kv_lens=131072), 48, 48),
]


HOST_PLANNED = ("mixed",)


@pytest.mark.parametrize("peaked", [False, True], ids=["normal", "peaked"])
@pytest.mark.parametrize("cfg,kw,n_normal,n_peaked", CONFIGS,
                         ids=[f"{c}-{'-'.join(f'{k}{v}' for k, v in kw.items())}"
                              for c, kw, _, _ in CONFIGS])
def test_config_parity(cfg, kw, n_normal, n_peaked, peaked):
    """The named workloads at their full sizes, in the planner's own launch
    configuration (the one the benchmark times). Outputs are compared in full
    where the oracle finishes within about a minute, else on sampled (row,
    head) items that include every windowed / edge request's first and last
    row."""
    n_sample = n_peaked if peaked else n_normal
    extra = dict(q_mult=4.0) if peaked else {}
    wl = config_workload(cfg, device=DEV, **kw, **extra)
    # the mixed batch is planned from its host lengths, rows and windows, as
    # the benchmark plans it
    out, lse, status, dec = run_decode(wl, host_plan=cfg in HOST_PLANNED)
    assert status == 0
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    if n_sample is None:
        ref_o, ref_l = oracle_ref(wl)
        assert_close(out, lse, ref_o, ref_l, tol_for(wl), what=cfg, output_rounding=peaked)
    else:
        must = []
        if wl.window is not None:
            w = wl.window.cpu().tolist()
            must = [b for b in range(wl.batch) if w[b] > 0][:8] + [0, wl.batch - 1]
        items = sample_items(wl, n_sample, seed=3, must=must)
        ref_o, ref_l = oracle_ref(wl, items=items)
        o = out.reshape(-1, dv_of(wl))[items]
        l_ = lse.reshape(-1)[items]
        assert_close(o, l_, ref_o, ref_l, tol_for(wl), what=f"{cfg} sampled",
                     output_rounding=peaked)


def test_tail_split_parity():
    """A plan whose last requests run with shorter chunks than the rest (the
    partial last wave cut finer) matches the oracle everywhere."""
    wl = config_workload("fp8_decode", device=DEV, batch=40)
    out, lse, status, dec = run_decode(wl)
    assert status == 0
    assert dec.plan.tail_from < wl.batch and dec.plan.tail_chunk_pages < dec.plan.chunk_pages
    ref_o, ref_l = oracle_ref(wl)
    assert_close(out, lse, ref_o, ref_l, tol_for(wl), what="tail split")


# ------------------------------------------------ bit-exact gather and masks
def _index_code(L, H, D):
    """v_j[c]: hex digit (c mod 4) of token j, negated for kv head 1 --
    integers 0..15, exact in bf16 and E4M3."""
    j = torch.arange(L)[:, None, None]
    c = torch.arange(D)[None, None, :]
    digit = ((j >> (4 * (c % 4))) & 15).float()
    sign = torch.ones(H)[None, :, None]
    if H > 1:
        sign[0, 1, 0] = -1.0
    return (digit * sign).expand(L, H, D).clone()


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("kind", ["bf16", "fp8_tensor", "fp8_pth", "fp8_qfp8"])
@pytest.mark.parametrize("chunk", [0, 4])
def test_causal_upper_bound_bit_exact(kind, chunk, kernel):
    """K channel 0 is 0 for old tokens and t+1 for the t-th new token; Q
    channel 0 is 128, sm_scale 1. Row i's own token then outweighs every other
    visible key by e^-128 (below the smallest fp32), so its output must be
    v_{p_i} bit for bit; a leaked future key would outweigh it and show a
    different token's code."""
    R_list, L_list = [8, 1, 5, 3], [700, 90, 64, 5]
    H, G, D, P = 2, 4, 128, 16

    def token_fn(which, b, L):
        if which == "v":
            return _index_code(L, H, D)
        x = torch.zeros(L, H, D)
        R = R_list[b]
        x[L - R:, :, 0] = torch.arange(1, R + 1, dtype=torch.float32)[:, None]
        return x

    def value_fn(which, shape, gen):
        x = torch.zeros(shape)
        if which == "q":
            x[..., 0] = 128.0
        return x

    kv, qd, sm = {"bf16": ("bf16", "bf16", SCALE_NONE), "fp8_tensor": ("e4m3", "bf16", SCALE_TENSOR),
                  "fp8_pth": ("e4m3", "bf16", SCALE_TOKEN_HEAD),
                  "fp8_qfp8": ("e4m3", "e4m3", SCALE_TENSOR)}[kind]
    wl = make_workload(batch=4, rows=R_list, kv_lens=L_list, num_qo_heads=H * G, num_kv_heads=H,
                       head_dim=D, page_size=P, kv_dtype=kv, q_dtype=qd, scale_mode=sm,
                       sm_scale=1.0, value_fn=value_fn, token_fn=token_fn, unit_scale=True,
                       seed=5, device=DEV)
    out, lse, status, _ = run_decode(wl, chunk_pages=chunk, kernel=KERNELS[kernel])
    assert status == 0
    r0 = 0
    for b, (R, L) in enumerate(zip(R_list, L_list)):
        code = _index_code(L, H, D)
        for i in range(R):
            pos = L - R + i
            for h in range(H * G):
                assert torch.equal(out[r0 + i, h], code[pos, h // G]), (b, i, h)
                assert math.isclose(float(lse[r0 + i, h]), 128.0 * (i + 1), rel_tol=1e-5)
        r0 += R


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("kind", ["bf16", "fp8_pth"])
def test_window_lower_bound_bit_exact(kind, kernel):
    """K channel 0 falls by one per token (bf16: 256 - j; per-token-head
    E4M3: code 1 with scale 256 - j), Q channel 0 is 128: the earliest visible
    key of each row outweighs the next by e^-128 (below the smallest fp32),
    and the key just below the window would dominate it if it were admitted.
    Output must be v at p_i - W + 1 bit for bit."""
    R_list, L_list, W_list = [8, 4, 2, 1, 3, 5], [200, 70, 33, 129, 250, 180], [1, 5, 64, 17, 63, 65]
    H, G, D, P = 2, 3, 128, 16

    def token_fn(which, b, L):
        if which == "v":
            return _index_code(L, H, D)
        x = torch.zeros(L, H, D)
        x[:, :, 0] = 1.0 if kind == "fp8_pth" else (256.0 - torch.arange(L).float())[:, None]
        return x

    def scale_fn(which, b, L):
        s = torch.ones(L, H)
        if which == "k":
            s = (256.0 - torch.arange(L).float())[:, None].expand(L, H).clone()
        return s

    def value_fn(which, shape, gen):
        x = torch.zeros(shape)
        if which == "q":
            x[..., 0] = 128.0
        return x

    kv, sm = ("bf16", SCALE_NONE) if kind == "bf16" else ("e4m3", SCALE_TOKEN_HEAD)
    wl = make_workload(batch=len(R_list), rows=R_list, kv_lens=L_list, windows=W_list,
                       num_qo_heads=H * G, num_kv_heads=H, head_dim=D, page_size=P, kv_dtype=kv,
                       scale_mode=sm, sm_scale=1.0, value_fn=value_fn, token_fn=token_fn,
                       scale_fn=scale_fn if kind != "bf16" else None, unit_scale=True, seed=9,
                       device=DEV)
    out, lse, status, _ = run_decode(wl, chunk_pages=4, kernel=KERNELS[kernel])
    assert status == 0
    r0 = 0
    for b, (R, L, W) in enumerate(zip(R_list, L_list, W_list)):
        code = _index_code(L, H, D)
        for i in range(R):
            lo = max(0, L - R + i - W + 1)
            for h in range(H * G):
                assert torch.equal(out[r0 + i, h], code[lo, h // G]), (b, i, h, lo)
        r0 += R


# ------------------------------------------------------------- invariants
def test_page_permutation_bitwise():
    wl, _ = _make("perm", dict(batch=3, rows=[2, 5, 1], kv_lens=[1333, 700, 81], num_qo_heads=16,
                               num_kv_heads=2, head_dim=128, page_size=16, kv_dtype="e4m3",
                               scale_mode=SCALE_TOKEN_HEAD, windows=[0, 99, 0]))
    out, lse, _, _ = run_decode(wl, chunk_pages=8)
    g = torch.Generator().manual_seed(4)
    pi = torch.randperm(wl.num_pages, generator=g).to(DEV)
    inv = torch.argsort(pi)
    wl.k_pages, wl.v_pages = wl.k_pages[inv].contiguous(), wl.v_pages[inv].contiguous()
    wl.k_scale, wl.v_scale = wl.k_scale[inv].contiguous(), wl.v_scale[inv].contiguous()
    wl.page_table = pi[wl.page_table.long()].to(torch.int32)
    out2, lse2, _, _ = run_decode(wl, chunk_pages=8)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_rows_equal_single_row_requests():
    R, L, P = 7, 1500, 16
    wl, _ = _make("rows", dict(batch=1, rows=R, kv_lens=L, num_qo_heads=16, num_kv_heads=2,
                               head_dim=256, page_size=P, windows=[200]))
    out, lse, _, _ = run_decode(wl, chunk_pages=16)
    pages = wl.page_table[: math.ceil(L / P)].cpu().tolist()
    table, kvi, lens = [], [0], []
    for i in range(R):
        Li = L - R + i + 1
        table.extend(pages[: math.ceil(Li / P)])
        kvi.append(len(table))
        lens.append(Li)
    wl.page_table = torch.tensor(table, dtype=torch.int32, device=DEV)
    wl.kv_indptr = torch.tensor(kvi, dtype=torch.int32, device=DEV)
    wl.kv_len = torch.tensor(lens, dtype=torch.int32, device=DEV)
    wl.qo_indptr = torch.arange(R + 1, dtype=torch.int32, device=DEV)
    wl.window = torch.full((R,), 200, dtype=torch.int32, device=DEV)
    out1, lse1, _, _ = run_decode(wl, chunk_pages=16)
    assert (out1 - out).abs().max() <= TOL_BF16["max"]
    assert (lse1 - lse).abs().max() <= TOL_BF16["lse"]


GRAPH_CASES = {
    "int8_pth_d256": dict(batch=2, rows=[3, 8], kv_lens=[1500, 700], num_qo_heads=16,
                          num_kv_heads=2, head_dim=256, page_size=16, kv_dtype="int8",
                          scale_mode=SCALE_TOKEN_HEAD),
    "mla_records": dict(batch=2, rows=[1, 2], kv_lens=[900, 333], num_qo_heads=16,
                        num_kv_heads=1, head_dim=576, head_dim_v=512, page_size=64,
                        kv_dtype="e4m3", scale_mode=3),
    "mla_bf16": dict(batch=2, rows=[2, 1], kv_lens=[1200, 64], num_qo_heads=16,
                     num_kv_heads=1, head_dim=576, head_dim_v=512, page_size=16),
}


@pytest.mark.parametrize("name", sorted(GRAPH_CASES))
def test_graph_replay_new_queries(name):
    """A captured call replayed with new query values (same buffers) matches
    the oracle each time: the converter and latent pipelines carry no state
    from one call to the next."""
    wl, _ = _make(name, GRAPH_CASES[name])
    dec = B.Decoder(B.params_for(wl), device=DEV)
    out = torch.empty(wl.total_rows, wl.num_qo_heads, dv_of(wl), dtype=torch.bfloat16,
                      device=DEV)
    lse = torch.empty(wl.total_rows, wl.num_qo_heads, dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dec.run(wl, out, lse, stream=s)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        dec.run(wl, out, lse, stream=s)
    g = torch.Generator(device="cpu").manual_seed(5)
    for step in range(3):
        if step:
            wl.q.copy_(torch.randn(wl.q.shape, generator=g).to(wl.q.dtype))
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        ref_o, ref_l = oracle_ref(wl)
        assert_close(out.float().cpu(), lse.cpu(), ref_o, ref_l, tol_for(wl),
                     what=f"{name} replay {step}")
    assert dec.status() == 0


def test_stages_apart_equal_one_call():
    """pda_decode_stages(PARTIAL) then (MERGE) on one stream writes the same
    bytes as pda_decode (a plan with tail splits: both launches run)."""
    wl = config_workload("fp8_decode", device=DEV, batch=40)
    dec = B.Decoder(B.params_for(wl), device=DEV)
    assert dec.plan.max_splits > 1
    outs = []
    for stages in (None, "apart"):
        out = torch.full((wl.total_rows, wl.num_qo_heads, wl.head_dim), float("nan"),
                         dtype=torch.bfloat16, device=DEV)
        lse = torch.full((wl.total_rows, wl.num_qo_heads), float("nan"), device=DEV)
        if stages is None:
            dec.run(wl, out, lse)
        else:
            dec.run(wl, out, lse, stages=B.PDA_STAGE_PARTIAL)
            dec.run(wl, out, lse, stages=B.PDA_STAGE_MERGE)
        torch.cuda.synchronize()
        outs.append((out.view(torch.int16).cpu(), lse.cpu()))
    assert dec.status() == 0
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_cuda_graph_replay_with_new_lengths():
    """One plan + one captured graph serve new kv_len / page_table / qo_indptr
    / window contents (same maxima): replay matches the oracle on each."""
    import types
    H, G, D, P = 2, 8, 128, 16
    cap_pages, cap_rows, cap_batch = 1024, 40, 4
    base = dict(batch=4, num_qo_heads=H * G, num_kv_heads=H, head_dim=D, page_size=P)
    w1, _ = _make("g1", dict(base, rows=[1, 8, 3, 2], kv_lens=[3000, 2500, 64, 1000],
                             windows=[0, 128, 0, 0]))
    w2, _ = _make("g2", dict(base, rows=[2, 4, 8, 1], kv_lens=[4096, 17, 800, 2222],
                             windows=[5, 0, 0, 64]), seed=1)
    buf = types.SimpleNamespace(
        num_qo_heads=H * G, num_kv_heads=H, head_dim=D, page_size=P, num_pages=cap_pages,
        q_e4m3=False, kv_e4m3=False, scale_mode=SCALE_NONE, strides=w1.strides,
        q=torch.zeros(cap_rows, H * G, D, dtype=torch.bfloat16, device=DEV),
        k_pages=torch.zeros(cap_pages, P, H, D, dtype=torch.bfloat16, device=DEV),
        v_pages=torch.zeros(cap_pages, P, H, D, dtype=torch.bfloat16, device=DEV),
        k_scale=None, v_scale=None,
        page_table=torch.zeros(2048, dtype=torch.int32, device=DEV),
        kv_indptr=torch.zeros(cap_batch + 1, dtype=torch.int32, device=DEV),
        kv_len=torch.ones(cap_batch, dtype=torch.int32, device=DEV),
        qo_indptr=torch.zeros(cap_batch + 1, dtype=torch.int32, device=DEV),
        window=torch.zeros(cap_batch, dtype=torch.int32, device=DEV),
        sm_scale=w1.sm_scale, batch=cap_batch, max_q_len=8)
    buf.kv_len.fill_(4096)

    def load(w):
        buf.q[: w.total_rows].copy_(w.q)
        buf.k_pages[: w.num_pages].copy_(w.k_pages)
        buf.v_pages[: w.num_pages].copy_(w.v_pages)
        buf.page_table[: w.page_table.numel()].copy_(w.page_table)
        for name in ("kv_indptr", "kv_len", "qo_indptr", "window"):
            getattr(buf, name).copy_(getattr(w, name))

    p = B.params_for(w1, max_batch=cap_batch, max_q_len=8, max_kv_len=4096)
    p.num_pages = cap_pages
    dec = B.Decoder(p)
    out = torch.zeros(cap_rows, H * G, D, dtype=torch.bfloat16, device=DEV)
    lse = torch.zeros(cap_rows, H * G, dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    load(w1)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        dec.run(buf, out, lse, max_q_len=8, stream=s)  # warm-up outside capture
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        dec.run(buf, out, lse, max_q_len=8, stream=s)
    for w in (w1, w2, w1):
        load(w)
        torch.cuda.synchronize()
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        ref_o, ref_l = oracle_ref(w)
        n = w.total_rows
        assert_close(out[:n].float().cpu(), lse[:n].cpu(), ref_o, ref_l, TOL_BF16,
                     what=f"graph replay {w.name}")
    assert dec.status() == 0


def test_status_bits_and_isolation():
    """Device-detected errors set status bits, skip only the bad request and
    leave the others correct."""
    wl, _ = _make("status", dict(batch=4, rows=[2, 3, 1, 2], kv_lens=[100, 400, 50, 300],
                                 num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=16))
    ref_o, ref_l = oracle_ref(wl)
    kv_len = wl.kv_len.clone()
    wl.kv_len[0] = 1                       # fewer tokens than rows
    pt = wl.page_table.clone()
    kvi = wl.kv_indptr.cpu().tolist()
    wl.page_table[kvi[2]] = wl.num_pages + 5   # page id out of range in request 2
    out, lse, status, dec = run_decode(wl, max_kv_len=512)
    assert status & B.PDA_STATUS_KV_LEN_LT_ROWS
    assert status & B.PDA_STATUS_PAGE_OOB
    qo = wl.qo_indptr.cpu().tolist()
    assert torch.isnan(out[qo[0]:qo[1]]).all()  # skipped rows left unwritten
    for b in (1, 3):
        sl = slice(qo[b], qo[b + 1])
        assert_close(out[sl], lse[sl], ref_o[sl], ref_l[sl], TOL_BF16, what=f"request {b}")
    dec.reset_status()
    torch.cuda.synchronize()
    assert dec.status() == 0
    wl.kv_len.copy_(kv_len)
    wl.page_table.copy_(pt)
    wl.kv_len[3] = 600                     # above the plan's max_kv_len
    out, lse, status, _ = run_decode(wl, max_kv_len=512, decoder=dec)
    assert status == B.PDA_STATUS_KV_LEN_GT_MAX


def test_rows_above_max_q_len_flagged():
    wl, _ = _make("rows_gt", dict(batch=2, rows=[4, 2], kv_lens=[100, 100], num_qo_heads=4,
                                  num_kv_heads=2, head_dim=64, page_size=16))
    out, lse, status, _ = run_decode(wl, max_q_len=2, max_batch=4)
    assert status & B.PDA_STATUS_ROWS_GT_MAX
    ref_o, ref_l = oracle_ref(wl)
    assert_close(out[4:], lse[4:], ref_o[4:], ref_l[4:], TOL_BF16, what="request 1")
