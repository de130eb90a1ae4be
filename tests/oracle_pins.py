"""Pins of the fp64 oracle to things other than itself.

Each ``pin_*`` function raises AssertionError when the oracle (optionally a
copy built with one planted mistake, ``mutation`` > 0) disagrees with:
  * torch's own float8_e4m3fn decoding of all 256 E4M3 codes;
  * dense torch attention with an explicit mask on tiny inputs (bruteforce);
  * closed forms: Q = 0 gives the mean of the visible values and
    lse = ln(number of visible keys); a window of 1 gives v at the row's own
    position and lse = its logit;
  * invariants: constant V returns V; permuting physical pages and remapping
    the page table changes nothing; cutting the keys into chunks and merging
    the chunks' (o, lse) equals one pass; R rows equal R single-row requests
    whose contexts end at the rows' positions.
The semantics pinned are those of "perf(attention): run up to 8 query rows
per request in the triton decode kernel", section "Changes" (per-row causal
limit and window, per-row merge of the KV split, GQA groups).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from bruteforce import dense_attention, dequant_cache, dequant_q, visibility_mask
from paged_split_kv_03_gb300.synth import (SCALE_NONE, SCALE_TENSOR, SCALE_TOKEN_HEAD,
                                           make_workload)

TOL = 1e-12


def _run(wl, mutation, **kw):
    out, lse, rc = oracle.attention_for(wl, mutation=mutation, **kw)
    total = wl.total_rows
    return (out.reshape(total, wl.num_qo_heads, wl.head_dim), lse.reshape(total, wl.num_qo_heads),
            rc)


def _close(a, b, tol=TOL, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    assert np.all(np.isfinite(a)) and np.all(np.isfinite(b)), f"{what}: non-finite values"
    err = np.max(np.abs(a - b) / np.maximum(1.0, np.abs(b))) if a.size else 0.0
    assert err <= tol, f"{what}: max rel err {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------------------

def pin_e4m3_all_codes(mutation=0):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).tolist()
    for c in range(256):
        got = oracle.e4m3_to_double(c, mutation=mutation)
        want = ref[c]
        if math.isnan(want):
            assert math.isnan(got), f"code {c:#x}: want NaN, got {got}"
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), \
                f"code {c:#x}: want {want}, got {got}"


def bruteforce_cases():
    """Tiny workloads spanning B <= 3, L <= 80, P in {1, 4, 16}, R in 0..8,
    W in {none, 1, 5}, G in {1, 3, 8, 24}, bf16 / e4m3 (both scale kinds),
    bf16 / e4m3 queries and both cache layouts."""
    cases = []
    rng = np.random.default_rng(7)
    groups = [(1, 1), (3, 3), (8, 1), (24, 2), (8, 2), (3, 1)]
    kinds = [("bf16", "bf16", SCALE_NONE), ("e4m3", "bf16", SCALE_TENSOR),
             ("e4m3", "bf16", SCALE_TOKEN_HEAD), ("e4m3", "e4m3", SCALE_TENSOR),
             ("e4m3", "e4m3", SCALE_TOKEN_HEAD)]
    n = 0
    for gi, (G, H) in enumerate(groups):
        for ki, (kvd, qd, sm) in enumerate(kinds):
            B = 1 + (n % 3)
            P = (1, 4, 16)[n % 3]
            rows = [int(r) for r in rng.integers(0, 9, size=B)]
            rows[0] = max(rows[0], 1)
            lens = [int(max(r, rng.integers(1, 81))) for r in rows]
            wsel = n % 3
            windows = None if wsel == 0 else [(1, 5)[wsel - 1] if b % 2 == 0 else 0
                                               for b in range(B)]
            cases.append(dict(batch=B, rows=rows, kv_lens=lens, num_qo_heads=G * H,
                              num_kv_heads=H, head_dim=(16, 32, 64)[n % 3], page_size=P,
                              kv_dtype=kvd, q_dtype=qd, scale_mode=sm, windows=windows,
                              layout=("NHD", "HND")[n % 2], seed=100 + n,
                              sm_scale=0.3 + 0.1 * (n % 4), q_mult=1.0 + (n % 2)))
            n += 1
    return cases


def pin_bruteforce(mutation=0):
    for args in bruteforce_cases():
        wl = make_workload(**args)
        out, lse, rc = _run(wl, mutation)
        assert rc == 0, rc
        ref_o, ref_l = dense_attention(wl)
        _close(out, ref_o.numpy(), what=f"out {args}")
        _close(lse, ref_l.numpy(), what=f"lse {args}")


def pin_q_zero_closed_form(mutation=0):
    """Q = 0: every visible logit is 0, so o = mean of visible v and
    lse = ln |visible| = ln(min(p_i + 1, W)) (no window: p_i + 1)."""
    for kvd, sm, P in (("bf16", SCALE_NONE, 4), ("e4m3", SCALE_TOKEN_HEAD, 16)):
        def vals(kind, shape, gen):
            x = torch.randn(shape, generator=gen)
            return torch.zeros(shape) if kind == "q" else x
        B = 3
        rows, lens, wins = [3, 8, 1], [40, 9, 70], [5, 0, 1]
        wl = make_workload(batch=B, rows=rows, kv_lens=lens, num_qo_heads=6, num_kv_heads=2,
                           head_dim=16, page_size=P, kv_dtype=kvd, scale_mode=sm, windows=wins,
                           seed=5, value_fn=vals)
        out, lse, rc = _run(wl, mutation)
        assert rc == 0
        vd = dequant_cache(wl, "v")
        table = wl.page_table.long()
        kvi = wl.kv_indptr.tolist()
        r0 = 0
        for b in range(B):
            L, R, W = lens[b], rows[b], wins[b]
            npg = math.ceil(L / P)
            V = vd[table[kvi[b]:kvi[b] + npg]].reshape(npg * P, 2, -1)[:L]
            for i in range(R):
                pos = L - R + i
                lo = max(0, pos - W + 1) if W > 0 else 0
                count = pos - lo + 1
                for h in range(6):
                    want = V[lo:pos + 1, h // 3].mean(dim=0).numpy()
                    _close(out[r0 + i, h], want, what=f"Q=0 mean b{b} i{i} h{h}")
                    _close(lse[r0 + i, h], math.log(count), what=f"Q=0 lse b{b} i{i} h{h}")
            r0 += R


def pin_single_visible_key(mutation=0):
    """W = 1: the only visible key is the row's own, so o = v_{p_i} exactly
    and lse = sm_scale * q . k_{p_i}."""
    for kvd, sm in (("bf16", SCALE_NONE), ("e4m3", SCALE_TENSOR)):
        rows, lens = [4, 2], [9, 30]
        wl = make_workload(batch=2, rows=rows, kv_lens=lens, num_qo_heads=4, num_kv_heads=2,
                           head_dim=32, page_size=4, kv_dtype=kvd, scale_mode=sm,
                           windows=[1, 1], seed=11)
        out, lse, rc = _run(wl, mutation)
        assert rc == 0
        kd, vd, qd = dequant_cache(wl, "k"), dequant_cache(wl, "v"), dequant_q(wl)
        table = wl.page_table.long()
        kvi = wl.kv_indptr.tolist()
        r0 = 0
        for b in range(2):
            L, R = lens[b], rows[b]
            for i in range(R):
                pos = L - R + i
                page = table[kvi[b] + pos // 4]
                for h in range(4):
                    v = vd[page, pos % 4, h // 2].numpy()
                    assert np.array_equal(out[r0 + i, h], v), f"W=1 b{b} i{i} h{h}"
                    s = wl.sm_scale * float(torch.dot(qd[r0 + i, h], kd[page, pos % 4, h // 2]))
                    _close(lse[r0 + i, h], s, what=f"W=1 lse b{b} i{i} h{h}")
            r0 += R


def pin_constant_v(mutation=0):
    """V equal to one vector c_h for every token of kv head h gives o = c_h."""
    for kvd, sm in (("bf16", SCALE_NONE), ("e4m3", SCALE_TENSOR), ("e4m3", SCALE_TOKEN_HEAD)):
        def vals(kind, shape, gen):
            x = torch.randn(shape, generator=gen)
            if kind == "v":
                c = torch.randn(shape[2], shape[3], generator=gen)
                x = c.expand(shape).clone()
            return x
        rows, lens = [8, 3], [50, 17]
        wl = make_workload(batch=2, rows=rows, kv_lens=lens, num_qo_heads=6, num_kv_heads=2,
                           head_dim=32, page_size=16, kv_dtype=kvd, scale_mode=sm,
                           windows=[0, 6], seed=21, value_fn=vals, poison=True)
        out, lse, rc = _run(wl, mutation)
        assert rc == 0
        vd = dequant_cache(wl, "v")
        page0 = int(wl.page_table[0])
        for h in range(6):
            c = vd[page0, 0, h // 3].numpy()
            _close(out[:, h], np.broadcast_to(c, out[:, h].shape), what=f"constant V h{h}")


def pin_page_permutation(mutation=0):
    """Permuting physical pages and remapping the table gives identical output."""
    wl = make_workload(batch=3, rows=[2, 5, 1], kv_lens=[33, 70, 8], num_qo_heads=8,
                       num_kv_heads=2, head_dim=16, page_size=4, kv_dtype="e4m3",
                       scale_mode=SCALE_TOKEN_HEAD, windows=[0, 9, 0], seed=31)
    out, lse, rc = _run(wl, mutation)
    assert rc == 0
    g = torch.Generator().manual_seed(3)
    pi = torch.randperm(wl.num_pages, generator=g)         # old page p -> new id pi[p]
    inv = torch.argsort(pi)                                 # new id n holds old page inv[n]
    wl2 = make_workload(batch=3, rows=[2, 5, 1], kv_lens=[33, 70, 8], num_qo_heads=8,
                        num_kv_heads=2, head_dim=16, page_size=4, kv_dtype="e4m3",
                        scale_mode=SCALE_TOKEN_HEAD, windows=[0, 9, 0], seed=31)
    wl2.k_pages = wl.k_pages[inv].clone()
    wl2.v_pages = wl.v_pages[inv].clone()
    wl2.k_scale = wl.k_scale[inv].clone()
    wl2.v_scale = wl.v_scale[inv].clone()
    wl2.page_table = pi[wl.page_table.long()].to(torch.int32)
    out2, lse2, rc2 = _run(wl2, mutation)
    assert rc2 == 0
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2), "page permutation changed output"


def pin_split_merge(mutation=0):
    """Chunked keys + log-sum-exp merge equals the one-pass result (fp64)."""
    wl = make_workload(batch=2, rows=[8, 3], kv_lens=[77, 40], num_qo_heads=6, num_kv_heads=3,
                       head_dim=32, page_size=4, windows=[0, 11], seed=41, q_mult=3.0)
    out, lse, _ = _run(wl, mutation)
    for chunk in (1, 5, 16, 64):
        o2, l2, rc = _run(wl, mutation, split_tokens=chunk)
        assert rc == 0
        _close(o2, out, what=f"split {chunk} out")
        _close(l2, lse, what=f"split {chunk} lse")


def pin_rows_vs_single(mutation=0):
    """R rows of one request equal R one-row requests with kv_len p_i + 1."""
    R, L, P = 6, 45, 4
    for W in (0, 7):
        wl = make_workload(batch=1, rows=R, kv_lens=L, num_qo_heads=4, num_kv_heads=2,
                           head_dim=16, page_size=P, windows=[W], seed=51)
        out, lse, rc = _run(wl, mutation)
        assert rc == 0
        npg = math.ceil(L / P)
        pages = wl.page_table[:npg].tolist()
        table, kvi, lens = [], [0], []
        for i in range(R):
            Li = L - R + i + 1
            table.extend(pages[:math.ceil(Li / P)])
            kvi.append(len(table))
            lens.append(Li)
        wl1 = make_workload(batch=R, rows=1, kv_lens=lens, num_qo_heads=4, num_kv_heads=2,
                            head_dim=16, page_size=P, windows=[W] * R, seed=51)
        wl1.q, wl1.k_pages, wl1.v_pages, wl1.num_pages = wl.q, wl.k_pages, wl.v_pages, wl.num_pages
        wl1.page_table = torch.tensor(table, dtype=torch.int32)
        wl1.kv_indptr = torch.tensor(kvi, dtype=torch.int32)
        out1, lse1, rc1 = _run(wl1, mutation)
        assert rc1 == 0
        _close(out1, out, what=f"rows vs single W={W}")
        _close(lse1, lse, what=f"rows vs single lse W={W}")


ALL_PINS = [pin_e4m3_all_codes, pin_bruteforce, pin_q_zero_closed_form, pin_single_visible_key,
            pin_constant_v, pin_page_permutation, pin_split_merge, pin_rows_vs_single]

# Planted mistakes compiled into copies of the oracle (see MUT(k) in pdo_oracle.c).
MUTATIONS = {
    1: "window admits one key too many",
    2: "every row sees the whole context (no per-row causal limit)",
    3: "GQA maps q head h to kv head h % Hkv",
    4: "per-(token, head) scale ignores the head",
    5: "lse drops the running max",
    6: "E4M3 exponent bias 8",
    7: "E4M3 subnormal step 2^-10",
    8: "split merge forgets to divide by the weight sum",
    9: "V dequantised with K's scale",
    10: "token and head strides swapped",
    11: "row position one short (p_i = L - R + i - 1)",
    12: "sm_scale not applied",
    13: "page table read one entry late",
    14: "query row read from the previous row",
    15: "softmax output not divided by its denominator",
}
