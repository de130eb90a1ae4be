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

The quantise-on-append oracle (the fp8_per_token_head cache of the same
page's "End-to-end A/B", per-tensor FP8 of "fp8 support") is pinned to
torch's float8_e4m3fn cast (codes within +-448, ties to even), to the
saturation of the format's largest finite value, to closed forms of the
scale (amax / 448, 1 for a zero row) and to the page-table placement of
token L - R + i read independently here.

MLA ("fp8 support", FlashMLA PR #54): a latent cache read as K (all its
channels) and as V (the first dv) is pinned through the same dense attention
with V sliced from the latent.

The int8 cache (beside bf16 and fp8 in the same page's "Tested on") is
pinned to dense torch attention over torch's own int8 decode, to a closed
form (a constant negative code times its scale), and its quantiser to
torch.round (ties to even) with the +-127 clamp and the amax / 127 scale.
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
    dv = getattr(wl, "head_dim_v", None) or wl.head_dim
    return out.reshape(total, wl.num_qo_heads, dv), lse.reshape(total, wl.num_qo_heads), rc


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
             ("e4m3", "e4m3", SCALE_TOKEN_HEAD), ("int8", "bf16", SCALE_TENSOR),
             ("int8", "bf16", SCALE_TOKEN_HEAD)]
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
    # MLA: one latent cache read as K (all channels) and as V (the first dv)
    for i, (kvd, qd, sm) in enumerate(kinds[:5]):
        cases.append(dict(batch=2, rows=[1 + i, 2], kv_lens=[30 + 7 * i, 9], num_qo_heads=8,
                          num_kv_heads=1, head_dim=48, head_dim_v=32, page_size=(4, 16)[i % 2],
                          kv_dtype=kvd, q_dtype=qd, scale_mode=sm, seed=300 + i,
                          windows=None if i % 2 else [5, 0]))
    # the mixed-precision MLA latent: E4M3 nope with a scale per 128 channels, bf16 rope
    for i in range(2):
        cases.append(dict(batch=2, rows=[1 + i, 2], kv_lens=[40 + 9 * i, 17], num_qo_heads=4,
                          num_kv_heads=1, head_dim=576, head_dim_v=512, page_size=(8, 16)[i],
                          kv_dtype="e4m3", q_dtype="bf16", scale_mode=3, seed=310 + i,
                          windows=[0, 6] if i else None, layout=("NHD", "HND")[i]))
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


# ------------------------------------------------------------ append pins
def _e4m3_torch(y: torch.Tensor) -> torch.Tensor:
    return y.to(torch.float8_e4m3fn).view(torch.uint8)


def pin_e4m3_encode_vs_torch(mutation=0):
    # every finite code's value, every midpoint between neighbours (a tie:
    # the even code), and random fp32 values, both signs, all within +-448
    codes = torch.arange(0, 0x7F, dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).float()
    mids = (vals[:-1] + vals[1:]) / 2
    g = torch.Generator().manual_seed(5)
    rnd = (torch.rand(4000, generator=g) * 2 - 1) * 448
    tiny = (torch.rand(1000, generator=g) * 2 - 1) * 2.0 ** -6
    ys = torch.cat([vals, mids, rnd, tiny]).float()
    ys = torch.cat([ys, -ys])
    got = torch.tensor([oracle.e4m3_encode(float(y), mutation) for y in ys], dtype=torch.uint8)
    ref = _e4m3_torch(ys)
    bad = (got != ref).nonzero()
    assert bad.numel() == 0, f"E4M3 encode differs from torch at {ys[bad[0]].item()!r}"


def pin_e4m3_encode_saturates(mutation=0):
    # the largest finite E4M3 value is 448 (S.1111.110); beyond it the code
    # saturates; S.1111.111 is NaN
    for y, code in [(448.0, 0x7E), (449.0, 0x7E), (1e30, 0x7E), (float("inf"), 0x7E),
                    (-449.0, 0xFE), (-float("inf"), 0xFE)]:
        assert oracle.e4m3_encode(y, mutation) == code, (y, code)
    assert oracle.e4m3_encode(float("nan"), mutation) == 0x7F


def _append_case(mode, D=8, P=4, H=2, lens=(9, 5), rows=(3, 2), seed=0):
    """Tiny cache with a shuffled page table; returns the pieces by name."""
    g = torch.Generator().manual_seed(seed)
    B = len(lens)
    pages_per = [math.ceil(L / P) for L in lens]
    num_pages = sum(pages_per) + 2
    perm = torch.randperm(num_pages, generator=g)[:sum(pages_per)].to(torch.int32)
    kv_indptr = torch.tensor([0] + list(np.cumsum(pages_per)), dtype=torch.int32)
    qo = torch.tensor([0] + list(np.cumsum(rows)), dtype=torch.int32)
    n = int(qo[-1])
    k_new = (torch.randn(n, H, D, generator=g) * 3).to(torch.bfloat16)
    v_new = (torch.randn(n, H, D, generator=g) * 3).to(torch.bfloat16)
    elt = 2 if mode == oracle.APPEND_BF16 else 1
    shape = (num_pages, P, H, D)
    fill = torch.randint(0, 256, (num_pages * P * H * D * elt,), generator=g, dtype=torch.uint8)
    k_pages = fill.clone().numpy()
    v_pages = fill.flip(0).clone().numpy()
    ks = vs = None
    if mode in (oracle.APPEND_TENSOR, oracle.APPEND_INT8_TENSOR):
        ks, vs = np.array([0.0125], np.float32), np.array([0.02], np.float32)
    elif mode in (oracle.APPEND_TOKEN_HEAD, oracle.APPEND_INT8_TOKEN_HEAD):
        ks = np.full(num_pages * P * H, -1.0, np.float32)
        vs = np.full(num_pages * P * H, -2.0, np.float32)
    return dict(k_new=k_new, v_new=v_new, page_table=perm, kv_indptr=kv_indptr,
                kv_len=torch.tensor(lens, dtype=torch.int32), qo_indptr=qo, k_pages=k_pages,
                v_pages=v_pages, k_scale=ks, v_scale=vs, num_kv_heads=H, head_dim=D,
                page_size=P, mode=mode, strides=(P * H * D, H * D, D), num_pages=num_pages)


def _slots(case):
    """(row, page, slot) of every new row, from the page table, read here."""
    P = case["page_size"]
    out = []
    qo = case["qo_indptr"].tolist()
    for b, L in enumerate(case["kv_len"].tolist()):
        R = qo[b + 1] - qo[b]
        for i in range(R):
            t = L - R + i
            page = int(case["page_table"][int(case["kv_indptr"][b]) + t // P])
            out.append((qo[b] + i, page, t % P))
    return out


def pin_append_token_head(mutation=0):
    case = _append_case(oracle.APPEND_TOKEN_HEAD)
    # closed forms: a row with one nonzero value, a zero row, a negative peak
    kn = case["k_new"].float()
    kn[0, 0] = 0
    kn[0, 0, 3] = 3.0
    kn[1, 1] = 0
    kn[2, 0] = torch.linspace(-5, 1, 8)
    case["k_new"] = kn.to(torch.bfloat16)
    kc, vc, ks, vs, rc = oracle.append_kv(**case, mutation=mutation)
    assert rc == 0
    P, H, D = case["page_size"], case["num_kv_heads"], case["head_dim"]
    kcache = kc.reshape(-1, P, H, D)
    touched = np.zeros((case["num_pages"], P), bool)
    for row, page, slot in _slots(case):
        touched[page, slot] = True
        for h in range(H):
            for new, cache, scales in ((case["k_new"], kcache, ks),
                                       (case["v_new"], vc.reshape(-1, P, H, D), vs)):
                x = new[row, h].float()
                amax = float(x.abs().max())
                s = np.float32(np.float32(amax) / np.float32(448.0)) if amax > 0 else np.float32(1.0)
                assert scales[(page * P + slot) * H + h] == s, (row, h)
                ref = _e4m3_torch((x / torch.tensor(float(s))).float()).numpy()
                assert np.array_equal(cache[page, slot, h], ref), (row, h)
    assert kcache[_slots(case)[0][1], _slots(case)[0][2], 0, 3] == 0x7E
    assert np.all(kcache[_slots(case)[1][1], _slots(case)[1][2], 1] == 0)
    assert ks[(_slots(case)[1][1] * P + _slots(case)[1][2]) * H + 1] == 1.0
    assert kcache[_slots(case)[2][1], _slots(case)[2][2], 0, 0] == 0xFE
    # nothing else changed
    before = case["k_pages"].reshape(-1, P, H, D)
    assert np.array_equal(kcache[~touched], before[~touched])
    assert np.all(ks.reshape(-1, P, H)[~touched] == -1.0)


def pin_append_per_tensor(mutation=0):
    case = _append_case(oracle.APPEND_TENSOR, seed=1)
    kc, vc, ks, vs, rc = oracle.append_kv(**case, mutation=mutation)
    assert rc == 0
    P, H, D = case["page_size"], case["num_kv_heads"], case["head_dim"]
    for row, page, slot in _slots(case):
        for new, cache, s in ((case["k_new"], kc, 0.0125), (case["v_new"], vc, 0.02)):
            y = new[row].float() / torch.tensor(s, dtype=torch.float32)
            ref = _e4m3_torch(y.clamp(-448, 448)).numpy()
            got = cache.reshape(-1, P, H, D)[page, slot]
            assert np.array_equal(got, ref), row


def pin_append_bf16_copy(mutation=0):
    case = _append_case(oracle.APPEND_BF16, seed=2)
    kc, vc, _, _, rc = oracle.append_kv(**case, mutation=mutation)
    assert rc == 0
    P, H, D = case["page_size"], case["num_kv_heads"], case["head_dim"]
    k16 = kc.view(np.uint16).reshape(-1, P, H, D)
    v16 = vc.view(np.uint16).reshape(-1, P, H, D)
    for row, page, slot in _slots(case):
        assert np.array_equal(k16[page, slot], case["k_new"][row].view(torch.int16).numpy().view(np.uint16))
        assert np.array_equal(v16[page, slot], case["v_new"][row].view(torch.int16).numpy().view(np.uint16))


# ------------------------------------------------------------- int8 pins
def pin_int8_constant_code(mutation=0):
    """Every V code -3 with v_scale 0.5 gives o = -1.5 exactly, whatever the
    logits; every K code equal gives lse = ln(visible count) + its logit."""
    def vals(kind, shape, gen):
        if kind == "v":
            return torch.full(shape, -3.0)
        if kind == "k":
            return torch.full(shape, -2.0)
        return torch.randn(shape, generator=gen)
    wl = make_workload(batch=2, rows=[3, 1], kv_lens=[40, 9], num_qo_heads=4, num_kv_heads=2,
                       head_dim=16, page_size=8, kv_dtype="int8", scale_mode=SCALE_TENSOR,
                       unit_scale=True, value_fn=vals, seed=4, poison=True)
    ks, vs = torch.tensor([0.25]), torch.tensor([0.5])
    out, lse, rc = _run(wl, mutation, k_scale=ks, v_scale=vs)
    assert rc == 0
    _close(out, np.full(out.shape, -1.5), what="int8 constant V")
    qd = dequant_q(wl)
    r0 = 0
    for b, (R, L) in enumerate(zip([3, 1], [40, 9])):
        for i in range(R):
            for h in range(4):
                s = wl.sm_scale * float(qd[r0 + i, h].sum()) * (-2.0 * 0.25)
                _close(lse[r0 + i, h], math.log(L - R + i + 1) + s, what=f"int8 lse b{b} i{i} h{h}")
        r0 += R


def pin_int8_encode_vs_torch(mutation=0):
    # integers, half-integers (ties: the even neighbour), random values and
    # values beyond +-127 (clamped), both signs
    g = torch.Generator().manual_seed(9)
    ints = torch.arange(-127, 128).float()
    halves = torch.arange(-130, 130).float() + 0.5
    rnd = (torch.rand(3000, generator=g) * 2 - 1) * 140
    ys = torch.cat([ints, halves, rnd, torch.tensor([1e6, -1e6, 127.5, -127.5])]).float()
    got = torch.tensor([oracle.int8_encode(float(y), mutation) for y in ys])
    ref = torch.round(ys).clamp(-127, 127).to(torch.int64)
    bad = (got != ref).nonzero()
    assert bad.numel() == 0, f"int8 encode differs from torch.round at {ys[bad[0]].item()!r}"


def pin_append_int8(mutation=0):
    for mode in (oracle.APPEND_INT8_TOKEN_HEAD, oracle.APPEND_INT8_TENSOR):
        case = _append_case(mode, seed=3)
        if mode == oracle.APPEND_INT8_TENSOR:
            case["k_scale"], case["v_scale"] = np.array([0.03], np.float32), np.array([0.05], np.float32)
        kn = case["k_new"].float()
        kn[0, 0] = 0                       # a zero row: scale 1, codes 0
        kn[1, 1] = torch.linspace(-4, 2, 8)  # amax 4 at a negative value
        case["k_new"] = kn.to(torch.bfloat16)
        kc, vc, ks, vs, rc = oracle.append_kv(**case, mutation=mutation)
        assert rc == 0
        P, H, D = case["page_size"], case["num_kv_heads"], case["head_dim"]
        for row, page, slot in _slots(case):
            for h in range(H):
                for new, cache, scales in ((case["k_new"], kc, ks), (case["v_new"], vc, vs)):
                    x = new[row, h].float()
                    if mode == oracle.APPEND_INT8_TENSOR:
                        s = np.float32(scales[0])
                    else:
                        amax = float(x.abs().max())
                        s = (np.float32(np.float32(amax) / np.float32(127.0)) if amax > 0
                             else np.float32(1.0))
                        assert scales[(page * P + slot) * H + h] == s, (row, h)
                    ref = torch.round(x / torch.tensor(float(s))).clamp(-127, 127).to(torch.int8)
                    got = cache.reshape(-1, P, H, D)[page, slot, h].view(np.int8)
                    assert np.array_equal(got, ref.numpy()), (mode, row, h)
        if mode == oracle.APPEND_INT8_TOKEN_HEAD:
            r1 = _slots(case)[1]
            assert kc.reshape(-1, P, H, D)[r1[1], r1[2], 1].view(np.int8)[0] == -127


def pin_append_mla_record(mutation=0):
    """MLA records: per 128-channel block s = fp32(amax / 448), codes = the
    E4M3 cast of x / s, the rope channels' bf16 bytes at byte 512; nothing
    else changes. A block's largest value sits in its second half."""
    g = torch.Generator().manual_seed(8)
    P, H, D, rec = 4, 2, 576, 640
    lens, rows = (9, 5), (3, 2)
    pages_per = [math.ceil(L / P) for L in lens]
    num_pages = sum(pages_per) + 2
    perm = torch.randperm(num_pages, generator=g)[:sum(pages_per)].to(torch.int32)
    kv_indptr = torch.tensor([0] + list(np.cumsum(pages_per)), dtype=torch.int32)
    qo = torch.tensor([0] + list(np.cumsum(rows)), dtype=torch.int32)
    n = int(qo[-1])
    x = torch.randn(n, H, D, generator=g)
    x[:, :, 100] = 9.0   # block 0's maximum in its second 64 channels
    x[1, 0, 256:384] = 0  # a zero block: scale 0, codes 0
    k_new = x.to(torch.bfloat16)
    fill = torch.randint(0, 256, (num_pages * P * H * rec,), generator=g, dtype=torch.uint8)
    case = dict(k_new=k_new, v_new=None, page_table=perm, kv_indptr=kv_indptr,
                kv_len=torch.tensor(lens, dtype=torch.int32), qo_indptr=qo,
                k_pages=fill.clone().numpy(), v_pages=None,
                k_scale=np.full(num_pages * P * H * 4, -1.0, np.float32), v_scale=None,
                num_kv_heads=H, head_dim=D, page_size=P, mode=oracle.APPEND_MLA_RECORD,
                strides=(P * H * rec, H * rec, rec), num_pages=num_pages)
    kc, _, ks, _, rc = oracle.append_kv(**case, mutation=mutation)
    assert rc == 0
    kc = kc.reshape(num_pages, P, H, rec)
    ks = ks.reshape(num_pages, P, H, 4)
    touched = np.zeros((num_pages, P), bool)
    for row, page, slot in _slots(case):
        touched[page, slot] = True
        for h in range(H):
            xr = k_new[row, h].float()
            for b in range(4):
                blk = xr[128 * b:128 * (b + 1)]
                amax = float(blk.abs().max())
                sc = np.float32(np.float32(amax) / np.float32(448.0)) if amax > 0 else np.float32(0.0)
                assert ks[page, slot, h, b] == sc, (row, h, b)
                div = float(sc) if amax > 0 else 1.0
                ref = _e4m3_torch((blk / torch.tensor(div)).clamp(-448, 448)).numpy()
                assert np.array_equal(kc[page, slot, h, 128 * b:128 * (b + 1)], ref), (row, h, b)
            rope = k_new[row, h, 512:].contiguous().view(torch.uint8).numpy()
            assert np.array_equal(kc[page, slot, h, 512:], rope), (row, h)
    before = fill.numpy().reshape(num_pages, P, H, rec)
    assert np.array_equal(kc[~touched], before[~touched])
    assert np.all(ks[~touched] == -1.0)


ALL_PINS = [pin_e4m3_all_codes, pin_bruteforce, pin_q_zero_closed_form, pin_single_visible_key,
            pin_constant_v, pin_page_permutation, pin_split_merge, pin_rows_vs_single,
            pin_e4m3_encode_vs_torch, pin_e4m3_encode_saturates, pin_append_token_head,
            pin_append_per_tensor, pin_append_bf16_copy, pin_int8_constant_code,
            pin_int8_encode_vs_torch, pin_append_int8, pin_append_mla_record]

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
    16: "append: per-token scale amax / 256",
    17: "append: E4M3 ties go to the odd code",
    18: "append: new row written one token early",
    19: "append: E4M3 sign dropped",
    24: "MLA: values read from the latent's last dv channels",
    25: "MLA record: nope scale block from 64-channel groups",
    26: "MLA record: rope read at a one-byte stride",
    27: "append: MLA record block amax over its first 64 channels only",
    28: "append: MLA record zero block given scale 1",
    20: "int8 cache bytes read as unsigned",
    21: "append: int8 per-token scale amax / 128",
    22: "append: int8 ties rounded away from zero",
    23: "append: int8 codes not clamped to +-127",
}
