"""Seeded synthetic workloads for paged decode attention.

This module only draws inputs: query rows, a paged K/V cache (bf16, OCP
E4M3 codes or int8 codes, with their scales), a shuffled page table and the CSR offsets. It
holds none of the attention arithmetic. Both the CUDA library's callers and
the fp64 oracle consume the arrays it returns, so neither side's arithmetic
can leak into the other's inputs.

Recipe (stated once here, used by the tests and the benchmark):
  * values: Q, K, V ~ N(0, 1) from a torch.Generator seeded per workload;
  * bf16 payloads are the round-to-nearest-even bf16 of those values;
  * FP8 payloads: scale = amax / 448 (1 if amax == 0), per tensor or per
    (token, kv head) over head_dim; code = e4m3(clamp(x / scale, +-448))
    by torch's float8_e4m3fn cast (RNE). int8 payloads: scale = amax / 127
    (1 if amax == 0), code = clamp(round-half-even(x / scale), +-127) by
    torch.round. A per-tensor E4M3 query folds its
    scale into the returned sm_scale, so a consumer multiplies decoded codes
    by sm_scale only;
  * optional K outliers: round(frac * head_dim) channels per kv head, chosen
    by the seed and fixed across tokens, multiplied by ``k_outlier_mult``
    before quantisation;
  * the page table is a random permutation of the physical pages; every
    request's CSR list gets ``extra_table_entries`` trailing entries that
    point at poison pages, and ``extra_pages`` poison pages exist;
  * poison: pages no request uses and the tail slots of each request's last
    page hold NaN (bf16 0x7FC0, e4m3 0x7F), and so do their per-token scales,
    so that any read of them shows up as NaN in the output (int8 has no NaN:
    its poison code is -128, which no quantiser produces, and only the
    per-token scales of those slots are NaN).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence, Union

import torch

E4M3_MAX = 448.0
BF16_NAN_BITS = 0x7FC0
E4M3_NAN_CODE = 0x7F
INT8_MAX = 127.0
INT8_POISON = -128

SCALE_NONE, SCALE_TENSOR, SCALE_TOKEN_HEAD = 0, 1, 2
# MLA latent records: 512 E4M3 nope codes (a scale per token, kv head and 128
# channels) then the 64 bf16 rope channels, 640 bytes per (token, kv head)
SCALE_MLA_BLOCK = 3
MLA_NOPE, MLA_ROPE, MLA_RECORD = 512, 64, 640


@dataclass
class Workload:
    name: str
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    q_e4m3: bool
    kv_e4m3: bool
    scale_mode: int
    layout: str                      # "NHD" = [page, slot, head, d]; "HND" = [page, head, slot, d]
    strides: tuple                   # (page, token, head) strides in elements
    q: torch.Tensor                  # [total_rows, Hq, D] bf16 or uint8 codes
    k_pages: torch.Tensor            # cache, bf16 or uint8 codes, layout as above
    v_pages: torch.Tensor
    k_scale: Optional[torch.Tensor]  # None, [1] or [num_pages, page_size, Hkv] float32
    v_scale: Optional[torch.Tensor]
    page_table: torch.Tensor         # int32 CSR page ids
    kv_indptr: torch.Tensor          # int32 [B+1]
    kv_len: torch.Tensor             # int32 [B]
    qo_indptr: torch.Tensor          # int32 [B+1]
    window: Optional[torch.Tensor]   # int32 [B] (<= 0: none) or None
    sm_scale: float
    q_scale: float = 1.0             # already folded into sm_scale when q_e4m3
    meta: dict = field(default_factory=dict)
    kv_int8: bool = False            # int8 cache codes (kv_e4m3 is then False)
    head_dim_v: Optional[int] = None # value channels (None: head_dim); MLA: v_pages is k_pages

    @property
    def batch(self) -> int:
        return int(self.kv_len.shape[0])

    @property
    def total_rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_q_len(self) -> int:
        """Largest rows-per-request (read from host-side metadata when the
        offsets live on a device, so that it never synchronises a stream)."""
        if self.qo_indptr.device.type == "cpu" or "rows" not in self.meta:
            r = self.qo_indptr[1:] - self.qo_indptr[:-1]
            return int(r.max().item()) if r.numel() else 0
        return max(self.meta["rows"]) if self.meta["rows"] else 0

    @property
    def group(self) -> int:
        return self.num_qo_heads // self.num_kv_heads

    def rows_per_request(self):
        return (self.qo_indptr[1:] - self.qo_indptr[:-1]).tolist()

    def to(self, device) -> "Workload":
        def mv(t):
            return None if t is None else t.to(device)
        k_pages, k_scale = mv(self.k_pages), mv(self.k_scale)
        # an MLA latent cache is one tensor read as K and as V: keep it one
        v_pages = k_pages if self.v_pages is self.k_pages else mv(self.v_pages)
        v_scale = k_scale if self.v_scale is self.k_scale else mv(self.v_scale)
        return Workload(self.name, self.num_qo_heads, self.num_kv_heads, self.head_dim,
                        self.page_size, self.num_pages, self.q_e4m3, self.kv_e4m3,
                        self.scale_mode, self.layout, self.strides, mv(self.q), k_pages,
                        v_pages, k_scale, v_scale,
                        mv(self.page_table), mv(self.kv_indptr), mv(self.kv_len),
                        mv(self.qo_indptr), mv(self.window), self.sm_scale, self.q_scale,
                        dict(self.meta), self.kv_int8, self.head_dim_v)


def _as_list(x, n):
    if isinstance(x, (list, tuple)):
        assert len(x) == n
        return [int(v) for v in x]
    return [int(x)] * n


def _quant_e4m3(x: torch.Tensor, amax_dims) -> tuple:
    """(codes uint8, scale float32) with scale = amax/448 over ``amax_dims``
    (None: whole tensor)."""
    if amax_dims is None:
        amax = x.abs().amax().float()
    else:
        amax = x.abs().amax(dim=amax_dims).float()
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    if amax_dims is None:
        y = x / scale
    else:
        y = x / scale.unsqueeze(-1)
    codes = y.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale.to(torch.float32)


def _quant_int8(x: torch.Tensor, amax_dims) -> tuple:
    """(codes int8, scale float32) with scale = amax/127 over ``amax_dims``
    (None: whole tensor); codes = clamp(round(x / scale), +-127), ties to even."""
    if amax_dims is None:
        amax = x.abs().amax().float()
    else:
        amax = x.abs().amax(dim=amax_dims).float()
    scale = torch.where(amax > 0, amax / INT8_MAX, torch.ones_like(amax))
    y = x / scale if amax_dims is None else x / scale.unsqueeze(-1)
    codes = torch.round(y).clamp(-INT8_MAX, INT8_MAX).to(torch.int8)
    return codes, scale.to(torch.float32)


def _exact_int8(x: torch.Tensor) -> torch.Tensor:
    """int8 codes of integer values in [-127, 127] (asserted)."""
    codes = x.to(torch.int8)
    assert torch.equal(codes.to(torch.float32), x), "value not an int8 code"
    assert int(codes.min()) >= -INT8_MAX, "-128 is the poison code"
    return codes


def _exact_e4m3(x: torch.Tensor) -> torch.Tensor:
    """E4M3 codes of values that E4M3 represents exactly (asserted)."""
    codes = x.to(torch.float8_e4m3fn)
    back = codes.to(torch.float32)
    assert torch.equal(back, x), "value not exactly representable in E4M3"
    return codes.view(torch.uint8)


def make_workload(*, name: str = "custom", batch: int, rows: Union[int, Sequence[int]],
                  kv_lens: Union[int, Sequence[int]], num_qo_heads: int, num_kv_heads: int,
                  head_dim: int, page_size: int, kv_dtype: str = "bf16", q_dtype: str = "bf16",
                  scale_mode: int = SCALE_NONE, windows=None, sm_scale: Optional[float] = None,
                  layout: str = "NHD", seed: int = 0, device="cpu",
                  k_outlier_frac: float = 0.0, k_outlier_mult: float = 20.0,
                  q_mult: float = 1.0, extra_pages: int = 4, extra_table_entries: int = 1,
                  poison: bool = True, value_fn=None, token_fn=None,
                  unit_scale: bool = False, scale_fn=None, head_dim_v: Optional[int] = None
                  ) -> Workload:
    """Draw one workload.

    Structured tests may replace the N(0,1) draws:
      ``value_fn(kind, shape, gen)`` -- kind in {"q", "k", "v"}, logical
          shapes [rows, Hq, D] and [num_pages, P, Hkv, D];
      ``token_fn(kind, b, L)`` -- kind in {"k", "v"}: values [L, Hkv, D] of
          request b's tokens in order, scattered through the page table;
      ``unit_scale`` -- E4M3 / int8 scales fixed at 1 (values must be exact
          E4M3, or integers in [-127, 127] for int8);
      ``scale_fn(kind, b, L)`` -- per-(token, kv head) scales [L, Hkv] of
          request b (with ``unit_scale``), e.g. to ramp logits per token.
    ``head_dim_v`` < head_dim makes an MLA latent cache: one tensor (and one
    scale) serves as K (all head_dim channels) and V (the first head_dim_v).
    """
    assert kv_dtype in ("bf16", "e4m3", "int8") and q_dtype in ("bf16", "e4m3")
    if scale_mode == SCALE_MLA_BLOCK:
        assert kv_dtype == "e4m3" and q_dtype == "bf16" and head_dim == 576 and head_dim_v == 512
    assert q_dtype == "bf16" or kv_dtype == "e4m3"
    assert num_qo_heads % num_kv_heads == 0
    if kv_dtype == "bf16":
        assert scale_mode == SCALE_NONE
    else:
        assert scale_mode in (SCALE_TENSOR, SCALE_TOKEN_HEAD, SCALE_MLA_BLOCK)
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(seed))
    R = _as_list(rows, batch)
    L = _as_list(kv_lens, batch)
    P, H, D = page_size, num_kv_heads, head_dim
    qo_indptr = [0]
    for r in R:
        qo_indptr.append(qo_indptr[-1] + r)
    npages_b = [-(-l // P) for l in L]
    used = sum(npages_b)
    num_pages = used + int(extra_pages)
    perm = torch.randperm(num_pages, generator=gen, device=dev).to(torch.int32).cpu().tolist()
    poison_pages = perm[used:]
    table, kv_indptr, cursor = [], [0], 0
    for b in range(batch):
        table.extend(perm[cursor:cursor + npages_b[b]])
        cursor += npages_b[b]
        for e in range(extra_table_entries):
            table.append(poison_pages[(b + e) % len(poison_pages)] if poison_pages else perm[0])
        kv_indptr.append(len(table))

    def draw(kind, shape):
        if value_fn is not None:
            return value_fn(kind, shape, gen).to(dev, torch.float32)
        return torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)

    total_rows = qo_indptr[-1]
    qf = draw("q", (total_rows, num_qo_heads, D)) * q_mult
    kf = draw("k", (num_pages, P, H, D))
    vf = draw("v", (num_pages, P, H, D)) if head_dim_v is None else kf
    if token_fn is not None or scale_fn is not None:
        cursor = 0
        for b in range(batch):
            pages = torch.tensor(perm[cursor:cursor + npages_b[b]], dtype=torch.long, device=dev)
            cursor += npages_b[b]
            tok = torch.arange(L[b], device=dev)
            pg, sl = pages[tok // P], tok % P
            if token_fn is not None:
                kf[pg, sl] = token_fn("k", b, L[b]).to(dev, torch.float32)
                if head_dim_v is None:
                    vf[pg, sl] = token_fn("v", b, L[b]).to(dev, torch.float32)
    outlier_channels = None
    if k_outlier_frac > 0:
        n_out = max(1, int(round(k_outlier_frac * D)))
        outlier_channels = torch.stack([torch.randperm(D, generator=gen, device=dev)[:n_out]
                                        for _ in range(H)])
        for h in range(H):
            kf[:, :, h, outlier_channels[h]] *= k_outlier_mult

    # valid-slot mask [num_pages, P]: which slots hold a real token
    valid = torch.zeros(num_pages, P, dtype=torch.bool, device=dev)
    cursor = 0
    for b in range(batch):
        pages = torch.tensor(perm[cursor:cursor + npages_b[b]], dtype=torch.long, device=dev)
        cursor += npages_b[b]
        if npages_b[b]:
            valid[pages] = True
            tail = L[b] - (npages_b[b] - 1) * P
            valid[pages[-1], tail:] = False

    q_scale = 1.0
    if q_dtype == "bf16":
        q = qf.to(torch.bfloat16)
    elif unit_scale:
        q = _exact_e4m3(qf)
    else:
        q, qs = _quant_e4m3(qf, None)
        q_scale = float(qs.item())
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    sm_eff = float(sm_scale) * q_scale

    k_scale = v_scale = None
    if kv_dtype == "bf16":
        kc, vc = kf.to(torch.bfloat16), vf.to(torch.bfloat16)
    elif unit_scale:
        if kv_dtype == "int8":
            kc, vc = _exact_int8(kf), _exact_int8(vf)
        else:
            kc, vc = _exact_e4m3(kf), _exact_e4m3(vf)
        if scale_mode == SCALE_TENSOR:
            k_scale = torch.ones(1, dtype=torch.float32, device=dev)
            v_scale = torch.ones(1, dtype=torch.float32, device=dev)
        else:
            k_scale = torch.ones(num_pages, P, H, dtype=torch.float32, device=dev)
            v_scale = torch.ones(num_pages, P, H, dtype=torch.float32, device=dev)
            if scale_fn is not None:
                cursor = 0
                for b in range(batch):
                    pages = torch.tensor(perm[cursor:cursor + npages_b[b]], dtype=torch.long,
                                         device=dev)
                    cursor += npages_b[b]
                    tok = torch.arange(L[b], device=dev)
                    pg, sl = pages[tok // P], tok % P
                    k_scale[pg, sl] = scale_fn("k", b, L[b]).to(dev, torch.float32)
                    v_scale[pg, sl] = scale_fn("v", b, L[b]).to(dev, torch.float32)
    elif scale_mode == SCALE_MLA_BLOCK:
        # nope: E4M3 with amax/448 per (token, kv head, 128 channels); rope: bf16
        nope = kf[..., :MLA_NOPE].reshape(num_pages, P, H, MLA_NOPE // 128, 128)
        codes, k_scale = _quant_e4m3(nope, -1)  # scale [pages, P, H, 4]
        rope = kf[..., MLA_NOPE:].to(torch.bfloat16).contiguous().view(torch.uint8)
        kc = torch.cat([codes.reshape(num_pages, P, H, MLA_NOPE), rope], dim=-1).contiguous()
        vc, v_scale = kc, k_scale
    elif scale_mode == SCALE_TENSOR:
        quant = _quant_int8 if kv_dtype == "int8" else _quant_e4m3
        kc, k_scale = quant(kf, None)
        vc, v_scale = quant(vf, None)
        k_scale, v_scale = k_scale.reshape(1), v_scale.reshape(1)
    else:
        quant = _quant_int8 if kv_dtype == "int8" else _quant_e4m3
        kc, k_scale = quant(kf, -1)
        vc, v_scale = quant(vf, -1)
    del kf, vf, qf

    if poison:
        bad = ~valid
        if kv_dtype == "bf16":
            nanb = torch.tensor(BF16_NAN_BITS, dtype=torch.int16, device=dev).view(torch.bfloat16)
            kc[bad] = nanb
            vc[bad] = nanb
        elif kv_dtype == "int8":
            kc[bad] = INT8_POISON
            vc[bad] = INT8_POISON
        elif scale_mode == SCALE_MLA_BLOCK:
            kc[..., :MLA_NOPE][bad] = E4M3_NAN_CODE
            nan_rope = torch.tensor([BF16_NAN_BITS], dtype=torch.int16, device=dev).view(torch.uint8)
            kc[..., MLA_NOPE:][bad] = nan_rope.repeat(MLA_ROPE)
        else:
            kc[bad] = E4M3_NAN_CODE
            vc[bad] = E4M3_NAN_CODE
        if scale_mode in (SCALE_TOKEN_HEAD, SCALE_MLA_BLOCK):
            k_scale[bad] = float("nan")
            v_scale[bad] = float("nan")

    Dc = MLA_RECORD if scale_mode == SCALE_MLA_BLOCK else D  # elements (bytes) per row
    if layout == "NHD":
        strides = (P * H * Dc, H * Dc, Dc)
    elif layout == "HND":
        kc = kc.permute(0, 2, 1, 3).contiguous()
        vc = vc.permute(0, 2, 1, 3).contiguous()
        strides = (H * P * Dc, Dc, P * Dc)
    else:
        raise ValueError(layout)
    if head_dim_v is not None:
        # MLA: one latent cache read as K and as V (its first head_dim_v channels)
        assert 0 < head_dim_v <= D
        vc, v_scale = kc, k_scale

    win = None
    if windows is not None:
        win = torch.tensor(_as_list(windows, batch), dtype=torch.int32, device=dev)

    i32 = dict(dtype=torch.int32, device=dev)
    return Workload(
        name=name, num_qo_heads=num_qo_heads, num_kv_heads=H, head_dim=D, page_size=P,
        num_pages=num_pages, q_e4m3=(q_dtype == "e4m3"), kv_e4m3=(kv_dtype == "e4m3"),
        scale_mode=scale_mode, layout=layout, strides=strides, q=q, k_pages=kc, v_pages=vc,
        k_scale=k_scale, v_scale=v_scale, page_table=torch.tensor(table, **i32),
        kv_indptr=torch.tensor(kv_indptr, **i32), kv_len=torch.tensor(L, **i32),
        qo_indptr=torch.tensor(qo_indptr, **i32), window=win, sm_scale=sm_eff, q_scale=q_scale,
        meta=dict(seed=seed, rows=R, kv_lens=L, outlier_channels=outlier_channels,
                  poison_pages=poison_pages), kv_int8=(kv_dtype == "int8"),
        head_dim_v=head_dim_v)


# ---------------------------------------------------------------------------
# The five workloads the benchmark and the parity tests use.

CONFIG_NAMES = ("tiny", "fp8_decode", "mtp_verify_bf16", "longctx_fp8_pth", "mixed")
# head_dim 512 with one kv head: the full-attention layers of the Gemma-4
# MTP runs ("perf(attention): run up to 8 query rows per request in the
# triton decode kernel", "Gemma-4 MTP at long context"); 16 query heads
# (the page gives no count), bs 1, R 1 / 4 / 8 (no spec, k = 3, k = 7)
D512_NAMES = ("d512_mtp_bf16", "d512_mtp_fp8")
# MLA decode ("fp8 support", FlashMLA PR #54): a 576-channel latent (512 +
# the 64-channel rope) per token, one kv head, V = its first 512 channels;
# 16 query heads (128 over 8-way tensor parallelism; the page gives none),
# pages of 64, bs 64, ctx 4096, R 1 (2); bf16, or E4M3 Q/K/V per tensor
MLA_NAMES = ("mla_bf16", "mla_fp8", "mla_fp8_mixed")


def config_workload(name: str, *, R: Optional[int] = None, bs: Optional[int] = None,
                    device="cpu", seed: Optional[int] = None, **kw) -> Workload:
    """The named workload at its stated sizes (seed 1000 + its index).

    tiny            bs 1, R 1, 16/2 heads, D 128, ctx 512, page 16, bf16, 4 poison pages
    fp8_decode      bs 128, R 1, 64/8 heads, D 128, ctx 2048, page 64, Q/K/V e4m3
                    with per-tensor scales, bf16 output
    mtp_verify_bf16 16/2 heads, D 256, R 4 (1, 8), ctx 32768, bs 1 or 16, page 16, bf16
    longctx_fp8_pth 16/2 heads, D 256, R 1 or 8 (4), ctx 131072, bs 1 or 16, page 16,
                    e4m3 K/V with a scale per (token, kv head), 1% K channels x20, Q bf16
    mixed           bs 64, 48/2 heads, D 128, R_b ~ U{1..8}, ctx_b ~ U[1024, 65536],
                    window 64 on half the requests, page 32, bf16
    longctx_int8_pth  the longctx_fp8_pth shape with int8 codes (scale amax / 127)
                    per (token, kv head) (seed 1200)
    mla_bf16        bs 64, R 1 (2), 16/1 heads, latent 576 (V its first 512), ctx 4096,
                    page 64, bf16 (seeds 1300 + index)
    mla_fp8         the same with E4M3 Q and latent, per-tensor scales
    mla_fp8_mixed   the same with latent records: E4M3 nope with a scale per token and
                    128 channels, bf16 rope; bf16 Q
    d512_mtp_bf16   bs 1 (16), R 4 (1, 8), 16/1 heads, D 512, ctx 32768, page 16, bf16
    d512_mtp_fp8    bs 1 (16), R 4 (1, 8), 16/1 heads, D 512, ctx 32768, page 16, e4m3
                    K/V with a scale per (token, kv head), Q bf16 (seeds 1100 + index)
    """
    if name == "longctx_int8_pth":
        # the longctx_fp8_pth shape over an int8 cache (same scale kind)
        seed = 1200 if seed is None else seed
        return config_workload("longctx_fp8_pth", R=R, bs=bs, device=device, seed=seed,
                               **dict(dict(kv_dtype="int8"), **kw))
    if name in MLA_NAMES:
        seed = 1300 + MLA_NAMES.index(name) if seed is None else seed
        args = dict(batch=bs or 64, rows=R or 1, kv_lens=4096, num_qo_heads=16, num_kv_heads=1,
                    head_dim=576, head_dim_v=512, page_size=64)
        if name == "mla_fp8":
            args.update(kv_dtype="e4m3", q_dtype="e4m3", scale_mode=SCALE_TENSOR)
        elif name == "mla_fp8_mixed":
            args.update(kv_dtype="e4m3", q_dtype="bf16", scale_mode=SCALE_MLA_BLOCK)
        args.update(kw)
        return make_workload(name=name, seed=seed, device=device, **args)
    if name in D512_NAMES:
        seed = 1100 + D512_NAMES.index(name) if seed is None else seed
        args = dict(batch=bs or 1, rows=R or 4, kv_lens=32768, num_qo_heads=16, num_kv_heads=1,
                    head_dim=512, page_size=16)
        if name == "d512_mtp_fp8":
            args.update(kv_dtype="e4m3", q_dtype="bf16", scale_mode=SCALE_TOKEN_HEAD)
        args.update(kw)
        return make_workload(name=name, seed=seed, device=device, **args)
    idx = CONFIG_NAMES.index(name)
    seed = 1000 + idx if seed is None else seed
    if name == "tiny":
        args = dict(batch=1, rows=1, kv_lens=512, num_qo_heads=16, num_kv_heads=2, head_dim=128,
                    page_size=16)
    elif name == "fp8_decode":
        args = dict(batch=128, rows=1, kv_lens=2048, num_qo_heads=64, num_kv_heads=8,
                    head_dim=128, page_size=64, kv_dtype="e4m3", q_dtype="e4m3",
                    scale_mode=SCALE_TENSOR)
    elif name == "mtp_verify_bf16":
        args = dict(batch=bs or 16, rows=R or 4, kv_lens=32768, num_qo_heads=16, num_kv_heads=2,
                    head_dim=256, page_size=16)
    elif name == "longctx_fp8_pth":
        args = dict(batch=bs or 16, rows=R or 8, kv_lens=131072, num_qo_heads=16,
                    num_kv_heads=2, head_dim=256, page_size=16, kv_dtype="e4m3",
                    q_dtype="bf16", scale_mode=SCALE_TOKEN_HEAD, k_outlier_frac=0.01)
    elif name == "mixed":
        g = torch.Generator().manual_seed(seed + 7)
        b = bs or 64
        rows = torch.randint(1, 9, (b,), generator=g).tolist()
        lens = torch.randint(1024, 65537, (b,), generator=g).tolist()
        order = torch.randperm(b, generator=g).tolist()
        win = [0] * b
        for pos, req in enumerate(order):
            if pos % 2 == 0:
                win[req] = 64
        args = dict(batch=b, rows=rows, kv_lens=lens, num_qo_heads=48, num_kv_heads=2,
                    head_dim=128, page_size=32, windows=win)
    else:
        raise KeyError(name)
    args.update(kw)
    return make_workload(name=name, seed=seed, device=device, **args)
