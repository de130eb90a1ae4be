"""The C ABI on the CPU: the library builds and loads, exports every entry
point include/pda.h declares, agrees with the binding's struct layouts, and
its planner and host-side checks behave (no kernel is launched here)."""
import ctypes
import os
import re

import pytest

from paged_split_kv_03_gb300 import binding as B
from paged_split_kv_03_gb300 import build as build_mod

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "pda.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w[\w\s\*]*?\b(pda_\w+)\s*\(", src, re.M)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"pda_plan", "pda_decode", "pda_get_status", "pda_reset_status",
            "pda_strerror"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pda.h but not exported"
    assert sorted(B.EXPORTED) == names, "binding's list of entry points differs from pda.h"


def test_struct_layouts_match(lib):
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.pda_struct_sizes(ctypes.byref(a), ctypes.byref(b)) == 0
    assert a.value == ctypes.sizeof(B.PdaParams)
    assert b.value == ctypes.sizeof(B.PdaPlan)


def _params(**kw):
    p = B.PdaParams()
    base = dict(num_qo_heads=16, num_kv_heads=2, head_dim=256, page_size=16, q_dtype=0,
                kv_dtype=0, scale_mode=0, max_batch=16, max_q_len=8, max_kv_len=32768,
                num_pages=40000, kv_stride_page=16 * 2 * 256, kv_stride_token=2 * 256,
                kv_stride_head=256, device=0, num_sms=152, batch=0, chunk_pages=0, kernel=0)
    base.update(kw)
    for k, v in base.items():
        setattr(p, k, v)
    return p


def test_plan_heads_divide_group(lib):
    # 48 query / 2 kv heads: group 24; heads per CTA must divide 24 at every R
    # (bf16 head_dim 128: the 96-column build, 24 heads up to R = 4, then 12)
    plan, nbytes, rc = B.pda_plan(_params(num_qo_heads=48, num_kv_heads=2, head_dim=128))
    assert plan.rows_per_cta == 96
    for R in range(1, 9):
        h = plan.heads_per_cta[R]
        assert 24 % h == 0 and R * h <= plan.rows_per_cta
    assert plan.heads_per_cta[1] == 24 and plan.heads_per_cta[4] == 24
    assert plan.heads_per_cta[5] == 12 and plan.heads_per_cta[8] == 12
    assert plan.head_blocks == 2
    # E4M3 at head_dim 128 keeps 64 columns: 8 heads at R = 8, 3 head blocks
    f8, _, rc = B.pda_plan(_params(num_qo_heads=48, num_kv_heads=2, head_dim=128, kv_dtype=1,
                                   scale_mode=1, kv_stride_page=16 * 2 * 128,
                                   kv_stride_token=2 * 128, kv_stride_head=128))
    assert rc == 0 and f8.rows_per_cta == 64 and f8.heads_per_cta[8] == 8 and f8.head_blocks == 3


def test_plan_splits_and_scratch(lib):
    plan, nbytes, _ = B.pda_plan(_params(max_batch=1, max_kv_len=32768))
    assert plan.max_splits > 1                      # bs 1: the KV split fills the GPU
    assert plan.grid_ctas <= 2 * 152                # ... in about one wave of CTAs
    assert plan.max_splits * plan.chunk_pages * 16 >= 32768
    rows = 1 * 8
    assert nbytes == plan.scratch_bytes >= 256 + plan.max_splits * rows * 16 * 257 * 4
    plan2, nbytes2, _ = B.pda_plan(_params(num_qo_heads=64, num_kv_heads=8, head_dim=128,
                                           page_size=64, q_dtype=1, kv_dtype=1, scale_mode=1,
                                           max_batch=128, max_q_len=1, max_kv_len=2048,
                                           kv_stride_page=64 * 8 * 128, kv_stride_token=8 * 128,
                                           kv_stride_head=128))
    assert plan2.grid_ctas >= 1024
    forced, _, _ = B.pda_plan(_params(chunk_pages=5))
    assert forced.chunk_pages == 5 and forced.max_splits == 32768 // (5 * 16) + 1


FP8_DECODE = dict(num_qo_heads=64, num_kv_heads=8, head_dim=128, page_size=64, q_dtype=1,
                  kv_dtype=1, scale_mode=1, max_batch=128, max_q_len=1, max_kv_len=2048,
                  kv_stride_page=64 * 8 * 128, kv_stride_token=8 * 128, kv_stride_head=128)


def test_plan_tail_split(lib):
    # 1024 one-split CTAs at 2 per SM are 3.37 waves of 304: the 14 requests
    # of the partial wave are cut into 2 chunks each and laid out last
    plan, _, rc = B.pda_plan(_params(**FP8_DECODE))
    assert rc == 0 and plan.kernel == B.PDA_KERNEL_TC
    assert plan.chunk_pages == 32 and plan.head_splits == 1
    assert (plan.tail_from, plan.tail_chunk_pages, plan.tail_splits) == (114, 16, 2)
    assert plan.max_splits == 2
    assert plan.grid_ctas == 114 * 8 + 14 * 8 * 2
    assert plan.scratch_bytes >= 256 + 2 * 128 * 64 * 129 * 4  # partials for max_splits
    # a forced chunk is used as it is, for every request
    forced, _, _ = B.pda_plan(_params(chunk_pages=8, **FP8_DECODE))
    assert forced.tail_from == forced.batch and forced.tail_chunk_pages == 8
    assert forced.grid_ctas == 128 * 8 * 4
    # a whole number of waves has no tail
    even, _, _ = B.pda_plan(_params(**dict(FP8_DECODE, max_batch=76)))
    assert even.tail_from == even.batch and even.grid_ctas == 76 * 8


def test_plan_one_per_sm_waves(lib):
    # bf16 head_dim 256 runs one CTA per SM; its CTAs start and drain in
    # step, so each wave costs a start-up with the SM idle, and one CTA can
    # stream faster than a 1/152 share of HBM: bs 16 x 2 kv heads at 32K
    # takes one wave of 4 splits (128 CTAs), not three
    plan, _, rc = B.pda_plan(_params(max_q_len=1))
    assert rc == 0 and plan.kernel == B.PDA_KERNEL_TC
    assert plan.rows_per_cta == 64 and plan.grid_ctas <= 152
    assert (plan.head_splits, plan.grid_ctas) == (4, 128)
    # int8 widens its codes at ~24 KB/us per CTA, below the SM's share of
    # HBM: more CTAs than SMs still pays, and it keeps several waves
    i8, _, rc = B.pda_plan(_params(max_q_len=1, kv_dtype=B.PDA_INT8, scale_mode=2,
                                   max_kv_len=131072, num_pages=140000))
    assert rc == 0 and i8.grid_ctas > 2 * 152
    # two CTAs per SM (E4M3 head_dim 256 at 16 columns): unchanged share model
    f8, _, rc = B.pda_plan(_params(max_q_len=1, kv_dtype=1, q_dtype=0, scale_mode=2,
                                   max_kv_len=131072, num_pages=140000))
    assert rc == 0 and f8.grid_ctas == 608


def test_plan_whole_tiles(lib):
    # a CTA works in 128-token tiles, so the planner's chunks at bs 1 leave
    # at most one page of their last tile unused (560 tokens would cost five
    # tiles, 512 four; 864 seven, as 896 would)
    for kw in (dict(max_batch=1, max_q_len=8), dict(max_batch=1, max_q_len=1),
               dict(max_batch=1, max_q_len=4, kv_dtype=1, scale_mode=2, max_kv_len=131072,
                    num_pages=140000)):
        plan, _, rc = B.pda_plan(_params(**kw))
        assert rc == 0 and plan.max_splits > 1
        tokens = plan.chunk_pages * 16
        assert -tokens % 128 <= 16, (kw, plan.chunk_pages)


D512 = dict(num_qo_heads=16, num_kv_heads=1, head_dim=512, page_size=16, max_batch=1,
            max_kv_len=131072, kv_stride_page=16 * 512, kv_stride_token=512, kv_stride_head=512)


def test_plan_head_dim_512(lib):
    # bf16: up to 64 rows x heads per CTA (R 8 -> 8 heads, 2 head blocks)
    plan, _, rc = B.pda_plan(_params(**D512))
    assert rc == 0 and plan.kernel == B.PDA_KERNEL_TC and plan.rows_per_cta == 64
    assert plan.heads_per_cta[1] == 16 and plan.heads_per_cta[8] == 8 and plan.head_blocks == 2
    assert plan.stage1_smem_bytes <= 227 * 1024
    # E4M3: 32 rows x heads (the two-term S and O accumulators' TMEM share)
    for sm in (1, 2):
        q, _, rc = B.pda_plan(_params(kv_dtype=1, scale_mode=sm, **D512))
        assert rc == 0 and q.rows_per_cta == 32
        assert [q.heads_per_cta[r] for r in (1, 2, 4, 8)] == [16, 16, 8, 4] and q.head_blocks == 4
        assert q.stage1_smem_bytes <= 227 * 1024
    # two rows over bf16: the 32-column build
    two, _, _ = B.pda_plan(_params(**dict(D512, max_q_len=2)))
    assert two.rows_per_cta == 32 and two.head_blocks == 1
    # R 1 over bf16 fits 16 columns: the 16-column build, still one CTA per SM
    one, _, _ = B.pda_plan(_params(**dict(D512, max_q_len=1)))
    assert one.rows_per_cta == 16 and one.head_blocks == 1
    # no mma.sync build for head_dim 512
    _, _, rc = B.pda_plan(_params(kernel=B.PDA_KERNEL_MMA, **D512), check=False)
    assert rc == B.PDA_ERR_UNSUPPORTED


MLA = dict(num_qo_heads=16, num_kv_heads=1, head_dim=576, head_dim_v=512, page_size=64,
           max_batch=64, max_q_len=2, max_kv_len=4096, kv_stride_page=64 * 576,
           kv_stride_token=576, kv_stride_head=576)


def test_plan_mla(lib):
    # the latent (576 channels, V its first 512) on the tcgen05 path; scratch
    # partials hold 512 channels
    plan, nbytes, rc = B.pda_plan(_params(**MLA))
    assert rc == 0 and plan.kernel == B.PDA_KERNEL_TC and plan.head_dim_v == 512
    assert plan.rows_per_cta == 32 and plan.head_blocks == 1
    rows = 64 * 2
    assert nbytes >= 256 + plan.max_splits * rows * 16 * (512 + 1) * 4
    assert plan.stage1_smem_bytes <= 227 * 1024
    q, _, rc = B.pda_plan(_params(kv_dtype=1, q_dtype=1, scale_mode=1, **MLA))
    assert rc == 0 and q.rows_per_cta == 32
    for bad in (dict(kv_dtype=1, scale_mode=1),              # E4M3 latent needs an E4M3 query
                dict(kv_dtype=2, scale_mode=1),              # no int8 latent
                dict(kernel=B.PDA_KERNEL_MMA),
                dict(head_dim_v=500)):
        _, _, rc = B.pda_plan(_params(**dict(MLA, **bad)), check=False)
        assert rc == B.PDA_ERR_UNSUPPORTED, bad
    _, _, rc = B.pda_plan(_params(head_dim_v=64), check=False)  # only the MLA pair differs
    assert rc == B.PDA_ERR_UNSUPPORTED
    # the mixed-precision records: E4M3 codes with block scales, bf16 query
    mix, _, rc = B.pda_plan(_params(kv_dtype=1, scale_mode=B.PDA_SCALE_MLA_BLOCK,
                                    **dict(MLA, kv_stride_page=64 * 640, kv_stride_token=640,
                                           kv_stride_head=640)))
    # (their per-block S^T fits TMEM at 16 columns: R = 2 runs two head blocks)
    assert rc == 0 and mix.kernel == B.PDA_KERNEL_TC and mix.rows_per_cta == 16
    assert list(mix.heads_per_cta)[1:3] == [16, 8] and mix.head_blocks == 2
    assert mix.stage1_smem_bytes <= 227 * 1024
    for bad in (dict(q_dtype=1), dict(kv_dtype=0), dict(head_dim=512, head_dim_v=0)):
        args = dict(MLA, kv_dtype=1, scale_mode=B.PDA_SCALE_MLA_BLOCK)
        args.update(bad)
        _, _, rc = B.pda_plan(_params(**args), check=False)
        assert rc == B.PDA_ERR_UNSUPPORTED, bad


def test_plan_int8(lib):
    # int8 caches: the tcgen05 path up to head_dim 256 (codes widened to f16
    # in shared memory, one CTA per SM), the mma.sync path at head_dim 64
    for sm in (1, 2):
        plan, _, rc = B.pda_plan(_params(kv_dtype=B.PDA_INT8, scale_mode=sm))
        assert rc == 0 and plan.kernel == B.PDA_KERNEL_TC and plan.kv_dtype == B.PDA_INT8
        assert plan.stage1_smem_bytes <= 227 * 1024
        d64, _, rc = B.pda_plan(_params(kv_dtype=B.PDA_INT8, scale_mode=sm, head_dim=64,
                                        kv_stride_page=16 * 2 * 64, kv_stride_token=2 * 64,
                                        kv_stride_head=64))
        assert rc == 0 and d64.kernel == B.PDA_KERNEL_MMA
    for bad in (dict(scale_mode=0), dict(q_dtype=1, scale_mode=1), dict(scale_mode=1, **D512)):
        args = dict(kv_dtype=B.PDA_INT8)
        args.update(bad)
        _, _, rc = B.pda_plan(_params(**args), check=False)
        assert rc == B.PDA_ERR_UNSUPPORTED, bad


@pytest.mark.parametrize("bad,code", [
    (dict(num_qo_heads=15), B.PDA_ERR_INVALID),
    (dict(head_dim=96), B.PDA_ERR_UNSUPPORTED),
    (dict(page_size=24), B.PDA_ERR_UNSUPPORTED),
    (dict(max_q_len=9), B.PDA_ERR_INVALID),
    (dict(max_q_len=0), B.PDA_ERR_INVALID),
    (dict(q_dtype=1), B.PDA_ERR_UNSUPPORTED),          # e4m3 Q needs e4m3 KV
    (dict(scale_mode=1), B.PDA_ERR_UNSUPPORTED),       # bf16 KV takes no scales
    (dict(kv_dtype=1, scale_mode=0, kv_stride_page=16 * 2 * 256 // 2 * 2), B.PDA_ERR_UNSUPPORTED),
    (dict(kv_stride_head=260), B.PDA_ERR_ALIGNMENT),   # 520 B: not a multiple of 16
    (dict(batch=17), B.PDA_ERR_INVALID),
    (dict(max_kv_len=0), B.PDA_ERR_INVALID),
    (dict(wait_limit_us=-1), B.PDA_ERR_INVALID),
    (dict(inject=0x80), B.PDA_ERR_INVALID),            # an unknown test hook
])
def test_plan_rejects(lib, bad, code):
    _, _, rc = B.pda_plan(_params(**bad), check=False)
    assert rc == code, (bad, rc, B.pda_strerror(rc))


def test_decode_host_checks_return_before_any_launch(lib):
    plan, _, _ = B.pda_plan(_params())
    fake = 1 << 20  # 16-byte aligned non-null address; never dereferenced on these paths
    args = dict(q=fake, k_pages=fake, v_pages=fake, page_table=fake, kv_indptr=fake,
                kv_len=fake, qo_indptr=fake, max_q_len=4, window=None, sm_scale=0.1,
                k_scale=None, v_scale=None, out=fake, lse=fake, split_scratch=fake, stream=0)

    def call(**over):
        a = dict(args)
        a.update(over)
        return B.pda_decode(plan, check=False, **a)

    assert call(q=None) == B.PDA_ERR_NULL
    assert call(split_scratch=None) == B.PDA_ERR_SCRATCH
    assert call(split_scratch=fake + 16) == B.PDA_ERR_SCRATCH
    assert call(max_q_len=0) == B.PDA_ERR_INVALID
    assert call(max_q_len=9) == B.PDA_ERR_INVALID
    assert call(k_pages=fake + 8) == B.PDA_ERR_ALIGNMENT
    assert call(out=fake + 2) == B.PDA_ERR_ALIGNMENT
    bad = B.PdaPlan()
    assert B.pda_decode(bad, check=False, **args) == B.PDA_ERR_PLAN
    fplan, _, _ = B.pda_plan(_params(kv_dtype=1, scale_mode=2, kv_stride_page=16 * 2 * 256,
                                     kv_stride_token=512, kv_stride_head=256))
    assert B.pda_decode(fplan, check=False, **args) == B.PDA_ERR_NULL  # scales missing
    # the two-stage entry point: a stage mask of 0 or with unknown bits is refused
    sargs = dict(args)
    stream = sargs.pop("stream")
    for mask in (0, 4, 7):
        assert B.pda_decode_stages(plan, check=False, stages=mask, stream=stream,
                                   **sargs) == B.PDA_ERR_INVALID
    assert B.pda_decode_stages(plan, check=False, stages=1, stream=stream,
                               **dict(sargs, q=None)) == B.PDA_ERR_NULL


def test_strerror(lib):
    for code in range(0, -8, -1):
        assert B.pda_strerror(code)
    assert "unknown" in B.pda_strerror(-99)


def test_missing_library_raises(tmp_path):
    # no fallback: a binding pointed at an absent library refuses to load
    with pytest.raises(RuntimeError, match="no fallback"):
        B.load_library(str(tmp_path / "libpda.so"))


def _random_params(rng):
    D = rng.choice([64, 128, 256, 512, 576])
    mla = D == 576
    hkv = 1 if (D >= 512 and rng.random() < 0.8) else rng.choice([1, 2, 4, 8])
    G = rng.choice([1, 2, 3, 4, 6, 8, 12, 16, 24, 48, 64])
    P = rng.choice([1, 2, 4, 8, 16, 32, 64, 128, 256])
    kvt = rng.choice([B.PDA_BF16, B.PDA_E4M3, B.PDA_INT8])
    qt = B.PDA_E4M3 if (kvt == B.PDA_E4M3 and rng.random() < 0.4) else B.PDA_BF16
    sm = B.PDA_SCALE_NONE if kvt == B.PDA_BF16 else rng.choice([1, 2])
    if mla and kvt == B.PDA_E4M3 and rng.random() < 0.5:
        sm, qt = B.PDA_SCALE_MLA_BLOCK, B.PDA_BF16
    Dc = 640 if sm == B.PDA_SCALE_MLA_BLOCK else D      # row elements (record bytes)
    mq, mb = rng.randint(1, 8), rng.choice([1, 2, 3, 7, 16, 64, 128, 256])
    L = rng.choice([1, 7, 64, 1000, 2048, 4096, 32768, 131072])
    return _params(num_qo_heads=G * hkv, num_kv_heads=hkv, head_dim=D, page_size=P,
                   q_dtype=qt, kv_dtype=kvt, scale_mode=sm, max_batch=mb, max_q_len=mq,
                   max_kv_len=L, num_pages=mb * -(-L // P) + 4, kv_stride_page=P * hkv * Dc,
                   kv_stride_token=hkv * Dc, kv_stride_head=Dc, batch=0,
                   chunk_pages=rng.choice([0, 0, 0, 1, 5, 64]), head_dim_v=512 if mla else 0)


def test_plan_invariants_random_shapes(lib):
    """Seeded sweep over shapes, dtypes, page sizes, rows and forced chunks:
    every accepted plan tiles its heads and tokens exactly, sizes its grid
    and scratch for them and fits shared memory; every refusal is a
    documented code."""
    import random
    rng = random.Random(5)
    accepted = 0
    for _ in range(800):
        p = _random_params(rng)
        plan, nbytes, rc = B.pda_plan(p, check=False)
        if rc != B.PDA_OK:
            assert rc in (B.PDA_ERR_UNSUPPORTED, B.PDA_ERR_INVALID, B.PDA_ERR_ALIGNMENT), rc
            continue
        accepted += 1
        G, mq, Hq = p.num_qo_heads // p.num_kv_heads, p.max_q_len, p.num_qo_heads
        for R in range(1, mq + 1):                      # q heads per CTA divide the group
            h = plan.heads_per_cta[R]
            assert G % h == 0 and R * h <= plan.rows_per_cta
        assert plan.head_blocks * plan.heads_per_cta[mq] == G
        pages = -(-p.max_kv_len // p.page_size)         # splits cover the context, none empty
        assert plan.head_splits * plan.chunk_pages >= pages
        assert (plan.head_splits - 1) * plan.chunk_pages < pages
        assert plan.tail_splits * plan.tail_chunk_pages >= pages
        tail = plan.tail_from < plan.batch
        assert plan.max_splits == max(plan.head_splits, plan.tail_splits if tail else 0)
        assert plan.grid_ctas == ((plan.tail_from * plan.head_splits +
                                   (plan.batch - plan.tail_from) * plan.tail_splits) *
                                  p.num_kv_heads * plan.head_blocks)
        assert plan.rows_cap == p.max_batch * mq
        dv = p.head_dim_v or p.head_dim
        assert plan.scratch_lse_offset >= 256 and plan.scratch_lse_offset % 16 == 0
        assert plan.scratch_o_offset % 16 == 0 and nbytes == plan.scratch_bytes
        if plan.max_splits > 1:
            n = plan.max_splits * plan.rows_cap * Hq
            assert plan.scratch_o_offset >= plan.scratch_lse_offset + 4 * n
            assert nbytes >= plan.scratch_o_offset + 4 * n * dv
        assert plan.stage1_smem_bytes <= 227 * 1024
    assert accepted > 500


def test_append_host_checks_return_before_any_launch(lib):
    fake = 1 << 20  # 16-byte aligned non-null address; never dereferenced on these paths
    args = dict(k_new=fake, v_new=fake, page_table=fake, kv_indptr=fake, kv_len=fake,
                qo_indptr=fake, max_q_len=4, k_pages=fake, v_pages=fake, k_scale=fake,
                v_scale=fake, split_scratch=fake, stream=0)

    def call(plan, **over):
        return B.pda_append_kv(plan, check=False, **dict(args, **over))

    fp8, _, _ = B.pda_plan(_params(kv_dtype=1, scale_mode=2, kv_stride_page=16 * 2 * 256,
                                   kv_stride_token=512, kv_stride_head=256))
    assert call(B.PdaPlan()) == B.PDA_ERR_PLAN
    assert call(fp8, k_new=None) == B.PDA_ERR_NULL
    assert call(fp8, v_new=None) == B.PDA_ERR_NULL
    assert call(fp8, v_pages=None) == B.PDA_ERR_NULL
    assert call(fp8, k_scale=None) == B.PDA_ERR_NULL
    assert call(fp8, split_scratch=None) == B.PDA_ERR_SCRATCH
    assert call(fp8, split_scratch=fake + 16) == B.PDA_ERR_SCRATCH
    assert call(fp8, max_q_len=0) == B.PDA_ERR_INVALID
    assert call(fp8, max_q_len=9) == B.PDA_ERR_INVALID
    assert call(fp8, k_new=fake + 2) == B.PDA_ERR_ALIGNMENT
    assert call(fp8, v_pages=fake + 8) == B.PDA_ERR_ALIGNMENT
    assert call(fp8, v_scale=fake + 2) == B.PDA_ERR_ALIGNMENT
    # MLA records: one latent, so the v arguments may be NULL; the block
    # scales are read as 16-byte vectors
    rec, _, _ = B.pda_plan(_params(**dict(MLA, kv_dtype=1, scale_mode=B.PDA_SCALE_MLA_BLOCK,
                                          kv_stride_page=64 * 640, kv_stride_token=640,
                                          kv_stride_head=640)))
    assert call(rec, v_new=None, v_pages=None, v_scale=None, k_scale=fake + 4,
                max_q_len=2) == B.PDA_ERR_ALIGNMENT
    assert call(rec, k_scale=None, max_q_len=2) == B.PDA_ERR_NULL
    # a latent without records has no append kernel
    lat, _, _ = B.pda_plan(_params(**MLA))
    assert call(lat, max_q_len=2) == B.PDA_ERR_UNSUPPORTED


def test_plan_from_host_lengths(lib):
    """Eager planning from the batch's host lengths, rows and windows (the
    mixed batch's shape: 48 / 2 heads, R 1..8, ctx 1K..64K, half windowed):
    the plan is a valid split plan for the same maxima, its chunk covers the
    longest request, and a batch of tiny windowed requests is not split."""
    import random
    rng = random.Random(3)
    bs = 64
    lens = [rng.randint(1024, 65536) for _ in range(bs)]
    rows = [rng.randint(1, 8) for _ in range(bs)]
    wins = [64 if b % 2 == 0 else 0 for b in range(bs)]
    qo = [0]
    for r in rows:
        qo.append(qo[-1] + r)

    def params(lens_, qo_, wins_):
        p = _params(num_qo_heads=48, num_kv_heads=2, head_dim=128, page_size=32, max_batch=bs,
                    max_q_len=8, max_kv_len=65536, num_pages=bs * 2048 + 4,
                    kv_stride_page=32 * 2 * 128, kv_stride_token=2 * 128, kv_stride_head=128)
        keep = [(ctypes.c_int32 * len(x))(*x) for x in (lens_, qo_, wins_)]
        p.host_kv_len, p.host_qo_indptr, p.host_window = (
            ctypes.cast(k, ctypes.POINTER(ctypes.c_int32)) for k in keep)
        return p, keep

    p, keep = params(lens, qo, wins)
    plan, nbytes, rc = B.pda_plan(p)
    assert rc == 0 and plan.kernel == B.PDA_KERNEL_TC
    pages_max = -(-max(lens) // 32)
    assert plan.head_splits * plan.chunk_pages >= pages_max
    assert plan.tail_from == plan.batch  # the simulated grid replaces the tail split
    assert plan.grid_ctas == bs * 2 * plan.head_blocks * plan.head_splits
    base, _ = B.pda_plan(_params(num_qo_heads=48, num_kv_heads=2, head_dim=128, page_size=32,
                                 max_batch=bs, max_q_len=8, max_kv_len=65536,
                                 num_pages=bs * 2048 + 4, kv_stride_page=32 * 2 * 128,
                                 kv_stride_token=2 * 128, kv_stride_head=128))[:2]
    assert plan.max_kv_len <= base.max_kv_len and plan.head_blocks == base.head_blocks
    # every request windowed to 64 keys: one or two pages each, no split
    p2, keep2 = params(lens, qo, [64] * bs)
    small, _, rc = B.pda_plan(p2)
    assert rc == 0 and small.max_splits == 1
