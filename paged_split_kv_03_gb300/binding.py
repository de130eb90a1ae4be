"""Thin ctypes binding of the C ABI in include/pda.h (argument marshalling only).

The names mirror the C entry points: ``pda_plan``, ``pda_decode``,
``pda_get_status``, ``pda_reset_status``, ``pda_strerror``. Tensors are
passed as raw pointers (``data_ptr()``) and streams as their CUDA handle;
every step of the computation runs in the library's kernels. There is no
fallback: if ``_lib/libpda.so`` has not been built, loading raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libpda.so")

PDA_BF16, PDA_E4M3, PDA_INT8 = 0, 1, 2
PDA_SCALE_MLA_BLOCK = 3
PDA_SCALE_NONE, PDA_SCALE_TENSOR, PDA_SCALE_TOKEN_HEAD = 0, 1, 2
PDA_KERNEL_AUTO, PDA_KERNEL_MMA, PDA_KERNEL_TC = 0, 1, 2
PDA_OK = 0
PDA_ERR_NULL, PDA_ERR_INVALID, PDA_ERR_UNSUPPORTED = -1, -2, -3
PDA_ERR_ALIGNMENT, PDA_ERR_SCRATCH, PDA_ERR_CUDA, PDA_ERR_PLAN = -4, -5, -6, -7
PDA_ERR_TOO_LARGE = -8
PDA_STATIC_SCRATCH_BYTES = 32 << 20
PDA_STATUS_KV_LEN_LT_ROWS = 0x1
PDA_STATUS_ROWS_GT_MAX = 0x2
PDA_STATUS_KV_LEN_GT_MAX = 0x4
PDA_STATUS_PAGE_OOB = 0x8
PDA_STATUS_ROWS_GT_CAP = 0x10
PDA_STATUS_WAIT_TIMEOUT = 0x20
PDA_STATUS_SMEM_MISALIGNED = 0x40
PDA_PLAN_MAGIC = 0x50444131
PDA_INJECT_WITHHOLD_KV = 0x1

# every entry point include/pda.h declares
EXPORTED = ("pda_plan", "pda_decode", "pda_decode_stages", "pda_decode_static", "pda_append_kv",
            "pda_get_status", "pda_reset_status", "pda_strerror", "pda_version",
            "pda_struct_sizes")

_i32, _i64, _u32, _vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_void_p


class PdaParams(ctypes.Structure):
    _fields_ = [("num_qo_heads", _i32), ("num_kv_heads", _i32), ("head_dim", _i32),
                ("page_size", _i32), ("q_dtype", _i32), ("kv_dtype", _i32),
                ("scale_mode", _i32), ("max_batch", _i32), ("max_q_len", _i32),
                ("max_kv_len", _i32), ("num_pages", _i32), ("kv_stride_page", _i64),
                ("kv_stride_token", _i64), ("kv_stride_head", _i64), ("device", _i32),
                ("num_sms", _i32), ("host_kv_len", ctypes.POINTER(_i32)), ("batch", _i32),
                ("chunk_pages", _i32), ("kernel", _i32), ("head_dim_v", _i32),
                ("wait_limit_us", _i32), ("inject", _u32),
                ("host_qo_indptr", ctypes.POINTER(_i32)), ("host_window", ctypes.POINTER(_i32))]


class PdaPlan(ctypes.Structure):
    _fields_ = [("magic", _u32), ("num_qo_heads", _i32), ("num_kv_heads", _i32),
                ("head_dim", _i32), ("page_size", _i32), ("q_dtype", _i32), ("kv_dtype", _i32),
                ("scale_mode", _i32), ("max_batch", _i32), ("max_q_len", _i32),
                ("max_kv_len", _i32), ("num_pages", _i32), ("batch", _i32),
                ("kv_stride_page", _i64), ("kv_stride_token", _i64), ("kv_stride_head", _i64),
                ("group", _i32), ("kernel", _i32), ("rows_per_cta", _i32),
                ("heads_per_cta", _i32 * 9), ("head_blocks", _i32), ("chunk_pages", _i32),
                ("max_splits", _i32), ("num_sms", _i32), ("grid_ctas", _i64),
                ("rows_cap", _i64), ("scratch_bytes", _i64), ("scratch_lse_offset", _i64),
                ("scratch_o_offset", _i64), ("stage1_smem_bytes", _i32),
                ("tail_from", _i32), ("tail_chunk_pages", _i32), ("head_splits", _i32),
                ("tail_splits", _i32), ("head_dim_v", _i32), ("device", _i32),
                ("wait_limit_us", _i32), ("inject", _u32), ("reserved", _i32 * 7)]


class PdaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where} failed: {pda_strerror(code)} ({code})")


_LIB = None


def load_library(path: Optional[str] = None):
    """Load libpda.so (built by paged_split_kv_03_gb300.build); raises if absent."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with paged_split_kv_03_gb300.build.build() "
                           "(there is no fallback implementation)")
    lib = ctypes.CDLL(p)
    lib.pda_plan.argtypes = [ctypes.POINTER(PdaParams), ctypes.POINTER(PdaPlan),
                             ctypes.POINTER(ctypes.c_size_t)]
    lib.pda_plan.restype = ctypes.c_int
    lib.pda_decode.argtypes = [ctypes.POINTER(PdaPlan), _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                               _i32, _vp, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.pda_decode.restype = ctypes.c_int
    lib.pda_decode_stages.argtypes = [ctypes.POINTER(PdaPlan), _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                      _i32, _vp, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _u32,
                                      _vp]
    lib.pda_decode_stages.restype = ctypes.c_int
    lib.pda_decode_static.argtypes = [ctypes.POINTER(PdaPlan), _vp, _vp, _vp, _vp, _vp, _vp,
                                      _vp, _i32, _vp, ctypes.c_float, _vp, _vp, _vp, _vp, _vp]
    lib.pda_decode_static.restype = ctypes.c_int
    lib.pda_append_kv.argtypes = [ctypes.POINTER(PdaPlan), _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                  _vp, _vp, _vp, _vp, _vp, _vp]
    lib.pda_append_kv.restype = ctypes.c_int
    lib.pda_get_status.argtypes = [ctypes.POINTER(PdaPlan), _vp, ctypes.POINTER(_u32), _vp]
    lib.pda_get_status.restype = ctypes.c_int
    lib.pda_reset_status.argtypes = [ctypes.POINTER(PdaPlan), _vp, _vp]
    lib.pda_reset_status.restype = ctypes.c_int
    lib.pda_strerror.argtypes = [ctypes.c_int]
    lib.pda_strerror.restype = ctypes.c_char_p
    lib.pda_version.restype = ctypes.c_int
    lib.pda_struct_sizes.argtypes = [ctypes.POINTER(ctypes.c_size_t),
                                     ctypes.POINTER(ctypes.c_size_t)]
    lib.pda_struct_sizes.restype = ctypes.c_int
    if path is None:
        _LIB = lib
    return lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def pda_strerror(code: int) -> str:
    return load_library().pda_strerror(int(code)).decode()


def pda_plan(params: PdaParams, check: bool = True):
    """-> (PdaPlan, scratch_bytes, rc)."""
    plan = PdaPlan()
    nbytes = ctypes.c_size_t(0)
    rc = load_library().pda_plan(ctypes.byref(params), ctypes.byref(plan), ctypes.byref(nbytes))
    if check and rc != PDA_OK:
        raise PdaError(rc, "pda_plan")
    return plan, int(nbytes.value), rc


def pda_decode(plan: PdaPlan, q, k_pages, v_pages, page_table, kv_indptr, kv_len, qo_indptr,
               max_q_len: int, window, sm_scale: float, k_scale, v_scale, out, lse,
               split_scratch, stream=None, check: bool = True) -> int:
    rc = load_library().pda_decode(
        ctypes.byref(plan), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
        _ptr(kv_indptr), _ptr(kv_len), _ptr(qo_indptr), int(max_q_len), _ptr(window),
        float(sm_scale), _ptr(k_scale), _ptr(v_scale), _ptr(out), _ptr(lse), _ptr(split_scratch),
        _stream(stream))
    if check and rc != PDA_OK:
        raise PdaError(rc, "pda_decode")
    return rc


PDA_STAGE_PARTIAL, PDA_STAGE_MERGE = 1, 2


def pda_decode_stages(plan: PdaPlan, q, k_pages, v_pages, page_table, kv_indptr, kv_len,
                      qo_indptr, max_q_len: int, window, sm_scale: float, k_scale, v_scale, out,
                      lse, split_scratch, stages: int, stream=None, check: bool = True) -> int:
    """pda_decode's stage 1 (PDA_STAGE_PARTIAL) and / or merge (PDA_STAGE_MERGE)."""
    rc = load_library().pda_decode_stages(
        ctypes.byref(plan), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
        _ptr(kv_indptr), _ptr(kv_len), _ptr(qo_indptr), int(max_q_len), _ptr(window),
        float(sm_scale), _ptr(k_scale), _ptr(v_scale), _ptr(out), _ptr(lse), _ptr(split_scratch),
        int(stages), _stream(stream))
    if check and rc != PDA_OK:
        raise PdaError(rc, "pda_decode_stages")
    return rc


def pda_decode_static(plan: PdaPlan, q, k_pages, v_pages, page_table, kv_indptr, kv_len,
                      qo_indptr, max_q_len: int, window, sm_scale: float, k_scale, v_scale, out,
                      lse, stream=None, check: bool = True) -> int:
    """pda_decode for callers that cannot allocate device memory: the split
    scratch is the library's own fixed array (PDA_STATIC_SCRATCH_BYTES), so
    nothing is allocated. Calls share that array: do not overlap them."""
    rc = load_library().pda_decode_static(
        ctypes.byref(plan), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
        _ptr(kv_indptr), _ptr(kv_len), _ptr(qo_indptr), int(max_q_len), _ptr(window),
        float(sm_scale), _ptr(k_scale), _ptr(v_scale), _ptr(out), _ptr(lse), _stream(stream))
    if check and rc != PDA_OK:
        raise PdaError(rc, "pda_decode_static")
    return rc


def pda_append_kv(plan: PdaPlan, k_new, v_new, page_table, kv_indptr, kv_len, qo_indptr,
                  max_q_len: int, k_pages, v_pages, k_scale, v_scale, split_scratch,
                  stream=None, check: bool = True) -> int:
    """Quantise-on-append of the new rows' K/V (bf16 [rows, Hkv, D]) into the
    paged cache of the plan's dtype and scale mode (see include/pda.h)."""
    rc = load_library().pda_append_kv(
        ctypes.byref(plan), _ptr(k_new), _ptr(v_new), _ptr(page_table), _ptr(kv_indptr),
        _ptr(kv_len), _ptr(qo_indptr), int(max_q_len), _ptr(k_pages), _ptr(v_pages),
        _ptr(k_scale), _ptr(v_scale), _ptr(split_scratch), _stream(stream))
    if check and rc != PDA_OK:
        raise PdaError(rc, "pda_append_kv")
    return rc


def pda_get_status(plan: PdaPlan, split_scratch, stream=None) -> int:
    """Device status bits; ``split_scratch=None`` reads those of the
    built-in array that pda_decode_static uses."""
    bits = _u32(0)
    rc = load_library().pda_get_status(ctypes.byref(plan), _ptr(split_scratch),
                                       ctypes.byref(bits), _stream(stream))
    if rc != PDA_OK:
        raise PdaError(rc, "pda_get_status")
    return int(bits.value)


def pda_reset_status(plan: PdaPlan, split_scratch, stream=None) -> None:
    rc = load_library().pda_reset_status(ctypes.byref(plan), _ptr(split_scratch),
                                         _stream(stream))
    if rc != PDA_OK:
        raise PdaError(rc, "pda_reset_status")


# ---------------------------------------------------------------- helpers

def params_for(wl, *, max_batch=None, max_q_len=None, max_kv_len=None, device=0, num_sms=0,
               chunk_pages=0, kernel=PDA_KERNEL_AUTO, batch=0, wait_limit_us=0,
               inject=0, host_plan=False) -> PdaParams:
    """PdaParams describing a workload object (synth.Workload or alike).
    ``host_plan``: pass the batch's host lengths, rows and windows, so the
    planner sizes the KV chunk for this batch (the plan still serves any
    lengths within its maxima)."""
    p = PdaParams()
    p.num_qo_heads = wl.num_qo_heads
    p.num_kv_heads = wl.num_kv_heads
    p.head_dim = wl.head_dim
    p.page_size = wl.page_size
    p.q_dtype = PDA_E4M3 if wl.q_e4m3 else PDA_BF16
    p.kv_dtype = (PDA_E4M3 if wl.kv_e4m3 else
                  PDA_INT8 if getattr(wl, "kv_int8", False) else PDA_BF16)
    p.scale_mode = wl.scale_mode
    p.max_batch = max_batch or wl.batch
    p.max_q_len = max_q_len or max(1, wl.max_q_len)
    p.max_kv_len = max_kv_len or max(1, int(wl.kv_len.max().item()))
    p.num_pages = wl.num_pages
    p.kv_stride_page, p.kv_stride_token, p.kv_stride_head = (int(s) for s in wl.strides)
    p.device = device
    p.num_sms = num_sms
    p.batch = batch or wl.batch
    p.chunk_pages = chunk_pages
    p.kernel = kernel
    p.head_dim_v = getattr(wl, "head_dim_v", None) or 0
    p.wait_limit_us = wait_limit_us
    p.inject = inject
    if host_plan:
        def arr(xs):
            a = (_i32 * len(xs))(*[int(x) for x in xs])
            return a, ctypes.cast(a, ctypes.POINTER(_i32))
        p._keep = [arr(wl.kv_len.cpu().tolist()), arr(wl.qo_indptr.cpu().tolist())]
        p.host_kv_len, p.host_qo_indptr = p._keep[0][1], p._keep[1][1]
        if wl.window is not None:
            p._keep.append(arr(wl.window.cpu().tolist()))
            p.host_window = p._keep[2][1]
    return p


class Decoder:
    """A plan plus its split scratch (allocated once with torch) for one
    workload shape; ``run`` enqueues one pda_decode on the current stream."""

    def __init__(self, params: PdaParams, device="cuda"):
        import torch
        self.params = params
        self.plan, self.scratch_bytes, _ = pda_plan(params)
        n = (max(self.scratch_bytes, 256) + 255) // 256 * 256
        self.scratch = torch.zeros(n, dtype=torch.uint8, device=device)

    def run(self, wl, out, lse, max_q_len=None, stream=None, sm_scale=None, stages=None):
        args = (self.plan, wl.q, wl.k_pages, wl.v_pages, wl.page_table, wl.kv_indptr, wl.kv_len,
                wl.qo_indptr, max_q_len or max(1, wl.max_q_len), wl.window,
                wl.sm_scale if sm_scale is None else sm_scale, wl.k_scale, wl.v_scale, out, lse,
                self.scratch)
        if stages is None:
            return pda_decode(*args, stream)
        return pda_decode_stages(*args, stages, stream)

    def status(self, stream=None) -> int:
        return pda_get_status(self.plan, self.scratch, stream)

    def reset_status(self, stream=None) -> None:
        pda_reset_status(self.plan, self.scratch, stream)
