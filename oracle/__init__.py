"""fp64 CPU oracle for paged split-KV decode attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm may import this package. The CUDA library never
links it and it imports nothing from the CUDA library's package: it takes
plain CPU arrays (torch CPU tensors or numpy arrays) and returns fp64 numpy
arrays.

The arithmetic lives in ``pdo_oracle.c`` (plain C, fp64, OpenMP over output
items); this module compiles it with gcc on first use and wraps it with
ctypes. The method it states, and the readings of the pages it takes, are in
that file's header: per-row causal limit p_i = L - R + i, optional sliding
window of W keys, contiguous GQA groups, bf16, OCP E4M3 or int8 cache values
with per-tensor or per-(token, kv head) scales ("perf(attention): run up to 8
query rows per request in the triton decode kernel", section "Changes";
"fp8 support", section "Functionality"; "Naive Support for Hopper FP8
Prefill Kernel with Per-Head Quantization", item 3).
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pdo_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict = {}

PDO_OK = 0
PDO_ERR_ARG = -1
PDO_ERR_KVLEN = -2
PDO_ERR_PAGE = -3


def lib_path(mutation: int = 0) -> str:
    name = "libpdo.so" if mutation == 0 else f"libpdo_mut{mutation}.so"
    return os.path.join(_BUILD, name)


def build(mutation: int = 0, force: bool = False) -> str:
    """Compile the oracle (gcc, -O2, no FP contraction) into oracle/_build.

    ``mutation`` > 0 builds a copy with one deliberate mistake planted
    (``PDO_MUTATION``); the test suite uses those copies to show that the
    pins catch each such mistake. The default build has none.
    """
    out = lib_path(mutation)
    stamp_path = out + ".stamp"
    with open(_SRC, "rb") as f:  # the source and the machine type it was built on
        stamp = hashlib.sha256(platform.machine().encode() + f.read()).hexdigest()
    with _LOCK:
        if not force and os.path.exists(out) and os.path.exists(stamp_path):
            with open(stamp_path) as f:
                if f.read().strip() == stamp:
                    return out
        os.makedirs(_BUILD, exist_ok=True)
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               _SRC, "-o", tmp, "-lm"]
        if mutation:
            cmd.insert(1, f"-DPDO_MUTATION={mutation}")
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
        with open(stamp_path, "w") as f:
            f.write(stamp + "\n")
    return out


def _load(mutation: int = 0):
    if mutation in _LIBS:
        return _LIBS[mutation]
    lib = ctypes.CDLL(build(mutation))
    i32, i64, vp, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
    lib.pdo_attention.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, i64, i64, i64, i64,
                                  vp, vp, vp, vp, vp, vp, vp, vp, dbl, vp, vp, i64, vp, i64,
                                  vp, vp, i32]
    lib.pdo_attention.restype = i32
    lib.pdo_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.pdo_e4m3_to_double.restype = dbl
    lib.pdo_max_threads.restype = i32
    lib.pdo_e4m3_encode.argtypes = [ctypes.c_float]
    lib.pdo_e4m3_encode.restype = ctypes.c_uint8
    lib.pdo_int8_encode.argtypes = [ctypes.c_float]
    lib.pdo_int8_encode.restype = ctypes.c_uint8
    lib.pdo_append.argtypes = [i32, i32, i32, i32, i32, i64, i64, i64, i64, vp, vp, vp, vp, vp,
                               vp, vp, vp, vp, vp]
    lib.pdo_append.restype = i32
    _LIBS[mutation] = lib
    return lib


def _np(x, dtype=None):
    """Contiguous numpy view of a CPU torch tensor / numpy array (None stays None)."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: reinterpret 16-/8-bit payloads as integers
        import torch
        t = x.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        elif t.dtype in (getattr(torch, "float8_e4m3fn", None),):
            t = t.view(torch.uint8)
        x = t.numpy()
    x = np.ascontiguousarray(x)
    if dtype is not None:
        x = x.astype(dtype, copy=False)
    return x


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def e4m3_to_double(code: int, mutation: int = 0) -> float:
    return _load(mutation).pdo_e4m3_to_double(int(code) & 0xFF)


def max_threads() -> int:
    return int(_load().pdo_max_threads())


def attention(*, q, k_pages, v_pages, page_table, kv_indptr, kv_len, qo_indptr, window,
              sm_scale, k_scale=None, v_scale=None, num_qo_heads, num_kv_heads, head_dim,
              page_size, q_e4m3, kv_e4m3, scale_mode, strides, num_pages, items=None,
              split_tokens=0, num_threads=0, mutation=0, check=True, kv_int8=False,
              head_dim_v=None):
    """fp64 attention for the given (row, q head) items.

    Arrays are CPU tensors / numpy arrays holding raw cache payloads (bf16 as
    16-bit words, e4m3 and int8 as bytes; ``kv_int8`` marks an int8 cache).
    ``strides`` = (page, token, head) in elements. ``items`` = flat indices
    row*Hq + h (None: every item). ``head_dim_v`` (default ``head_dim``): the
    value channels, the first ones of each v row (MLA: the latent cache is
    passed as both k and v, 576 channels, V the first 512).
    Returns (out [n, D] float64, lse [n] float64, status).
    """
    lib = _load(mutation)
    q_ = _np(q)
    k_ = _np(k_pages)
    v_ = _np(v_pages)
    pt = _np(page_table, np.int32)
    ki = _np(kv_indptr, np.int32)
    kl = _np(kv_len, np.int32)
    qi = _np(qo_indptr, np.int32)
    win = _np(window, np.int32)
    ks = _np(k_scale, np.float32)
    vs = _np(v_scale, np.float32)
    it = _np(items, np.int64)
    batch = int(kl.shape[0])
    total_rows = int(qi[batch]) if batch else 0
    n = int(it.shape[0]) if it is not None else total_rows * num_qo_heads
    dv = int(head_dim_v or head_dim)
    out = np.zeros((max(n, 0), dv), dtype=np.float64)
    lse = np.zeros((max(n, 0),), dtype=np.float64)
    sp, st, sh = (int(s) for s in strides)
    kv_dtype = 2 if kv_int8 else int(bool(kv_e4m3))
    rc = lib.pdo_attention(batch, num_qo_heads, num_kv_heads, head_dim, dv, page_size, int(q_e4m3),
                           kv_dtype, int(scale_mode), sp, st, sh, int(num_pages), _ptr(q_),
                           _ptr(k_), _ptr(v_), _ptr(pt), _ptr(ki), _ptr(kl), _ptr(qi), _ptr(win),
                           float(sm_scale), _ptr(ks), _ptr(vs), int(split_tokens), _ptr(it),
                           n if it is not None else 0, _ptr(out), _ptr(lse), int(num_threads))
    if check and rc == PDO_ERR_ARG:
        raise ValueError("oracle rejected its arguments")
    return out, lse, rc


def attention_for(wl, items=None, split_tokens=0, num_threads=0, mutation=0, **overrides):
    """``attention`` on a workload object that carries the fields by name
    (q, k_pages, ..., num_qo_heads, ...). The object only transports arrays;
    nothing of its arithmetic is used."""
    args = dict(q=wl.q, k_pages=wl.k_pages, v_pages=wl.v_pages, page_table=wl.page_table,
                kv_indptr=wl.kv_indptr, kv_len=wl.kv_len, qo_indptr=wl.qo_indptr,
                window=wl.window, sm_scale=wl.sm_scale, k_scale=wl.k_scale, v_scale=wl.v_scale,
                num_qo_heads=wl.num_qo_heads, num_kv_heads=wl.num_kv_heads,
                head_dim=wl.head_dim, page_size=wl.page_size, q_e4m3=wl.q_e4m3,
                kv_e4m3=wl.kv_e4m3, scale_mode=wl.scale_mode, strides=wl.strides,
                num_pages=wl.num_pages, kv_int8=getattr(wl, "kv_int8", False),
                head_dim_v=getattr(wl, "head_dim_v", None))
    args.update(overrides)
    return attention(items=items, split_tokens=split_tokens, num_threads=num_threads,
                     mutation=mutation, **args)


def e4m3_encode(y: float, mutation: int = 0) -> int:
    """Nearest E4M3 code to the fp32 value y (ties to even, saturating)."""
    return int(_load(mutation).pdo_e4m3_encode(float(y)))


def int8_encode(y: float, mutation: int = 0) -> int:
    """Symmetric int8 code (as a signed integer) of the fp32 value y: nearest
    integer, ties to even, clamped to [-127, 127]."""
    b = int(_load(mutation).pdo_int8_encode(float(y)))
    return b - 256 if b >= 128 else b


APPEND_BF16, APPEND_TENSOR, APPEND_TOKEN_HEAD = 0, 1, 2
APPEND_INT8_TENSOR, APPEND_INT8_TOKEN_HEAD = 3, 4
APPEND_MLA_RECORD = 5  # 576-channel latent -> 640-byte record + four block scales


def append_kv(*, k_new, v_new, page_table, kv_indptr, kv_len, qo_indptr, k_pages, v_pages,
              k_scale, v_scale, num_kv_heads, head_dim, page_size, mode, strides, num_pages,
              mutation=0):
    """Quantise-on-append into copies of the given caches.

    ``k_new`` / ``v_new``: bf16 [rows, Hkv, D] (CPU tensors or 16-bit words);
    ``k_pages`` / ``v_pages``: the caches before the append (bytes, or bf16
    words for mode 0); ``k_scale`` / ``v_scale``: fp32 arrays (read for
    modes 1 and 3, written for modes 2 and 4, None for mode 0). Modes 3 / 4
    are the int8 counterparts of 1 / 2 (scale amax / 127). Mode 5 writes MLA
    records (head_dim 576: E4M3 nope with a scale per 128 channels, bf16
    rope) from ``k_new`` alone into ``k_pages`` / ``k_scale``. Returns (k_pages, v_pages,
    k_scale, v_scale, status) as numpy arrays (caches as raw bytes).
    """
    lib = _load(mutation)
    kn = _np(k_new).view(np.uint16)
    vn = _np(v_new if v_new is not None else k_new).view(np.uint16)
    kc = np.array(_np(k_pages), copy=True).view(np.uint8)
    vc = kc if v_pages is None else np.array(_np(v_pages), copy=True).view(np.uint8)
    ks = None if k_scale is None else np.array(_np(k_scale, np.float32), copy=True)
    vs = None if v_scale is None else np.array(_np(v_scale, np.float32), copy=True)
    pt = _np(page_table, np.int32)
    ki = _np(kv_indptr, np.int32)
    kl = _np(kv_len, np.int32)
    qi = _np(qo_indptr, np.int32)
    sp, st, sh = (int(s) for s in strides)
    rc = lib.pdo_append(int(kl.shape[0]), num_kv_heads, head_dim, page_size, int(mode), sp, st, sh,
                        int(num_pages), _ptr(kn), _ptr(vn), _ptr(pt), _ptr(ki), _ptr(kl), _ptr(qi),
                        _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs))
    if rc == PDO_ERR_ARG:
        raise ValueError("oracle rejected its arguments")
    return kc, vc, ks, vs, rc
