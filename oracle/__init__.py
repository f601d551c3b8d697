"""Oracle for paged FP8 MLA decode: a plain fp64 CPU implementation.

TEST INFRASTRUCTURE ONLY.  Only tests, the smoke check and the CPU-baseline
leg of the benchmark may import this package.  It shares no code with the CUDA
path (the product never imports it), and it is built from `mla_oracle.c` with
the host C compiler.

Functions follow "CuTe DSL FP8 MLA decode regression" (TensorRT-LLM issue
#20510, "Setup": 512 latent + 64 rope E4M3 rows, page size 32; "Analysis": V
is the latent part of K) for the attention itself, and "split the KV partials
of a row across thread groups in fmhaReductionKernel" (TensorRT-LLM PR #20380,
"Description") for the merge of split partials.  See `mla_oracle.c` for the
formulas.

Parity pins: every function here is pinned by tests in tests/test_oracle.py
(E4M3 against torch's float8 widening, single key, equal scores, split
invariance, causal reduction, page permutation, brute force against torch's
float64 attention, and a hand-expanded two-key case).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmla_oracle.so")
_lock = threading.Lock()
_lib = None

HEAD_DIM = 576
LATENT_DIM = 512


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.mla_oracle_e4m3_decode.restype = ctypes.c_double
            lib.mla_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.mla_oracle_max_threads.restype = ctypes.c_int
            p = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.mla_oracle_decode_rows.restype = ctypes.c_int
            lib.mla_oracle_decode_rows.argtypes = [
                p, p, i64, p, i32, p, i32, i32, i32, i32, f64, f64, f64, p, i64, i64, i64, i32,
                p, p, p, p, i32]
            lib.mla_oracle_decode_rows_ex.restype = ctypes.c_int
            lib.mla_oracle_decode_rows_ex.argtypes = [
                p, p, i32, i64, p, i32, p, i32, i32, i32, i32, f64, f64, f64, p, f64, p, i64,
                i64, i64, i32, p, p, p, p, i32]
            lib.mla_oracle_decode_rows_v2.restype = ctypes.c_int
            lib.mla_oracle_decode_rows_v2.argtypes = [
                p, p, i32, i64, p, i32, p, i32, i32, i32, i32, f64, f64, f64, p, f64, p, p, p,
                i32, p, i64, i64, i64, i32, p, p, p, p, i32]
            lib.mla_oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.mla_oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.mla_oracle_kv_append.restype = ctypes.c_int
            lib.mla_oracle_kv_append.argtypes = [p, i64, p, p, p, i32, i32, p, i64, ctypes.c_float]
            lib.mla_oracle_merge.restype = None
            lib.mla_oracle_merge.argtypes = [p, p, i64, i32, p, p]
            _lib = lib
    return _lib


def _np(x, dtype):
    """Host numpy view of a torch tensor or array-like, contiguous, given dtype."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x), dtype=dtype)


def max_threads() -> int:
    return int(_load().mla_oracle_max_threads())


def e4m3_decode(codes) -> np.ndarray:
    """Exact E4M3 decode of uint8 codes (fp64)."""
    lib = _load()
    c = _np(codes, np.uint8)
    out = np.array([lib.mla_oracle_e4m3_decode(int(v)) for v in c.reshape(-1)], dtype=np.float64)
    return out.reshape(c.shape)


def decode_rows(q, kv, page_table, kv_lens, *, q_len: int, num_heads: int, causal: bool,
                softmax_scale: float, q_scale: float = 1.0, kv_scale: float = 1.0,
                rows=None, tok_begin: int = -1, tok_end: int = -1, partial: bool = False,
                n_threads: int = 0, sinks=None, output_scale: float = 1.0, query_lens=None,
                kv_bounds=None, block_idx=None):
    """Run the fp64 oracle on the given rows.

    q: uint8 [B, q_len, H, 576]; kv: uint8 [P, 32, 576] (E4M3 codes), or both
    torch bfloat16 tensors (the BF16-KV variant); page_table int32
    [B, max_pages]; kv_lens int32 [B].  rows: flat row ids (b*q_len+qi)*H+h,
    default all.  sinks: optional per-head sink logits [H] (natural-log units);
    output_scale multiplies O.  query_lens int32 [B] (per-request query tokens in
    the padded q_len slots), kv_bounds int32 [B, 2] (key window [lo, hi)) and
    block_idx int32 [B, topk] (selected logical pages, negative = unused)
    restrict the visible keys; see mla_oracle.c.  Returns (O [n, 512], LSE [n])
    or, with partial=True, (O_unnormalised [n, 512], m_log2 [n], l [n]).
    """
    lib = _load()
    dtype = 0
    try:
        import torch
        if isinstance(q, torch.Tensor) and q.dtype in (torch.bfloat16, torch.int16):
            dtype = 1
            q = q.view(torch.int16)
            kv = kv.view(torch.int16)
    except ImportError:  # pragma: no cover
        pass
    if dtype == 0:
        qa = _np(q, np.uint8)
        kva = _np(kv, np.uint8)
    else:
        qa = _np(q, np.int16)
        kva = _np(kv, np.int16)
    pt = _np(page_table, np.int32)
    lens = _np(kv_lens, np.int32)
    batch = int(lens.shape[0])
    if rows is None:
        rows = np.arange(batch * q_len * num_heads, dtype=np.int64)
    ra = _np(rows, np.int64)
    n = int(ra.shape[0])
    out = np.zeros((n, LATENT_DIM), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    m = np.zeros((n,), dtype=np.float64)
    l = np.zeros((n,), dtype=np.float64)
    num_pages = int(kva.shape[0])
    sk = None if sinks is None else _np(sinks, np.float64)
    ql = None if query_lens is None else _np(query_lens, np.int32)
    kb = None if kv_bounds is None else _np(kv_bounds, np.int32).reshape(batch, 2)
    bi = None if block_idx is None else _np(block_idx, np.int32).reshape(batch, -1)
    st = lib.mla_oracle_decode_rows_v2(
        qa.ctypes.data, kva.ctypes.data, dtype, num_pages, pt.ctypes.data, int(pt.shape[1]),
        lens.ctypes.data, batch, int(q_len), int(num_heads), int(bool(causal)), float(q_scale),
        float(kv_scale), float(softmax_scale), None if sk is None else sk.ctypes.data,
        float(output_scale), None if ql is None else ql.ctypes.data,
        None if kb is None else kb.ctypes.data, None if bi is None else bi.ctypes.data,
        0 if bi is None else int(bi.shape[1]), ra.ctypes.data, n, int(tok_begin), int(tok_end),
        1 if partial else 0, out.ctypes.data, lse.ctypes.data, m.ctypes.data, l.ctypes.data,
        int(n_threads))
    if st != 0:
        raise RuntimeError(f"oracle decode failed with status {st}")
    if partial:
        return out, m, l
    return out, lse


def merge(partial_o, partial_ml):
    """Closed-form merge of split partials (fp64).

    partial_o [rows, S, 512], partial_ml [rows, S, 2] = (m in log2 units, l).
    Returns (O [rows, 512], LSE [rows]) with LSE in natural-log units.
    """
    lib = _load()
    o = _np(partial_o, np.float64)
    ml = _np(partial_ml, np.float64)
    rows, S = int(o.shape[0]), int(o.shape[1])
    out = np.zeros((rows, LATENT_DIM), dtype=np.float64)
    lse = np.zeros((rows,), dtype=np.float64)
    lib.mla_oracle_merge(ml.ctypes.data, o.ctypes.data, rows, S, out.ctypes.data, lse.ctypes.data)
    return out, lse


def e4m3_encode(values) -> np.ndarray:
    """Nearest E4M3 codes (ties to even, saturating at 448) of float32 values."""
    lib = _load()
    v = _np(values, np.float32)
    out = np.array([lib.mla_oracle_e4m3_encode(float(x)) for x in v.reshape(-1)], dtype=np.uint8)
    return out.reshape(v.shape)


def kv_append(rows_bf16, req, pos, page_table, kv, kv_scale: float):
    """Quantize bf16 rows [n, 576] (given as uint16/int16 bit patterns or a torch
    bfloat16 tensor) into a copy of the uint8 pool kv [P, 32, 576]; returns the
    new pool and the status (0, or -1 if some row had an invalid target)."""
    lib = _load()
    try:
        import torch
        if isinstance(rows_bf16, torch.Tensor) and rows_bf16.dtype == torch.bfloat16:
            rows_bf16 = rows_bf16.view(torch.int16)
    except ImportError:  # pragma: no cover
        pass
    r = _np(rows_bf16, np.int16).view(np.uint16)
    rq = _np(req, np.int32)
    ps = _np(pos, np.int32)
    pt = _np(page_table, np.int32)
    pool = _np(kv, np.uint8).copy()
    st = lib.mla_oracle_kv_append(r.ctypes.data, int(r.shape[0]), rq.ctypes.data, ps.ctypes.data,
                                  pt.ctypes.data, int(pt.shape[1]), int(pt.shape[0]),
                                  pool.ctypes.data, int(pool.shape[0]), float(kv_scale))
    return pool, int(st)
