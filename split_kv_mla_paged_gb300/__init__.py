"""Paged FP8 MLA split-KV decode for GB300 (sm_103a).

A thin ctypes binding over libmla_decode.so (declared in include/mla_decode.h).
The functions keep the C names and only marshal arguments: every step of the
decode runs in the library's CUDA kernels.  PyTorch supplies device memory and
streams.  There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading
from typing import Optional, Sequence

import numpy as np

from . import build as _build

__all__ = [
    "MLA_OK", "MLA_ERR_INVALID_ARG", "MLA_ERR_UNSUPPORTED", "MLA_ERR_WORKSPACE_TOO_SMALL",
    "MLA_ERR_CUDA", "MLA_ERR_TIMEOUT", "MlaError", "Plan", "load_library", "library_path",
    "mla_decode_plan", "mla_decode_workspace_size", "mla_decode_workspace_init", "mla_decode",
    "mla_decode_splitkv", "mla_decode_merge", "mla_merge", "mla_decode_status", "mla_last_error",
    "mla_decode_static_ws", "mla_decode_static_ws_status", "mla_kv_append", "mla_decode_ex",
    "mla_decode_bf16", "mla_decode_sparse", "mla_decode_plan_items", "mla_decode_bf16_ex",
    "mla_decode_bf16_sparse", "mla_decode_plan_items_bf16", "DecodeOptions",
    "decode", "merge",
    "EXPORTED_SYMBOLS",
]

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE_TOO_SMALL = 3
MLA_ERR_CUDA = 4
MLA_ERR_TIMEOUT = 5
_STATUS_NAMES = {
    0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED",
    3: "MLA_ERR_WORKSPACE_TOO_SMALL", 4: "MLA_ERR_CUDA", 5: "MLA_ERR_TIMEOUT",
}
EXPORTED_SYMBOLS = ("mla_decode_plan", "mla_decode_workspace_size", "mla_decode_workspace_init",
                    "mla_decode", "mla_decode_splitkv", "mla_decode_merge", "mla_merge",
                    "mla_decode_status", "mla_last_error", "mla_debug_set_wait_limit",
                    "mla_decode_static_ws", "mla_decode_static_ws_status", "mla_kv_append",
                    "mla_decode_ex", "mla_decode_bf16", "mla_decode_sparse",
                    "mla_decode_plan_items", "mla_decode_bf16_ex", "mla_decode_bf16_sparse",
                    "mla_decode_plan_items_bf16", "mla_debug_set_expire")

HEAD_DIM = 576
LATENT_DIM = 512
PAGE_SIZE = 32
TILE_TOKENS = 128
MAX_SPLITS = 256
PAGES_SPLIT_CAP = 128


class DecodeOptions(ctypes.Structure):
    """mla_decode_options_t (include/mla_decode.h)."""
    _fields_ = [("q_scale_dev", ctypes.c_void_p), ("kv_scale_dev", ctypes.c_void_p),
                ("softmax_scale_dev", ctypes.c_void_p), ("output_scale", ctypes.c_float),
                ("sinks", ctypes.c_void_p), ("query_lens", ctypes.c_void_p),
                ("kv_bounds", ctypes.c_void_p), ("cta_items", ctypes.c_void_p),
                ("num_ctas", ctypes.c_int32), ("persistent_ctas", ctypes.c_int32),
                ("phases", ctypes.c_int32)]


# mla_decode_options_t.phases: both phases, the split-KV kernel only, the merge only.
PHASE_ALL, PHASE_SPLIT, PHASE_MERGE = 0, 1, 2


class MlaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load libmla_decode.so (built by `build.build()`); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with split_kv_mla_paged_gb300.build.build() "
                "(there is no fallback implementation)")
        lib = ctypes.CDLL(path)
        vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                 ctypes.c_size_t)
        lib.mla_decode_plan.restype = ctypes.c_int
        lib.mla_decode_plan.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp]
        for name in ("mla_decode_plan_items", "mla_decode_plan_items_bf16"):
            getattr(lib, name).restype = ctypes.c_int
            getattr(lib, name).argtypes = [vp, i32, i32, i32, vp, i32, vp]
        lib.mla_decode_workspace_size.restype = sz
        lib.mla_decode_workspace_size.argtypes = [i32, i32, i32, i32]
        dec_args = [vp, vp, i64, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, f32, f32,
                    vp, sz, vp, vp, vp, vp]
        for name in ("mla_decode", "mla_decode_splitkv", "mla_decode_merge"):
            getattr(lib, name).restype = ctypes.c_int
            getattr(lib, name).argtypes = dec_args
        lib.mla_decode_ex.restype = ctypes.c_int
        lib.mla_decode_ex.argtypes = dec_args[:-1] + [ctypes.POINTER(DecodeOptions), vp]
        lib.mla_decode_sparse.restype = ctypes.c_int
        lib.mla_decode_sparse.argtypes = (dec_args[:6] + [vp, i32] + dec_args[6:-1]
                                          + [ctypes.POINTER(DecodeOptions), vp])
        lib.mla_decode_bf16.restype = ctypes.c_int
        lib.mla_decode_bf16.argtypes = dec_args[:14] + [f32] + dec_args[17:]
        lib.mla_decode_bf16_ex.restype = ctypes.c_int
        lib.mla_decode_bf16_ex.argtypes = (dec_args[:14] + [f32] + dec_args[17:-1]
                                           + [ctypes.POINTER(DecodeOptions), vp])
        lib.mla_decode_bf16_sparse.restype = ctypes.c_int
        lib.mla_decode_bf16_sparse.argtypes = (dec_args[:6] + [vp, i32] + dec_args[6:14] + [f32]
                                               + dec_args[17:-1]
                                               + [ctypes.POINTER(DecodeOptions), vp])
        lib.mla_decode_workspace_init.restype = ctypes.c_int
        lib.mla_decode_workspace_init.argtypes = [vp, sz, vp]
        lib.mla_merge.restype = ctypes.c_int
        lib.mla_merge.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp]
        lib.mla_decode_status.restype = ctypes.c_int
        lib.mla_decode_status.argtypes = [vp, vp]
        lib.mla_decode_static_ws.restype = ctypes.c_int
        lib.mla_decode_static_ws.argtypes = [vp, vp, i64, vp, i32, vp, vp, vp, i32, i32, i32, i32,
                                             i32, i32, f32, f32, f32, vp, vp, vp, vp]
        lib.mla_decode_static_ws_status.restype = ctypes.c_int
        lib.mla_decode_static_ws_status.argtypes = [vp]
        lib.mla_kv_append.restype = ctypes.c_int
        lib.mla_kv_append.argtypes = [vp, i64, vp, vp, vp, i32, i32, vp, i64, f32, vp, vp]
        lib.mla_debug_set_wait_limit.restype = None
        lib.mla_debug_set_wait_limit.argtypes = [ctypes.c_longlong]
        lib.mla_debug_set_expire.restype = None
        lib.mla_debug_set_expire.argtypes = [i32, i32]
        lib.mla_last_error.restype = ctypes.c_char_p
        lib.mla_last_error.argtypes = []
        _lib = lib
        return lib


def mla_last_error() -> str:
    return load_library().mla_last_error().decode("utf-8", "replace")


def _check(status: int) -> None:
    if status != MLA_OK:
        raise MlaError(status, mla_last_error())


def _ptr(t) -> Optional[int]:
    """Address of a torch tensor / numpy array, or None."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


@dataclasses.dataclass
class Plan:
    splits: np.ndarray   # int32 [B]
    chunks: np.ndarray   # int32 [B]
    kv_split: int
    workspace_bytes: int

    @property
    def max_splits(self) -> int:
        return int(self.splits.max())


def mla_decode_plan(kv_lens: Sequence[int], num_heads: int, q_len: int, sm_count: int = 0,
                    target_ctas: int = 0) -> Plan:
    lib = load_library()
    lens = np.ascontiguousarray(np.asarray(kv_lens, dtype=np.int32))
    b = int(lens.shape[0])
    splits = np.zeros(b, dtype=np.int32)
    chunks = np.zeros(b, dtype=np.int32)
    kvs = ctypes.c_int32(0)
    ws = ctypes.c_size_t(0)
    _check(lib.mla_decode_plan(lens.ctypes.data, b, int(num_heads), int(q_len), int(sm_count),
                               int(target_ctas), splits.ctypes.data, chunks.ctypes.data,
                               ctypes.addressof(kvs), ctypes.addressof(ws)))
    return Plan(splits=splits, chunks=chunks, kv_split=int(kvs.value), workspace_bytes=int(ws.value))


def mla_decode_plan_items(splits, num_heads: int, q_len: int, bf16: bool = False) -> np.ndarray:
    """CTA item list of a plan (one int32 per CTA that has work, split-major);
    bf16=True builds it with the BF16 kernels' row groups."""
    lib = load_library()
    fn = lib.mla_decode_plan_items_bf16 if bf16 else lib.mla_decode_plan_items
    sp = np.ascontiguousarray(np.asarray(splits, dtype=np.int32))
    n = ctypes.c_int32(0)
    _check(fn(sp.ctypes.data, int(sp.shape[0]), int(num_heads), int(q_len), None, 0,
              ctypes.addressof(n)))
    items = np.zeros(int(n.value), dtype=np.int32)
    _check(fn(sp.ctypes.data, int(sp.shape[0]), int(num_heads), int(q_len), items.ctypes.data,
              int(items.shape[0]), ctypes.addressof(n)))
    return items


def mla_decode_plan_items_bf16(splits, num_heads: int, q_len: int) -> np.ndarray:
    """The CTA item list for the BF16 entry points."""
    return mla_decode_plan_items(splits, num_heads, q_len, bf16=True)


def mla_decode_workspace_size(batch: int, q_len: int, num_heads: int, max_splits: int) -> int:
    return int(load_library().mla_decode_workspace_size(batch, q_len, num_heads, max_splits))


def mla_decode(q_fp8, kv_pages_fp8, num_pages: int, page_table, max_pages_per_req: int,
               kv_lens, splits, chunks, max_splits: int, kv_split: int, batch: int, q_len: int,
               num_heads: int, causal: bool, q_scale: float, kv_scale: float,
               softmax_scale: float, workspace, workspace_bytes: int, out_bf16, lse_f32=None,
               out_f32_debug=None, stream=None) -> None:
    """Enqueue one decode (split-KV kernel + merge) on `stream`; see mla_decode.h."""
    _decode_call("mla_decode", q_fp8, kv_pages_fp8, num_pages, page_table, max_pages_per_req,
                 kv_lens, splits, chunks, max_splits, kv_split, batch, q_len, num_heads, causal,
                 q_scale, kv_scale, softmax_scale, workspace, workspace_bytes, out_bf16, lse_f32,
                 out_f32_debug, stream)


def _decode_call(fn_name, q_fp8, kv_pages_fp8, num_pages, page_table, max_pages_per_req, kv_lens,
                 splits, chunks, max_splits, kv_split, batch, q_len, num_heads, causal, q_scale,
                 kv_scale, softmax_scale, workspace, workspace_bytes, out_bf16, lse_f32,
                 out_f32_debug, stream):
    fn = getattr(load_library(), fn_name)
    _check(fn(_ptr(q_fp8), _ptr(kv_pages_fp8), int(num_pages), _ptr(page_table),
              int(max_pages_per_req), _ptr(kv_lens), _ptr(splits), _ptr(chunks), int(max_splits),
              int(kv_split), int(batch), int(q_len), int(num_heads), 1 if causal else 0,
              float(q_scale), float(kv_scale), float(softmax_scale), _ptr(workspace),
              int(workspace_bytes), _ptr(out_bf16), _ptr(lse_f32), _ptr(out_f32_debug),
              _stream_handle(stream)))


def mla_decode_ex(q_fp8, kv_pages_fp8, num_pages, page_table, max_pages_per_req, kv_lens, splits,
                  chunks, max_splits, kv_split, batch, q_len, num_heads, causal, q_scale,
                  kv_scale, softmax_scale, workspace, workspace_bytes, out_bf16, lse_f32=None,
                  out_f32_debug=None, *, q_scale_dev=None, kv_scale_dev=None,
                  softmax_scale_dev=None, output_scale: float = 1.0, sinks=None,
                  query_lens=None, kv_bounds=None, cta_items=None, persistent_ctas: int = 0,
                  phases: int = PHASE_ALL, stream=None) -> None:
    """mla_decode with device-side scales, an output scale, attention sinks,
    ragged query counts, key windows and a CTA item list (a device int32
    tensor from mla_decode_plan_items), optionally run by persistent_ctas
    CTAs that loop over the list; phases selects the split-KV kernel or the
    merge alone."""
    opts = DecodeOptions(_ptr(q_scale_dev), _ptr(kv_scale_dev), _ptr(softmax_scale_dev),
                         float(output_scale), _ptr(sinks), _ptr(query_lens), _ptr(kv_bounds),
                         _ptr(cta_items), 0 if cta_items is None else int(cta_items.numel()),
                         int(persistent_ctas), int(phases))
    lib = load_library()
    _check(lib.mla_decode_ex(_ptr(q_fp8), _ptr(kv_pages_fp8), int(num_pages), _ptr(page_table),
                             int(max_pages_per_req), _ptr(kv_lens), _ptr(splits), _ptr(chunks),
                             int(max_splits), int(kv_split), int(batch), int(q_len),
                             int(num_heads), 1 if causal else 0, float(q_scale), float(kv_scale),
                             float(softmax_scale), _ptr(workspace), int(workspace_bytes),
                             _ptr(out_bf16), _ptr(lse_f32), _ptr(out_f32_debug),
                             ctypes.byref(opts), _stream_handle(stream)))


def mla_decode_bf16(q_bf16, kv_pages_bf16, num_pages: int, page_table, max_pages_per_req: int,
                    kv_lens, splits, chunks, max_splits: int, kv_split: int, batch: int,
                    q_len: int, num_heads: int, causal: bool, softmax_scale: float, workspace,
                    workspace_bytes: int, out_bf16, lse_f32=None, out_f32_debug=None,
                    stream=None) -> None:
    """Enqueue one BF16-KV decode (split-KV kernel + merge) on `stream`."""
    lib = load_library()
    _check(lib.mla_decode_bf16(_ptr(q_bf16), _ptr(kv_pages_bf16), int(num_pages),
                               _ptr(page_table), int(max_pages_per_req), _ptr(kv_lens),
                               _ptr(splits), _ptr(chunks), int(max_splits), int(kv_split),
                               int(batch), int(q_len), int(num_heads), 1 if causal else 0,
                               float(softmax_scale), _ptr(workspace), int(workspace_bytes),
                               _ptr(out_bf16), _ptr(lse_f32), _ptr(out_f32_debug),
                               _stream_handle(stream)))


def mla_decode_bf16_ex(q_bf16, kv_pages_bf16, num_pages, page_table, max_pages_per_req, kv_lens,
                       splits, chunks, max_splits, kv_split, batch, q_len, num_heads, causal,
                       softmax_scale, workspace, workspace_bytes, out_bf16, lse_f32=None,
                       out_f32_debug=None, *, softmax_scale_dev=None, output_scale: float = 1.0,
                       sinks=None, query_lens=None, kv_bounds=None, cta_items=None,
                       phases: int = PHASE_ALL, stream=None) -> None:
    """mla_decode_bf16 with a device softmax scale, output scale, sinks,
    ragged query counts, key windows and a CTA item list (a device int32
    tensor from mla_decode_plan_items_bf16); phases as for mla_decode_ex."""
    opts = DecodeOptions(None, None, _ptr(softmax_scale_dev), float(output_scale), _ptr(sinks),
                         _ptr(query_lens), _ptr(kv_bounds), _ptr(cta_items),
                         0 if cta_items is None else int(cta_items.numel()), 0, int(phases))
    lib = load_library()
    _check(lib.mla_decode_bf16_ex(_ptr(q_bf16), _ptr(kv_pages_bf16), int(num_pages),
                                  _ptr(page_table), int(max_pages_per_req), _ptr(kv_lens),
                                  _ptr(splits), _ptr(chunks), int(max_splits), int(kv_split),
                                  int(batch), int(q_len), int(num_heads), 1 if causal else 0,
                                  float(softmax_scale), _ptr(workspace), int(workspace_bytes),
                                  _ptr(out_bf16), _ptr(lse_f32), _ptr(out_f32_debug),
                                  ctypes.byref(opts), _stream_handle(stream)))


def mla_decode_bf16_sparse(q_bf16, kv_pages_bf16, num_pages, page_table, max_pages_per_req,
                           kv_lens, block_idx, topk, splits, chunks, max_splits, kv_split, batch,
                           q_len, num_heads, causal, softmax_scale, workspace, workspace_bytes,
                           out_bf16, lse_f32=None, out_f32_debug=None, *, softmax_scale_dev=None,
                           output_scale: float = 1.0, sinks=None, query_lens=None,
                           kv_bounds=None, cta_items=None, phases: int = PHASE_ALL,
                           stream=None) -> None:
    """BF16 sparse decode over the selected pages block_idx [batch, topk]
    (plan with the compact lengths 32 * topk)."""
    opts = DecodeOptions(None, None, _ptr(softmax_scale_dev), float(output_scale), _ptr(sinks),
                         _ptr(query_lens), _ptr(kv_bounds), _ptr(cta_items),
                         0 if cta_items is None else int(cta_items.numel()), 0, int(phases))
    lib = load_library()
    _check(lib.mla_decode_bf16_sparse(_ptr(q_bf16), _ptr(kv_pages_bf16), int(num_pages),
                                      _ptr(page_table), int(max_pages_per_req), _ptr(kv_lens),
                                      _ptr(block_idx), int(topk), _ptr(splits), _ptr(chunks),
                                      int(max_splits), int(kv_split), int(batch), int(q_len),
                                      int(num_heads), 1 if causal else 0, float(softmax_scale),
                                      _ptr(workspace), int(workspace_bytes), _ptr(out_bf16),
                                      _ptr(lse_f32), _ptr(out_f32_debug), ctypes.byref(opts),
                                      _stream_handle(stream)))


def mla_decode_sparse(q_fp8, kv_pages_fp8, num_pages, page_table, max_pages_per_req, kv_lens,
                      block_idx, topk, splits, chunks, max_splits, kv_split, batch, q_len,
                      num_heads, causal, q_scale, kv_scale, softmax_scale, workspace,
                      workspace_bytes, out_bf16, lse_f32=None, out_f32_debug=None, *,
                      q_scale_dev=None, kv_scale_dev=None, softmax_scale_dev=None,
                      output_scale: float = 1.0, sinks=None, query_lens=None, kv_bounds=None,
                      cta_items=None, persistent_ctas: int = 0, phases: int = PHASE_ALL,
                      stream=None) -> None:
    """Sparse decode over the selected pages block_idx [batch, topk] (plan with
    the compact lengths 32 * topk)."""
    opts = DecodeOptions(_ptr(q_scale_dev), _ptr(kv_scale_dev), _ptr(softmax_scale_dev),
                         float(output_scale), _ptr(sinks), _ptr(query_lens), _ptr(kv_bounds),
                         _ptr(cta_items), 0 if cta_items is None else int(cta_items.numel()),
                         int(persistent_ctas), int(phases))
    lib = load_library()
    _check(lib.mla_decode_sparse(_ptr(q_fp8), _ptr(kv_pages_fp8), int(num_pages),
                                 _ptr(page_table), int(max_pages_per_req), _ptr(kv_lens),
                                 _ptr(block_idx), int(topk), _ptr(splits), _ptr(chunks),
                                 int(max_splits), int(kv_split), int(batch), int(q_len),
                                 int(num_heads), 1 if causal else 0, float(q_scale),
                                 float(kv_scale), float(softmax_scale), _ptr(workspace),
                                 int(workspace_bytes), _ptr(out_bf16), _ptr(lse_f32),
                                 _ptr(out_f32_debug), ctypes.byref(opts),
                                 _stream_handle(stream)))


def mla_decode_splitkv(*args, **kw) -> None:
    """Split-KV phase of mla_decode (same arguments)."""
    _decode_call("mla_decode_splitkv", *args, **kw)


def mla_decode_merge(*args, **kw) -> None:
    """Merge phase of mla_decode (same arguments)."""
    _decode_call("mla_decode_merge", *args, **kw)


def mla_decode_workspace_init(workspace, workspace_bytes: int, stream=None) -> None:
    _check(load_library().mla_decode_workspace_init(_ptr(workspace), int(workspace_bytes),
                                                    _stream_handle(stream)))


def mla_merge(partial_o, partial_ml, rows: int, num_ctas_kv: int, kv_split: int, out_bf16,
              lse_f32=None, out_f32_debug=None, stream=None) -> None:
    lib = load_library()
    _check(lib.mla_merge(_ptr(partial_o), _ptr(partial_ml), int(rows), int(num_ctas_kv),
                         int(kv_split), _ptr(out_bf16), _ptr(lse_f32), _ptr(out_f32_debug),
                         _stream_handle(stream)))


def mla_decode_static_ws(q_fp8, kv_pages_fp8, num_pages: int, page_table,
                         max_pages_per_req: int, kv_lens, splits, chunks, max_splits: int,
                         kv_split: int, batch: int, q_len: int, num_heads: int, causal: bool,
                         q_scale: float, kv_scale: float, softmax_scale: float, out_bf16,
                         lse_f32=None, out_f32_debug=None, stream=None) -> None:
    """mla_decode for callers that cannot allocate device memory.

    The scratch lives in a fixed array inside the library
    (MLA_STATIC_WS_BYTES = 16 MiB per GPU), so no workspace is passed.  The
    first call on a device resolves that array's address and should come
    before any stream capture; calls that overlap on the GPU race on the array.
    Device-detected conditions are read with mla_decode_static_ws_status().
    """
    lib = load_library()
    _check(lib.mla_decode_static_ws(
        _ptr(q_fp8), _ptr(kv_pages_fp8), int(num_pages), _ptr(page_table), int(max_pages_per_req),
        _ptr(kv_lens), _ptr(splits), _ptr(chunks), int(max_splits), int(kv_split), int(batch),
        int(q_len), int(num_heads), 1 if causal else 0, float(q_scale), float(kv_scale),
        float(softmax_scale), _ptr(out_bf16), _ptr(lse_f32), _ptr(out_f32_debug),
        _stream_handle(stream)))


STATIC_WS_BYTES = 16 * 1024 * 1024


def mla_decode_static_ws_status(stream=None) -> int:
    """Read and clear the status word of mla_decode_static_ws's fixed scratch
    array (after `stream` drains); raises MlaError on a non-OK status."""
    st = load_library().mla_decode_static_ws_status(_stream_handle(stream))
    _check(st)
    return st


def mla_kv_append(rows_bf16, n_tokens: int, req_idx, positions, page_table,
                  max_pages_per_req: int, batch: int, kv_pages_fp8, num_pages: int,
                  kv_scale: float, status=None, stream=None) -> None:
    """Quantize BF16 latent rows to E4M3 and scatter them into the paged cache."""
    _check(load_library().mla_kv_append(
        _ptr(rows_bf16), int(n_tokens), _ptr(req_idx), _ptr(positions), _ptr(page_table),
        int(max_pages_per_req), int(batch), _ptr(kv_pages_fp8), int(num_pages), float(kv_scale),
        _ptr(status), _stream_handle(stream)))


def mla_debug_set_wait_limit(cycles: int) -> None:
    """Test hook: limit of the kernel's pipeline waits (0 = default)."""
    load_library().mla_debug_set_wait_limit(int(cycles))


def mla_debug_set_expire(role: int, tile: int = 0) -> None:
    """Test hook: the pipeline wait `role` at tile `tile` of later launches
    reads as expired (role < 0 = off); see mla_decode.h."""
    load_library().mla_debug_set_expire(int(role), int(tile))


def mla_decode_status(workspace, stream=None) -> int:
    """Read and clear the device status word; raises MlaError on a non-OK status."""
    lib = load_library()
    st = lib.mla_decode_status(_ptr(workspace), _stream_handle(stream))
    _check(st)
    return st


# ---------------------------------------------------------------------------
# Convenience wrappers over torch tensors (allocation on the caller's side).
# ---------------------------------------------------------------------------

def decode(q_fp8, kv_pages_fp8, page_table, kv_lens, *, num_heads: int, q_len: int,
           causal: bool, softmax_scale: float, q_scale: float = 1.0, kv_scale: float = 1.0,
           plan: Optional[Plan] = None, sm_count: Optional[int] = None, target_ctas: int = 0,
           kv_split: Optional[int] = None, want_f32: bool = False, stream=None,
           check_status: bool = True, sinks=None, output_scale: float = 1.0,
           device_scales: bool = False, query_lens=None, kv_bounds=None, block_idx=None,
           use_items: Optional[bool] = None, persistent_ctas: int = 0):
    """Plan, allocate outputs and a workspace with torch, and run mla_decode.

    q_fp8 uint8 [B, q, H, 576] and kv_pages_fp8 uint8 [P, 32, 576] (E4M3 codes)
    and page_table int32 [B, max_pages] are CUDA tensors; kv_lens is a host
    sequence.  With torch.bfloat16 q and kv this runs mla_decode_bf16 (no
    q/kv scales there).  query_lens [B], kv_bounds [B, 2] and block_idx
    [B, topk] (selected pages: mla_decode_sparse / mla_decode_bf16_sparse,
    planned on the compact lengths) restrict the visible keys.  use_items
    (default: when the plan has empty split slots) launches the split kernel
    over the plan's CTA item list; persistent_ctas > 0 (FP8) runs that list
    with that many persistent CTAs.  Returns (out_bf16, lse, out_f32 or None).
    """
    import torch
    dev = q_fp8.device
    lens = np.asarray(kv_lens.cpu() if hasattr(kv_lens, "cpu") else kv_lens, dtype=np.int32)
    batch = int(lens.shape[0])
    topk = 0 if block_idx is None else int(block_idx.shape[1])
    if plan is None:
        if sm_count is None:
            sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
        plan_lens = lens if block_idx is None else np.full_like(lens, PAGE_SIZE * topk)
        plan = mla_decode_plan(plan_lens, num_heads, q_len, sm_count=sm_count,
                               target_ctas=target_ctas)
    ks = plan.kv_split if kv_split is None else int(kv_split)
    lens_d = torch.from_numpy(lens).to(dev)
    splits_d = torch.from_numpy(plan.splits).to(dev)
    chunks_d = torch.from_numpy(plan.chunks).to(dev)
    ws_bytes = mla_decode_workspace_size(batch, q_len, num_heads, plan.max_splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    mla_decode_workspace_init(ws, ws_bytes, stream)
    out = torch.empty((batch, q_len, num_heads, LATENT_DIM), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((batch, q_len, num_heads), dtype=torch.float32, device=dev)
    out_f32 = (torch.empty((batch, q_len, num_heads, LATENT_DIM), dtype=torch.float32, device=dev)
               if want_f32 else None)
    common = (q_fp8, kv_pages_fp8, kv_pages_fp8.shape[0], page_table, page_table.shape[1],
              lens_d, splits_d, chunks_d, plan.max_splits, ks, batch, q_len, num_heads, causal)
    restricted = query_lens is not None or kv_bounds is not None or block_idx is not None
    if use_items is None:
        use_items = bool(np.any(plan.splits < plan.max_splits)) or persistent_ctas > 0
    is_bf16 = q_fp8.dtype == torch.bfloat16
    items_d = None
    if use_items:
        items_d = torch.from_numpy(
            mla_decode_plan_items(plan.splits, num_heads, q_len, bf16=is_bf16)).to(dev)

    def _dev_i32(x):
        return None if x is None else torch.as_tensor(x, dtype=torch.int32).to(dev).contiguous()
    if is_bf16:
        if kv_pages_fp8.dtype != torch.bfloat16 or q_scale != 1.0 or kv_scale != 1.0:
            raise ValueError("BF16 decode takes BF16 q and kv and no q/kv scales")
        if (sinks is None and output_scale == 1.0 and not device_scales and not restricted
                and items_d is None):
            mla_decode_bf16(*common, softmax_scale, ws, ws_bytes, out, lse, out_f32, stream)
        else:
            sm_d = (torch.tensor([softmax_scale], dtype=torch.float32, device=dev)
                    if device_scales else None)
            sk = None if sinks is None else torch.as_tensor(sinks, dtype=torch.float32).to(dev)
            extra = dict(softmax_scale_dev=sm_d, output_scale=output_scale, sinks=sk,
                         query_lens=_dev_i32(query_lens), kv_bounds=_dev_i32(kv_bounds),
                         cta_items=items_d, stream=stream)
            # With a device scale the host value is a placeholder the kernel must ignore.
            sm_h = 99.0 if device_scales else softmax_scale
            bi_d = _dev_i32(block_idx)
            if bi_d is None:
                mla_decode_bf16_ex(*common, sm_h, ws, ws_bytes, out, lse, out_f32, **extra)
            else:
                mla_decode_bf16_sparse(*common[:6], bi_d, topk, *common[6:], sm_h, ws, ws_bytes,
                                       out, lse, out_f32, **extra)
    elif (sinks is None and output_scale == 1.0 and not device_scales and not restricted
          and items_d is None and persistent_ctas == 0):
        mla_decode(*common, q_scale, kv_scale, softmax_scale, ws, ws_bytes, out, lse, out_f32,
                   stream)
    else:
        dev_s = None
        if device_scales:
            dev_s = torch.tensor([q_scale, kv_scale, softmax_scale], dtype=torch.float32,
                                 device=dev)
        sk = None if sinks is None else torch.as_tensor(sinks, dtype=torch.float32).to(dev)
        # With device scales the host values are placeholders the kernel must
        # ignore (deliberately wrong, so a kernel that used them would fail).
        host = (99.0,) * 3 if device_scales else (q_scale, kv_scale, softmax_scale)
        ql_d, kb_d, bi_d = _dev_i32(query_lens), _dev_i32(kv_bounds), _dev_i32(block_idx)
        extra = dict(q_scale_dev=None if dev_s is None else dev_s[0:1],
                     kv_scale_dev=None if dev_s is None else dev_s[1:2],
                     softmax_scale_dev=None if dev_s is None else dev_s[2:3],
                     output_scale=output_scale, sinks=sk, query_lens=ql_d, kv_bounds=kb_d,
                     cta_items=items_d, persistent_ctas=persistent_ctas, stream=stream)
        if bi_d is None:
            mla_decode_ex(*common, *host, ws, ws_bytes, out, lse, out_f32, **extra)
        else:
            mla_decode_sparse(*common[:6], bi_d, topk, *common[6:], *host, ws, ws_bytes, out,
                              lse, out_f32, **extra)
    if check_status:
        mla_decode_status(ws, stream)
    return out, lse, out_f32


def merge(partial_o, partial_ml, kv_split: int, want_f32: bool = True, stream=None):
    """Run mla_merge on CUDA tensors partial_o [rows, S, 512], partial_ml [rows, S, 2]."""
    import torch
    rows, s = int(partial_o.shape[0]), int(partial_o.shape[1])
    out = torch.empty((rows, LATENT_DIM), dtype=torch.bfloat16, device=partial_o.device)
    lse = torch.empty((rows,), dtype=torch.float32, device=partial_o.device)
    out_f32 = (torch.empty((rows, LATENT_DIM), dtype=torch.float32, device=partial_o.device)
               if want_f32 else None)
    mla_merge(partial_o, partial_ml, rows, s, kv_split, out, lse, out_f32, stream)
    return out, lse, out_f32
