"""The C-ABI library loads and exports what include/mla_decode.h declares.

No compute call here: host-side argument checks return before any CUDA call.
"""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import split_kv_mla_paged_gb300 as mla
from split_kv_mla_paged_gb300 import build as mla_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "mla_decode.h")


@pytest.fixture(scope="module")
def lib():
    mla_build.build()
    return mla.load_library()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", text)))


def test_header_declares_the_exported_set():
    assert _declared() == sorted(mla.EXPORTED_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(mla.library_path())
    for name in _declared():
        assert hasattr(raw, name), name


def test_workspace_size_layout(lib):
    rows, s = 12 * 8 * 3, 7
    ml = rows * s * 8
    ml_aligned = (ml + 255) // 256 * 256
    assert mla.mla_decode_workspace_size(3, 8, 12, s) == 256 + ml_aligned + rows * s * 2048
    assert mla.mla_decode_workspace_size(0, 8, 12, s) == 0


def test_decode_rejects_null_pointers_without_gpu(lib):
    st = lib.mla_decode(None, None, 1, None, 1, None, None, None, 1, 1, 1, 1, 12, 0, 1.0, 1.0,
                        0.1, None, 0, None, None, None, None)
    assert st == mla.MLA_ERR_INVALID_ARG
    assert "null" in mla.mla_last_error()


def test_decode_rejects_small_workspace_without_gpu(lib):
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced on this path
    st = lib.mla_decode(fake, fake, 4, fake, 4, fake, fake, fake, 2, 2, 1, 1, 12, 0, 1.0, 1.0,
                        0.1, fake, 16, fake, None, None, None)
    assert st == mla.MLA_ERR_WORKSPACE_TOO_SMALL


def test_decode_rejects_bad_kv_split_and_rows(lib):
    fake = ctypes.c_void_p(1 << 20)
    st = lib.mla_decode(fake, fake, 4, fake, 4, fake, fake, fake, 2, 3, 1, 1, 12, 0, 1.0, 1.0,
                        0.1, fake, 1 << 30, fake, None, None, None)
    assert st == mla.MLA_ERR_INVALID_ARG
    st = lib.mla_decode(fake, fake, 4, fake, 4, fake, fake, fake, 2, 2, 1, 8, 256, 0, 1.0, 1.0,
                        0.1, fake, 1 << 30, fake, None, None, None)
    assert st == mla.MLA_ERR_UNSUPPORTED


def test_decode_rejects_misaligned_inputs(lib):
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 8)
    st = lib.mla_decode(odd, fake, 4, fake, 4, fake, fake, fake, 2, 2, 1, 1, 12, 0, 1.0, 1.0,
                        0.1, fake, 1 << 30, fake, None, None, None)
    assert st == mla.MLA_ERR_INVALID_ARG


def test_merge_rejects_bad_arguments(lib):
    assert lib.mla_merge(None, None, 4, 4, 1, None, None, None, None) == mla.MLA_ERR_INVALID_ARG
    fake = ctypes.c_void_p(1 << 20)
    assert lib.mla_merge(fake, fake, 4, 4, 5, fake, None, None, None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_merge(fake, fake, 0, 4, 4, fake, None, None, None) == mla.MLA_ERR_INVALID_ARG


def test_status_rejects_null(lib):
    assert lib.mla_decode_status(None, None) == mla.MLA_ERR_INVALID_ARG


def test_bf16_decode_host_checks(lib):
    fake = ctypes.c_void_p(1 << 20)
    st = lib.mla_decode_bf16(None, fake, 4, fake, 4, fake, fake, fake, 2, 2, 1, 1, 12, 0, 0.1,
                             fake, 1 << 30, fake, None, None, None)
    assert st == mla.MLA_ERR_INVALID_ARG and "null" in mla.mla_last_error()
    st = lib.mla_decode_bf16(fake, fake, 4, fake, 4, fake, fake, fake, 2, 2, 1, 8, 256, 0, 0.1,
                             fake, 1 << 30, fake, None, None, None)
    assert st == mla.MLA_ERR_UNSUPPORTED
    st = lib.mla_decode_bf16(fake, fake, 4, fake, 4, fake, fake, fake, 2, 2, 1, 1, 12, 0,
                             float("nan"), fake, 1 << 30, fake, None, None, None)
    assert st == mla.MLA_ERR_INVALID_ARG
    st = lib.mla_decode_bf16(fake, fake, 4, fake, 4, fake, fake, fake, 2, 2, 1, 1, 12, 0, 0.1,
                             fake, 16, fake, None, None, None)
    assert st == mla.MLA_ERR_WORKSPACE_TOO_SMALL


def test_sparse_decode_host_checks(lib):
    fake = ctypes.c_void_p(1 << 20)
    args = [fake, fake, 4, fake, 4, fake]
    tail = [fake, fake, 2, 2, 1, 1, 12, 0, 1.0, 1.0, 0.1, fake, 1 << 30, fake, None, None, None,
            None]
    assert lib.mla_decode_sparse(*args, None, 8, *tail) == mla.MLA_ERR_INVALID_ARG
    assert "block_idx" in mla.mla_last_error()
    assert lib.mla_decode_sparse(*args, fake, 0, *tail) == mla.MLA_ERR_INVALID_ARG
    assert "topk" in mla.mla_last_error()
    small = list(tail)
    small[12] = 16  # workspace bytes
    assert lib.mla_decode_sparse(*args, fake, 8, *small) == mla.MLA_ERR_WORKSPACE_TOO_SMALL


def test_decode_ex_rejects_nonfinite_output_scale(lib):
    fake = ctypes.c_void_p(1 << 20)
    opts = mla.DecodeOptions(None, None, None, float("inf"), None, None, None)
    st = lib.mla_decode_ex(fake, fake, 4, fake, 4, fake, fake, fake, 2, 2, 1, 1, 12, 0, 1.0, 1.0,
                           0.1, fake, 1 << 30, fake, None, None, ctypes.byref(opts), None)
    assert st == mla.MLA_ERR_INVALID_ARG and "output_scale" in mla.mla_last_error()


def test_kv_append_host_checks(lib):
    fake = ctypes.c_void_p(1 << 20)
    # Zero tokens is a no-op that touches nothing.
    assert lib.mla_kv_append(None, 0, None, None, None, 1, 1, None, 1, 1.0, None, None) == mla.MLA_OK
    assert lib.mla_kv_append(None, 4, fake, fake, fake, 1, 1, fake, 1, 1.0, None,
                             None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_kv_append(fake, 4, fake, fake, fake, 1, 1, fake, 1, 0.0, None,
                             None) == mla.MLA_ERR_INVALID_ARG


def test_bf16_ex_rejects_fp8_only_options(lib):
    fake = ctypes.c_void_p(1 << 20)
    opts = mla.DecodeOptions(fake, None, None, 1.0, None, None, None, None, 0)
    st = lib.mla_decode_bf16_ex(fake, fake, 4, fake, 4, fake, fake, fake, 2, 2, 1, 1, 12, 0, 0.1,
                                fake, 1 << 30, fake, None, None, ctypes.byref(opts), None)
    assert st == mla.MLA_ERR_UNSUPPORTED and "FP8-only" in mla.mla_last_error()


def test_bf16_item_list_size_is_checked(lib):
    fake = ctypes.c_void_p(1 << 20)
    opts = mla.DecodeOptions(None, None, None, 1.0, None, None, None, fake, 0)
    st = lib.mla_decode_bf16_ex(fake, fake, 4, fake, 4, fake, fake, fake, 2, 2, 1, 1, 12, 0, 0.1,
                                fake, 1 << 30, fake, None, None, ctypes.byref(opts), None)
    assert st == mla.MLA_ERR_INVALID_ARG and "num_ctas" in mla.mla_last_error()


def test_bf16_sparse_host_checks(lib):
    fake = ctypes.c_void_p(1 << 20)
    args = [fake, fake, 4, fake, 4, fake]
    tail = [fake, fake, 2, 2, 1, 1, 12, 0, 0.1, fake, 1 << 30, fake, None, None, None, None]
    assert lib.mla_decode_bf16_sparse(*args, None, 8, *tail) == mla.MLA_ERR_INVALID_ARG
    assert "block_idx" in mla.mla_last_error()
    assert lib.mla_decode_bf16_sparse(*args, fake, 0, *tail) == mla.MLA_ERR_INVALID_ARG
    assert "topk" in mla.mla_last_error()
    small = list(tail)
    small[10] = 16  # workspace bytes
    assert lib.mla_decode_bf16_sparse(*args, fake, 8, *small) == mla.MLA_ERR_WORKSPACE_TOO_SMALL


def test_bf16_item_lists_use_the_bf16_row_groups(lib):
    splits = [3, 1, 2]
    # Up to 48 rows both kernels run one CTA per split.
    assert np.array_equal(mla.mla_decode_plan_items(splits, 12, 4),
                          mla.mla_decode_plan_items_bf16(splits, 12, 4))
    # 96 rows: one FP8 CTA per split, two BF16 CTAs (48 rows each).
    fp8 = mla.mla_decode_plan_items(splits, 12, 8)
    bf16 = mla.mla_decode_plan_items_bf16(splits, 12, 8)
    assert len(fp8) == sum(splits) and len(bf16) == 2 * sum(splits)
    groups = bf16 & ((1 << 5) - 1)
    assert sorted(set(groups.tolist())) == [0, 1]


def test_persistent_ctas_host_checks(lib):
    fake = ctypes.c_void_p(1 << 20)
    args = [fake, fake, 4, fake, 4, fake, fake, fake, 2, 2, 1, 1, 12, 0, 1.0, 1.0, 0.1, fake,
            1 << 30, fake, None, None]
    # Persistent CTAs need an item list; a negative count is refused.
    opts = mla.DecodeOptions(None, None, None, 1.0, None, None, None, None, 0, 4)
    assert lib.mla_decode_ex(*args, ctypes.byref(opts), None) == mla.MLA_ERR_INVALID_ARG
    assert "persistent" in mla.mla_last_error()
    opts = mla.DecodeOptions(None, None, None, 1.0, None, None, None, fake, 2, -1)
    assert lib.mla_decode_ex(*args, ctypes.byref(opts), None) == mla.MLA_ERR_INVALID_ARG
    # The BF16 entry points have no persistent mode.
    opts = mla.DecodeOptions(None, None, None, 1.0, None, None, None, fake, 2, 4)
    st = lib.mla_decode_bf16_ex(fake, fake, 4, fake, 4, fake, fake, fake, 2, 2, 1, 1, 12, 0, 0.1,
                                fake, 1 << 30, fake, None, None, ctypes.byref(opts), None)
    assert st == mla.MLA_ERR_UNSUPPORTED and "persistent" in mla.mla_last_error()


def test_phases_are_checked(lib):
    fake = ctypes.c_void_p(1 << 20)
    args = [fake, fake, 4, fake, 4, fake, fake, fake, 2, 2, 1, 1, 12, 0, 1.0, 1.0, 0.1, fake,
            1 << 30, fake, None, None]
    for bad in (-1, 3):
        opts = mla.DecodeOptions(None, None, None, 1.0, None, None, None, None, 0, 0, bad)
        assert lib.mla_decode_ex(*args, ctypes.byref(opts), None) == mla.MLA_ERR_INVALID_ARG
        assert "phases" in mla.mla_last_error()
        st = lib.mla_decode_sparse(*args[:6], fake, 8, *args[6:], ctypes.byref(opts), None)
        assert st == mla.MLA_ERR_INVALID_ARG and "phases" in mla.mla_last_error()
        st = lib.mla_decode_bf16_ex(fake, fake, 4, fake, 4, fake, fake, fake, 2, 2, 1, 1, 12, 0,
                                    0.1, fake, 1 << 30, fake, None, None, ctypes.byref(opts),
                                    None)
        assert st == mla.MLA_ERR_INVALID_ARG and "phases" in mla.mla_last_error()


def test_options_struct_matches_the_header(tmp_path):
    # The binding's ctypes mirror of mla_decode_options_t against the C
    # compiler's layout of the header's structure.
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stddef.h>\n#include <stdio.h>\n#include "mla_decode.h"\n'
        "int main(void) {\n"
        '  printf("%zu", sizeof(mla_decode_options_t));\n'
        + "".join(f'  printf(" %zu", offsetof(mla_decode_options_t, {name}));\n'
                  for name, _ in mla.DecodeOptions._fields_)
        + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)],
                   check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [ctypes.sizeof(mla.DecodeOptions)] + [getattr(mla.DecodeOptions, name).offset
                                                 for name, _ in mla.DecodeOptions._fields_]
    assert got == want
