"""The no-allocation decode entry point (mla_decode_static_ws).

Callers that cannot allocate device memory (a host runtime that owns every
allocation, or a latency-critical path that cannot take cudaMalloc's implicit
synchronisation) use this entry point: its scratch is a fixed array inside the
library instead of a caller-provided workspace.  These tests check, through the
C ABI, that it returns what mla_decode returns on two calls in a row (the
second call sees the first call's leftovers in the shared array), that a call
needing more scratch than the array holds is refused with a clear error, and
that a condition the device detects (a bad page id) is reported by
mla_decode_static_ws_status, which reads and clears the array's status word.

This file is collected last on purpose; it passes alone in a fresh process
and after the other tests.
"""
import numpy as np
import pytest
import torch

import split_kv_mla_paged_gb300 as mla
from split_kv_mla_paged_gb300 import build as mla_build
from synth import SOFTMAX_SCALE, decode_inputs
from mla_testutil import PLAN_ABS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mla_build.build()
    mla.load_library()


def _device_args(inp, plan):
    dev = torch.device("cuda")
    return dict(q=inp.q.to(dev), kv=inp.kv.to(dev), pt=inp.page_table.to(dev),
                lens=inp.kv_lens.to(dev), splits=torch.from_numpy(plan.splits).to(dev),
                chunks=torch.from_numpy(plan.chunks).to(dev))


def _outputs(inp):
    dev = torch.device("cuda")
    shape = (inp.batch, inp.q_len, inp.num_heads, 512)
    return (torch.full(shape, float("nan"), dtype=torch.bfloat16, device=dev),
            torch.full(shape[:3], float("nan"), dtype=torch.float32, device=dev),
            torch.full(shape, float("nan"), dtype=torch.float32, device=dev))


def _run_both(inp, causal, target_ctas=0):
    plan = mla.mla_decode_plan(inp.kv_lens.tolist(), inp.num_heads, inp.q_len, sm_count=152,
                               target_ctas=target_ctas)
    assert plan.workspace_bytes <= mla.STATIC_WS_BYTES
    a = _device_args(inp, plan)
    common = (a["q"], a["kv"], inp.num_pages, a["pt"], inp.max_pages, a["lens"], a["splits"],
              a["chunks"], plan.max_splits, plan.kv_split, inp.batch, inp.q_len, inp.num_heads,
              causal, 1.0, 1.0, SOFTMAX_SCALE)
    ref = _outputs(inp)
    ws_bytes = mla.mla_decode_workspace_size(inp.batch, inp.q_len, inp.num_heads,
                                             plan.max_splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    mla.mla_decode_workspace_init(ws, ws_bytes)
    mla.mla_decode(*common, ws, ws_bytes, *ref)
    got = _outputs(inp)
    mla.mla_decode_static_ws(*common, *got)
    torch.cuda.synchronize()
    mla.mla_decode_status(ws)
    assert mla.mla_decode_static_ws_status() == mla.MLA_OK
    return ref, got, plan


def _assert_same(ref, got):
    out_r, lse_r, f_r = ref
    out_g, lse_g, f_g = got
    assert torch.isfinite(f_g).all() and torch.isfinite(lse_g).all()
    assert (f_g - f_r).abs().max().item() <= PLAN_ABS
    assert (lse_g - lse_r).abs().max().item() <= PLAN_ABS
    assert (out_g.float() - out_r.float()).abs().max().item() <= 2.0 ** -8 * max(
        1.0, out_r.float().abs().max().item())


def test_static_ws_matches_mla_decode_two_calls_in_a_row():
    # First call: many splits per request, so the partial area is well used.
    inp1 = decode_inputs(2, 12, 8, [20000, 7777], seed=31, extra_pages=1)
    ref1, got1, plan1 = _run_both(inp1, causal=True, target_ctas=24)
    assert plan1.max_splits > 1
    _assert_same(ref1, got1)
    # Second call, different inputs and shapes: the array still holds the
    # first call's partials and must not leak into the result.
    inp2 = decode_inputs(3, 12, 1, [5000, 300, 12345], seed=32)
    ref2, got2, _ = _run_both(inp2, causal=False)
    _assert_same(ref2, got2)


def test_static_ws_refuses_oversized_scratch():
    rows, splits = 16 * 8 * 12, 128
    need = mla.mla_decode_workspace_size(16, 8, 12, splits)
    assert need > mla.STATIC_WS_BYTES
    dev = torch.device("cuda")
    dummy = torch.zeros(16, dtype=torch.uint8, device=dev)
    lens = torch.full((16,), 1 << 20, dtype=torch.int32, device=dev)
    out = torch.empty((rows, 512), dtype=torch.bfloat16, device=dev)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_static_ws(dummy, dummy, 1, lens, 1, lens, lens, lens, splits, 16, 16, 8, 12,
                                 True, 1.0, 1.0, SOFTMAX_SCALE, out)
    assert e.value.status == mla.MLA_ERR_WORKSPACE_TOO_SMALL
    assert "MLA_STATIC_WS_BYTES" in mla.mla_last_error()


def test_static_ws_status_reports_a_bad_page_id():
    # The split CTAs that meet a page id outside the pool stop early, so that
    # call's output is not valid; the status word says so until it is read.
    inp = decode_inputs(1, 12, 8, [6000], seed=33)
    plan = mla.mla_decode_plan([6000], 12, 8, target_ctas=6)
    assert plan.max_splits > 1
    a = _device_args(inp, plan)
    bad_pt = a["pt"].clone()
    bad_pt[0, 40] = inp.num_pages + 9
    out = _outputs(inp)
    args = (a["q"], a["kv"], inp.num_pages, bad_pt, inp.max_pages, a["lens"], a["splits"],
            a["chunks"], plan.max_splits, plan.kv_split, 1, 8, 12, True, 1.0, 1.0,
            SOFTMAX_SCALE)
    mla.mla_decode_static_ws(*args, *out)
    # A second call with the same bad id: the word stays set (not reset per call).
    mla.mla_decode_static_ws(*args, *out)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_static_ws_status()
    assert e.value.status == mla.MLA_ERR_INVALID_ARG
    # Read and cleared: the next good call reports OK and matches mla_decode.
    assert mla.mla_decode_static_ws_status() == mla.MLA_OK
    ref, got, _ = _run_both(inp, causal=True, target_ctas=6)
    _assert_same(ref, got)
