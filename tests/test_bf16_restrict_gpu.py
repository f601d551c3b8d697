"""GPU parity of the BF16-KV decode with restricted key sets and CTA item
lists against the fp64 oracle, through the C ABI: key windows (kv_bounds of
issue #20510 "Repro 1"), the sparse decode over selected pages
(mla_decode_bf16_sparse; PR #17441 "m3 decode perf") and the item list of a
skewed batch (the follow-up comment of issue #20510: skip the empty split
slots), on both BF16 kernels (16-row groups with Q in TMEM, and 32/48-row
groups)."""
import numpy as np
import pytest
import torch

import oracle
import split_kv_mla_paged_gb300 as mla
from split_kv_mla_paged_gb300 import build as mla_build
from synth import PAGE_SIZE, SOFTMAX_SCALE, decode_inputs, kv_windows, page_selection
from mla_testutil import PLAN_ABS, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mla_build.build()
    mla.load_library()
    yield
    torch.cuda.synchronize()


def _run(inp, causal, plan=None, target_ctas=0, **kw):
    dev = torch.device("cuda")
    out, lse, o32 = mla.decode(inp.q.to(dev), inp.kv.to(dev), inp.page_table.to(dev),
                               inp.kv_lens, num_heads=inp.num_heads, q_len=inp.q_len,
                               causal=causal, softmax_scale=SOFTMAX_SCALE, plan=plan,
                               target_ctas=target_ctas, want_f32=True, **kw)
    torch.cuda.synchronize()
    return out, lse, o32


def _check(inp, causal, ref_kw, run_kw=None, **plan_kw):
    run_kw = dict(ref_kw if run_kw is None else run_kw)
    out, lse, o32 = _run(inp, causal, **plan_kw, **run_kw)
    ref_o, ref_l = oracle.decode_rows(inp.q, inp.kv.cpu(), inp.page_table.cpu(), inp.kv_lens,
                                      q_len=inp.q_len, num_heads=inp.num_heads, causal=causal,
                                      softmax_scale=SOFTMAX_SCALE, **ref_kw)
    lse_np = lse.cpu().numpy().reshape(-1)
    fin = np.isfinite(ref_l)
    # Rows that see no key: O = 0 and LSE = -inf, exactly.
    assert np.array_equal(np.isfinite(lse_np), fin)
    assert torch.all(out.reshape(-1, 512)[torch.from_numpy(~fin).cuda()] == 0)
    assert_parity(out.reshape(-1, 512)[torch.from_numpy(fin).cuda()],
                  lse.reshape(-1)[torch.from_numpy(fin).cuda()], ref_o[fin], ref_l[fin])
    assert torch.equal(o32.to(torch.bfloat16), out)
    return out, lse, o32


# 12 rows -> the 16-row kernel; 20 rows -> 32; 96 rows -> two 48-row groups.
@pytest.mark.parametrize("B,H,q_len,lens,causal", [
    (4, 12, 1, [1000, 5000, 777, 130], False),
    (4, 12, 8, [3000, 1029, 4100, 900], True),
    (3, 20, 1, [2500, 300, 1300], False),
])
def test_bf16_kv_bounds_parity(B, H, q_len, lens, causal):
    inp = decode_inputs(B, H, q_len, lens, seed=520 + B, extra_pages=2, dtype="bf16")
    win = kv_windows(lens, seed=B + H)
    base = None
    for target in (0, 1, 9, 60):
        plan = mla.mla_decode_plan(lens, H, q_len, target_ctas=target) if target else None
        _, _, o32 = _check(inp, causal, dict(kv_bounds=win), plan=plan)
        if base is None:
            base = o32
        else:
            assert (o32 - base).abs().max().item() <= PLAN_ABS


def test_bf16_kv_bounds_empty_window_ragged_q_and_sinks():
    inp = decode_inputs(3, 12, 4, [2000, 640, 1500], seed=530, dtype="bf16")
    win = np.array([[500, 500], [0, 640], [1400, 1450]], np.int32)  # empty, whole, inner
    ql = np.array([4, 2, 3], np.int32)
    for target in (0, 8):
        plan = mla.mla_decode_plan([2000, 640, 1500], 12, 4, target_ctas=target) if target else None
        _check(inp, True, dict(kv_bounds=win, query_lens=ql), plan=plan)
    sinks = np.linspace(-1.0, 2.0, 12)
    out, lse, _ = _run(inp, True, kv_bounds=win, query_lens=ql, sinks=sinks)
    ref_o, ref_l = oracle.decode_rows(inp.q, inp.kv.cpu(), inp.page_table.cpu(), inp.kv_lens,
                                      q_len=4, num_heads=12, causal=True,
                                      softmax_scale=SOFTMAX_SCALE, kv_bounds=win, query_lens=ql,
                                      sinks=sinks)
    assert_parity(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("B,H,q_len,lens,topk,causal,keep_last", [
    (2, 12, 1, [5000, 3000], 20, False, True),
    (3, 12, 1, [4000, 100, 2200], 16, False, False),   # short request: -1 slots
    (2, 12, 8, [6000, 1500], 24, True, True),           # 96 rows: two 48-row groups
    (1, 16, 2, [9000], 40, True, True),                 # 32 rows
    (2, 1, 1, [700, 33], 8, False, True),               # 33 tokens: last page has 1
])
def test_bf16_sparse_parity(B, H, q_len, lens, topk, causal, keep_last):
    inp = decode_inputs(B, H, q_len, lens, seed=540 + topk, extra_pages=2, dtype="bf16")
    sel = page_selection(lens, topk, seed=topk + B, keep_last=keep_last)
    base = None
    for target in (0, 1, 5, 30):
        plan = None
        if target:
            plan = mla.mla_decode_plan([PAGE_SIZE * topk] * B, H, q_len, target_ctas=target)
        _, _, o32 = _check(inp, causal, dict(block_idx=sel), plan=plan)
        if base is None:
            base = o32
        else:
            assert (o32 - base).abs().max().item() <= PLAN_ABS


def test_bf16_sparse_with_window_and_ragged_q():
    lens = [6000, 2500]
    inp = decode_inputs(2, 12, 8, lens, seed=550, dtype="bf16")
    sel = page_selection(lens, 30, seed=551)
    win = np.array([[1000, 6000], [0, 2000]], np.int32)
    ql = np.array([5, 8], np.int32)
    _check(inp, True, dict(block_idx=sel, kv_bounds=win, query_lens=ql))


def test_bf16_sparse_all_pages_equals_dense():
    lens = [3000, 1111]
    inp = decode_inputs(2, 12, 1, lens, seed=552, dtype="bf16")
    n = max((L + 31) // 32 for L in lens)
    sel = np.full((2, n), -1, np.int32)
    for b, L in enumerate(lens):
        k = (L + 31) // 32
        sel[b, :k] = np.arange(k)
    out_s, lse_s, o32_s = _run(inp, False, block_idx=sel)
    out_d, lse_d, o32_d = _run(inp, False)
    ref_o, ref_l = oracle.decode_rows(inp.q, inp.kv.cpu(), inp.page_table.cpu(), inp.kv_lens,
                                      q_len=1, num_heads=12, causal=False,
                                      softmax_scale=SOFTMAX_SCALE)
    assert_parity(out_s, lse_s, ref_o, ref_l)
    assert_parity(out_d, lse_d, ref_o, ref_l)


def test_bf16_sparse_unordered_selection_is_reported():
    inp = decode_inputs(1, 12, 1, [3000], seed=553, dtype="bf16")
    sel = np.array([[3, 9, 7, 20]], np.int32)
    with pytest.raises(mla.MlaError) as e:
        _run(inp, False, block_idx=sel)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG


@pytest.mark.parametrize("H,q_len", [(12, 1), (12, 8), (10, 4)])
def test_bf16_item_list_matches_the_grid_launch(H, q_len):
    # A skewed batch: the item list launches only the CTAs with work; the
    # results are the same numbers as the full grid's.
    lens = [9000, 300, 129, 2000, 4100]
    inp = decode_inputs(5, H, q_len, lens, seed=560 + H, extra_pages=1, dtype="bf16")
    causal = q_len > 1
    for target in (0, 40):
        plan = (mla.mla_decode_plan(lens, H, q_len, target_ctas=target) if target
                else mla.mla_decode_plan(lens, H, q_len, sm_count=152))
        assert np.any(plan.splits < plan.max_splits)
        out_i, lse_i, o32_i = _run(inp, causal, plan=plan, use_items=True)
        out_g, lse_g, o32_g = _run(inp, causal, plan=plan, use_items=False)
        assert torch.equal(o32_i, o32_g) and torch.equal(lse_i, lse_g)
        ref_o, ref_l = oracle.decode_rows(inp.q, inp.kv.cpu(), inp.page_table.cpu(), inp.kv_lens,
                                          q_len=q_len, num_heads=H, causal=causal,
                                          softmax_scale=SOFTMAX_SCALE)
        assert_parity(out_i, lse_i, ref_o, ref_l)


def test_bf16_sparse_with_item_list_and_window():
    lens = [6000, 200, 3000]
    inp = decode_inputs(3, 12, 1, lens, seed=570, dtype="bf16")
    sel = page_selection(lens, 24, seed=571, keep_last=False)
    win = np.array([[0, 6000], [10, 150], [500, 2900]], np.int32)
    plan = mla.mla_decode_plan([PAGE_SIZE * 24] * 3, 12, 1, target_ctas=30)
    _check(inp, False, dict(block_idx=sel, kv_bounds=win),
           run_kw=dict(block_idx=sel, kv_bounds=win, use_items=True), plan=plan)
