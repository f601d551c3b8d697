"""Persistent CTAs (issue #20510, "Repro 1": the run() argument is_persistent):
a few CTAs loop over the CTA item list, carrying their barrier phases from one
item to the next.  Through the C ABI, against the one-CTA-per-item launch
(bit-identical fp32 output and LSE) and the fp64 oracle, on every FP8 kernel
configuration, with restricted key sets, skewed batches, and an expired wait.
"""
import numpy as np
import pytest
import torch

import oracle
import split_kv_mla_paged_gb300 as mla
from split_kv_mla_paged_gb300 import build as mla_build
from synth import PAGE_SIZE, SOFTMAX_SCALE, decode_inputs, kv_windows, page_selection
from mla_testutil import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mla_build.build()
    mla.load_library()
    yield
    mla.mla_debug_set_expire(-1)
    torch.cuda.synchronize()


def _run(inp, causal, plan, persistent_ctas=0, **kw):
    dev = torch.device("cuda")
    out, lse, o32 = mla.decode(inp.q.to(dev), inp.kv.to(dev), inp.page_table.to(dev),
                               inp.kv_lens, num_heads=inp.num_heads, q_len=inp.q_len,
                               causal=causal, softmax_scale=SOFTMAX_SCALE, plan=plan,
                               want_f32=True, use_items=True, persistent_ctas=persistent_ctas,
                               **kw)
    torch.cuda.synchronize()
    return out, lse, o32


def _oracle(inp, causal, **kw):
    return oracle.decode_rows(inp.q, inp.kv.cpu(), inp.page_table.cpu(), inp.kv_lens,
                              q_len=inp.q_len, num_heads=inp.num_heads, causal=causal,
                              softmax_scale=SOFTMAX_SCALE, **kw)


# 12 rows -> 16-row CTAs; 20 -> 32; 40 -> 48; 96 -> one 96-row CTA; 768 -> 8.
@pytest.mark.parametrize("B,H,q_len,lens,causal,target", [
    (4, 12, 1, [5000, 777, 3000, 130], False, 40),
    (3, 20, 1, [2500, 300, 4100], False, 30),
    (3, 10, 4, [3000, 700, 2000], True, 30),
    (2, 12, 8, [6000, 1500], True, 24),
    (1, 96, 8, [2000], True, 6),
])
@pytest.mark.parametrize("ctas", [1, 5, 13])
def test_persistent_matches_one_cta_per_item(B, H, q_len, lens, causal, target, ctas):
    inp = decode_inputs(B, H, q_len, lens, seed=800 + B * H + q_len, extra_pages=1)
    plan = mla.mla_decode_plan(lens, H, q_len, target_ctas=target)
    out_i, lse_i, o32_i = _run(inp, causal, plan)
    out_p, lse_p, o32_p = _run(inp, causal, plan, persistent_ctas=ctas)
    assert torch.equal(o32_p, o32_i) and torch.equal(lse_p, lse_i)
    ref_o, ref_l = _oracle(inp, causal)
    assert_parity(out_p, lse_p, ref_o, ref_l)


def test_persistent_skewed_batch_and_more_ctas_than_items():
    lens = [9000, 300, 129, 2000, 4100]
    inp = decode_inputs(5, 12, 8, lens, seed=820, extra_pages=1)
    plan = mla.mla_decode_plan(lens, 12, 8, sm_count=152)
    assert np.any(plan.splits < plan.max_splits)
    base = _run(inp, True, plan)
    for ctas in (3, 152, 10 ** 6):  # above the item count: one CTA per item
        got = _run(inp, True, plan, persistent_ctas=ctas)
        assert torch.equal(got[2], base[2]) and torch.equal(got[1], base[1])


def test_persistent_with_windows_selections_and_ragged_q():
    lens = [6000, 2500, 4000]
    inp = decode_inputs(3, 12, 4, lens, seed=830)
    win = kv_windows(lens, seed=831)
    ql = np.array([4, 1, 3], np.int32)
    plan = mla.mla_decode_plan(lens, 12, 4, target_ctas=30)
    base = _run(inp, True, plan, kv_bounds=win, query_lens=ql)
    got = _run(inp, True, plan, persistent_ctas=4, kv_bounds=win, query_lens=ql)
    assert torch.equal(got[2], base[2]) and torch.equal(got[1], base[1])
    ref_o, ref_l = _oracle(inp, True, kv_bounds=win, query_lens=ql)
    fin = np.isfinite(ref_l)
    idx = torch.from_numpy(fin).cuda()
    assert_parity(got[0].reshape(-1, 512)[idx], got[1].reshape(-1)[idx], ref_o[fin], ref_l[fin])
    sel = page_selection(lens, 40, seed=832)
    plan_s = mla.mla_decode_plan([PAGE_SIZE * 40] * 3, 12, 4, target_ctas=12)
    base = _run(inp, True, plan_s, block_idx=sel)
    got = _run(inp, True, plan_s, persistent_ctas=5, block_idx=sel)
    assert torch.equal(got[2], base[2]) and torch.equal(got[1], base[1])
    ref_o, ref_l = _oracle(inp, True, block_idx=sel)
    assert_parity(got[0], got[1], ref_o, ref_l)


@pytest.mark.parametrize("H,q_len", [(12, 1), (12, 8)])
def test_persistent_expired_wait_then_exact(H, q_len):
    lens = [5000, 3000]
    inp = decode_inputs(2, H, q_len, lens, seed=840 + q_len)
    plan = mla.mla_decode_plan(lens, H, q_len, target_ctas=8)
    mla.mla_debug_set_expire(3, 2)  # the softmax's S^T wait, tile 2 of an item
    try:
        with pytest.raises(mla.MlaError) as e:
            _run(inp, q_len > 1, plan, persistent_ctas=3)
        assert e.value.status == mla.MLA_ERR_TIMEOUT
    finally:
        mla.mla_debug_set_expire(-1)
    out, lse, _ = _run(inp, q_len > 1, plan, persistent_ctas=3)
    ref_o, ref_l = _oracle(inp, q_len > 1)
    assert_parity(out, lse, ref_o, ref_l)


def test_persistent_bad_item_is_reported():
    inp = decode_inputs(2, 12, 1, [3000, 300], seed=850)
    dev = torch.device("cuda")
    plan = mla.mla_decode_plan([3000, 300], 12, 1, target_ctas=6)
    items = torch.from_numpy(mla.mla_decode_plan_items(plan.splits, 12, 1)).to(dev)
    items[1] = (7 << 14)  # request 7 of a batch of 2
    ws_bytes = mla.mla_decode_workspace_size(2, 1, 12, plan.max_splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    mla.mla_decode_workspace_init(ws, ws_bytes)
    out = torch.empty((2, 1, 12, 512), dtype=torch.bfloat16, device=dev)
    lens = torch.tensor([3000, 300], dtype=torch.int32, device=dev)
    mla.mla_decode_ex(inp.q.to(dev), inp.kv.to(dev), inp.num_pages, inp.page_table.to(dev),
                      inp.max_pages, lens, torch.from_numpy(plan.splits).to(dev),
                      torch.from_numpy(plan.chunks).to(dev), plan.max_splits, plan.kv_split, 2, 1,
                      12, False, 1.0, 1.0, SOFTMAX_SCALE, ws, ws_bytes, out, cta_items=items,
                      persistent_ctas=2)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_status(ws)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG
