"""GPU parity of the restricted-key-set variants against the fp64 oracle:
ragged query counts (query_lens), key windows (kv_bounds) and the sparse decode
over selected pages (mla_decode_sparse), through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import split_kv_mla_paged_gb300 as mla
from split_kv_mla_paged_gb300 import build as mla_build
from synth import (PAGE_SIZE, SOFTMAX_SCALE, decode_inputs, kv_windows, page_selection,
                   query_lens_ragged)
from mla_testutil import PLAN_ABS, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mla_build.build()
    mla.load_library()
    yield
    torch.cuda.synchronize()


def _run(inp, causal, scale=SOFTMAX_SCALE, plan=None, target_ctas=0, **kw):
    dev = torch.device("cuda")
    out, lse, o32 = mla.decode(inp.q.to(dev), inp.kv.to(dev), inp.page_table.to(dev),
                               inp.kv_lens, num_heads=inp.num_heads, q_len=inp.q_len,
                               causal=causal, softmax_scale=scale, plan=plan,
                               target_ctas=target_ctas, want_f32=True, **kw)
    torch.cuda.synchronize()
    return out, lse, o32


def _oracle(inp, causal, scale=SOFTMAX_SCALE, **kw):
    return oracle.decode_rows(inp.q, inp.kv.cpu(), inp.page_table.cpu(), inp.kv_lens,
                              q_len=inp.q_len, num_heads=inp.num_heads, causal=causal,
                              softmax_scale=scale, **kw)


def _check(inp, causal, ref_kw, run_kw=None, scale=SOFTMAX_SCALE, **plan_kw):
    run_kw = dict(ref_kw if run_kw is None else run_kw)
    out, lse, o32 = _run(inp, causal, scale, **plan_kw, **run_kw)
    ref_o, ref_l = _oracle(inp, causal, scale, **ref_kw)
    lse_np = lse.cpu().numpy().reshape(-1)
    fin = np.isfinite(ref_l)
    # Rows that see no key: O = 0 and LSE = -inf, exactly.
    assert np.array_equal(np.isfinite(lse_np), fin)
    assert torch.all(out.reshape(-1, 512)[torch.from_numpy(~fin).cuda()] == 0)
    assert_parity(out.reshape(-1, 512)[torch.from_numpy(fin).cuda()],
                  lse.reshape(-1)[torch.from_numpy(fin).cuda()], ref_o[fin], ref_l[fin])
    assert torch.equal(o32.to(torch.bfloat16), out)
    return out, lse, o32


# ---- ragged query counts ------------------------------------------------------

@pytest.mark.parametrize("B,H,q_len,lens,causal", [
    (4, 12, 8, [300, 1029, 4000, 900], True),   # 96 rows -> two groups of 48
    (3, 16, 4, [2000, 700, 129], True),         # 64 rows -> two groups of 32
    (3, 12, 2, [513, 64, 5000], False),         # 24 rows -> 32
    (2, 3, 5, [40, 1000], True),                # 15 rows -> 16
])
def test_query_lens_parity(B, H, q_len, lens, causal):
    inp = decode_inputs(B, H, q_len, lens, seed=400 + B * H, extra_pages=1)
    ql = query_lens_ragged(B, q_len, seed=B + q_len)
    ql[0] = 1
    for target in (0, 3, 40):
        plan = mla.mla_decode_plan(lens, H, q_len, target_ctas=target) if target else None
        _check(inp, causal, dict(query_lens=np.asarray(ql, np.int32)), plan=plan)


@pytest.mark.parametrize("H", [12, 16])
def test_query_lens_whole_padding_group_and_sinks(H):
    # q_b = 1 of 8: with H = 12 the 96-row group holds 12 real rows; with
    # H = 16 (128 rows, two groups of 64) the second group of the request is
    # all padding (no tile runs there).  Sinks give padding rows LSE = sink.
    inp = decode_inputs(2, H, 8, [3000, 700], seed=410)
    ql = np.array([1, 8], np.int32)
    sinks = np.linspace(-1.0, 2.0, H)
    for target in (2, 30):
        plan = mla.mla_decode_plan([3000, 700], H, 8, target_ctas=target)
        out, lse, _ = _run(inp, True, plan=plan, query_lens=ql, sinks=sinks)
        ref_o, ref_l = _oracle(inp, True, query_lens=ql, sinks=sinks)
        assert_parity(out, lse, ref_o, ref_l)


# ---- key windows --------------------------------------------------------------

@pytest.mark.parametrize("B,H,q_len,lens,causal", [
    (4, 12, 1, [1000, 5000, 777, 130], False),
    (4, 12, 8, [3000, 1029, 4100, 900], True),
    (3, 20, 1, [2500, 300, 1300], False),
])
def test_kv_bounds_parity(B, H, q_len, lens, causal):
    inp = decode_inputs(B, H, q_len, lens, seed=420 + B, extra_pages=2)
    win = kv_windows(lens, seed=B + H)
    base = None
    for target in (0, 1, 9, 60):
        plan = mla.mla_decode_plan(lens, H, q_len, target_ctas=target) if target else None
        _, _, o32 = _check(inp, causal, dict(kv_bounds=win), plan=plan)
        if base is None:
            base = o32
        else:
            assert (o32 - base).abs().max().item() <= PLAN_ABS


def test_kv_bounds_empty_window_and_ragged_q_together():
    inp = decode_inputs(3, 12, 4, [2000, 640, 1500], seed=430)
    win = np.array([[500, 500], [0, 640], [1400, 1450]], np.int32)  # empty, whole, inner
    ql = np.array([4, 2, 3], np.int32)
    for target in (0, 8):
        plan = mla.mla_decode_plan([2000, 640, 1500], 12, 4, target_ctas=target) if target else None
        _check(inp, True, dict(kv_bounds=win, query_lens=ql), plan=plan)


# ---- sparse decode over selected pages ----------------------------------------

@pytest.mark.parametrize("B,H,q_len,lens,topk,causal,keep_last", [
    (2, 12, 1, [5000, 3000], 20, False, True),
    (3, 12, 1, [4000, 100, 2200], 16, False, False),   # short request: -1 slots
    (2, 12, 8, [6000, 1500], 24, True, True),
    (1, 16, 4, [9000], 40, True, True),
    (2, 1, 1, [700, 33], 8, False, True),               # 33 tokens: last page has 1
])
def test_sparse_parity(B, H, q_len, lens, topk, causal, keep_last):
    inp = decode_inputs(B, H, q_len, lens, seed=440 + topk, extra_pages=2)
    sel = page_selection(lens, topk, seed=topk + B, keep_last=keep_last)
    for target in (0, 1, 5, 30):
        plan = None
        if target:
            plan = mla.mla_decode_plan([PAGE_SIZE * topk] * B, H, q_len, target_ctas=target)
        _check(inp, causal, dict(block_idx=sel), plan=plan)


def test_sparse_with_window_and_ragged_q():
    lens = [6000, 2500]
    inp = decode_inputs(2, 12, 8, lens, seed=450)
    sel = page_selection(lens, 30, seed=451)
    win = np.array([[1000, 6000], [0, 2000]], np.int32)
    ql = np.array([5, 8], np.int32)
    _check(inp, True, dict(block_idx=sel, kv_bounds=win, query_lens=ql))


def test_sparse_all_pages_equals_dense():
    # Selecting every page in order is the dense decode.
    lens = [3000, 1111]
    inp = decode_inputs(2, 12, 1, lens, seed=452)
    n = max((L + 31) // 32 for L in lens)
    sel = np.full((2, n), -1, np.int32)
    for b, L in enumerate(lens):
        k = (L + 31) // 32
        sel[b, :k] = np.arange(k)
    out_s, lse_s, _ = _run(inp, False, block_idx=sel)
    out_d, lse_d, _ = _run(inp, False)
    ref_o, ref_l = _oracle(inp, False)
    assert_parity(out_s, lse_s, ref_o, ref_l)
    assert_parity(out_d, lse_d, ref_o, ref_l)


def test_sparse_unordered_selection_is_reported():
    inp = decode_inputs(1, 12, 1, [3000], seed=453)
    sel = np.array([[3, 9, 7, 20]], np.int32)
    with pytest.raises(mla.MlaError) as e:
        _run(inp, False, block_idx=sel)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG


def test_query_lens_out_of_range_is_reported():
    inp = decode_inputs(2, 12, 4, [300, 500], seed=454)
    with pytest.raises(mla.MlaError) as e:
        _run(inp, True, query_lens=np.array([2, 5], np.int32))
    assert e.value.status == mla.MLA_ERR_INVALID_ARG


def test_sparse_full_size_sampled_rows():
    # 16 requests of 1M keys with 256 selected pages (8192 keys) each, the
    # plan and launch of the sparse bench line; rows sampled for the oracle.
    B, L, topk = 16, 1048576, 256
    inp = decode_inputs(B, 12, 1, [L] * B, seed=460, device="cuda")
    sel = page_selection([L] * B, topk, seed=461)
    out, lse, o32 = _run(inp, False, block_idx=sel)
    g = np.random.default_rng(7)
    rows = np.sort(g.choice(B * 12, size=6, replace=False))
    ref_o = np.zeros((len(rows), 512))
    ref_l = np.zeros(len(rows))
    for i, r in enumerate(rows):
        b = int(r // 12)
        # Oracle over only this request's selected pages (a gathered cache).
        pages = inp.page_table[b].cpu()[torch.from_numpy(sel[b].astype(np.int64))]
        kv_b = inp.kv[pages.cuda().long()].cpu()
        table = torch.arange(topk, dtype=torch.int32)[None, :]
        o, l = oracle.decode_rows(inp.q[b:b + 1].cpu(), kv_b, table,
                                  torch.tensor([topk * PAGE_SIZE], dtype=torch.int32),
                                  q_len=1, num_heads=12, causal=False,
                                  softmax_scale=SOFTMAX_SCALE, rows=[int(r % 12)])
        ref_o[i], ref_l[i] = o[0], l[0]
    idx = torch.from_numpy(rows).cuda()
    assert_parity(out.reshape(-1, 512)[idx], lse.reshape(-1)[idx], ref_o, ref_l)
    assert torch.isfinite(o32).all()
    del inp
    torch.cuda.empty_cache()


def test_sparse_with_item_list():
    lens = [6000, 200, 3000]
    inp = decode_inputs(3, 12, 1, lens, seed=470)
    sel = page_selection(lens, 24, seed=471, keep_last=False)
    plan = mla.mla_decode_plan([PAGE_SIZE * 24] * 3, 12, 1, target_ctas=30)
    _check(inp, False, dict(block_idx=sel), run_kw=dict(block_idx=sel, use_items=True), plan=plan)


def test_graph_replay_picks_up_new_selection():
    # The selection is a device input: a captured sparse decode reads the new
    # pages on every replay (the block selector runs before it each step).
    lens = [7000, 4000]
    inp = decode_inputs(2, 12, 1, lens, seed=480)
    dev = torch.device("cuda")
    topk = 20
    plan = mla.mla_decode_plan([PAGE_SIZE * topk] * 2, 12, 1, sm_count=152)
    sel_d = torch.from_numpy(page_selection(lens, topk, seed=481)).to(dev)
    q, kv, pt = inp.q.to(dev), inp.kv.to(dev), inp.page_table.to(dev)
    lens_d = inp.kv_lens.to(dev)
    ws_bytes = plan.workspace_bytes
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    mla.mla_decode_workspace_init(ws, ws_bytes)
    out = torch.empty((2, 1, 12, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((2, 1, 12), dtype=torch.float32, device=dev)
    args = (q, kv, inp.num_pages, pt, inp.max_pages, lens_d, sel_d, topk,
            torch.from_numpy(plan.splits).to(dev), torch.from_numpy(plan.chunks).to(dev),
            plan.max_splits, plan.kv_split, 2, 1, 12, False, 1.0, 1.0, SOFTMAX_SCALE, ws,
            ws_bytes, out, lse, None)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        mla.mla_decode_sparse(*args, stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        mla.mla_decode_sparse(*args)
    for s in (481, 482, 483):
        sel = page_selection(lens, topk, seed=s)
        sel_d.copy_(torch.from_numpy(sel))
        g.replay()
        torch.cuda.synchronize()
        ref_o, ref_l = _oracle(inp, False, block_idx=sel)
        assert_parity(out, lse, ref_o, ref_l, what=f"selection {s}")
    mla.mla_decode_status(ws, stream)
