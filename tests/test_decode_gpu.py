"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import split_kv_mla_paged_gb300 as mla
from split_kv_mla_paged_gb300 import build as mla_build
from synth import SOFTMAX_SCALE, WORKLOADS, decode_inputs, merge_partials, workload_inputs
from mla_testutil import PLAN_ABS, assert_parity, oracle_rows, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mla_build.build()
    mla.load_library()
    yield
    torch.cuda.synchronize()


def _full_check(inp, causal, scale, o_tol=None, **kw):
    out, lse, out_f32 = run_decode(inp, causal, scale, **kw)
    ref_o, ref_l = oracle.decode_rows(inp.q, inp.kv.cpu(), inp.page_table.cpu(), inp.kv_lens,
                                      q_len=inp.q_len, num_heads=inp.num_heads, causal=causal,
                                      softmax_scale=scale, q_scale=kw.get("q_scale", 1.0),
                                      kv_scale=kw.get("kv_scale", 1.0))
    assert_parity(out, lse, ref_o, ref_l, o_tol=o_tol)
    # The fp32 pre-store output rounds to the BF16 output exactly.
    assert torch.equal(out_f32.to(torch.bfloat16), out)
    return out, lse, out_f32


def test_tiny_config_pages_plan():
    w = WORKLOADS["tiny_b1_h12_q1_l4096"]
    inp = workload_inputs("tiny_b1_h12_q1_l4096")
    plan = mla.mla_decode_plan(inp.kv_lens.tolist(), 12, 1, target_ctas=w["target"])
    assert plan.splits.tolist() == [4]
    _full_check(inp, False, SOFTMAX_SCALE, plan=plan)


def test_tiny_config_gb300_plan():
    inp = workload_inputs("tiny_b1_h12_q1_l4096")
    _full_check(inp, False, SOFTMAX_SCALE)


@pytest.mark.parametrize("B,H,q_len,lens,causal", [
    (1, 12, 1, [1], False),
    (1, 12, 1, [31], False),
    (1, 12, 1, [129], False),
    (2, 12, 1, [1000, 77], False),
    (1, 12, 8, [8], True),
    (2, 12, 8, [300, 1029], True),
    (1, 1, 1, [5000], False),
    (1, 3, 2, [513], True),
    (1, 20, 1, [333], False),       # 20 rows -> 32 columns
    (1, 10, 4, [700], True),        # 40 rows -> 48
    (1, 16, 4, [2000], True),       # 64 rows
    (1, 16, 5, [900], True),        # 80 rows
    (2, 12, 8, [4096, 2500], True), # 96 rows
    (1, 16, 8, [1500], True),       # 128 rows -> two groups of 64
    (2, 25, 4, [1200, 700], True),  # 100 rows -> two groups of 50 in 96-row CTAs
    (1, 96, 8, [600], True),        # 768 rows -> eight groups of 96
])
def test_parity_shapes(B, H, q_len, lens, causal):
    inp = decode_inputs(B, H, q_len, lens, seed=100 + B * H + q_len, extra_pages=2)
    _full_check(inp, causal, SOFTMAX_SCALE)


@pytest.mark.parametrize("target", [1, 3, 7, 50])
def test_parity_pages_planner_targets(target):
    inp = decode_inputs(2, 12, 8, [3000, 1111], seed=7, extra_pages=1)
    plan = mla.mla_decode_plan(inp.kv_lens.tolist(), 12, 8, target_ctas=target)
    _full_check(inp, True, SOFTMAX_SCALE, plan=plan)


def test_parity_scales_and_peaked_softmax():
    inp = decode_inputs(1, 12, 2, [3333], seed=8)
    _full_check(inp, True, 0.11, q_scale=1.5, kv_scale=0.75)
    # Large logits: many reference moves and strongly peaked rows.
    _full_check(inp, False, 1.0)


def test_split_plans_agree_in_fp32():
    inp = decode_inputs(2, 12, 8, [5000, 2345], seed=9, extra_pages=1)
    lens = inp.kv_lens.tolist()
    plans = [mla.mla_decode_plan(lens, 12, 8, target_ctas=t) for t in (1, 2, 6, 20, 100)]
    plans.append(mla.mla_decode_plan(lens, 12, 8, sm_count=152))
    base = None
    for plan in plans:
        for ks in (1, 2, 4, 8, 16):
            if ks > plan.max_splits and ks != 1:
                continue
            _, lse, o32 = run_decode(inp, True, SOFTMAX_SCALE, plan=plan, kv_split=ks)
            if base is None:
                base = (o32.clone(), lse.clone())
                continue
            d = (o32 - base[0]).abs().max().item()
            dl = (lse - base[1]).abs().max().item()
            assert d <= PLAN_ABS, f"plan {plan.splits.tolist()} kv_split {ks}: {d:.3e}"
            assert dl <= PLAN_ABS, f"plan {plan.splits.tolist()} kv_split {ks}: lse {dl:.3e}"


def test_maximum_rows_per_request():
    # H * q = 1024 = MLA_MAX_ROWS: 11 row groups of at most 94 rows (96-row CTAs).
    inp = decode_inputs(2, 128, 8, [700, 300], seed=21, extra_pages=1)
    _full_check(inp, True, SOFTMAX_SCALE)


def test_maximum_splits_per_request():
    # 256 splits (MLA_MAX_SPLITS) of one 128-token tile each, merged by 16 groups.
    inp = decode_inputs(1, 12, 1, [32768], seed=22)
    plan = mla.mla_decode_plan([32768], 12, 1, sm_count=256)
    assert plan.max_splits == mla.MAX_SPLITS == 256 and plan.kv_split == 16
    _full_check(inp, False, SOFTMAX_SCALE, plan=plan)


def test_many_row_merge_fits_one_wave():
    # 96 rows over ~96 splits merged by 16 groups (an explicit KvSplit; the
    # planner picks 8 here): rows x 4 CTAs above two per SM, the case the
    # one-wave merge kernel serves.
    inp = decode_inputs(1, 12, 8, [12288], seed=24)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = mla.mla_decode_plan([12288], 12, 8, sm_count=sms)
    assert plan.max_splits >= 32 and 96 * 4 > 2 * sms
    _full_check(inp, True, SOFTMAX_SCALE, plan=plan, kv_split=16)


def test_deterministic_run_to_run():
    inp = decode_inputs(1, 12, 1, [9000], seed=10)
    a = run_decode(inp, False, SOFTMAX_SCALE)
    b = run_decode(inp, False, SOFTMAX_SCALE)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_page_permutation_changes_nothing():
    inp = decode_inputs(1, 12, 1, [2500], seed=11, extra_pages=3)
    a = run_decode(inp, False, SOFTMAX_SCALE)
    P = inp.num_pages
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    inp.kv = inp.kv[perm]
    pt = inp.page_table.clone()
    m = pt >= 0
    pt[m] = inv[pt[m].long()].to(torch.int32)
    inp.page_table = pt
    b = run_decode(inp, False, SOFTMAX_SCALE)
    assert torch.equal(a[2], b[2]) and torch.equal(a[1], b[1])


# ---------------------------------------------------------------- merge alone

@pytest.mark.parametrize("rows,S", [(12, 6), (96, 25), (192, 128), (7, 1), (40, 33)])
@pytest.mark.parametrize("kv_split", [1, 2, 4, 8, 16])
def test_merge_against_oracle(rows, S, kv_split):
    o, ml = merge_partials(rows, S, seed=rows * 131 + S, all_empty_rows=[rows // 2])
    ref_o, ref_l = oracle.merge(o, ml)
    out, lse, out_f32 = mla.merge(torch.from_numpy(o).cuda(), torch.from_numpy(ml).cuda(), kv_split)
    torch.cuda.synchronize()
    f = out_f32.cpu().numpy().astype(np.float64)
    scale = np.max(np.abs(ref_o))
    assert np.max(np.abs(f - ref_o)) <= 2e-6 * scale
    l = lse.cpu().numpy()
    e = rows // 2
    assert l[e] == -np.inf and np.all(f[e] == 0.0)
    # Rows whose slots all came out empty (the forced one, or by chance) give
    # -inf on both sides; the others agree to fp32 rounding.
    empty = ref_l == -np.inf
    assert np.array_equal(l == -np.inf, empty)
    assert np.max(np.abs(l[~empty] - ref_l[~empty])) <= 1e-5
    assert torch.equal(out_f32.to(torch.bfloat16), out)


def test_merge_kv_split_invariance():
    o, ml = merge_partials(24, 100, seed=5)
    res = [mla.merge(torch.from_numpy(o).cuda(), torch.from_numpy(ml).cuda(), g)
           for g in (1, 2, 4, 8, 16)]
    for _, lse, f in res[1:]:
        assert (f - res[0][2]).abs().max().item() <= PLAN_ABS * res[0][2].abs().max().item()
        assert (lse - res[0][1]).abs().max().item() <= PLAN_ABS


# ---------------------------------------------------------------- device status

def test_bad_page_id_is_reported():
    inp = decode_inputs(1, 12, 1, [200], seed=12)
    inp.page_table[0, 2] = inp.num_pages + 5
    with pytest.raises(mla.MlaError) as e:
        run_decode(inp, False, SOFTMAX_SCALE)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG


def test_inconsistent_plan_is_reported():
    inp = decode_inputs(1, 12, 1, [1000], seed=13)
    plan = mla.mla_decode_plan(inp.kv_lens.tolist(), 12, 1, target_ctas=4)
    plan.chunks[:] = 100  # not a multiple of the 128-token tile
    with pytest.raises(mla.MlaError) as e:
        run_decode(inp, False, SOFTMAX_SCALE, plan=plan)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG


@pytest.mark.parametrize("H,q_len", [(12, 1), (12, 8)])
def test_tiny_wait_limit_times_out_or_completes_and_context_survives(H, q_len):
    # With a wait limit of 64 cycles a pipeline wait may run out or not (the
    # waits block in mbarrier.try_wait, whose hardware suspend window can
    # outlast so short a limit; tests/test_expire_gpu.py drives the expiry
    # path deterministically).  Either the call completes with the right
    # result or it reports MLA_ERR_TIMEOUT, and the next call on the same
    # context is exact.
    inp = decode_inputs(1, H, q_len, [60000], seed=14)
    rows = np.array([0, 5, 11]) if q_len == 1 else np.array([0, 17, 50, 95])
    ref_o, ref_l = oracle_rows(inp, rows, q_len > 1, SOFTMAX_SCALE)
    idx = torch.from_numpy(rows).cuda()
    mla.mla_debug_set_wait_limit(64)
    try:
        out, lse, _ = run_decode(inp, q_len > 1, SOFTMAX_SCALE)
        assert_parity(out.reshape(-1, 512)[idx], lse.reshape(-1)[idx], ref_o, ref_l)
    except mla.MlaError as e:
        assert e.status == mla.MLA_ERR_TIMEOUT
    finally:
        mla.mla_debug_set_wait_limit(0)
    out, lse, _ = run_decode(inp, q_len > 1, SOFTMAX_SCALE)
    assert_parity(out.reshape(-1, 512)[idx], lse.reshape(-1)[idx], ref_o, ref_l)


# ---------------------------------------------------------------- full-size workloads

def _sample_rows(inp, n, seed):
    """Rows to check against the oracle: in the first and the last request,
    one row of every 96-row group (so every CTA row group of a packed request
    is hit), the first and the last query token of the block (MTP verify: the
    fewest and the most visible keys), then seeded random rows up to n."""
    g = np.random.default_rng(seed)
    per_req = inp.num_heads * inp.q_len
    picks = set()
    for b in sorted({0, inp.batch - 1}):
        base = b * per_req
        for grp in range(0, per_req, 96):
            picks.add(base + grp + int(g.integers(0, min(96, per_req - grp))))
        for qi in (0, inp.q_len - 1):
            picks.add(base + qi * inp.num_heads + int(g.integers(0, inp.num_heads)))
    while len(picks) < min(n, inp.rows):
        picks.add(int(g.integers(0, inp.rows)))
    return np.array(sorted(picks), dtype=np.int64)


# Every configuration of the workload list at its own size: the tiny case and
# B1-B16 at 128K are covered above and here; the 1M q1/q8 batches, the MTP
# verify block at B1-B16, the H96 packed heads at 128K/1M and B1/B4, the
# ragged batch and the skewed batch.
@pytest.mark.parametrize("name,nrows", [
    ("h12_q1_l128k_b1", 8),
    ("h12_q1_l128k_b16", 8),
    ("mtp_h12_q8_l128k_b1", 8),
    ("mtp_h12_q8_l128k_b4", 10),
    ("mtp_h12_q8_l128k_b8", 8),
    ("mtp_h12_q8_l128k_b16", 10),
    ("ragged_h12_q1_b16", 16),
    ("packed_h96_q8_l128k_b1", 12),
    ("packed_h96_q8_l128k_b4", 20),
    ("packed_h96_q8_l1m_b1", 12),
    ("packed_h96_q8_l1m_b4", 20),
    ("long_h12_q1_l1m_b16", 6),
    ("long_h12_q8_l1m_b1", 8),
    ("long_h12_q8_l1m_b16", 8),
    ("skewed_h12_q8_1m_plus_7x4k", 8),
])
def test_full_size_sampled_rows(name, nrows):
    w = WORKLOADS[name]
    inp = workload_inputs(name, device="cuda")
    out, lse, o32 = run_decode(inp, w["causal"], SOFTMAX_SCALE)
    rows = _sample_rows(inp, nrows, seed=len(name))
    ref_o, ref_l = oracle_rows(inp, rows, w["causal"], SOFTMAX_SCALE)
    flat_o = out.reshape(-1, 512)[torch.from_numpy(rows).cuda()]
    flat_l = lse.reshape(-1)[torch.from_numpy(rows).cuda()]
    assert_parity(flat_o, flat_l, ref_o, ref_l, what=name)
    assert torch.isfinite(o32).all() and torch.isfinite(lse).all()
    # Properties over every row at full size: a second split plan (the pages'
    # planner, or a smaller CTA target for the packed-heads batches) agrees in
    # fp32 before the store.
    target = w["target"] if w["target"] is not None else 40
    plan = mla.mla_decode_plan(inp.kv_lens.tolist(), w["num_heads"], w["q_len"],
                               target_ctas=target)
    _, lse2, o32b = run_decode(inp, w["causal"], SOFTMAX_SCALE, plan=plan)
    assert (o32b - o32).abs().max().item() <= PLAN_ABS
    assert (lse2 - lse).abs().max().item() <= PLAN_ABS
    del inp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,scale", [
    ("long_h12_q8_l1m_b1", 0.5),
    ("long_h12_q1_l1m_b16", 1.0),
])
def test_full_length_peaked_rows(name, scale):
    # At 1M keys with softmax_scale 0.0722 every row is nearly uniform and
    # |O| ~ 5e-4, below the absolute term of the tolerance.  A larger scale
    # makes the rows peaked (a few hundred effective keys at 0.5, a handful at
    # 1.0), so |O| is far above 2e-3 and the O comparison can fail.
    w = WORKLOADS[name]
    inp = workload_inputs(name, device="cuda")
    out, lse, o32 = run_decode(inp, w["causal"], scale)
    rows = _sample_rows(inp, 12, seed=7)
    ref_o, ref_l = oracle_rows(inp, rows, w["causal"], scale)
    flat_o = out.reshape(-1, 512)[torch.from_numpy(rows).cuda()]
    flat_l = lse.reshape(-1)[torch.from_numpy(rows).cuda()]
    o_max = float(np.abs(ref_o).max())
    assert o_max > 10 * 2e-3, f"{name}: rows not peaked (max |O| {o_max:.2e})"
    worst, lerr = assert_parity(flat_o, flat_l, ref_o, ref_l, what=f"{name} scale {scale}")
    f32 = o32.reshape(-1, 512)[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    rel32 = float(np.abs(f32 - ref_o).max()) / o_max
    print(f"{name} softmax_scale {scale}: max|O_ref| {o_max:.3e}, max |O err| (BF16) "
          f"{worst:.3e} = {worst / o_max:.2e} of max|O_ref|, fp32 before the store "
          f"{rel32:.2e} of max|O_ref|, max |LSE err| {lerr:.2e}")
    del inp
    torch.cuda.empty_cache()


def test_item_list_matches_the_grid_launch():
    # A skewed batch: the item list launches only the CTAs with work; the
    # results are the same numbers as the full grid's.
    lens = [9000, 300, 129, 2000, 4100]
    inp = decode_inputs(5, 12, 8, lens, seed=23, extra_pages=1)
    for target in (0, 40):
        plan = (mla.mla_decode_plan(lens, 12, 8, target_ctas=target) if target
                else mla.mla_decode_plan(lens, 12, 8, sm_count=152))
        assert np.any(plan.splits < plan.max_splits)
        dev = torch.device("cuda")
        kw = dict(num_heads=12, q_len=8, causal=True, softmax_scale=SOFTMAX_SCALE, plan=plan,
                  want_f32=True)
        out_i, lse_i, o32_i = mla.decode(inp.q.to(dev), inp.kv.to(dev), inp.page_table.to(dev),
                                         inp.kv_lens, use_items=True, **kw)
        out_g, lse_g, o32_g = mla.decode(inp.q.to(dev), inp.kv.to(dev), inp.page_table.to(dev),
                                         inp.kv_lens, use_items=False, **kw)
        torch.cuda.synchronize()
        assert torch.equal(o32_i, o32_g) and torch.equal(lse_i, lse_g)
        ref_o, ref_l = oracle.decode_rows(inp.q, inp.kv.cpu(), inp.page_table.cpu(), inp.kv_lens,
                                          q_len=8, num_heads=12, causal=True,
                                          softmax_scale=SOFTMAX_SCALE)
        assert_parity(out_i, lse_i, ref_o, ref_l)


def test_bad_item_is_reported():
    inp = decode_inputs(2, 12, 1, [3000, 300], seed=24)
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
                      12, False, 1.0, 1.0, SOFTMAX_SCALE, ws, ws_bytes, out, cta_items=items)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_status(ws)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG
