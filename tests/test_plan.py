"""Host planner: the pages' printed plans, and invariants of the GB300 planner."""
import json
import os

import numpy as np
import pytest

import split_kv_mla_paged_gb300 as mla
from split_kv_mla_paged_gb300 import build as mla_build

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "p4_split_plans.json")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mla_build.build()
    mla.load_library()


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden()["repro2_q8_target100"],
                         ids=lambda c: f"B{c['batch']}_L{c['kv_len']}")
def test_repro2_plans_reproduced(case):
    p = mla.mla_decode_plan([case["kv_len"]] * case["batch"], num_heads=12, q_len=8,
                            target_ctas=100)
    assert p.splits.tolist() == [case["splits"]] * case["batch"]
    assert np.all(p.chunks % 128 == 0)
    assert np.all(p.splits.astype(np.int64) * p.chunks >= case["kv_len"])
    assert np.all((p.splits.astype(np.int64) - 1) * p.chunks < case["kv_len"])


@pytest.mark.parametrize("case", _golden()["repro1_q1_uniform"], ids=lambda c: f"B{c['batch']}")
@pytest.mark.parametrize("kv_len", [131072, 1048576])
def test_repro1_uniform_splits(case, kv_len):
    b, split = case["batch"], case["split"]
    p = mla.mla_decode_plan([kv_len] * b, num_heads=12, q_len=1, target_ctas=b * split)
    assert p.splits.tolist() == [split] * b


def test_tiny_plan():
    t = _golden()["tiny"]
    p = mla.mla_decode_plan([t["kv_len"]], num_heads=12, q_len=t["q_len"], target_ctas=t["target"])
    assert p.splits.tolist() == [t["splits"]] and p.chunks.tolist() == [1024]


@pytest.mark.parametrize("lens,H,q", [
    ([1048576] * 16, 12, 1), ([1048576] * 16, 12, 8), ([131072] * 4, 12, 8), ([4096], 12, 1),
    ([131072], 12, 8), ([1048576], 96, 8), ([1024, 131072, 5000, 77777, 1048576], 12, 1),
    ([8] * 3, 12, 8), ([1], 1, 1),
])
@pytest.mark.parametrize("sm_count", [152, 148, 7])
def test_gb300_planner_invariants(lens, H, q, sm_count):
    p = mla.mla_decode_plan(lens, num_heads=H, q_len=q, sm_count=sm_count)
    L = np.asarray(lens, dtype=np.int64)
    assert np.all(p.chunks % 128 == 0) and np.all(p.chunks >= 128)
    assert np.all(p.splits >= 1) and np.all(p.splits <= mla.MAX_SPLITS)
    assert np.all(p.splits * p.chunks.astype(np.int64) >= L)
    assert np.all((p.splits - 1) * p.chunks.astype(np.int64) < L)
    assert p.kv_split in (1, 2, 4, 8, 16) and p.kv_split <= max(1, p.max_splits)
    assert p.workspace_bytes == mla.mla_decode_workspace_size(len(lens), q, H, p.max_splits)
    # CTA budget: at most two waves (2 x SMs) of split-kernel CTAs, unless one
    # split per request already exceeds it (then every request has one split).
    ctas = int(p.splits.sum()) * _row_groups(H * q)
    if len(lens) * _row_groups(H * q) <= 2 * sm_count:
        assert ctas <= 2 * sm_count, (ctas, sm_count)
    else:
        assert np.all(p.splits == 1)


def _row_groups(rows):
    """CTAs per (request, split) of the FP8 split kernel: one CTA of up to 48
    rows, else groups of at most 96 rows."""
    return 1 if rows <= 48 else -(-rows // 96)


def test_gb300_planner_stays_within_two_waves_on_every_workload():
    from synth import WORKLOADS
    for name, w in WORKLOADS.items():
        lens = [32 * w["topk"]] * w["batch"] if w.get("topk") else w["kv_lens"]
        p = mla.mla_decode_plan(lens, num_heads=w["num_heads"], q_len=w["q_len"], sm_count=152)
        ctas = int(p.splits.sum()) * _row_groups(w["num_heads"] * w["q_len"])
        assert ctas <= 2 * 152, (name, ctas)


def test_gb300_planner_budget_with_many_requests():
    # 64 requests x 8 row groups (H96 q8) exceed two waves with one split
    # each: every request keeps one split.
    p = mla.mla_decode_plan([100000] * 64, num_heads=96, q_len=8, sm_count=152)
    assert np.all(p.splits == 1)


def test_gb300_planner_fills_one_wave_for_uniform_long_batch():
    p = mla.mla_decode_plan([1048576] * 16, num_heads=12, q_len=1, sm_count=152)
    ctas = int(p.splits.sum())
    # Whole waves of 152 CTAs, at least 90% busy.
    waves = -(-ctas // 152)
    assert ctas >= 0.9 * waves * 152


def test_skewed_batch_gets_common_chunk():
    lens = [1048576] + [2048] * 7
    p = mla.mla_decode_plan(lens, num_heads=12, q_len=1, sm_count=152)
    assert len(set(p.chunks.tolist())) == 1
    assert p.splits[0] > 8 * p.splits[1]


@pytest.mark.parametrize("bad", [
    dict(kv_lens=[4, 10], q_len=8),       # kv_len below q_len
    dict(kv_lens=[0], q_len=1),           # empty request
    dict(kv_lens=[100], q_len=0),
])
def test_plan_rejects_bad_arguments(bad):
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_plan(bad["kv_lens"], num_heads=12, q_len=bad["q_len"], sm_count=152)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG


def test_plan_rejects_too_many_rows():
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_plan([4096], num_heads=256, q_len=8, sm_count=152)
    assert e.value.status == mla.MLA_ERR_UNSUPPORTED


def test_plan_needs_sm_count_without_target():
    with pytest.raises(mla.MlaError):
        mla.mla_decode_plan([4096], num_heads=12, q_len=1, sm_count=0, target_ctas=0)


def test_plan_items_are_the_ctas_with_work_in_split_major_order():
    splits = np.array([3, 1, 2], dtype=np.int32)
    for H, q, groups in ((12, 1, 1), (12, 4, 1), (12, 8, 1), (16, 8, 2), (96, 8, 8)):
        items = mla.mla_decode_plan_items(splits, H, q)
        assert items.shape[0] == int(splits.sum()) * groups
        b = items >> 14
        s = (items >> 5) & 511
        g = items & 31
        # every (request, split < splits[b], group) exactly once
        got = sorted(zip(b.tolist(), s.tolist(), g.tolist()))
        want = sorted((bb, ss, gg) for bb in range(3) for ss in range(int(splits[bb]))
                      for gg in range(groups))
        assert got == want
        # split-major, row groups adjacent
        assert np.all(np.diff(s) >= 0)
        key = s * 1000 + b
        assert np.all(np.diff(key) >= 0)


def test_fp8_row_groups_over_all_row_counts():
    # Up to 48 rows run in one CTA; above that, groups of at most 96 rows.
    for rows in list(range(1, 200)) + [255, 256, 287, 288, 289, 767, 768, 769, 1000, 1024]:
        items = mla.mla_decode_plan_items(np.array([1], np.int32), rows, 1)
        want = 1 if rows <= 48 else -(-rows // 96)
        assert items.shape[0] == want, rows
        assert sorted((items & 31).tolist()) == list(range(want))


def test_plan_items_rejects_bad_splits():
    with pytest.raises(mla.MlaError):
        mla.mla_decode_plan_items([2, 0], 12, 1)
    with pytest.raises(mla.MlaError):
        mla.mla_decode_plan_items([2, mla.MAX_SPLITS + 1], 12, 1)


@pytest.mark.parametrize("rows_hq,splits,expect", [
    ((12, 1), 6, 2), ((12, 1), 12, 4), ((12, 1), 25, 8), ((12, 1), 128, 16),
    ((12, 8), 25, 8), ((12, 8), 128, 8), ((12, 16), 50, 4), ((96, 8), 19, 1), ((12, 1), 1, 1),
])
def test_merge_kv_split_rule(rows_hq, splits, expect):
    # KvSplit = the largest of 16/8/4/2/1 with >= 2 partials per group and
    # rows x groups <= 6 x SMs (152 SMs: 912); one request planned by the
    # pages' planner to exactly `splits` splits of one tile each.
    H, q = rows_hq
    p = mla.mla_decode_plan([splits * 128], num_heads=H, q_len=q, sm_count=152,
                            target_ctas=splits)
    assert p.max_splits == splits and p.kv_split == expect


def test_merge_kv_split_counts_only_merged_rows():
    # A skewed batch: one long request (many splits) and short ones (one split
    # each, written directly): only the long request's 96 rows are merged.
    lens = [1048576] + [4096] * 7
    p = mla.mla_decode_plan(lens, num_heads=12, q_len=8, sm_count=152)
    assert p.splits[0] > 100 and np.all(p.splits[1:] == 1)
    assert p.kv_split == 8  # 96 rows x 8 groups <= 912; 768 rows would give 1
