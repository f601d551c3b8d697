"""GPU parity of the BF16-KV decode (mla_decode_bf16, through the C ABI) against
the fp64 oracle on the same BF16 inputs (issue #20510, "Repro 2": the BF16
kernel with the FP8 kernel's geometry)."""
import numpy as np
import pytest
import torch

import oracle
import split_kv_mla_paged_gb300 as mla
from split_kv_mla_paged_gb300 import build as mla_build
from synth import SOFTMAX_SCALE, WORKLOADS, decode_inputs, workload_inputs
from mla_testutil import PLAN_ABS, assert_parity, oracle_rows, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mla_build.build()
    mla.load_library()
    yield
    torch.cuda.synchronize()


def _full_check(inp, causal, scale, **kw):
    out, lse, out_f32 = run_decode(inp, causal, scale, **kw)
    ref_o, ref_l = oracle.decode_rows(inp.q, inp.kv.cpu(), inp.page_table.cpu(), inp.kv_lens,
                                      q_len=inp.q_len, num_heads=inp.num_heads, causal=causal,
                                      softmax_scale=scale)
    assert_parity(out, lse, ref_o, ref_l)
    assert torch.equal(out_f32.to(torch.bfloat16), out)
    return out, lse, out_f32


# Shapes span one and several 64-token tiles, ragged page tails, every row
# grouping (16, 32 and 48 rows per CTA, several groups), MTP causal blocks and
# single-split and multi-split plans.
@pytest.mark.parametrize("B,H,q_len,lens,causal", [
    (1, 12, 1, [1], False),
    (1, 12, 1, [31], False),
    (1, 12, 1, [65], False),
    (1, 12, 1, [129], False),
    (2, 12, 1, [1000, 77], False),
    (1, 12, 8, [8], True),
    (2, 12, 8, [300, 1029], True),
    (1, 1, 1, [5000], False),
    (1, 3, 2, [513], True),
    (1, 20, 1, [333], False),
    (1, 10, 4, [700], True),
    (1, 16, 5, [900], True),
    (1, 16, 8, [1500], True),
    (1, 96, 8, [600], True),
])
def test_bf16_parity_shapes(B, H, q_len, lens, causal):
    inp = decode_inputs(B, H, q_len, lens, seed=300 + B * H + q_len, extra_pages=2,
                        dtype="bf16")
    _full_check(inp, causal, SOFTMAX_SCALE)


@pytest.mark.parametrize("target", [1, 3, 50])
def test_bf16_parity_pages_planner_targets(target):
    inp = decode_inputs(2, 12, 8, [3000, 1111], seed=9, extra_pages=1, dtype="bf16")
    plan = mla.mla_decode_plan(inp.kv_lens.tolist(), 12, 8, target_ctas=target)
    _full_check(inp, True, SOFTMAX_SCALE, plan=plan)


def test_bf16_peaked_softmax_and_plan_agreement():
    # Large logits: many reference moves, strongly peaked rows.
    inp = decode_inputs(1, 12, 2, [4500], seed=10, std=1.5, dtype="bf16")
    out, lse, o32 = _full_check(inp, True, 0.3)
    for target in (1, 7, 40):
        plan = mla.mla_decode_plan(inp.kv_lens.tolist(), 12, 2, target_ctas=target)
        _, lse2, o32b = run_decode(inp, True, 0.3, plan=plan)
        assert (o32b - o32).abs().max().item() <= PLAN_ABS
        assert (lse2 - lse).abs().max().item() <= PLAN_ABS


def test_bf16_bad_page_id_is_reported():
    inp = decode_inputs(1, 12, 1, [700], seed=11, dtype="bf16")
    inp.page_table[0, 3] = inp.kv.shape[0] + 5
    with pytest.raises(mla.MlaError) as e:
        run_decode(inp, False, SOFTMAX_SCALE)
    assert e.value.status == mla.MLA_ERR_INVALID_ARG


def _sample_rows(inp, n, seed):
    g = np.random.default_rng(seed)
    return np.sort(g.choice(inp.rows, size=min(n, inp.rows), replace=False))


@pytest.mark.parametrize("name,nrows", [
    ("bf16_h12_q1_l1m_b1", 4),
    ("bf16_h12_q8_l1m_b1", 4),
    ("bf16_h12_q1_l1m_b16", 4),
])
def test_bf16_full_size_sampled_rows(name, nrows):
    w = WORKLOADS[name]
    inp = workload_inputs(name, device="cuda")
    out, lse, o32 = run_decode(inp, w["causal"], SOFTMAX_SCALE)
    rows = _sample_rows(inp, nrows, seed=len(name))
    ref_o, ref_l = oracle_rows(inp, rows, w["causal"], SOFTMAX_SCALE)
    flat_o = out.reshape(-1, 512)[torch.from_numpy(rows).cuda()]
    flat_l = lse.reshape(-1)[torch.from_numpy(rows).cuda()]
    assert_parity(flat_o, flat_l, ref_o, ref_l, what=name)
    assert torch.isfinite(o32).all() and torch.isfinite(lse).all()
    del inp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,H,q_len,lens,causal", [
    (2, 12, 1, [3000, 700], False),     # 16-row groups: Q in TMEM
    (2, 12, 4, [2000, 900], True),      # one 48-row group
    (2, 12, 8, [1500, 4100], True),     # two 48-row groups
])
def test_bf16_options_parity(B, H, q_len, lens, causal):
    from synth import query_lens_ragged
    inp = decode_inputs(B, H, q_len, lens, seed=320 + q_len, extra_pages=1, dtype="bf16")
    sinks = np.linspace(-2.0, 3.0, H)
    ql = np.asarray(query_lens_ragged(B, q_len, seed=q_len), np.int32) if q_len > 1 else None
    dev = torch.device("cuda")
    for target in (0, 1, 9):
        plan = (mla.mla_decode_plan(lens, H, q_len, target_ctas=target) if target else None)
        for device_scales in (False, True):
            out, lse, o32 = mla.decode(inp.q.to(dev), inp.kv.to(dev), inp.page_table.to(dev),
                                       inp.kv_lens, num_heads=H, q_len=q_len, causal=causal,
                                       softmax_scale=0.13, plan=plan, want_f32=True,
                                       sinks=sinks, output_scale=1.7, query_lens=ql,
                                       device_scales=device_scales)
            torch.cuda.synchronize()
            ref_o, ref_l = oracle.decode_rows(inp.q, inp.kv.cpu(), inp.page_table.cpu(),
                                              inp.kv_lens, q_len=q_len, num_heads=H,
                                              causal=causal, softmax_scale=0.13, sinks=sinks,
                                              output_scale=1.7, query_lens=ql)
            assert_parity(out, lse, ref_o, ref_l, what=f"target {target} dev {device_scales}")
            assert torch.equal(o32.to(torch.bfloat16), out)
