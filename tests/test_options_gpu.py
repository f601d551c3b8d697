"""GPU: mla_decode_ex options (device-side scales, output scale, attention
sinks) against the oracle, including a CUDA-graph replay that picks up a
changed device scale."""
import numpy as np
import pytest
import torch

import oracle
import split_kv_mla_paged_gb300 as mla
from split_kv_mla_paged_gb300 import build as mla_build
from synth import SOFTMAX_SCALE, decode_inputs
from mla_testutil import PLAN_ABS, assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mla_build.build()
    mla.load_library()


def _dev(inp):
    d = torch.device("cuda")
    return inp.q.to(d), inp.kv.to(d), inp.page_table.to(d)


@pytest.mark.parametrize("target", [1, 5, 0])
@pytest.mark.parametrize("B,H,q_len,lens,causal", [
    (2, 12, 1, [3000, 700], False),
    (1, 12, 8, [2500], True),
    (1, 24, 2, [900], True),
])
def test_sinks_and_output_scale(target, B, H, q_len, lens, causal):
    inp = decode_inputs(B, H, q_len, lens, seed=51 + H)
    sinks = np.linspace(-1.0, 2.5, H).astype(np.float32)
    plan = mla.mla_decode_plan(lens, H, q_len, sm_count=152, target_ctas=target)
    q, kv, pt = _dev(inp)
    out, lse, o32 = mla.decode(q, kv, pt, inp.kv_lens, num_heads=H, q_len=q_len, causal=causal,
                               softmax_scale=SOFTMAX_SCALE, plan=plan, sinks=sinks,
                               output_scale=0.8, want_f32=True)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=q_len,
                                      num_heads=H, causal=causal, softmax_scale=SOFTMAX_SCALE,
                                      sinks=sinks.astype(np.float64), output_scale=0.8)
    assert_parity(out, lse, ref_o, ref_l)


def test_sinks_agree_across_plans():
    inp = decode_inputs(1, 12, 8, [4000], seed=55)
    sinks = np.full(12, 1.5, np.float32)
    q, kv, pt = _dev(inp)
    res = []
    for target in (1, 3, 30):
        plan = mla.mla_decode_plan([4000], 12, 8, target_ctas=target)
        res.append(mla.decode(q, kv, pt, inp.kv_lens, num_heads=12, q_len=8, causal=True,
                              softmax_scale=SOFTMAX_SCALE, plan=plan, sinks=sinks,
                              want_f32=True))
    torch.cuda.synchronize()
    for _, lse, o32 in res[1:]:
        assert (o32 - res[0][2]).abs().max().item() <= PLAN_ABS
        assert (lse - res[0][1]).abs().max().item() <= PLAN_ABS


def test_device_scales_match_oracle():
    inp = decode_inputs(2, 12, 2, [1500, 400], seed=56)
    q, kv, pt = _dev(inp)
    out, lse, _ = mla.decode(q, kv, pt, inp.kv_lens, num_heads=12, q_len=2, causal=True,
                             softmax_scale=0.09, q_scale=1.3, kv_scale=0.6, device_scales=True)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=2,
                                      num_heads=12, causal=True, softmax_scale=0.09,
                                      q_scale=1.3, kv_scale=0.6)
    assert_parity(out, lse, ref_o, ref_l)


def test_graph_replay_reads_new_device_scale():
    inp = decode_inputs(1, 12, 1, [3000], seed=57)
    q, kv, pt = _dev(inp)
    dev = q.device
    plan = mla.mla_decode_plan([3000], 12, 1, sm_count=152)
    lens_d = inp.kv_lens.to(dev)
    splits_d = torch.from_numpy(plan.splits).to(dev)
    chunks_d = torch.from_numpy(plan.chunks).to(dev)
    ws_bytes = plan.workspace_bytes
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    mla.mla_decode_workspace_init(ws, ws_bytes)
    out = torch.empty((1, 1, 12, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((1, 1, 12), dtype=torch.float32, device=dev)
    scales = torch.tensor([1.0, 1.0, SOFTMAX_SCALE], dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)
    args = (q, kv, inp.num_pages, pt, inp.max_pages, lens_d, splits_d, chunks_d,
            plan.max_splits, plan.kv_split, 1, 1, 12, False, 99.0, 99.0, 99.0, ws, ws_bytes,
            out, lse, None)
    kw = dict(q_scale_dev=scales[0:1], kv_scale_dev=scales[1:2], softmax_scale_dev=scales[2:3])
    with torch.cuda.stream(stream):  # first call outside the capture
        mla.mla_decode_ex(*args, **kw, stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        mla.mla_decode_ex(*args, **kw)
    for sm_scale in (SOFTMAX_SCALE, 0.3):
        scales[2] = sm_scale
        g.replay()
        torch.cuda.synchronize()
        ref_o, ref_l = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=1,
                                          num_heads=12, causal=False, softmax_scale=sm_scale)
        assert_parity(out, lse, ref_o, ref_l, what=f"softmax_scale {sm_scale}")
    mla.mla_decode_status(ws, stream)


# Negative and zero scales on every FP8 kernel configuration (12 rows -> the
# 16-row CTA, 20 -> 32, 40 -> 48, 96 -> the 96-row CTA, whose softmax keeps
# scores unscaled and applies the scale's sign and magnitude separately).
@pytest.mark.parametrize("H,q_len,causal", [(12, 1, False), (20, 1, False), (10, 4, True),
                                            (12, 8, True)])
@pytest.mark.parametrize("scales", [
    dict(softmax_scale=-SOFTMAX_SCALE),
    dict(softmax_scale=0.0),
    dict(softmax_scale=SOFTMAX_SCALE, q_scale=-1.3, kv_scale=0.6),
    dict(softmax_scale=0.09, q_scale=1.1, kv_scale=-0.7),
])
def test_negative_and_zero_scales(H, q_len, causal, scales):
    lens = [3000, 1100]
    inp = decode_inputs(2, H, q_len, lens, seed=60 + H + q_len)
    q, kv, pt = _dev(inp)
    for target in (0, 6):
        plan = mla.mla_decode_plan(lens, H, q_len, target_ctas=target) if target else None
        out, lse, _ = mla.decode(q, kv, pt, inp.kv_lens, num_heads=H, q_len=q_len,
                                 causal=causal, plan=plan, **scales)
        torch.cuda.synchronize()
        ref_o, ref_l = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens,
                                          q_len=q_len, num_heads=H, causal=causal, **scales)
        assert_parity(out, lse, ref_o, ref_l)
