"""Seeded randomized parity sweep of the BF16-KV decode against the oracle:
random shapes (heads, query tokens, batch, lengths with ragged tails) on both
BF16 kernels (16-row groups with Q in TMEM; 32/48-row groups with 128-token
tiles released block by block), split plans (the pages' targets and the
GB300 planner, with and without the CTA item list) and options (sinks, output
scale, ragged q, key windows, page selections).  Every case is small enough
for the oracle."""
import numpy as np
import pytest
import torch

import oracle
import split_kv_mla_paged_gb300 as mla
from split_kv_mla_paged_gb300 import build as mla_build
from synth import PAGE_SIZE, decode_inputs, kv_windows, page_selection, query_lens_ragged
from mla_testutil import assert_parity

pytestmark = pytest.mark.gpu

N_CASES = 40


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mla_build.build()
    mla.load_library()
    yield
    torch.cuda.synchronize()


def _case(seed):
    g = np.random.default_rng(5000 + seed)
    H = int(g.choice([1, 4, 8, 12, 16, 24]))
    q_len = int(g.choice([1, 2, 4, 8]))
    while H * q_len > 96:
        q_len //= 2
    q_len = max(q_len, 1)
    B = int(g.integers(1, 5))
    lens = [int(x) for x in g.integers(max(q_len, 1), 2500, size=B)]
    causal = bool(q_len > 1 and g.random() < 0.7)
    opts = {}
    if g.random() < 0.25:
        opts["sinks"] = g.normal(0, 2, size=H)
    if g.random() < 0.25:
        opts["output_scale"] = float(g.uniform(0.25, 3))
    if q_len > 1 and g.random() < 0.3:
        opts["query_lens"] = np.asarray(query_lens_ragged(B, q_len, seed=seed), np.int32)
    if g.random() < 0.3:
        opts["kv_bounds"] = kv_windows(lens, seed=seed)
    if g.random() < 0.3:
        topk = int(g.integers(1, 30))
        opts["block_idx"] = page_selection(lens, topk, seed=seed, keep_last=bool(g.random() < 0.5))
    plan_kind = str(g.choice(["gb300", "target"]))
    target = int(g.integers(1, 60))
    scale = float(g.uniform(0.03, 0.3))
    return H, q_len, B, lens, causal, opts, plan_kind, target, scale


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_bf16_case(seed):
    H, q_len, B, lens, causal, opts, plan_kind, target, scale = _case(seed)
    inp = decode_inputs(B, H, q_len, lens, seed=seed, extra_pages=1, dtype="bf16")
    sel = opts.get("block_idx")
    plan_lens = lens if sel is None else [PAGE_SIZE * sel.shape[1]] * B
    if plan_kind == "gb300":
        plan = mla.mla_decode_plan(plan_lens, H, q_len, sm_count=152)
    else:
        plan = mla.mla_decode_plan(plan_lens, H, q_len, target_ctas=target)
    dev = torch.device("cuda")
    results = []
    for use_items in (False, True):
        out, lse, o32 = mla.decode(inp.q.to(dev), inp.kv.to(dev), inp.page_table.to(dev),
                                   inp.kv_lens, num_heads=H, q_len=q_len, causal=causal,
                                   softmax_scale=scale, plan=plan, want_f32=True,
                                   use_items=use_items, **opts)
        torch.cuda.synchronize()
        results.append((out, lse, o32))
    # The item list launches the same CTAs: the same numbers.
    assert torch.equal(results[0][2], results[1][2]) and torch.equal(results[0][1], results[1][1])
    ref_o, ref_l = oracle.decode_rows(inp.q, inp.kv.cpu(), inp.page_table.cpu(), inp.kv_lens,
                                      q_len=q_len, num_heads=H, causal=causal,
                                      softmax_scale=scale, **opts)
    out, lse, o32 = results[0]
    fin = np.isfinite(ref_l)
    lse_np = lse.cpu().numpy().reshape(-1)
    assert np.array_equal(np.isfinite(lse_np), fin), "empty-row pattern"
    o = out.reshape(-1, 512)
    if (~fin).any():
        assert torch.all(o[torch.from_numpy(~fin).cuda()] == 0)
    if fin.any():
        assert_parity(o[torch.from_numpy(fin).cuda()], lse.reshape(-1)[torch.from_numpy(fin).cuda()],
                      ref_o[fin], ref_l[fin], what=f"case {seed}")
    assert torch.equal(o32.to(torch.bfloat16), out)
