"""GPU: an options call split into its two phases (mla_decode_options_t.phases:
the split-KV kernel, then the merge, enqueued one after the other on one
stream) writes the same bytes as the whole call, on the FP8 grid, item-list,
persistent, sparse, BF16 and BF16 sparse paths, for batches that mix one-split
and many-split requests."""
import numpy as np
import pytest
import torch

import split_kv_mla_paged_gb300 as mla
from split_kv_mla_paged_gb300 import build as mla_build
from synth import PAGE_SIZE, SOFTMAX_SCALE, decode_inputs, page_selection

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mla_build.build()
    mla.load_library()


def _run(kind, inp, lens, H, q_len, causal, sel, phase_seq):
    dev = torch.device("cuda")
    q, kv, pt = inp.q.to(dev), inp.kv.to(dev), inp.page_table.to(dev)
    B = len(lens)
    sparse = kind.endswith("sparse")
    bf16 = kind.startswith("bf16")
    plan_lens = [PAGE_SIZE * sel.shape[1]] * B if sparse else lens
    plan = mla.mla_decode_plan(plan_lens, H, q_len, sm_count=152)
    ws_bytes = mla.mla_decode_workspace_size(B, q_len, H, plan.max_splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    mla.mla_decode_workspace_init(ws, ws_bytes)
    out = torch.full((B, q_len, H, 512), 7.0, dtype=torch.bfloat16, device=dev)
    lse = torch.full((B, q_len, H), 7.0, dtype=torch.float32, device=dev)
    o32 = torch.full((B, q_len, H, 512), 7.0, dtype=torch.float32, device=dev)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev)
    splits_d = torch.from_numpy(plan.splits).to(dev)
    chunks_d = torch.from_numpy(plan.chunks).to(dev)
    items = torch.from_numpy(mla.mla_decode_plan_items(plan.splits, H, q_len, bf16=bf16)).to(dev)
    sel_d = None if sel is None else torch.from_numpy(sel).to(dev)
    common = (q, kv, kv.shape[0], pt, pt.shape[1], lens_d, splits_d, chunks_d, plan.max_splits,
              plan.kv_split, B, q_len, H, causal)
    for ph in phase_seq:
        if kind == "fp8_items":
            mla.mla_decode_ex(*common, 1.0, 1.0, SOFTMAX_SCALE, ws, ws_bytes, out, lse, o32,
                              cta_items=items, phases=ph)
        elif kind == "fp8_persistent":
            mla.mla_decode_ex(*common, 1.0, 1.0, SOFTMAX_SCALE, ws, ws_bytes, out, lse, o32,
                              cta_items=items, persistent_ctas=16, phases=ph)
        elif kind == "fp8_grid":
            mla.mla_decode_ex(*common, 1.0, 1.0, SOFTMAX_SCALE, ws, ws_bytes, out, lse, o32,
                              output_scale=0.5, phases=ph)
        elif kind == "fp8_sparse":
            mla.mla_decode_sparse(*common[:6], sel_d, sel.shape[1], *common[6:], 1.0, 1.0,
                                  SOFTMAX_SCALE, ws, ws_bytes, out, lse, o32, phases=ph)
        elif kind == "bf16":
            mla.mla_decode_bf16_ex(*common, SOFTMAX_SCALE, ws, ws_bytes, out, lse, o32,
                                   cta_items=items, phases=ph)
        else:
            mla.mla_decode_bf16_sparse(*common[:6], sel_d, sel.shape[1], *common[6:],
                                       SOFTMAX_SCALE, ws, ws_bytes, out, lse, o32, phases=ph)
    torch.cuda.synchronize()
    mla.mla_decode_status(ws)
    return plan, out, lse, o32


@pytest.mark.parametrize("kind", ["fp8_grid", "fp8_items", "fp8_persistent", "fp8_sparse", "bf16",
                                  "bf16_sparse"])
@pytest.mark.parametrize("H,q_len,lens", [
    (12, 1, [9000, 100, 3000]),
    (12, 8, [6000, 200]),
])
def test_split_then_merge_is_the_whole_call(kind, H, q_len, lens):
    causal = q_len > 1
    inp = decode_inputs(len(lens), H, q_len, lens, seed=900 + q_len,
                        dtype="bf16" if kind.startswith("bf16") else "e4m3")
    sel = page_selection(lens, 40, seed=901) if kind.endswith("sparse") else None
    plan, *whole = _run(kind, inp, lens, H, q_len, causal, sel, [mla.PHASE_ALL])
    _, *two = _run(kind, inp, lens, H, q_len, causal, sel, [mla.PHASE_SPLIT, mla.PHASE_MERGE])
    assert plan.max_splits > 1 and np.any(plan.splits > 1)
    for a, b in zip(whole, two):
        assert torch.equal(a, b)
    # The split phase alone finishes the one-split requests and leaves the
    # rows of the others to the merge.
    _, out, lse, _ = _run(kind, inp, lens, H, q_len, causal, sel, [mla.PHASE_SPLIT])
    for b, ns in enumerate(plan.splits):
        if ns == 1:
            assert torch.equal(out[b], whole[0][b]) and torch.equal(lse[b], whole[1][b])
        else:
            assert torch.all(out[b] == 7.0) and torch.all(lse[b] == 7.0)
