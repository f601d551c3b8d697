"""Pins for the fp64 oracle, checked against things other than itself.

Each test names what fixes the expected value: a library routine (torch's
float8 widening, torch's float64 attention), a closed form, or an invariance
of the method (split-KV is an exact refactoring of softmax; pages are only an
indirection; the MTP-verify mask truncates the key range).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from synth import (HEAD_DIM, LATENT_DIM, PAGE_SIZE, SOFTMAX_SCALE, decode_inputs, kv_windows,
                   merge_partials, page_selection, query_lens_ragged)


def _gather_keys(inp, b):
    """Dense [L, 576] uint8 keys of request b, gathered page by page in Python."""
    L = int(inp.kv_lens[b])
    pages = inp.page_table[b].cpu()
    rows = []
    for j in range(L):
        rows.append(inp.kv[int(pages[j // PAGE_SIZE]), j % PAGE_SIZE])
    return torch.stack(rows) if rows else torch.empty((0, HEAD_DIM), dtype=torch.uint8)


def _widen(u8):
    return u8.view(torch.float8_e4m3fn).to(torch.float64)


# --- (1) E4M3 codec ---------------------------------------------------------

def test_e4m3_all_codes_match_torch_widening():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], ref[~nan])
    # Signed zero is kept.
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_e4m3_landmarks():
    # Largest finite, smallest normal, smallest subnormal and one (E4M3 "FN").
    assert oracle.e4m3_decode(np.array([0x7E]))[0] == 448.0
    assert oracle.e4m3_decode(np.array([0x08]))[0] == 2.0 ** -6
    assert oracle.e4m3_decode(np.array([0x01]))[0] == 2.0 ** -9
    assert oracle.e4m3_decode(np.array([0x38]))[0] == 1.0
    assert oracle.e4m3_decode(np.array([0xB8]))[0] == -1.0


def test_e4m3_widening_to_bf16_is_exact():
    # "Sparse MLA decode" page: widening E4M3 to BF16 loses nothing.
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    finite = ~np.isnan(vals)
    bf = torch.from_numpy(vals[finite]).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(bf, vals[finite])


# --- (2) single key, (3) equal scores --------------------------------------

@pytest.mark.parametrize("q_scale,kv_scale", [(1.0, 1.0), (0.5, 2.0)])
def test_single_key_returns_v(q_scale, kv_scale):
    inp = decode_inputs(1, 3, 1, [1], seed=11)
    out, lse = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=1,
                                  num_heads=3, causal=False, softmax_scale=0.3,
                                  q_scale=q_scale, kv_scale=kv_scale)
    k = _widen(inp.kv[int(inp.page_table[0, 0]), 0]) * kv_scale
    for h in range(3):
        q = _widen(inp.q[0, 0, h]) * q_scale
        assert np.array_equal(out[h], k[:LATENT_DIM].numpy())
        assert lse[h] == pytest.approx(0.3 * float(q @ k), abs=1e-12)


def test_equal_scores_give_mean_of_v_and_log_n():
    # Zero latent query: every score comes from the rope dims.  Give every key
    # the same rope part, so every score is equal while V varies.
    inp = decode_inputs(1, 2, 1, [77], seed=12)
    inp.q[..., :LATENT_DIM] = 0
    inp.kv[..., LATENT_DIM:] = inp.kv[0, 0, LATENT_DIM:]
    out, lse = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=1,
                                  num_heads=2, causal=False, softmax_scale=SOFTMAX_SCALE)
    keys = _widen(_gather_keys(inp, 0))
    mean_v = keys[:, :LATENT_DIM].mean(dim=0).numpy()
    for h in range(2):
        s = SOFTMAX_SCALE * float(_widen(inp.q[0, 0, h]) @ keys[0])
        np.testing.assert_allclose(out[h], mean_v, rtol=0, atol=1e-13)
        assert lse[h] == pytest.approx(s + math.log(77), abs=1e-12)


# --- (7) brute force and the two-key closed form ---------------------------

def _sdpa_reference(inp, causal, scale, q_scale=1.0, kv_scale=1.0):
    """Attention through torch's float64 scaled_dot_product_attention."""
    outs, lses = [], []
    B, q_len, H = inp.batch, inp.q_len, inp.num_heads
    for b in range(B):
        keys = _widen(_gather_keys(inp, b)) * kv_scale          # [L, 576]
        L = keys.shape[0]
        q = _widen(inp.q[b]).reshape(q_len * H, HEAD_DIM) * q_scale
        mask = torch.ones((q_len * H, L), dtype=torch.bool)
        if causal:
            for qi in range(q_len):
                mask[qi * H:(qi + 1) * H, L - q_len + qi + 1:] = False
        o = torch.nn.functional.scaled_dot_product_attention(
            q[None, None], keys[None, None], keys[None, None, :, :LATENT_DIM],
            attn_mask=mask[None, None], scale=scale)[0, 0]
        logits = (q @ keys.T) * scale
        logits = logits.masked_fill(~mask, -math.inf)
        outs.append(o)
        lses.append(torch.logsumexp(logits, dim=-1))
    return torch.cat(outs).numpy(), torch.cat(lses).numpy()


@pytest.mark.parametrize("B,H,q_len,lens,causal", [
    (1, 4, 1, [64], False),
    (2, 3, 1, [33, 7], False),
    (2, 2, 4, [40, 9], True),
    (1, 1, 8, [61], True),
])
def test_bruteforce_matches_torch_attention(B, H, q_len, lens, causal):
    inp = decode_inputs(B, H, q_len, lens, seed=13, extra_pages=3)
    out, lse = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=q_len,
                                  num_heads=H, causal=causal, softmax_scale=0.11,
                                  q_scale=1.5, kv_scale=0.75)
    ref_o, ref_lse = _sdpa_reference(inp, causal, 0.11, q_scale=1.5, kv_scale=0.75)
    np.testing.assert_allclose(out, ref_o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_two_key_closed_form():
    inp = decode_inputs(1, 1, 1, [2], seed=14)
    out, lse = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=1,
                                  num_heads=1, causal=False, softmax_scale=0.25)
    q = _widen(inp.q[0, 0, 0]).numpy()
    page = int(inp.page_table[0, 0])
    k0 = _widen(inp.kv[page, 0]).numpy()
    k1 = _widen(inp.kv[page, 1]).numpy()
    s0, s1 = 0.25 * float(q @ k0), 0.25 * float(q @ k1)
    e0, e1 = math.exp(s0), math.exp(s1)
    expect = (e0 * k0[:LATENT_DIM] + e1 * k1[:LATENT_DIM]) / (e0 + e1)
    np.testing.assert_allclose(out[0], expect, rtol=1e-13, atol=1e-15)
    assert lse[0] == pytest.approx(math.log(e0 + e1), abs=1e-13)


# --- (4) split invariance, (5) causal reduction, (6) permutation -----------

@pytest.mark.parametrize("bounds", [[0, 100], [0, 1, 100], [0, 32, 64, 96, 100], [0, 3, 50, 51, 99, 100]])
def test_split_partials_merge_to_unsplit(bounds):
    inp = decode_inputs(1, 3, 2, [100], seed=15)
    kw = dict(q_len=2, num_heads=3, causal=True, softmax_scale=0.2)
    full_o, full_lse = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, **kw)
    parts_o, parts_ml = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        o, m, l = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, tok_begin=a,
                                     tok_end=b, partial=True, **kw)
        parts_o.append(o)
        parts_ml.append(np.stack([m, l], axis=-1))
    po = np.stack(parts_o, axis=1)
    pml = np.stack(parts_ml, axis=1)
    o, lse = oracle.merge(po, pml)
    np.testing.assert_allclose(o, full_o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, full_lse, rtol=0, atol=1e-12)


def test_causal_row_equals_truncated_noncausal():
    L, q_len, H = 70, 8, 2
    inp = decode_inputs(1, H, q_len, [L], seed=16)
    oc, lc = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=q_len,
                                num_heads=H, causal=True, softmax_scale=0.3)
    for qi in range(q_len):
        n = L - q_len + qi + 1
        on, ln = oracle.decode_rows(inp.q, inp.kv, inp.page_table, torch.tensor([n], dtype=torch.int32),
                                    q_len=q_len, num_heads=H, causal=False, softmax_scale=0.3)
        sl = slice(qi * H, (qi + 1) * H)
        np.testing.assert_array_equal(oc[sl], on[sl])
        np.testing.assert_array_equal(lc[sl], ln[sl])


def test_page_permutation_invariance():
    inp = decode_inputs(2, 2, 1, [90, 45], seed=17, extra_pages=2)
    kw = dict(q_len=1, num_heads=2, causal=False, softmax_scale=0.3)
    o1, l1 = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, **kw)
    P = inp.num_pages
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    kv2 = inp.kv[perm]                        # new page i holds old page perm[i]
    pt = inp.page_table.clone()
    valid = pt >= 0
    pt[valid] = inv[pt[valid].long()].to(torch.int32)
    o2, l2 = oracle.decode_rows(inp.q, kv2, pt, inp.kv_lens, **kw)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_scale_placement():
    # q_scale and kv_scale multiply the logits; kv_scale also scales V.
    inp = decode_inputs(1, 2, 1, [50], seed=18)
    kw = dict(q_len=1, num_heads=2, causal=False)
    o1, l1 = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, softmax_scale=0.3,
                                q_scale=2.0, kv_scale=0.5, **kw)
    o2, l2 = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, softmax_scale=0.3,
                                **kw)
    np.testing.assert_allclose(o1, 0.5 * o2, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


# --- merge pins ------------------------------------------------------------

def test_merge_single_slot_and_empty_slots():
    o, ml = merge_partials(rows=5, num_splits=6, seed=3, empty_frac=0.0)
    # Only slot 2 is kept in each row: the merge must return O_2 / l_2.
    ml_one = ml.copy()
    o_one = o.copy()
    keep = 2
    for s in range(6):
        if s != keep:
            ml_one[:, s, 0] = -np.inf
            ml_one[:, s, 1] = 0.0
            o_one[:, s, :] = 0.0
    out, lse = oracle.merge(o_one, ml_one)
    np.testing.assert_allclose(out, o[:, keep, :].astype(np.float64) / ml[:, keep, 1:2], rtol=1e-15)
    expect_lse = math.log(2.0) * ml[:, keep, 0].astype(np.float64) + np.log(ml[:, keep, 1].astype(np.float64))
    np.testing.assert_allclose(lse, expect_lse, rtol=0, atol=1e-12)


def test_merge_all_empty_row():
    o, ml = merge_partials(rows=3, num_splits=4, seed=4, all_empty_rows=[1])
    out, lse = oracle.merge(o, ml)
    assert np.all(out[1] == 0.0) and lse[1] == -np.inf
    assert np.all(np.isfinite(out[[0, 2]]))


def test_merge_equals_pairwise_combination():
    # Merging three slots at once equals merging two, then the third: the
    # closed form is associative.  Written through the partial convention
    # (m, l, O) -> (m, l, O) of two merged slots, with no reference to the
    # oracle's own code.
    o, ml = merge_partials(rows=4, num_splits=3, seed=5, empty_frac=0.0)
    out3, lse3 = oracle.merge(o, ml)
    m0, l0 = ml[:, 0, 0].astype(np.float64), ml[:, 0, 1].astype(np.float64)
    m1, l1 = ml[:, 1, 0].astype(np.float64), ml[:, 1, 1].astype(np.float64)
    mm = np.maximum(m0, m1)
    a0, a1 = np.exp2(m0 - mm), np.exp2(m1 - mm)
    o01 = a0[:, None] * o[:, 0] + a1[:, None] * o[:, 1]
    l01 = a0 * l0 + a1 * l1
    o2 = np.stack([o01, o[:, 2].astype(np.float64)], axis=1)
    ml2 = np.stack([np.stack([mm, l01], -1), ml[:, 2].astype(np.float64)], axis=1)
    out2, lse2 = oracle.merge(o2, ml2)
    np.testing.assert_allclose(out3, out2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse3, lse2, rtol=0, atol=1e-12)


# --- KV append: E4M3 encoder ----------------------------------------------

def test_e4m3_encode_roundtrips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    enc = oracle.e4m3_encode(vals)
    # -0.0 encodes to 0x80, +0.0 to 0x00: every code comes back.
    assert np.array_equal(enc, codes)


def test_e4m3_encode_matches_torch_cast_in_range():
    g = torch.Generator().manual_seed(21)
    x = (torch.randn(20000, generator=g) * torch.exp2(torch.randint(-12, 9, (20000,), generator=g)))
    x = x.clamp(-440, 440).to(torch.float32)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x.numpy()), ref)


def test_e4m3_encode_ties_go_to_even_and_saturate():
    # 1.0 + 1/16 lies halfway between 1.0 (0x38) and 1.125 (0x39): even code wins.
    assert oracle.e4m3_encode(np.array([1.0625], np.float32))[0] == 0x38
    # 1.125 + 1/16 lies between 0x39 and 0x3A: 0x3A is even.
    assert oracle.e4m3_encode(np.array([1.1875], np.float32))[0] == 0x3A
    # Halfway between the two smallest subnormals 2^-9 and 2^-8: 0x02 is even.
    assert oracle.e4m3_encode(np.array([1.5 * 2.0 ** -9], np.float32))[0] == 0x02
    assert oracle.e4m3_encode(np.array([1000.0, -1e30], np.float32)).tolist() == [0x7E, 0xFE]
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F


def test_kv_append_scatters_through_page_table():
    pool = np.full((5, 32, 576), 0x7F, dtype=np.uint8)
    table = np.array([[3, 1], [0, 4]], dtype=np.int32)
    g = torch.Generator().manual_seed(22)
    rows = (torch.randn(3, 576, generator=g)).to(torch.bfloat16)
    req = np.array([0, 0, 1], np.int32)
    pos = np.array([0, 33, 40], np.int32)
    new, st = oracle.kv_append(rows, req, pos, table, pool, kv_scale=0.5)
    assert st == 0
    want = (rows.float() / 0.5).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(new[3, 0], want[0])
    assert np.array_equal(new[1, 1], want[1])
    assert np.array_equal(new[4, 8], want[2])
    touched = {(3, 0), (1, 1), (4, 8)}
    for pg in range(5):
        for sl in range(32):
            if (pg, sl) not in touched:
                assert np.all(new[pg, sl] == 0x7F)
    _, st = oracle.kv_append(rows[:1], np.array([2], np.int32), np.array([0], np.int32), table,
                             pool, kv_scale=1.0)
    assert st == -1


# --- sinks and output scale --------------------------------------------------

def test_sink_at_minus_infinity_changes_nothing_and_output_scale_is_linear():
    inp = decode_inputs(1, 3, 2, [90], seed=23)
    kw = dict(q_len=2, num_heads=3, causal=True, softmax_scale=0.2)
    o1, l1 = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, **kw)
    o2, l2 = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens,
                                sinks=np.full(3, -np.inf), output_scale=2.5, **kw)
    np.testing.assert_array_equal(l1, l2)
    np.testing.assert_allclose(o2, 2.5 * o1, rtol=1e-15, atol=0)


def test_sink_single_key_closed_form():
    inp = decode_inputs(1, 2, 1, [1], seed=24)
    sinks = np.array([0.3, -1.7])
    o, l = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=1, num_heads=2,
                              causal=False, softmax_scale=0.25, sinks=sinks)
    k = _widen(inp.kv[int(inp.page_table[0, 0]), 0]).numpy()
    for h in range(2):
        s0 = 0.25 * float(_widen(inp.q[0, 0, h]).numpy() @ k)
        w = math.exp(s0) / (math.exp(s0) + math.exp(sinks[h]))
        np.testing.assert_allclose(o[h], w * k[:LATENT_DIM], rtol=1e-13, atol=1e-15)
        assert l[h] == pytest.approx(math.log(math.exp(s0) + math.exp(sinks[h])), abs=1e-13)


def test_sink_equal_scores_mean_shrinks():
    inp = decode_inputs(1, 1, 1, [40], seed=25)
    inp.q[..., :LATENT_DIM] = 0
    inp.kv[..., LATENT_DIM:] = inp.kv[0, 0, LATENT_DIM:]
    keys = _widen(_gather_keys(inp, 0))
    s = SOFTMAX_SCALE * float(_widen(inp.q[0, 0, 0]) @ keys[0])
    sink = s + math.log(10.0)  # the sink weighs as much as 10 keys
    o, l = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=1, num_heads=1,
                              causal=False, softmax_scale=SOFTMAX_SCALE, sinks=np.array([sink]))
    np.testing.assert_allclose(o[0], keys[:, :LATENT_DIM].mean(0).numpy() * 40 / 50, rtol=1e-12,
                               atol=1e-15)
    assert l[0] == pytest.approx(s + math.log(50.0), abs=1e-12)


# --- BF16 KV variant -----------------------------------------------------------

@pytest.mark.parametrize("B,H,q_len,lens,causal", [(1, 4, 1, [64], False), (2, 2, 4, [40, 9], True)])
def test_bf16_oracle_matches_torch_attention(B, H, q_len, lens, causal):
    inp = decode_inputs(B, H, q_len, lens, seed=26, extra_pages=2, dtype="bf16")
    out, lse = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=q_len,
                                  num_heads=H, causal=causal, softmax_scale=0.11)
    outs, lses = [], []
    for b in range(B):
        L = int(inp.kv_lens[b])
        keys = torch.stack([inp.kv[int(inp.page_table[b, j // PAGE_SIZE]), j % PAGE_SIZE]
                            for j in range(L)]).to(torch.float64)
        q = inp.q[b].reshape(q_len * H, HEAD_DIM).to(torch.float64)
        mask = torch.ones((q_len * H, L), dtype=torch.bool)
        if causal:
            for qi in range(q_len):
                mask[qi * H:(qi + 1) * H, L - q_len + qi + 1:] = False
        outs.append(torch.nn.functional.scaled_dot_product_attention(
            q[None, None], keys[None, None], keys[None, None, :, :LATENT_DIM],
            attn_mask=mask[None, None], scale=0.11)[0, 0])
        lses.append(torch.logsumexp(((q @ keys.T) * 0.11).masked_fill(~mask, -math.inf), -1))
    np.testing.assert_allclose(out, torch.cat(outs).numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, torch.cat(lses).numpy(), rtol=1e-12, atol=1e-12)


# --- Restricted key sets: ragged q, key windows, page selection ----------------
#
# Readings of the run() arguments is_var_q/query_lens and kv_bounds (issue
# #20510, "Repro 1") and of the sparse decode over selected pages (PR #17441):
# query_lens[b] real query tokens in the first slots of the padded q_len block
# (the request's last positions), a key window [lo, hi), and a set of logical
# pages.  Pinned against torch's float64 attention with the visibility mask
# written from those definitions, and against the unrestricted oracle on
# caches rebuilt to hold only the visible keys.

def _visible(L, q_b, qi, causal, window, pages):
    """Boolean [L] visibility of keys for query slot qi (test-side definition)."""
    j = torch.arange(L)
    vis = torch.full((L,), qi < q_b, dtype=torch.bool)
    if causal:
        vis &= j <= L - q_b + qi
    if window is not None:
        vis &= (j >= int(window[0])) & (j < int(window[1]))
    if pages is not None:
        sel = torch.zeros(((L + PAGE_SIZE - 1) // PAGE_SIZE,), dtype=torch.bool)
        for p in pages:
            if p >= 0:
                sel[int(p)] = True
        vis &= sel[j // PAGE_SIZE]
    return vis


def _restricted_reference(inp, causal, scale, qlens=None, windows=None, sel=None):
    outs, lses = [], []
    B, q_len, H = inp.batch, inp.q_len, inp.num_heads
    for b in range(B):
        keys = _widen(_gather_keys(inp, b))
        L = keys.shape[0]
        q = _widen(inp.q[b]).reshape(q_len * H, HEAD_DIM)
        q_b = q_len if qlens is None else int(qlens[b])
        for qi in range(q_len):
            vis = _visible(L, q_b, qi, causal, None if windows is None else windows[b],
                           None if sel is None else sel[b])
            for h in range(H):
                if not bool(vis.any()):
                    outs.append(torch.zeros(LATENT_DIM, dtype=torch.float64))
                    lses.append(torch.tensor(-math.inf, dtype=torch.float64))
                    continue
                qr = q[qi * H + h]
                o = torch.nn.functional.scaled_dot_product_attention(
                    qr[None, None, None], keys[None, None], keys[None, None, :, :LATENT_DIM],
                    attn_mask=vis[None, None, None], scale=scale)[0, 0, 0]
                logits = ((keys @ qr) * scale).masked_fill(~vis, -math.inf)
                outs.append(o)
                lses.append(torch.logsumexp(logits, dim=0))
    return torch.stack(outs).numpy(), torch.stack(lses).numpy()


@pytest.mark.parametrize("kind", ["query_lens", "window", "pages", "all"])
@pytest.mark.parametrize("causal", [False, True])
def test_restricted_keys_match_torch_attention(kind, causal):
    lens = [77, 130, 41]
    inp = decode_inputs(3, 2, 4, lens, seed=31, extra_pages=2)
    ql = query_lens_ragged(3, 4, seed=5) if kind in ("query_lens", "all") else None
    win = kv_windows(lens, seed=6, full_every=0) if kind in ("window", "all") else None
    sel = page_selection(lens, 3, seed=7, keep_last=False) if kind in ("pages", "all") else None
    out, lse = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=4,
                                  num_heads=2, causal=causal, softmax_scale=0.2,
                                  query_lens=ql, kv_bounds=win, block_idx=sel)
    ref_o, ref_l = _restricted_reference(inp, causal, 0.2, ql, win, sel)
    np.testing.assert_allclose(out, ref_o, rtol=1e-12, atol=1e-12)
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], ref_l[fin], rtol=1e-12, atol=1e-12)


def test_query_lens_padding_rows_are_empty_and_sinks_fill_them():
    inp = decode_inputs(2, 3, 4, [50, 60], seed=32)
    ql = [2, 4]
    sinks = np.array([0.5, -1.0, 2.0])
    out, lse = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=4,
                                  num_heads=3, causal=True, softmax_scale=0.2, query_lens=ql,
                                  sinks=sinks)
    rows = np.arange(2 * 4 * 3)
    qi = (rows // 3) % 4
    b = rows // 12
    pad = qi >= np.array(ql)[b]
    assert pad.sum() == 2 * 3
    # A row that sees no key is the sink alone: O = 0, LSE = the sink logit.
    assert np.all(out[pad] == 0.0)
    np.testing.assert_array_equal(lse[pad], sinks[rows[pad] % 3])


def _repaged(inp, b, tokens):
    """A one-request cache holding the given token positions of request b, in
    order, packed from position 0 (pages filled in order)."""
    keys = _gather_keys(inp, b)[tokens]
    n = keys.shape[0]
    n_pages = (n + PAGE_SIZE - 1) // PAGE_SIZE
    pool = torch.zeros((n_pages, PAGE_SIZE, HEAD_DIM), dtype=torch.uint8)
    pool.view(-1, HEAD_DIM)[:n] = keys
    table = torch.arange(n_pages, dtype=torch.int32)[None, :]
    return pool, table, n


@pytest.mark.parametrize("causal", [False, True])
def test_trailing_window_equals_cache_of_the_window(causal):
    # A window [lo, L) equals attention over a cache that holds only those keys
    # (the causal limit moves with the end of the cache).
    inp = decode_inputs(1, 2, 3, [150], seed=33)
    lo = 37
    out, lse = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=3,
                                  num_heads=2, causal=causal, softmax_scale=0.2,
                                  kv_bounds=[[lo, 150]])
    pool, table, n = _repaged(inp, 0, torch.arange(lo, 150))
    ref_o, ref_l = oracle.decode_rows(inp.q, pool, table, [n], q_len=3, num_heads=2,
                                      causal=causal, softmax_scale=0.2)
    np.testing.assert_allclose(out, ref_o, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-13, atol=1e-13)


def test_page_selection_equals_gathered_cache():
    # Selected pages (ascending, last page partial) equal attention over a cache
    # made of those pages alone.
    lens = [300]
    inp = decode_inputs(1, 3, 1, lens, seed=34)
    sel = np.array([[1, 4, 5, 9]], dtype=np.int32)  # page 9 holds tokens 288..299
    out, lse = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=1,
                                  num_heads=3, causal=False, softmax_scale=0.2, block_idx=sel)
    toks = torch.cat([torch.arange(p * PAGE_SIZE, min((p + 1) * PAGE_SIZE, 300))
                      for p in sel[0]])
    pool, table, n = _repaged(inp, 0, toks)
    ref_o, ref_l = oracle.decode_rows(inp.q, pool, table, [n], q_len=1, num_heads=3,
                                      causal=False, softmax_scale=0.2)
    np.testing.assert_allclose(out, ref_o, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-13, atol=1e-13)
    # Unused (-1) slots and a repeated page change nothing.
    sel2 = np.array([[1, 4, 4, 5, 9, -1, -1]], dtype=np.int32)
    out2, lse2 = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=1,
                                    num_heads=3, causal=False, softmax_scale=0.2, block_idx=sel2)
    np.testing.assert_array_equal(out2, out)
    np.testing.assert_array_equal(lse2, lse)


def test_window_split_partials_merge_to_the_window():
    # Split invariance holds on a restricted key set too: partials over two
    # halves of the token range merge to the whole.
    inp = decode_inputs(1, 2, 1, [260], seed=35)
    win = [[50, 230]]
    o_all, l_all = oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=1,
                                      num_heads=2, causal=False, softmax_scale=0.2,
                                      kv_bounds=win)
    parts = [oracle.decode_rows(inp.q, inp.kv, inp.page_table, inp.kv_lens, q_len=1,
                                num_heads=2, causal=False, softmax_scale=0.2, kv_bounds=win,
                                tok_begin=a, tok_end=e, partial=True)
             for a, e in ((0, 128), (128, 260))]
    po = np.stack([p[0] for p in parts], axis=1)
    pml = np.stack([np.stack([p[1], p[2]], axis=-1) for p in parts], axis=1)
    o, l = oracle.merge(po, pml)
    np.testing.assert_allclose(o, o_all, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l, l_all, rtol=1e-12, atol=1e-12)
