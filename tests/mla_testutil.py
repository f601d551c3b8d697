"""Shared helpers for the GPU parity tests (compare the CUDA path to the oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import split_kv_mla_paged_gb300 as mla

# Parity tolerances of the decode: per element of O,
# |err| <= 1e-2 * max|O_ref| + 2e-3 (BF16 store); LSE within 1e-4 absolute;
# different split plans agree within 1e-5 in fp32 before the store.
O_REL = 1e-2
O_ABS = 2e-3
LSE_ABS = 1e-4
PLAN_ABS = 1e-5


def run_decode(inp, causal, softmax_scale, *, plan=None, target_ctas=0, kv_split=None,
               q_scale=1.0, kv_scale=1.0):
    dev = torch.device("cuda")
    q = inp.q.to(dev)
    kv = inp.kv.to(dev)
    pt = inp.page_table.to(dev)
    out, lse, out_f32 = mla.decode(q, kv, pt, inp.kv_lens, num_heads=inp.num_heads,
                                   q_len=inp.q_len, causal=causal, softmax_scale=softmax_scale,
                                   q_scale=q_scale, kv_scale=kv_scale, plan=plan,
                                   target_ctas=target_ctas, kv_split=kv_split, want_f32=True)
    torch.cuda.synchronize()
    return out, lse, out_f32


def oracle_rows(inp, rows, causal, softmax_scale, q_scale=1.0, kv_scale=1.0):
    """Oracle on selected flat rows.  Copies only the needed requests' pages."""
    rows = np.asarray(rows, dtype=np.int64)
    H, q_len = inp.num_heads, inp.q_len
    per_req = H * q_len
    out = np.zeros((len(rows), 512))
    lse = np.zeros((len(rows),))
    reqs = sorted(set((rows // per_req).tolist()))
    for b in reqs:
        sel = np.nonzero(rows // per_req == b)[0]
        L = int(inp.kv_lens[b])
        n_pages = (L + 31) // 32
        pages = inp.page_table[b, :n_pages].to(torch.int64)
        kv_b = inp.kv[pages.to(inp.kv.device)].cpu()
        table = torch.arange(n_pages, dtype=torch.int32)[None, :]
        q_b = inp.q[b:b + 1].cpu()
        local = rows[sel] - b * per_req
        o, l = oracle.decode_rows(q_b, kv_b, table, torch.tensor([L], dtype=torch.int32),
                                  q_len=q_len, num_heads=H, causal=causal,
                                  softmax_scale=softmax_scale, q_scale=q_scale,
                                  kv_scale=kv_scale, rows=local)
        out[sel] = o
        lse[sel] = l
    return out, lse


def assert_parity(out_bf16, lse, out_ref, lse_ref, what="", o_tol=None):
    """Element-wise check of the BF16 output and fp32 LSE against the oracle."""
    o = out_bf16.float().cpu().numpy().reshape(out_ref.shape).astype(np.float64)
    l = lse.cpu().numpy().reshape(lse_ref.shape).astype(np.float64)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    tol = O_REL * np.max(np.abs(out_ref)) + O_ABS if o_tol is None else o_tol
    err = np.abs(o - out_ref)
    worst = float(err.max())
    assert worst <= tol, f"{what}: max |O err| {worst:.3e} > tol {tol:.3e}"
    lerr = float(np.max(np.abs(l - lse_ref)))
    assert lerr <= LSE_ABS, f"{what}: max |LSE err| {lerr:.3e} > {LSE_ABS}"
    return worst, lerr

