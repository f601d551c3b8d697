"""GPU: the FP8 paged KV append (through the C ABI) against the oracle, byte
for byte, and a decode over an appended cache against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import split_kv_mla_paged_gb300 as mla
from split_kv_mla_paged_gb300 import build as mla_build
from synth import SOFTMAX_SCALE, decode_inputs
from mla_testutil import assert_parity, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mla_build.build()
    mla.load_library()


def _append(rows, req, pos, table, pool, kv_scale):
    dev = torch.device("cuda")
    kv_d = torch.from_numpy(pool).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    rq = torch.from_numpy(req).to(dev)
    ps = torch.from_numpy(pos).to(dev)
    pt = torch.from_numpy(table).to(dev)
    rows_d = rows.to(dev).contiguous()
    mla.mla_kv_append(rows_d, rows.shape[0], rq, ps, pt, table.shape[1], table.shape[0], kv_d,
                      pool.shape[0], kv_scale, st)
    torch.cuda.synchronize()
    return kv_d.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("kv_scale", [1.0, 0.37, 4.0, 0.125, -2.0, 3.0e-5])
def test_append_bytes_match_oracle(kv_scale):
    g = torch.Generator().manual_seed(41)
    n_pages, batch = 40, 3
    pool = np.full((n_pages, 32, 576), 0x7F, dtype=np.uint8)
    table = np.random.default_rng(41).permutation(n_pages).astype(np.int32)[:36].reshape(3, 12)
    req = np.repeat(np.arange(batch, dtype=np.int32), 97)
    pos = np.concatenate([np.random.default_rng(b).permutation(12 * 32)[:97] for b in range(3)])
    pos = pos.astype(np.int32)
    # Values spanning E4M3's range: normals, subnormals, saturating ones.
    mag = torch.exp2(torch.randint(-14, 10, (req.size, 576), generator=g).float())
    rows = (torch.randn(req.size, 576, generator=g) * mag).to(torch.bfloat16)
    got, st = _append(rows, req, pos, table, pool, kv_scale)
    want, st_o = oracle.kv_append(rows, req, pos, table, pool, kv_scale)
    assert st == 0 and st_o == 0
    assert np.array_equal(got, want)


# Scales for each way the kernel forms x / kv_scale: powers of two (a
# multiplication), positive scales in [2^-32, 2^32] (reciprocal and one
# correction) and the rest (the IEEE division).
ALL_MODE_SCALES = [1.0, 4.0, -2.0, 2.0 ** -20,
                   0.37, 3.0e-5, 1.0 / 448.0, 0.1, 1.5 * 2.0 ** -32, 1.3 * 2.0 ** 31,
                   -0.37, 1.0e-12, 1.0e12]


@pytest.mark.parametrize("kv_scale", ALL_MODE_SCALES)
def test_append_every_bf16_pattern(kv_scale):
    # All 65,536 BF16 bit patterns (zeros, subnormals, +-inf, NaN included):
    # the codes equal the oracle's (IEEE fp32 quotient, then E4M3).
    bits = np.zeros(114 * 576, dtype=np.uint16)
    bits[:65536] = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    rows = torch.from_numpy(bits.view(np.int16).reshape(114, 576)).view(torch.bfloat16)
    pool = np.full((4, 32, 576), 0x55, dtype=np.uint8)
    table = np.array([[2, 0, 3, 1]], dtype=np.int32)
    req = np.zeros(114, np.int32)
    pos = np.arange(114, dtype=np.int32)
    got, st = _append(rows, req, pos, table, pool, kv_scale)
    want, st_o = oracle.kv_append(rows, req, pos, table, pool, kv_scale)
    assert st == 0 and st_o == 0
    assert np.array_equal(got, want)


def test_append_reports_bad_targets_and_skips_them():
    pool = np.full((4, 32, 576), 0x7F, dtype=np.uint8)
    table = np.array([[0, 1], [2, 99]], dtype=np.int32)
    rows = torch.randn(3, 576, generator=torch.Generator().manual_seed(42)).to(torch.bfloat16)
    req = np.array([0, 1, 5], np.int32)
    pos = np.array([3, 40, 0], np.int32)  # row 1 hits page id 99, row 2 request 5
    got, st = _append(rows, req, pos, table, pool, 1.0)
    assert st == mla.MLA_ERR_INVALID_ARG
    want, _ = oracle.kv_append(rows[:1], req[:1], pos[:1], table, pool, 1.0)
    assert np.array_equal(got, want)


def test_decode_over_appended_cache():
    # Build a cache by appending, then decode it: same result as the oracle
    # on the appended bytes.
    base = decode_inputs(2, 12, 2, [700, 333], seed=43, extra_pages=2)
    L = base.kv_lens.tolist()
    g = torch.Generator().manual_seed(44)
    req = np.concatenate([np.full(n, b, np.int32) for b, n in enumerate(L)])
    pos = np.concatenate([np.arange(n, dtype=np.int32) for n in L])
    rows = (torch.randn(req.size, 576, generator=g) * 0.8).to(torch.bfloat16)
    kv, st = _append(rows, req, pos, base.page_table.numpy(), base.kv.numpy(), 0.5)
    assert st == 0
    base.kv = torch.from_numpy(kv)
    out, lse, _ = run_decode(base, True, SOFTMAX_SCALE, kv_scale=0.5)
    ref_o, ref_l = oracle.decode_rows(base.q, base.kv, base.page_table, base.kv_lens, q_len=2,
                                      num_heads=12, causal=True, softmax_scale=SOFTMAX_SCALE,
                                      kv_scale=0.5)
    assert_parity(out, lse, ref_o, ref_l)
