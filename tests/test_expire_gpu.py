"""The expiry-and-drain path of every split-KV kernel configuration.

Each pipeline wait is bounded; when one runs out the kernel records
MLA_ERR_TIMEOUT in the workspace status word, stops its other roles, lets its
own copies and MMAs finish, frees TMEM and exits, and the context stays usable.
The test hook mla_debug_set_expire makes one chosen wait (role, tile) read as
expired without any real stall, so the path runs in every configuration: the
16/32/48/96-row FP8 kernels and the 16-row (Q in TMEM), 32-row and 48-row
BF16 kernels, for each role whose wait the configuration has.  After each expired
call the next call on the same context must match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import split_kv_mla_paged_gb300 as mla
from split_kv_mla_paged_gb300 import build as mla_build
from synth import SOFTMAX_SCALE, decode_inputs
from mla_testutil import assert_parity

pytestmark = pytest.mark.gpu

STAGE_FREE, TILE_FULL, P_FULL, S_FULL, P_FREE, FINAL = range(6)

# name: (dtype, H, q_len, kv_len, causal, roles with a wait in this configuration)
CONFIGS = {
    "fp8_16rows": ("e4m3", 12, 1, 4000, False, (STAGE_FREE, TILE_FULL, P_FULL, S_FULL, FINAL)),
    "fp8_32rows": ("e4m3", 20, 1, 4000, False, (STAGE_FREE, TILE_FULL, P_FULL, S_FULL, P_FREE,
                                                FINAL)),
    "fp8_48rows": ("e4m3", 10, 4, 4000, True, (STAGE_FREE, TILE_FULL, P_FULL, S_FULL, P_FREE,
                                               FINAL)),
    "fp8_96rows": ("e4m3", 12, 8, 4000, True, (STAGE_FREE, TILE_FULL, P_FULL, S_FULL, P_FREE,
                                               FINAL)),
    "bf16_16rows": ("bf16", 12, 1, 4000, False, (STAGE_FREE, TILE_FULL, P_FULL, S_FULL, FINAL)),
    "bf16_48rows": ("bf16", 12, 4, 4000, True, (STAGE_FREE, TILE_FULL, P_FULL, S_FULL, P_FREE,
                                                FINAL)),
    "bf16_32rows": ("bf16", 16, 2, 4000, True, (STAGE_FREE, TILE_FULL, P_FULL, S_FULL, P_FREE,
                                                FINAL)),
}
CASES = [(name, role) for name, cfg in CONFIGS.items() for role in cfg[5]]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mla_build.build()
    mla.load_library()
    yield
    mla.mla_debug_set_expire(-1)
    torch.cuda.synchronize()


def _inputs(name):
    dtype, H, q_len, L, causal, _ = CONFIGS[name]
    inp = decode_inputs(2, H, q_len, [L, L - 777], seed=700 + H + q_len, dtype=dtype)
    return inp, causal


def _decode(inp, causal, plan):
    dev = torch.device("cuda")
    out, lse, _ = mla.decode(inp.q.to(dev), inp.kv.to(dev), inp.page_table.to(dev), inp.kv_lens,
                             num_heads=inp.num_heads, q_len=inp.q_len, causal=causal,
                             softmax_scale=SOFTMAX_SCALE, plan=plan)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("name,role", CASES)
def test_expired_wait_is_reported_and_the_next_call_is_exact(name, role):
    inp, causal = _inputs(name)
    # Two splits per request, so every CTA runs many tiles past the expired one.
    plan = mla.mla_decode_plan(inp.kv_lens.tolist(), inp.num_heads, inp.q_len, target_ctas=4)
    tile = 0 if role == FINAL else 2
    mla.mla_debug_set_expire(role, tile)
    try:
        with pytest.raises(mla.MlaError) as e:
            _decode(inp, causal, plan)
        assert e.value.status == mla.MLA_ERR_TIMEOUT
    finally:
        mla.mla_debug_set_expire(-1)
    out, lse = _decode(inp, causal, plan)
    ref_o, ref_l = oracle.decode_rows(inp.q, inp.kv.cpu(), inp.page_table.cpu(), inp.kv_lens,
                                      q_len=inp.q_len, num_heads=inp.num_heads, causal=causal,
                                      softmax_scale=SOFTMAX_SCALE)
    assert_parity(out, lse, ref_o, ref_l, what=f"{name} after role {role}")


def test_expire_hook_off_changes_nothing():
    inp, causal = _inputs("fp8_96rows")
    plan = mla.mla_decode_plan(inp.kv_lens.tolist(), inp.num_heads, inp.q_len, target_ctas=4)
    a = _decode(inp, causal, plan)
    mla.mla_debug_set_expire(S_FULL, 10 ** 6)  # a tile no CTA reaches
    try:
        b = _decode(inp, causal, plan)
    finally:
        mla.mla_debug_set_expire(-1)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
