"""Seeded synthetic workloads for paged FP8 MLA decode.

Shapes follow the issue "CuTe DSL FP8 MLA decode regression" (TensorRT-LLM
issue #20510, section "Setup" and the two repro tables): latent 512 + rope 64,
page size 32, FP8 E4M3 Q and KV, softmax_scale 0.0722, 12 heads per rank, q = 1
or 8 (MTP verify), KV 128K or 1M tokens, batch 1-16; and the H = 96, q = 8
packed-heads case from the same issue.  The pages use no public dataset; every
value here is drawn from a seeded generator.

Value recipe (both Q and KV): N(0, std^2) float32 with std = 0.5, then cast to
torch.float8_e4m3fn (round to nearest even), stored as raw uint8 codes.  The
page pool is shuffled with a seeded permutation and dealt to the requests in
order; the slots of a request's last page that lie past its KV length are
filled with 0x7F (an E4M3 NaN) so that any read of them poisons the result.

Nothing in this module decodes E4M3 or computes any part of attention.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

LATENT_DIM = 512
ROPE_DIM = 64
HEAD_DIM = LATENT_DIM + ROPE_DIM
PAGE_SIZE = 32
SOFTMAX_SCALE = 0.0722
E4M3_NAN_CODE = 0x7F

_CHUNK_ELEMS = 16 * 1024 * 1024  # 64 MB of float32 per draw


@dataclasses.dataclass
class DecodeInputs:
    """One decode batch. All tensors live on `device` unless noted."""

    q: torch.Tensor            # uint8 [B, q_len, H, 576] E4M3 codes
    kv: torch.Tensor           # uint8 [num_pages, 32, 576] E4M3 codes
    page_table: torch.Tensor   # int32 [B, max_pages]; -1 past a request's pages
    kv_lens: torch.Tensor      # int32 [B] (always on the host)
    batch: int
    q_len: int
    num_heads: int
    seed: int

    @property
    def num_pages(self) -> int:
        return int(self.kv.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def rows(self) -> int:
        return self.batch * self.q_len * self.num_heads

    def kv_bytes(self) -> int:
        return int(self.kv_lens.to(torch.int64).sum().item()) * HEAD_DIM * self.kv.element_size()


def _fill_e4m3(out_u8: torch.Tensor, gen: torch.Generator, std: float) -> None:
    """Fill a flat uint8 tensor with E4M3 codes of N(0, std^2) draws."""
    flat = out_u8.view(-1)
    n = flat.numel()
    for start in range(0, n, _CHUNK_ELEMS):
        cnt = min(_CHUNK_ELEMS, n - start)
        vals = torch.randn(cnt, generator=gen, device=flat.device, dtype=torch.float32)
        vals.mul_(std)
        flat[start:start + cnt].copy_(vals.to(torch.float8_e4m3fn).view(torch.uint8))


def _generator(device: torch.device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _fill_bf16(out: torch.Tensor, gen: torch.Generator, std: float) -> None:
    """Fill a flat bfloat16 tensor with N(0, std^2) draws (round to nearest even)."""
    flat = out.view(-1)
    n = flat.numel()
    for start in range(0, n, _CHUNK_ELEMS):
        cnt = min(_CHUNK_ELEMS, n - start)
        vals = torch.randn(cnt, generator=gen, device=flat.device, dtype=torch.float32)
        vals.mul_(std)
        flat[start:start + cnt].copy_(vals.to(torch.bfloat16))


BF16_NAN = float("nan")


def decode_inputs(batch: int, num_heads: int, q_len: int, kv_lens: Sequence[int],
                  seed: int, device: str | torch.device = "cpu", std: float = 0.5,
                  extra_pages: int = 0, dtype: str = "e4m3") -> DecodeInputs:
    """Draw one seeded decode batch.

    kv_lens: per-request KV lengths (len == batch).  extra_pages adds unused,
    NaN-filled pages to the pool (shuffled in with the used ones).  dtype
    "e4m3" gives uint8 E4M3 codes; "bf16" gives bfloat16 Q and KV.
    """
    device = torch.device(device)
    lens = [int(x) for x in kv_lens]
    if len(lens) != batch:
        raise ValueError("kv_lens must have one entry per request")
    pages_per_req = [(n + PAGE_SIZE - 1) // PAGE_SIZE for n in lens]
    used = sum(pages_per_req)
    total_pages = used + int(extra_pages)
    max_pages = max(1, max(pages_per_req))

    g = _generator(device, seed)
    if dtype == "e4m3":
        q = torch.empty((batch, q_len, num_heads, HEAD_DIM), dtype=torch.uint8, device=device)
        _fill_e4m3(q, g, std)
        kv = torch.empty((total_pages, PAGE_SIZE, HEAD_DIM), dtype=torch.uint8, device=device)
        _fill_e4m3(kv, g, std)
        poison = E4M3_NAN_CODE
    elif dtype == "bf16":
        q = torch.empty((batch, q_len, num_heads, HEAD_DIM), dtype=torch.bfloat16, device=device)
        _fill_bf16(q, g, std)
        kv = torch.empty((total_pages, PAGE_SIZE, HEAD_DIM), dtype=torch.bfloat16, device=device)
        _fill_bf16(kv, g, std)
        poison = BF16_NAN
    else:
        raise ValueError(f"unknown dtype {dtype}")

    # Page permutation is drawn on the host so that it does not depend on the device.
    gh = _generator(torch.device("cpu"), seed * 7919 + 17)
    perm = torch.randperm(total_pages, generator=gh).to(torch.int32)
    table = torch.full((batch, max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per_req):
        table[b, :n] = perm[off:off + n]
        off += n
    # Unused pool pages and the tail slots past each request's length are poison.
    if extra_pages:
        kv[perm[used:].to(torch.int64).to(device)] = poison
    for b, n in enumerate(lens):
        tail = n % PAGE_SIZE
        if n > 0 and tail:
            last = int(table[b, pages_per_req[b] - 1])
            kv[last, tail:, :] = poison
    return DecodeInputs(q=q, kv=kv, page_table=table.to(device),
                        kv_lens=torch.tensor(lens, dtype=torch.int32),
                        batch=batch, q_len=q_len, num_heads=num_heads, seed=seed)


def ragged_lens(seed: int = 4, n: int = 16, lo: int = 1024, hi: int = 131072) -> List[int]:
    """Mixed-length batch: lengths uniform in [lo, hi] (inclusive), seeded."""
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(lo, hi, size=n, endpoint=True)]


def query_lens_ragged(batch: int, q_len: int, seed: int) -> List[int]:
    """Per-request query-token counts, uniform in [1, q_len], seeded."""
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(1, q_len, size=batch, endpoint=True)]


def kv_windows(kv_lens: Sequence[int], seed: int, full_every: int = 4) -> np.ndarray:
    """Key windows [lo, hi) per request, int32 [B, 2], seeded.

    lo is uniform in [0, L - 1] and hi uniform in [lo + 1, L]; every
    full_every-th request keeps its whole range and every other one ends at L
    (a sliding window), so whole, trailing and inner windows all occur.
    """
    rng = np.random.default_rng(seed)
    out = np.zeros((len(kv_lens), 2), dtype=np.int32)
    for b, L in enumerate(kv_lens):
        L = int(L)
        if full_every and b % full_every == 0:
            out[b] = (0, L)
            continue
        lo = int(rng.integers(0, L))
        hi = L if b % 2 == 1 else int(rng.integers(lo + 1, L, endpoint=True))
        out[b] = (lo, hi)
    return out


def page_selection(kv_lens: Sequence[int], topk: int, seed: int,
                   keep_last: bool = True) -> np.ndarray:
    """Selected logical pages per request, int32 [B, topk], seeded.

    Each request gets min(topk, pages) distinct pages in ascending order
    (with keep_last, always including its last, possibly partial, page, as a
    local window does); unused slots at the end are -1.
    """
    rng = np.random.default_rng(seed)
    out = np.full((len(kv_lens), topk), -1, dtype=np.int32)
    for b, L in enumerate(kv_lens):
        n_pages = (int(L) + PAGE_SIZE - 1) // PAGE_SIZE
        k = min(topk, n_pages)
        if keep_last:
            rest = rng.choice(n_pages - 1, size=k - 1, replace=False) if k > 1 else []
            pages = np.sort(np.concatenate([np.asarray(rest, dtype=np.int64), [n_pages - 1]]))
        else:
            pages = np.sort(rng.choice(n_pages, size=k, replace=False))
        out[b, :k] = pages
    return out


def merge_partials(rows: int, num_splits: int, seed: int, empty_frac: float = 0.1,
                   all_empty_rows: Sequence[int] = ()):
    """Synthetic split partials for the merge alone.

    Returns (o, ml): o float32 [rows, S, 512] holds un-normalised outputs,
    ml float32 [rows, S, 2] holds (m in log2 units, l).  m ~ N(0, 2^2),
    l ~ U[1, 4096], o = l * N(0, 0.5^2).  A fraction empty_frac of the slots
    is empty: (m, l, o) = (-inf, 0, 0).  Rows listed in all_empty_rows are
    empty in every slot.
    """
    rng = np.random.default_rng(seed)
    m = rng.normal(0.0, 2.0, size=(rows, num_splits)).astype(np.float32)
    l = rng.uniform(1.0, 4096.0, size=(rows, num_splits)).astype(np.float32)
    o = (rng.normal(0.0, 0.5, size=(rows, num_splits, LATENT_DIM)).astype(np.float32)
         * l[:, :, None])
    empty = rng.random(size=(rows, num_splits)) < empty_frac
    for r in all_empty_rows:
        empty[r, :] = True
    m[empty] = -np.inf
    l[empty] = 0.0
    o[empty] = 0.0
    ml = np.stack([m, l], axis=-1).astype(np.float32)
    return np.ascontiguousarray(o), np.ascontiguousarray(ml)


# Named workloads.  "target" is the CTA target handed to the split planner when
# the pages' printed plan is reproduced; None means "derive it from the SM count".
WORKLOADS: Dict[str, dict] = {}


def _add(name: str, **kw) -> None:
    WORKLOADS[name] = kw


_add("tiny_b1_h12_q1_l4096", batch=1, num_heads=12, q_len=1, kv_lens=[4096],
     causal=False, target=4, seed=0)
for _b, _split in [(1, 32), (2, 32), (4, 25), (8, 12), (16, 6)]:
    _add(f"h12_q1_l128k_b{_b}", batch=_b, num_heads=12, q_len=1, kv_lens=[131072] * _b,
         causal=False, target=_b * _split, seed=1)
for _b in (1, 2, 4, 8, 16):
    _add(f"mtp_h12_q8_l128k_b{_b}", batch=_b, num_heads=12, q_len=8, kv_lens=[131072] * _b,
         causal=True, target=100, seed=2)
for _q in (1, 8):
    for _b in (1, 2, 4, 8, 16):
        _add(f"long_h12_q{_q}_l1m_b{_b}", batch=_b, num_heads=12, q_len=_q,
             kv_lens=[1048576] * _b, causal=(_q > 1), target=100, seed=3)
for _b in (1, 4):
    for _l, _tag in ((131072, "128k"), (1048576, "1m")):
        _add(f"packed_h96_q8_l{_tag}_b{_b}", batch=_b, num_heads=96, q_len=8,
             kv_lens=[_l] * _b, causal=True, target=None, seed=4)
_add("ragged_h12_q1_b16", batch=16, num_heads=12, q_len=1, kv_lens=ragged_lens(4),
     causal=False, target=None, seed=4)
# Skewed batch (issue #20510 follow-up: "one 1M request plus short ones";
# the count and lengths of the short ones are not given: seven of 4K here).
for _q in (1, 8):
    _add(f"skewed_h12_q{_q}_1m_plus_7x4k", batch=8, num_heads=12, q_len=_q,
         kv_lens=[1048576] + [4096] * 7, causal=(_q > 1), target=None, seed=7)
# BF16 KV cache (the pages' BF16 kernel is quoted at H12 q8 B1 1M).
for _q in (1, 8):
    _add(f"bf16_h12_q{_q}_l1m_b1", batch=1, num_heads=12, q_len=_q, kv_lens=[1048576],
         causal=(_q > 1), target=None, seed=5, dtype="bf16")
_add("bf16_h12_q1_l1m_b16", batch=16, num_heads=12, q_len=1, kv_lens=[1048576] * 16,
     causal=False, target=None, seed=5, dtype="bf16")
# Sparse decode over selected pages: 256 pages (8192 keys) of each 1M-key
# request, picked by a seeded stand-in for the block selector (the last page
# always included).
for _q in (1, 8):
    _add(f"sparse_h12_q{_q}_l1m_b16_top256", batch=16, num_heads=12, q_len=_q,
         kv_lens=[1048576] * 16, causal=(_q > 1), target=None, seed=6, topk=256)
# The same selections in 128K-key requests: the same CTAs and tiles over a
# 1.2 GB pool (a size for full-set profiler captures).
for _q in (1, 8):
    _add(f"sparse_h12_q{_q}_l128k_b16_top256", batch=16, num_heads=12, q_len=_q,
         kv_lens=[131072] * 16, causal=(_q > 1), target=None, seed=6, topk=256)


def workload_inputs(name: str, device: str | torch.device = "cpu",
                    kv_lens_override: Optional[Sequence[int]] = None,
                    seed_offset: int = 0) -> DecodeInputs:
    """Inputs of a named workload; seed_offset draws further distinct pools."""
    w = WORKLOADS[name]
    lens = list(kv_lens_override) if kv_lens_override is not None else w["kv_lens"]
    return decode_inputs(w["batch"], w["num_heads"], w["q_len"], lens,
                         w["seed"] + 1000 * seed_offset, device=device,
                         dtype=w.get("dtype", "e4m3"))
