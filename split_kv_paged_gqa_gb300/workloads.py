"""Seeded synthetic decode workloads for split-KV paged GQA flash decode.

This is the only module that both the CUDA path (tests, bench) and the float64
oracle read from. It draws random numbers, assigns KV lengths and cache pages,
and writes quantised KV caches the way a serving engine's cache writer would.
It holds none of the decode arithmetic (no scores, no softmax, no merge, no
dequantisation).

Recipe (every draw is seeded):

* Lengths and page placement come from ``numpy.random.default_rng(seed)``
  (PCG64): lengths first, then one permutation of the page pool. Request ``b``
  takes the next ``ceil(L_b / P)`` entries of that permutation; page-table
  columns past a request's last page hold the ``-1`` sentinel (the fused
  graph-metadata kernel of sglang PR 29843, section "implementation", guards
  the same sentinel).
* Q, K and V values are i.i.d. N(0, 1) float32 drawn by a
  ``torch.Generator`` on the target device (q first, then the K pool, then the
  V pool), cast to bf16 by round-to-nearest-even, or quantised:

  - int8: one fp32 scale per (token, KV head): ``scale = max|x| / 127``,
    ``code = clamp(round_half_even(x / scale), -127, 127)``;
  - int4: one fp32 scale per (token, KV head, 32-channel group):
    ``scale = max|x| / 7``, ``code = clamp(round_half_even(x / scale), -8, 7)``,
    two codes per byte, the even channel in the low nibble.

  An all-zero group gets scale 0 and codes 0.
* ``kv_scales`` is fp32 ``[2, num_pages, P, Hkv, n_g]`` (index 0 = K, 1 = V),
  ``n_g = 1`` for int8 and ``D / 32`` for int4: the scale of a cache row sits
  at the same (page, slot, head) index as the row. In memory the scales are
  stored head-major within a page (``[2, num_pages, Hkv, P, n_g]``, handed
  out as a strided view with the logical index order above), so the scales of
  one (page, head) are one contiguous run, as a cache writer that keeps a
  page's per-head metadata together stores them.

Optional structure used by the parity tests:

* ``poison``: tail slots past each request's length in its last page, and every
  pool page no request owns, are overwritten with values that break any kernel
  that reads them without masking (bf16 K = +1e4, V = NaN; quantised caches
  get NaN scales).
* ``needles``: for every (request, KV head) one random key position ``j*`` gets
  a K row aligned with the last query token's first query head of the group,
  so that head's score at ``j*`` is ``needle_score`` and its attention output
  is, to many digits, V[j*]. A kernel that skips or misaddresses a page fails.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

KV_DTYPES = ("bf16", "int8", "int4")


@dataclasses.dataclass(frozen=True)
class DecodeShape:
    """Shape and length recipe of one decode workload.

    ``lengths`` is a recipe string:
      ``fixed:a,b,...``  explicit lengths (one per request)
      ``const:L``        every request has length L
      ``uniform:lo,hi``  integers uniform on [lo, hi], both ends included
      ``lognormal:median,sigma,lo,hi``  round(exp(N(ln median, sigma))) clipped
    """

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    q_per_req: int
    kv_dtype: str
    lengths: str
    pool_pages: Optional[int] = None

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def with_(self, **kw) -> "DecodeShape":
        return dataclasses.replace(self, **kw)


# The five workloads of the decode study, named by what they are.
CONFIGS = {
    # batch 2, 8/2 heads, D64, page 16, lengths {100, 257}, 64-page pool
    "tiny_bf16": DecodeShape("tiny_bf16", 2, 8, 2, 64, 16, 1, "bf16", "fixed:100,257", 64),
    # batch 32, 40/8 heads (group 5), D128, page 16, lengths U[1024, 32768]
    "mixed_bf16": DecodeShape("mixed_bf16", 32, 40, 8, 128, 16, 1, "bf16", "uniform:1024,32768"),
    # every length 32768, 64/8 heads, D128, page 64; batch 1, 16 or 64
    "long_bf16_b1": DecodeShape("long_bf16_b1", 1, 64, 8, 128, 64, 1, "bf16", "const:32768"),
    "long_bf16_b16": DecodeShape("long_bf16_b16", 16, 64, 8, 128, 64, 1, "bf16", "const:32768"),
    "long_bf16_b64": DecodeShape("long_bf16_b64", 64, 64, 8, 128, 64, 1, "bf16", "const:32768"),
    # batch 64, 32/8 heads, D128, page 16, int8 KV, lognormal lengths (median 4096)
    "int8_lognormal": DecodeShape("int8_lognormal", 64, 32, 8, 128, 16, 1, "int8",
                                  "lognormal:4096,1.0,16,32768"),
    # batch 64, 4 causal query tokens, 32/8 heads, D128, page 16, int4 KV, U[4096, 32768]
    "int4_mtp": DecodeShape("int4_mtp", 64, 32, 8, 128, 16, 4, "int4", "uniform:4096,32768"),
}

# Fixed seed per workload so every consumer sees the same inputs.
CONFIG_SEEDS = {name: 1000 + i for i, name in enumerate(CONFIGS)}

# The sigma of the lognormal length mix is not stated anywhere; 1.0 is used.
LOGNORMAL_SIGMA = 1.0


@dataclasses.dataclass
class Workload:
    shape: DecodeShape
    seed: int
    q: torch.Tensor                 # bf16 [B, Tq, Hq, D]
    k_cache: torch.Tensor           # bf16/int8 [N, P, Hkv, D] or uint8 [N, P, Hkv, D/2]
    v_cache: torch.Tensor
    kv_scales: Optional[torch.Tensor]  # fp32 [2, N, P, Hkv, n_g] (head-major in memory) or None
    page_table: torch.Tensor        # int32 [B, max_pages], -1 padded
    cache_seqlens: torch.Tensor     # int32 [B]
    lengths: np.ndarray             # int64 [B], host copy
    softmax_scale: float
    needles: List[Tuple[int, int, int]]  # (request, kv_head, key position)

    @property
    def device(self) -> torch.device:
        return self.q.device

    def kv_bytes(self) -> int:
        """Bytes of K, V and scales for the keys the requests own (read once)."""
        return int(self.lengths.sum()) * kv_bytes_per_token(self.shape)


def kv_bytes_per_token(shape: DecodeShape) -> int:
    """Bytes of K + V (+ their fp32 scales) for one token over all KV heads."""
    d = shape.head_dim
    if shape.kv_dtype == "bf16":
        row = 2 * d
        scales = 0
    elif shape.kv_dtype == "int8":
        row = d
        scales = 4
    else:
        row = d // 2
        scales = 4 * (d // 32)
    return shape.num_kv_heads * 2 * (row + scales)


def draw_lengths(recipe: str, batch: int, rng: np.random.Generator) -> np.ndarray:
    kind, _, args = recipe.partition(":")
    vals = [float(a) for a in args.split(",")] if args else []
    if kind == "fixed":
        if len(vals) != batch:
            raise ValueError(f"fixed lengths {vals} do not match batch {batch}")
        return np.array([int(v) for v in vals], dtype=np.int64)
    if kind == "const":
        return np.full(batch, int(vals[0]), dtype=np.int64)
    if kind == "uniform":
        return rng.integers(int(vals[0]), int(vals[1]), size=batch, endpoint=True).astype(np.int64)
    if kind == "lognormal":
        median, sigma, lo, hi = vals
        x = rng.normal(math.log(median), sigma, size=batch)
        return np.clip(np.rint(np.exp(x)), lo, hi).astype(np.int64)
    raise ValueError(f"unknown length recipe {recipe!r}")


def assign_pages(lengths: np.ndarray, page_size: int, pool_pages: Optional[int],
                 extra_pages: int, rng: np.random.Generator, capacity_pages: Optional[int] = None):
    """Random page placement: one permutation of the pool, consecutive slices."""
    need = [int(-(-int(L) // page_size)) for L in lengths]
    total = sum(need)
    pool = (pool_pages if pool_pages is not None else total) + extra_pages
    if pool < total:
        raise ValueError(f"pool of {pool} pages is smaller than the {total} pages needed")
    perm = rng.permutation(pool)
    width = max(max(need) if need else 1, 1)
    if capacity_pages is not None:
        width = max(width, capacity_pages)
    table = np.full((len(lengths), width), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[pos:pos + n]
        pos += n
    return table, pool


def quantize_int8(x: torch.Tensor):
    """Symmetric int8 per last-dim row. Returns (codes int8, scale fp32 [..., 1])."""
    x = x.float()
    scale = x.abs().amax(dim=-1, keepdim=True) / 127.0
    codes = torch.where(scale > 0, torch.round(x / scale), torch.zeros_like(x))
    return codes.clamp_(-127, 127).to(torch.int8), scale


def quantize_int4(x: torch.Tensor):
    """Symmetric int4 per 32-channel group, packed low-nibble-first.

    Returns (packed uint8 [..., D/2], scale fp32 [..., D/32]).
    """
    x = x.float()
    d = x.shape[-1]
    if d % 32:
        raise ValueError("int4 groups need head_dim divisible by 32")
    g = x.reshape(*x.shape[:-1], d // 32, 32)
    scale = g.abs().amax(dim=-1) / 7.0
    s = scale.unsqueeze(-1)
    codes = torch.where(s > 0, torch.round(g / s), torch.zeros_like(g)).clamp_(-8, 7)
    codes = codes.reshape(*x.shape[:-1], d).to(torch.int16)
    lo = codes[..., 0::2] & 0xF
    hi = codes[..., 1::2] & 0xF
    return (lo | (hi << 4)).to(torch.uint8), scale


def _cast_or_quantize(x: torch.Tensor, kv_dtype: str):
    if kv_dtype == "bf16":
        return x.to(torch.bfloat16), None
    if kv_dtype == "int8":
        return quantize_int8(x)
    if kv_dtype == "int4":
        return quantize_int4(x)
    raise ValueError(kv_dtype)


def make_workload(shape: DecodeShape, seed: int, device="cpu", *, poison: bool = False,
                  needles: bool = False, needle_score: float = 30.0,
                  lengths: Optional[Sequence[int]] = None, extra_pages: int = 0,
                  capacity_pages: Optional[int] = None,
                  chunk_elems: int = 1 << 26) -> Workload:
    """Build one seeded workload on ``device``.

    ``lengths`` overrides the recipe; ``extra_pages`` adds unowned pool pages
    (poisoned when ``poison``); ``capacity_pages`` widens the page table.
    """
    if shape.kv_dtype not in KV_DTYPES:
        raise ValueError(shape.kv_dtype)
    device = torch.device(device)
    B, Tq, Hq, Hkv, D, P = (shape.batch, shape.q_per_req, shape.num_q_heads,
                            shape.num_kv_heads, shape.head_dim, shape.page_size)
    G = Hq // Hkv
    rng = np.random.default_rng(seed)
    L = (np.asarray(lengths, dtype=np.int64) if lengths is not None
         else draw_lengths(shape.lengths, B, rng))
    table, pool = assign_pages(L, P, shape.pool_pages, extra_pages, rng, capacity_pages)
    softmax_scale = 1.0 / math.sqrt(D)

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = torch.randn((B, Tq, Hq, D), generator=gen, device=device, dtype=torch.float32)
    q = q.to(torch.bfloat16)

    # Needle positions are drawn from the host rng after the page placement.
    needle_list: List[Tuple[int, int, int]] = []
    needle_rows = {}
    if needles:
        qf = q.double().cpu()
        for b in range(B):
            hi = int(L[b]) - Tq + 1
            if hi <= 0:
                continue
            for h in range(Hkv):
                j = int(rng.integers(0, hi))
                qv = qf[b, Tq - 1, h * G]
                row = (needle_score / softmax_scale) * qv / float((qv * qv).sum())
                page = int(table[b, j // P])
                needle_rows.setdefault(page, []).append((j % P, h, row.float()))
                needle_list.append((b, h, j))

    row_dim = D if shape.kv_dtype != "int4" else D // 2
    cache_dtype = {"bf16": torch.bfloat16, "int8": torch.int8, "int4": torch.uint8}[shape.kv_dtype]
    k_cache = torch.empty((pool, P, Hkv, row_dim), dtype=cache_dtype, device=device)
    v_cache = torch.empty_like(k_cache)
    n_g = 1 if shape.kv_dtype == "int8" else D // 32
    kv_scales = (torch.empty((2, pool, Hkv, P, n_g), dtype=torch.float32, device=device).permute(0, 1, 3, 2, 4)
                 if shape.kv_dtype != "bf16" else None)

    pages_per_chunk = max(1, chunk_elems // (P * Hkv * D))
    for which, cache in ((0, k_cache), (1, v_cache)):
        for p0 in range(0, pool, pages_per_chunk):
            p1 = min(pool, p0 + pages_per_chunk)
            x = torch.randn((p1 - p0, P, Hkv, D), generator=gen, device=device,
                            dtype=torch.float32)
            if which == 0 and needle_rows:
                for page in range(p0, p1):
                    for slot, h, row in needle_rows.get(page, ()):
                        x[page - p0, slot, h] = row.to(device)
            codes, scale = _cast_or_quantize(x, shape.kv_dtype)
            cache[p0:p1] = codes
            if kv_scales is not None:
                kv_scales[which, p0:p1] = scale.reshape(p1 - p0, P, Hkv, n_g)
            del x, codes, scale

    if poison:
        _poison(shape, L, table, pool, k_cache, v_cache, kv_scales)

    return Workload(
        shape=shape, seed=seed, q=q, k_cache=k_cache, v_cache=v_cache, kv_scales=kv_scales,
        page_table=torch.from_numpy(table).to(device),
        cache_seqlens=torch.from_numpy(L.astype(np.int32)).to(device),
        lengths=L, softmax_scale=softmax_scale, needles=needle_list)


def _poison(shape, L, table, pool, k_cache, v_cache, kv_scales):
    P = shape.page_size
    owned = set()
    for b in range(len(L)):
        n = int(-(-int(L[b]) // P))
        owned.update(int(p) for p in table[b, :n])
        tail = int(L[b]) % P
        if n and tail:
            last = int(table[b, n - 1])
            _poison_rows(shape, k_cache, v_cache, kv_scales, last, slice(tail, P))
    for page in range(pool):
        if page not in owned:
            _poison_rows(shape, k_cache, v_cache, kv_scales, page, slice(0, P))


def _poison_rows(shape, k_cache, v_cache, kv_scales, page, slots):
    if shape.kv_dtype == "bf16":
        k_cache[page, slots] = 1.0e4
        v_cache[page, slots] = float("nan")
    else:
        kv_scales[:, page, slots] = float("nan")


# ---------------------------------------------------------------------------
# Host views for the oracle (marshalling only)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (no rounding, no arithmetic)."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_inputs(w: Workload, requests: Optional[Sequence[int]] = None) -> dict:
    """Numpy copies of the inputs, optionally for a subset of requests.

    With ``requests`` the caches are compacted to just those requests' pages
    and the page table relabelled to match (the result does not depend on
    where pages sit in the pool).
    """
    L = w.lengths
    P = w.shape.page_size
    if requests is None:
        req = list(range(w.shape.batch))
        pt = w.page_table.cpu().numpy()
        k, v = w.k_cache, w.v_cache
        sc = w.kv_scales
    else:
        req = list(requests)
        table = w.page_table.cpu().numpy()
        pages, rows = [], []
        for b in req:
            n = int(-(-int(L[b]) // P))
            rows.append((len(pages), n))
            pages.extend(int(p) for p in table[b, :n])
        width = max([n for _, n in rows] + [1])
        pt = np.full((len(req), width), -1, dtype=np.int32)
        for i, (start, n) in enumerate(rows):
            pt[i, :n] = np.arange(start, start + n, dtype=np.int32)
        idx = torch.tensor(pages if pages else [0], dtype=torch.long, device=w.k_cache.device)
        k, v = w.k_cache.index_select(0, idx), w.v_cache.index_select(0, idx)
        sc = w.kv_scales.index_select(1, idx) if w.kv_scales is not None else None
    sel = torch.tensor(req, dtype=torch.long, device=w.q.device)
    q = w.q.index_select(0, sel)
    if w.shape.kv_dtype == "bf16":
        k_np, v_np = bf16_bits(k), bf16_bits(v)
    else:
        k_np, v_np = k.cpu().numpy(), v.cpu().numpy()
    return dict(
        q=bf16_bits(q), k_cache=k_np, v_cache=v_np,
        kv_scales=None if sc is None else sc.cpu().numpy(),
        page_table=pt.astype(np.int32), cache_seqlens=L[req].astype(np.int32),
        q_per_req=w.shape.q_per_req, kv_dtype=w.shape.kv_dtype,
        softmax_scale=w.softmax_scale)


def make_token_pool(seed: int, lengths: Sequence[int], page_size: int, max_ctx: Optional[int] = None,
                    extra_rows: int = 0, unallocated_frac: float = 0.0) -> Tuple[np.ndarray, np.ndarray]:
    """A serving engine's request-to-token pool, seeded: int32 [R, C] KV slots.

    Pool row r (one per entry of ``lengths``, plus ``extra_rows`` empty rows)
    holds, for token positions 0 .. ceil(len_r / P) * P - 1, the slots of the
    pages an allocator handed it: pages are a random permutation of the whole
    page pool, consecutive per request, and the slot of position c is
    page * P + c % P. Positions past the request's pages hold -1. With
    ``unallocated_frac`` that share of the pages is left without slots (-1 on
    all its positions). Returns (req_to_token, page_of_row_pages) where the
    second is the list of page ids per row (for checks that need no slots).
    """
    rng = np.random.default_rng(seed)
    L = np.asarray(lengths, dtype=np.int64)
    P = int(page_size)
    n_pages = -(-L // P)
    total = int(n_pages.sum())
    C = int(max_ctx or max(int(n_pages.max(initial=0)) * P, 1))
    R = len(L) + extra_rows
    perm = rng.permutation(max(total, 1))
    pool = np.full((R, C), -1, dtype=np.int32)
    pages = []
    k = 0
    for r in range(len(L)):
        row_pages = perm[k:k + n_pages[r]]
        k += int(n_pages[r])
        pages.append(row_pages.copy())
        n = min(int(n_pages[r]) * P, C)
        if n == 0:
            continue
        pos = np.arange(n)
        slots = row_pages[pos // P] * P + pos % P
        if unallocated_frac > 0:
            gone = rng.random(len(row_pages)) < unallocated_frac
            slots = np.where(gone[pos // P], -1, slots)
        pool[r, :n] = slots.astype(np.int32)
    return pool, pages
