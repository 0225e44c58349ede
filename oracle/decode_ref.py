"""Float64 CPU oracle for split-KV paged grouped-query flash decode.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` import this module. The CUDA library never
calls it and shares no code, header, table or helper with it.

What it computes is the plain definition of the operation the decode kernels of
"feat(autotune): separate general and decode attention warmup" (LightLLM
PR 1549, section "Covered decode kernels": Triton GQA flash decode, INT8 and
INT4 KV flash decode, MTP attention, FA3 KV-cache decode) compute faster:
softmax attention of each query row over the keys of its request, read through
a page table from a paged KV cache. Flash decode, split-KV and the stage-2
merge reorganise this computation without changing its result, so the oracle
does none of them: per (request, query token, query head) it gathers every
visible key, forms every score, materialises the full softmax in float64 and
takes the weighted sum of V rows.

Inputs are numpy arrays (bf16 passed as uint16 bit patterns, so no library
rounds them on the way in):

* ``q``            uint16 (bf16 bits) [B, Tq, Hq, D]
* ``k_cache``      bf16 bits uint16 / int8 [N, P, Hkv, D], or uint8 [N, P, Hkv, D/2] (int4)
* ``v_cache``      same as ``k_cache``
* ``kv_scales``    float32 [2, N, P, Hkv, n_g] (0 = K, 1 = V) or None for bf16
* ``page_table``   int32 [B, W]; entries past a request's last page are -1 and never read
* ``cache_seqlens`` int32 [B]

Readings taken where the pages are silent (each is a plain reading):

* GQA head map: query head h reads KV head h // G with G = Hq / Hkv.
* Causal multi-token decode (MTP): query token t of a request with L cached
  keys sees the first L - (Tq - 1) + t keys; the last token sees all L.
* LSE is the natural log of the sum of exp of the *scaled* scores.
* A row that sees no key returns out = 0 and lse = -inf.
* Scale defaults to 1 / sqrt(D).

Parity status: every function here is pinned by the CPU tests (brute force on
tiny inputs, closed forms, invariants, a library attention routine and hand
computed quantiser bytes); none is unpinned.
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import numpy as np


# ---------------------------------------------------------------------------
# Element decoding (the cache formats)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns: a bf16 is the top half of a float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def dequant_int8(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """INT8 KV (section "Covered decode kernels", INT8 KV flash decode).

    ``codes`` int8 [..., D]; ``scale`` float32 [..., 1], one per (token, KV
    head). Value = code * scale, evaluated in float64.
    """
    return codes.astype(np.float64) * scale.astype(np.float64)


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    """Two signed 4-bit codes per byte, even channel in the low nibble.

    ``packed`` uint8 [..., D/2] -> int64 [..., D] in [-8, 7].
    """
    p = packed.astype(np.int64)
    lo = p & 0xF
    hi = (p >> 4) & 0xF
    codes = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int64)
    codes[..., 0::2] = lo
    codes[..., 1::2] = hi
    return np.where(codes >= 8, codes - 16, codes)


def dequant_int4(packed: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """INT4 KV (section "Covered decode kernels", INT4 KV flash decode).

    ``scale`` float32 [..., D/32], one per (token, KV head, 32-channel group);
    channel c uses group c // 32.
    """
    codes = unpack_int4(packed).astype(np.float64)
    d = codes.shape[-1]
    s = np.repeat(scale.astype(np.float64), 32, axis=-1)[..., :d]
    return codes * s


# ---------------------------------------------------------------------------
# Page walk


def gather_kv(cache: np.ndarray, scales: Optional[np.ndarray], page_row: np.ndarray,
              n_keys: int, page_size: int, kv_dtype: str) -> np.ndarray:
    """Rows of keys 0..n_keys-1 of one request as float64 [n_keys, Hkv, D].

    Key j lives in page ``page_row[j // P]`` at slot ``j % P`` (the
    page_table / cache_seqlens metadata of sglang PR 29843, section
    "motivation"). Only the first ceil(n_keys / P) table entries are read.
    """
    j = np.arange(n_keys)
    pages = page_row[j // page_size].astype(np.int64)
    slots = j % page_size
    if n_keys and (pages.min() < 0 or pages.max() >= cache.shape[0]):
        raise IndexError("page table entry outside the cache for a visible key")
    raw = cache[pages, slots]                     # [n, Hkv, row]
    if kv_dtype == "bf16":
        return bf16_to_f64(raw)
    s = scales[pages, slots]                      # [n, Hkv, n_g]
    if kv_dtype == "int8":
        return dequant_int8(raw, s)
    if kv_dtype == "int4":
        return dequant_int4(raw, s)
    raise ValueError(kv_dtype)


# ---------------------------------------------------------------------------
# Attention by definition


def attend(q_row: np.ndarray, keys: np.ndarray, vals: np.ndarray,
           scale: float) -> Tuple[np.ndarray, float]:
    """Softmax attention of one query row over explicit keys, full softmax.

    s_j = scale * <q, k_j>;  p_j = exp(s_j - max s) / sum_i exp(s_i - max s);
    out = sum_j p_j v_j;  lse = max s + ln sum_i exp(s_i - max s).
    No keys: out = 0, lse = -inf.
    """
    if keys.shape[0] == 0:
        return np.zeros(vals.shape[-1], dtype=np.float64), -math.inf
    s = scale * (keys @ q_row)
    m = s.max()
    e = np.exp(s - m)
    z = e.sum()
    p = e / z
    return p @ vals, float(m + math.log(z))


def decode_ref(q, k_cache, v_cache, kv_scales, page_table, cache_seqlens, q_per_req,
               kv_dtype, softmax_scale: Optional[float] = None,
               key_range: Optional[Tuple[int, int]] = None,
               requests=None) -> Tuple[np.ndarray, np.ndarray]:
    """Paged GQA decode attention, float64.

    Returns ``out`` [B, Tq, Hq, D] and ``lse`` [B, Tq, Hq] (float64).

    ``key_range=(lo, hi)`` restricts every row to keys in [lo, hi) on top of
    its causal limit: that is the slice of the computation one KV split owns,
    used only to check the split/merge invariant of this oracle.
    ``requests`` limits the work to a subset of batch rows (others stay 0/-inf).
    """
    qf = bf16_to_f64(q)
    B, Tq, Hq, D = qf.shape
    if Tq != q_per_req:
        raise ValueError("q_per_req must equal q.shape[1]")
    P = k_cache.shape[1]
    Hkv = k_cache.shape[2]
    if Hq % Hkv:
        raise ValueError("query heads must be a multiple of KV heads")
    G = Hq // Hkv
    scale = (1.0 / math.sqrt(D)) if softmax_scale is None else float(softmax_scale)
    out = np.zeros((B, Tq, Hq, D), dtype=np.float64)
    lse = np.full((B, Tq, Hq), -math.inf, dtype=np.float64)
    k_sc = kv_scales[0] if kv_scales is not None else None
    v_sc = kv_scales[1] if kv_scales is not None else None
    for b in (range(B) if requests is None else requests):
        L = int(cache_seqlens[b])
        K = gather_kv(k_cache, k_sc, page_table[b], L, P, kv_dtype)
        V = gather_kv(v_cache, v_sc, page_table[b], L, P, kv_dtype)
        for t in range(Tq):
            n = L - (Tq - 1) + t                  # causal limit of token t
            lo, hi = 0, max(n, 0)
            if key_range is not None:
                lo, hi = max(lo, key_range[0]), min(hi, key_range[1])
            hi = max(hi, lo)
            for h in range(Hq):
                hk = h // G
                o, l = attend(qf[b, t, h], K[lo:hi, hk], V[lo:hi, hk], scale)
                out[b, t, h] = o
                lse[b, t, h] = l
    return out, lse


def decode_ref_inputs(inp: dict, **kw):
    """``decode_ref`` over a dict laid out like the workload host view."""
    return decode_ref(inp["q"], inp["k_cache"], inp["v_cache"], inp["kv_scales"],
                      inp["page_table"], inp["cache_seqlens"], inp["q_per_req"],
                      inp["kv_dtype"], inp.get("softmax_scale"), **kw)


def merge_splits(o_parts: np.ndarray, lse_parts: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Combine partial results by their LSE (the stage-2 merge), float64.

    ``o_parts`` [S, ..., D] each normalised over its own keys; ``lse_parts``
    [S, ...]. out = sum_s w_s o_s / sum_s w_s with w_s = exp(lse_s - max lse);
    lse = max lse + ln sum_s w_s. Splits with lse = -inf carry no weight;
    if every split is empty the result is out = 0, lse = -inf.
    """
    o = np.asarray(o_parts, dtype=np.float64)
    l = np.asarray(lse_parts, dtype=np.float64)
    m = l.max(axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(l), np.exp(l - m_safe), 0.0)
    z = w.sum(axis=0)
    z_safe = np.where(z > 0, z, 1.0)
    out = (w[..., None] * o).sum(axis=0) / z_safe[..., None]
    out = np.where(finite[..., None], out, 0.0)
    lse = np.where(finite, m_safe + np.log(z_safe), -math.inf)
    return out, lse
