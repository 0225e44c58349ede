"""CPU oracle for the decode metadata a CUDA-graph replay rebuilds per step.

TEST INFRASTRUCTURE. Only the test suite imports this module; the CUDA library
never calls it and shares no code with it.

What it computes: the metadata the decode path consumes, built from a serving
engine's request-to-token pool, as the fused graph-metadata kernel of "sglang
PR 29843" (section 实现拆解, item 1: one program per batch row computes
cache_seqlens, cu_seqlens_k / cu_seqlens_q and page_table at once, with three
q modes (preset / cumsum / strided) and a -1 sentinel guard) does in place of
about 25 small host-dispatched operations (section 功能与动机). The pages give
no formulas; the readings below are the plain ones:

* ``req_to_token[r, j]`` is the KV slot of token position j of pool request r;
  a slot s lives in page s // P at offset s % P, and a request's pages start
  on page boundaries, so page j of a request is ``req_to_token[r, j * P] // P``.
  A slot below 0 marks a position with no KV slot.
* Batch row b reads pool row ``req_pool_indices[b]``; an index below 0 marks a
  padding row (a graph captured for more rows than the step has).
* ``cache_seqlens[b] = seq_lens[b]`` (0 for a padding row).
* ``page_table[b, j]`` = page j of the request for j < ceil(L_b / P); -1 past
  the request's last page, for an unallocated slot, and for every entry of a
  padding row (the -1 sentinel the decode path never reads).
* ``cu_seqlens_k[b] = sum_{b' < b} cache_seqlens[b']`` for b in [0, B]
  (exclusive prefix sum with a leading 0).
* ``cu_seqlens_q``: ``preset`` copies a given [B + 1] array; ``cumsum`` takes
  the exclusive prefix sum of per-request query-token counts (0 for a padding
  row); ``strided`` is ``b * q_stride`` (a fixed number of query tokens per
  request, as in MTP verification).

Parity status: pinned by the CPU tests (a hand-worked example, prefix-sum
invariants, brute-force loops on tiny pools); no function here is unpinned.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

Q_PRESET, Q_CUMSUM, Q_STRIDED = 0, 1, 2


def graph_metadata_ref(req_to_token: np.ndarray, req_pool_indices: np.ndarray, seq_lens: np.ndarray,
                       page_size: int, width: int, q_mode: int, q_in: Optional[np.ndarray] = None,
                       q_stride: int = 1) -> Dict[str, np.ndarray]:
    """Returns page_table [B, width], cache_seqlens [B], cu_seqlens_k [B+1], cu_seqlens_q [B+1] (int32)."""
    req_to_token = np.asarray(req_to_token, dtype=np.int64)
    idx = np.asarray(req_pool_indices, dtype=np.int64)
    lens = np.asarray(seq_lens, dtype=np.int64)
    B = idx.shape[0]
    P = int(page_size)
    page_table = np.full((B, width), -1, dtype=np.int64)
    cache_seqlens = np.zeros(B, dtype=np.int64)
    for b in range(B):
        r = int(idx[b])
        if r < 0:  # padding row
            continue
        L = int(lens[b])
        cache_seqlens[b] = L
        n_pages = (L + P - 1) // P
        for j in range(min(n_pages, width)):
            slot = int(req_to_token[r, j * P])
            page_table[b, j] = slot // P if slot >= 0 else -1
    cu_k = np.zeros(B + 1, dtype=np.int64)
    for b in range(B):
        cu_k[b + 1] = cu_k[b] + cache_seqlens[b]
    if q_mode == Q_PRESET:
        cu_q = np.asarray(q_in, dtype=np.int64).copy()
    elif q_mode == Q_CUMSUM:
        cu_q = np.zeros(B + 1, dtype=np.int64)
        for b in range(B):
            cu_q[b + 1] = cu_q[b] + (int(q_in[b]) if idx[b] >= 0 else 0)
    elif q_mode == Q_STRIDED:
        cu_q = np.arange(B + 1, dtype=np.int64) * int(q_stride)
    else:
        raise ValueError(q_mode)
    return {"page_table": page_table.astype(np.int32), "cache_seqlens": cache_seqlens.astype(np.int32),
            "cu_seqlens_k": cu_k.astype(np.int32), "cu_seqlens_q": cu_q.astype(np.int32)}
