"""The decode entry point that allocates no device memory.

Some callers cannot call cudaMalloc: an engine that has reserved all GPU memory
for its own pool, or a plugin in a process that forbids foreign allocations.
They call fd_decode_paged_static, which runs the same kernels with a fixed
scratch array inside the library. Here it is checked, through the C ABI,
against the plan-based fd_decode_paged on the same inputs, on two calls in a
row (the second reuses the scratch the first left behind). This file is
collected last and must pass alone in a fresh process too.
"""
import numpy as np
import pytest
import torch

import split_kv_paged_gqa_gb300 as fd
from split_kv_paged_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

OUT_ATOL = 8e-3
LSE_ATOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _plan_call(w, S):
    s = w.shape
    plan = fd.fd_plan_create(0, s.batch, s.q_per_req, s.num_q_heads, s.num_kv_heads, s.head_dim, s.page_size,
                             s.kv_dtype, 64)
    try:
        fd.fd_set_plan(plan)
        out = torch.empty_like(w.q)
        lse = torch.empty(w.q.shape[:3], dtype=torch.float32, device=w.q.device)
        fd.fd_decode_paged(w.q, w.k_cache, w.v_cache, w.kv_scales, w.page_table, w.cache_seqlens,
                           s.q_per_req, S, out, lse)
        torch.cuda.synchronize()
    finally:
        fd.fd_set_plan(None)
        fd.fd_plan_destroy(plan)
    return out, lse


def _close(a_out, a_lse, b_out, b_lse):
    assert torch.equal(torch.isneginf(a_lse), torch.isneginf(b_lse))
    fin = torch.isfinite(b_lse)
    assert (a_out.float() - b_out.float()).abs().max().item() <= OUT_ATOL
    assert (a_lse[fin] - b_lse[fin]).abs().max().item() <= LSE_ATOL


CASES = [
    # kind, B, Tq, Hq, Hkv, D, P, lengths, num_splits
    ("bf16", 3, 1, 16, 4, 128, 16, (700, 1500, 33), 4),
    ("int8", 2, 1, 32, 8, 128, 16, (2000, 900), 8),
    ("int4", 2, 4, 32, 8, 128, 16, (1500, 333), 3),
    ("bf16", 2, 1, 8, 2, 64, 64, (300, 1), 1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-D{c[5]}-S{c[8]}")
def test_static_entry_matches_plan_entry_on_two_calls(case):
    kind, B, Tq, Hq, Hkv, D, P, lengths, S = case
    shape = wl.DecodeShape("static", B, Hq, Hkv, D, P, Tq, kind, "fixed:" + ",".join(map(str, lengths)))
    w = wl.make_workload(shape, 500 + CASES.index(case), "cuda", poison=True)
    ref_out, ref_lse = _plan_call(w, S)
    for _ in range(2):
        out = torch.full_like(w.q, float("nan"))
        lse = torch.full(w.q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
        fd.fd_decode_paged_static(w.q, w.k_cache, w.v_cache, w.kv_scales, w.page_table, w.cache_seqlens,
                                  Tq, S, 0.0, out, lse)
        torch.cuda.synchronize()
        _close(out, lse, ref_out, ref_lse)


def test_static_entry_rejects_workspace_beyond_its_array():
    shape = wl.DecodeShape("big", 64, 64, 8, 128, 64, 1, "bf16", "const:64")
    w = wl.make_workload(shape, 7, "cuda")
    out = torch.empty_like(w.q)
    lse = torch.empty(w.q.shape[:3], dtype=torch.float32, device="cuda")
    with pytest.raises(fd.FdError) as e:
        # 64 x 64 x 64 rows of 129 floats = 135 MB > the 32 MiB array
        fd.fd_decode_paged_static(w.q, w.k_cache, w.v_cache, None, w.page_table, w.cache_seqlens, 1, 64, 0.0,
                                  out, lse)
    assert e.value.status == fd.FD_ERR_WORKSPACE
