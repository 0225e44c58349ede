"""The decode entry point that allocates no device memory.

Some callers cannot call cudaMalloc: an engine that has reserved all GPU memory
for its own pool, or a plugin in a process that forbids foreign allocations.
They call fd_decode_paged_static, which runs the same kernels with a fixed
scratch array inside the library. Here it is checked, through the C ABI, on
two calls in a row (the second reuses the scratch the first left behind):

* against the float64 oracle, with the parity bar, the tighter gates and the
  needle rows of the other parity tests;
* against the plan-based fd_decode_paged on the same inputs;
* for allocations: after the first calls, further calls leave the device's
  free memory unchanged.

This file is collected last and must pass alone in a fresh process too.
"""
import pytest
import torch

import split_kv_paged_gqa_gb300 as fd
from oracle import decode_ref_inputs
from split_kv_paged_gqa_gb300 import workloads as wl
from tests.gpu_common import LSE_ATOL, OUT_ATOL, assert_needles, assert_parity

pytestmark = pytest.mark.gpu


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
        fd.fd_plan_set_split_policy(plan, "equal")   # the static path always splits equally
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


def _static_call(w, S, out, lse):
    fd.fd_decode_paged_static(w.q, w.k_cache, w.v_cache, w.kv_scales, w.page_table, w.cache_seqlens,
                              w.shape.q_per_req, S, 0.0, out, lse)


CASES = [
    # kind, B, Tq, Hq, Hkv, D, P, lengths, num_splits
    ("bf16", 3, 1, 16, 4, 128, 16, (700, 1500, 33), 4),
    ("int8", 2, 1, 32, 8, 128, 16, (2000, 900), 8),
    ("int4", 2, 4, 32, 8, 128, 16, (1500, 333), 3),
    ("bf16", 2, 1, 8, 2, 64, 64, (300, 1), 1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-D{c[5]}-S{c[8]}")
def test_static_entry_matches_oracle_and_plan_entry_on_two_calls(case):
    kind, B, Tq, Hq, Hkv, D, P, lengths, S = case
    shape = wl.DecodeShape("static", B, Hq, Hkv, D, P, Tq, kind, "fixed:" + ",".join(map(str, lengths)))
    w = wl.make_workload(shape, 500 + CASES.index(case), "cuda", poison=True, needles=True, extra_pages=2)
    inp = wl.oracle_inputs(w)
    ref_out, ref_lse = decode_ref_inputs(inp)
    plan_out, plan_lse = _plan_call(w, S)
    for call in range(2):
        out = torch.full_like(w.q, float("nan"))
        lse = torch.full(w.q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
        _static_call(w, S, out, lse)
        torch.cuda.synchronize()
        assert_parity(out, lse, ref_out, ref_lse, label=f"static {kind} S={S} call {call}", bf16_rounding=True)
        assert_needles(w, out, inp)
        _close(out, lse, plan_out, plan_lse)


def test_static_entry_allocates_nothing_on_later_calls():
    shape = wl.DecodeShape("static", 3, 32, 8, 128, 16, 4, "int4", "fixed:1500,333,2600")
    w = wl.make_workload(shape, 509, "cuda")
    out = torch.empty_like(w.q)
    lse = torch.empty(w.q.shape[:3], dtype=torch.float32, device="cuda")
    for S in (1, 3):                         # first calls: set-up, both kernels loaded
        _static_call(w, S, out, lse)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        for S in (1, 3, 8):
            _static_call(w, S, out, lse)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes across static calls"


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
