"""GPU parity of the CUDA path (through the C ABI) against the float64 oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import split_kv_paged_gqa_gb300 as fd
from oracle import decode_ref_inputs
from split_kv_paged_gqa_gb300 import workloads as wl
from tests.gpu_common import (OUT_ATOL, SPLIT_ATOL, assert_needles, assert_parity, plan_for, run)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _shape(kind, B, Tq, Hq, Hkv, D, P, lengths):
    return wl.DecodeShape("case", B, Hq, Hkv, D, P, Tq, kind, "fixed:" + ",".join(map(str, lengths)))


# ---------------------------------------------------------------------------
# the tiny workload, both split counts, bf16 and fp32 outputs


@pytest.mark.parametrize("S", [1, 4])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_tiny_bf16(S, out_dtype):
    shape = wl.CONFIGS["tiny_bf16"]
    w = wl.make_workload(shape, wl.CONFIG_SEEDS["tiny_bf16"], "cuda", poison=True)
    ref_out, ref_lse = decode_ref_inputs(wl.oracle_inputs(w))
    out, lse = run(w, S, out_dtype)
    assert_parity(out, lse, ref_out, ref_lse, label=f"tiny S={S}")


# ---------------------------------------------------------------------------
# several tiles, ragged tails, every cache format, GQA groups, MTP, page sizes

CASES = [
    # kind, B, Tq, Hq, Hkv, D, P, lengths
    ("bf16", 3, 1, 8, 2, 64, 16, (1, 300, 1023)),
    ("bf16", 2, 1, 40, 8, 128, 16, (777, 2050)),
    ("bf16", 2, 1, 64, 8, 128, 64, (4096, 1000)),
    ("bf16", 2, 4, 32, 8, 128, 16, (517, 1290)),
    ("bf16", 2, 1, 16, 1, 128, 256, (600, 129)),        # G=16, sub-page stages
    ("bf16", 2, 4, 32, 4, 128, 32, (99, 400)),          # R = 32 rows: two row tiles
    ("bf16", 2, 1, 4, 4, 64, 8, (70, 3)),               # smallest page size
    ("bf16", 2, 2, 12, 2, 64, 8, (45, 200)),
    ("int8", 3, 1, 32, 8, 128, 16, (16, 900, 2500)),
    ("int8", 2, 1, 8, 2, 64, 64, (300, 130)),
    ("int8", 2, 4, 32, 8, 128, 16, (1000, 67)),
    ("int4", 2, 4, 32, 8, 128, 16, (4096, 1111)),
    ("int4", 3, 1, 8, 2, 128, 64, (70, 640, 2000)),
    ("int4", 2, 1, 16, 4, 64, 16, (333, 48)),
    # quantised tiles of <= 8 rows run keys-as-M ("narrow"): causal MTP rows,
    # one row (MHA), and a 12-row tile that stays on the 16-row layout
    ("int8", 2, 2, 16, 4, 128, 16, (700, 33)),          # R = 8, causal
    ("int4", 2, 4, 8, 4, 128, 32, (260, 1500)),         # R = 8, causal
    ("int4", 2, 1, 8, 8, 128, 16, (129, 2000)),         # R = 1
    ("int8", 2, 3, 32, 8, 64, 16, (500, 81)),           # R = 12
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-B{c[1]}-T{c[2]}-H{c[3]}/{c[4]}-D{c[5]}-P{c[6]}")
@pytest.mark.parametrize("S", [1, 3, 8])
def test_parity_cases(case, S):
    shape = _shape(*case)
    w = wl.make_workload(shape, 100 + CASES.index(case), "cuda", poison=True, needles=True, extra_pages=3)
    inp = wl.oracle_inputs(w)
    ref_out, ref_lse = decode_ref_inputs(inp)
    out32, lse32 = run(w, S, torch.float32)
    assert_parity(out32, lse32, ref_out, ref_lse, label=f"{case} S={S} fp32 out")
    out, lse = run(w, S)
    assert_parity(out, lse, ref_out, ref_lse, label=f"{case} S={S} bf16 out", bf16_rounding=True)
    assert_needles(w, out, inp)


# The scales of a quantised cache in two memory orders: head-major within a
# page (the workloads' order: the scales of one (page, head) are contiguous)
# and the logical order [2, N, P, Hkv, n_g] made contiguous (the 8 heads of a
# slot interleaved).
@pytest.mark.parametrize("case", [c for c in CASES if c[0] != "bf16"],
                         ids=lambda c: f"{c[0]}-B{c[1]}-T{c[2]}-H{c[3]}/{c[4]}-D{c[5]}-P{c[6]}")
def test_parity_scale_memory_orders(case):
    shape = _shape(*case)
    w = wl.make_workload(shape, 300 + CASES.index(case), "cuda", poison=True, needles=True, extra_pages=2)
    inp = wl.oracle_inputs(w)
    ref_out, ref_lse = decode_ref_inputs(inp)
    assert w.kv_scales.stride(2) == w.kv_scales.shape[4]          # head-major: slots contiguous
    for scales in (w.kv_scales, w.kv_scales.contiguous()):
        w2 = dataclasses.replace(w, kv_scales=scales)
        for S in (1, 3):
            out32, lse32 = run(w2, S, torch.float32)
            assert_parity(out32, lse32, ref_out, ref_lse, label=f"{case} S={S} strides {scales.stride()}")


# Stage tails. The 16-row INT4 tile and the narrow INT8 tile take 32 keys per
# consumer warp in two 16-key sub-blocks (128-key stages), so a split's last
# stage can end inside a warp's first or second sub-block, on a sub-block
# edge, or leave whole warps idle. One length for each of those residues
# (mod 128), with causal MTP rows whose limits fall inside the last stage. The
# narrow INT4 tile (16 keys per warp, 64-key stages) runs the same lengths.
TAIL_LENGTHS = tuple(256 + r for r in (1, 2, 15, 16, 17, 31, 32, 33, 47, 63, 64, 65, 95, 96, 97, 111, 127, 128))


@pytest.mark.parametrize("kind,Tq,Hq,D", [("int4", 4, 32, 128), ("int4", 1, 128, 128), ("int4", 4, 32, 64),
                                          ("int4", 1, 32, 128), ("int4", 2, 32, 128),
                                          ("int8", 1, 32, 128), ("int8", 2, 32, 128), ("int8", 1, 32, 64)])
@pytest.mark.parametrize("S", [1, 3])
def test_stage_tail_residues(kind, Tq, Hq, D, S):
    shape = _shape(kind, len(TAIL_LENGTHS), Tq, Hq, 8, D, 16, TAIL_LENGTHS)
    w = wl.make_workload(shape, 7 + Tq + S, "cuda", poison=True, needles=True, extra_pages=2)
    inp = wl.oracle_inputs(w)
    ref_out, ref_lse = decode_ref_inputs(inp)
    label = f"{kind} Tq={Tq} Hq={Hq} D={D} S={S} tails"
    out32, lse32 = run(w, S, torch.float32)
    assert_parity(out32, lse32, ref_out, ref_lse, label=label + " fp32 out")
    out, lse = run(w, S)
    assert_parity(out, lse, ref_out, ref_lse, label=label, bf16_rounding=True)
    assert_needles(w, out, inp)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-B{c[1]}-T{c[2]}-H{c[3]}/{c[4]}-D{c[5]}-P{c[6]}")
@pytest.mark.parametrize("S", [3, 8])
def test_parity_cases_equal_policy(case, S):
    """The same cases with equal splits per request (FD_SPLIT_EQUAL)."""
    shape = _shape(*case)
    w = wl.make_workload(shape, 100 + CASES.index(case), "cuda", poison=True, needles=True, extra_pages=3)
    inp = wl.oracle_inputs(w)
    ref_out, ref_lse = decode_ref_inputs(inp)
    plan = fd.fd_plan_create(0, shape.batch, shape.q_per_req, shape.num_q_heads, shape.num_kv_heads,
                             shape.head_dim, shape.page_size, shape.kv_dtype, 64)
    try:
        fd.fd_plan_set_split_policy(plan, "equal")
        out32, lse32 = run(w, S, torch.float32, plan=plan)
        assert_parity(out32, lse32, ref_out, ref_lse, label=f"{case} S={S} equal")
        assert_needles(w, out32, inp)
    finally:
        fd.fd_set_plan(None)
        fd.fd_plan_destroy(plan)


def _plan_with_env(shape, monkeypatch, max_splits=64, **env):
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    plan = fd.fd_plan_create(0, shape.batch, shape.q_per_req, shape.num_q_heads, shape.num_kv_heads,
                             shape.head_dim, shape.page_size, shape.kv_dtype, max_splits)
    for k in env:
        monkeypatch.delenv(k)
    return plan


@pytest.mark.parametrize("case", [c for c in CASES if c[0] != "bf16" and c[5] == 128],
                         ids=lambda c: f"{c[0]}-B{c[1]}-T{c[2]}-H{c[3]}/{c[4]}-D{c[5]}-P{c[6]}")
@pytest.mark.parametrize("S", [1, 3, 8])
def test_parity_cases_tcgen05_kernel(case, S, monkeypatch):
    """Quantised head_dim-128 cases on the tcgen05 stage-1 kernel (FD_QUANT_KERNEL=tc)."""
    shape = _shape(*case)
    w = wl.make_workload(shape, 100 + CASES.index(case), "cuda", poison=True, needles=True, extra_pages=3)
    inp = wl.oracle_inputs(w)
    ref_out, ref_lse = decode_ref_inputs(inp)
    plan = _plan_with_env(shape, monkeypatch, FD_QUANT_KERNEL="tc")
    try:
        out32, lse32 = run(w, S, torch.float32, plan=plan)
        assert_parity(out32, lse32, ref_out, ref_lse, label=f"{case} S={S} tcgen05 kernel")
        assert_needles(w, out32, inp)
        out, lse = run(w, S, plan=plan)
        assert_parity(out, lse, ref_out, ref_lse, label=f"{case} S={S} tcgen05 bf16 out", bf16_rounding=True)
    finally:
        fd.fd_set_plan(None)
        fd.fd_plan_destroy(plan)


@pytest.mark.parametrize("kind", ["int8", "int4"])
def test_tcgen05_kernel_skewed_batch_and_split_agreement(kind, monkeypatch):
    Tq = 4 if kind == "int4" else 1
    lengths = (0, 9000, 3, 40, 0, 129, 1, 2000)
    shape = _shape(kind, len(lengths), Tq, 16, 4, 128, 16, lengths)
    w = wl.make_workload(shape, 56, "cuda", poison=True, needles=True)
    inp = wl.oracle_inputs(w)
    ref_out, ref_lse = decode_ref_inputs(inp)
    plan = _plan_with_env(shape, monkeypatch, FD_QUANT_KERNEL="tc")
    try:
        base = None
        for S in (1, 2, 7, 64):
            out32, lse32 = run(w, S, torch.float32, plan=plan)
            assert_parity(out32, lse32, ref_out, ref_lse, label=f"{kind} tcgen05 S={S}")
            assert_needles(w, out32, inp)
            if base is None:
                base = out32
            assert (out32 - base).abs().max().item() <= SPLIT_ATOL
        assert fd.fd_read_device_status(plan) == 0
    finally:
        fd.fd_set_plan(None)
        fd.fd_plan_destroy(plan)


# ---------------------------------------------------------------------------
# balanced splits on skewed batches: empty requests, one long request among
# short ones, and a workspace so small that long requests hit its split cap


@pytest.mark.parametrize("kind", ["bf16", "int8", "int4"])
@pytest.mark.parametrize("max_splits", [2, 64])
def test_balanced_splits_on_skewed_batches(kind, max_splits):
    Tq = 4 if kind == "int4" else 1
    lengths = (0, 9000, 3, 40, 0, 129, 1, 2000)
    shape = _shape(kind, len(lengths), Tq, 16, 4, 128, 16, lengths)
    w = wl.make_workload(shape, 55, "cuda", poison=True, needles=True)
    inp = wl.oracle_inputs(w)
    ref_out, ref_lse = decode_ref_inputs(inp)
    # max_splits 2: the workspace holds 2 partials per output row, so the long
    # request is cut into 2 splits however many the balanced map asks for
    plan = fd.fd_plan_create(0, shape.batch, Tq, 16, 4, 128, 16, kind, max_splits)
    try:
        for S in sorted({1, 2, min(4, max_splits), max_splits}):
            out32, lse32 = run(w, S, torch.float32, plan=plan)
            assert_parity(out32, lse32, ref_out, ref_lse, label=f"{kind} balanced S={S} cap={max_splits}")
            assert_needles(w, out32, inp)
    finally:
        fd.fd_set_plan(None)
        fd.fd_plan_destroy(plan)


# ---------------------------------------------------------------------------
# results for different num_splits agree


@pytest.mark.parametrize("policy", ["balanced", "equal"])
@pytest.mark.parametrize("kind", ["bf16", "int8", "int4"])
def test_cross_split_agreement(kind, policy):
    shape = _shape(kind, 3, 1, 32, 8, 128, 16, (3000, 5000, 129))
    w = wl.make_workload(shape, 7, "cuda", poison=True)
    plan = plan_for(shape)
    fd.fd_plan_set_split_policy(plan, policy)
    base_f, base_l = run(w, 1, torch.float32)
    base_b, _ = run(w, 1, torch.bfloat16)
    for S in (2, 4, 8, 16, 32, 64):
        of, lf = run(w, S, torch.float32)
        assert (of - base_f).abs().max().item() <= SPLIT_ATOL, f"fp32 out S={S}"
        assert (lf - base_l).abs().max().item() <= SPLIT_ATOL, f"lse S={S}"
        ob, _ = run(w, S, torch.bfloat16)
        d = (ob.float() - base_b.float()).abs()
        ulp = torch.where(base_b.float().abs() >= 0.5, 2.0 ** -7, 0.0)   # one bf16 rounding flip
        assert (d <= SPLIT_ATOL + ulp).all(), f"bf16 out S={S}: {d.max().item()}"
    fd.fd_plan_set_split_policy(plan, "balanced")


# ---------------------------------------------------------------------------
# mixed lengths with any max-length hint (exact, stale, loose) and many splits


@pytest.mark.parametrize("kind", ["bf16", "int8", "int4"])
def test_mixed_lengths_with_max_length_hints(kind):
    Tq = 4 if kind == "int4" else 1
    shape = _shape(kind, 5, Tq, 32, 8, 128, 16, (50, 3000, 12000, 700, 4))
    w = wl.make_workload(shape, 77, "cuda", poison=True)
    ref_out, ref_lse = decode_ref_inputs(wl.oracle_inputs(w))
    plan = fd.fd_plan_create(0, 5, Tq, 32, 8, 128, 16, kind, 64)
    try:
        for hint in (12000, 1000, 16384):          # exact, stale (too small), loose
            fd.fd_set_max_seqlen_hint(plan, hint)
            for S in (4, 16, 64):
                out32, lse32 = run(w, S, torch.float32, plan=plan)
                assert_parity(out32, lse32, ref_out, ref_lse, label=f"{kind} hint={hint} S={S}")
    finally:
        fd.fd_set_plan(None)
        fd.fd_plan_destroy(plan)


# ---------------------------------------------------------------------------
# split merge: the stage-2 kernel (default) and, under the equal split
# policy, the opt-in fused merge in stage 1


@pytest.mark.parametrize("kind", ["bf16", "int4"])
def test_fused_merge_matches_oracle_and_stage2_merge(kind, monkeypatch):
    Tq = 4 if kind == "int4" else 1
    shape = _shape(kind, 4, Tq, 32, 8, 128, 16, (2000, 37, 0, 5000))
    w = wl.make_workload(shape, 88, "cuda", poison=True)
    ref_out, ref_lse = decode_ref_inputs(wl.oracle_inputs(w))
    monkeypatch.delenv("FD_MERGE", raising=False)
    # the fused merge runs in the register stage-1 kernel: compare it with the
    # stage-2 merge on the same stage-1 kernel
    monkeypatch.setenv("FD_QUANT_KERNEL", "mma")
    plan2 = fd.fd_plan_create(0, 4, Tq, 32, 8, 128, 16, kind, 64)
    monkeypatch.setenv("FD_MERGE", "fused")
    plan1 = fd.fd_plan_create(0, 4, Tq, 32, 8, 128, 16, kind, 64)
    monkeypatch.delenv("FD_MERGE")
    monkeypatch.delenv("FD_QUANT_KERNEL")
    # the fused merge serves the equal policy; both plans use it so that their
    # splits, and so their rounding, are the same
    fd.fd_plan_set_split_policy(plan1, "equal")
    fd.fd_plan_set_split_policy(plan2, "equal")
    try:
        for S in (2, 7, 64):   # plan2: stage-2 kernel; plan1: fused merge, including an empty request
            o2, l2 = run(w, S, torch.float32, plan=plan2)
            assert_parity(o2, l2, ref_out, ref_lse, label=f"stage-2 merge S={S}")
            o1, l1 = run(w, S, torch.float32, plan=plan1)
            assert_parity(o1, l1, ref_out, ref_lse, label=f"fused merge S={S}")
            assert (o1 - o2).abs().max().item() <= 1e-5
    finally:
        fd.fd_set_plan(None)
        fd.fd_plan_destroy(plan1)
        fd.fd_plan_destroy(plan2)


# ---------------------------------------------------------------------------
# edge cases


@pytest.mark.parametrize("kind,Tq", [("bf16", 4), ("int8", 4), ("int4", 4), ("int8", 2), ("int4", 2)])
def test_rows_without_keys(kind, Tq):
    # L = 0 and L < Tq: rows with no visible key get out = 0, lse = -inf
    # (quantised: 16-row tiles at Tq 4, narrow 8-row tiles at Tq 2)
    shape = _shape(kind, 3, Tq, 8, 2, 64, 16, (0, 2, 17))
    w = wl.make_workload(shape, 3, "cuda", poison=True, capacity_pages=2)
    ref_out, ref_lse = decode_ref_inputs(wl.oracle_inputs(w))
    for S in (1, 4):
        out, lse = run(w, S)
        # rows that see one or two keys return (nearly) a V row, |out| up to ~4:
        # rounding to bf16 alone then takes up to half a bf16 ulp
        assert_parity(out, lse, ref_out, ref_lse, label=f"{kind} empty S={S}", bf16_rounding=True)
        assert torch.isneginf(lse[0]).all() and (out[0] == 0).all()


@pytest.mark.parametrize("kind", ["bf16", "int8", "int4"])
def test_more_splits_than_pages(kind):
    shape = _shape(kind, 2, 1, 8, 2, 64, 16, (20, 33))
    w = wl.make_workload(shape, 5, "cuda", poison=True)
    ref_out, ref_lse = decode_ref_inputs(wl.oracle_inputs(w))
    out, lse = run(w, 64)
    assert_parity(out, lse, ref_out, ref_lse, label=f"{kind} S=64 on 2-3 pages")


@pytest.mark.parametrize("kind", ["bf16", "int8", "int4"])
def test_strided_outputs_and_queries(kind):
    shape = _shape(kind, 2, 1, 16, 4, 128, 16, (500, 901))
    w = wl.make_workload(shape, 9, "cuda")
    ref_out, ref_lse = decode_ref_inputs(wl.oracle_inputs(w))
    big_q = torch.zeros((2, 1, 16, 256), dtype=torch.bfloat16, device="cuda")
    big_q[..., 64:192] = w.q
    q_view = big_q[..., 64:192]                      # non-contiguous query rows
    out_big = torch.full((2, 1, 16, 136), 7.0, dtype=torch.bfloat16, device="cuda")
    out_view = out_big[..., :128]
    lse_big = torch.zeros((2, 1, 16, 2), dtype=torch.float32, device="cuda")
    lse_view = lse_big[..., 0]
    fd.fd_set_plan(plan_for(shape))
    for S in (1, 4):
        fd.fd_decode_paged(q_view, w.k_cache, w.v_cache, w.kv_scales, w.page_table, w.cache_seqlens, 1, S,
                           out_view, lse_view)
        torch.cuda.synchronize()
        assert_parity(out_view, lse_view, ref_out, ref_lse, label=f"{kind} strided S={S}")
        assert (out_big[..., 128:] == 7.0).all()       # padding untouched


@pytest.mark.parametrize("kind,Tq", [("int4", 4), ("int8", 1), ("bf16", 1)])
def test_deterministic(kind, Tq):
    shape = _shape(kind, 2, Tq, 32, 8, 128, 16, (3000, 1700))
    w = wl.make_workload(shape, 13, "cuda")
    a, la = run(w, 8)
    for _ in range(5):
        b, lb = run(w, 8)
        assert torch.equal(a, b) and torch.equal(la, lb)


# ---------------------------------------------------------------------------
# bad metadata is reported, not faulted on


@pytest.mark.parametrize("kind", ["bf16", "int8", "int4"])
def test_bad_page_id_sets_status(kind):
    shape = _shape(kind, 2, 1, 8, 2, 64, 16, (100, 40))
    w = wl.make_workload(shape, 21, "cuda")
    plan = plan_for(shape)
    fd.fd_read_device_status(plan)                     # clear
    pt = w.page_table.clone()
    pt[0, 2] = w.k_cache.shape[0] + 5                   # outside the pool
    w.page_table = pt
    out, lse = run(w, 2)
    assert fd.fd_read_device_status(plan) & fd.FD_DEVSTAT_BAD_PAGE
    assert fd.fd_read_device_status(plan) == 0          # reading cleared it
    assert torch.isfinite(out.float()).all()


def test_seqlen_over_capacity_sets_status():
    shape = _shape("bf16", 2, 1, 8, 2, 64, 16, (100, 40))
    w = wl.make_workload(shape, 22, "cuda")
    plan = plan_for(shape)
    fd.fd_read_device_status(plan)
    w.cache_seqlens = torch.tensor([100, 40 + 10 * 16 * 7], dtype=torch.int32, device="cuda")
    run(w, 1)
    assert fd.fd_read_device_status(plan) & fd.FD_DEVSTAT_SEQLEN_OVERFLOW


def test_wait_that_never_completes_times_out_and_the_context_stays_usable():
    # The kernels' bounded wait on a barrier that nothing arrives on gives up
    # after its limit, records the status bit and returns; a decode call on the
    # same plan afterwards still matches the oracle.
    import time
    shape = _shape("bf16", 2, 1, 8, 2, 64, 16, (100, 40))
    w = wl.make_workload(shape, 23, "cuda")
    plan = fd.fd_plan_create(0, 2, 1, 8, 2, 64, 16, "bf16", 4)
    try:
        assert fd.fd_read_device_status(plan) == 0
        t0 = time.perf_counter()
        fd.fd_selftest_wait_timeout(plan, 2000)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        assert fd.fd_read_device_status(plan) == fd.FD_DEVSTAT_WAIT_TIMEOUT
        assert elapsed < 1.0, f"the 2 ms wait took {elapsed:.3f} s"
        ref_out, ref_lse = decode_ref_inputs(wl.oracle_inputs(w))
        out, lse = run(w, 4, plan=plan)
        assert_parity(out, lse, ref_out, ref_lse, label="decode after a timed-out wait")
        assert fd.fd_read_device_status(plan) == 0
        with pytest.raises(fd.FdError):
            fd.fd_selftest_wait_timeout(plan, 0)
    finally:
        fd.fd_set_plan(None)
        fd.fd_plan_destroy(plan)


# ---------------------------------------------------------------------------
# CUDA graph capture and replay with new metadata contents


def test_graph_capture_replay_picks_up_new_metadata():
    shape = _shape("bf16", 2, 1, 16, 4, 128, 16, (700, 1500))
    w = wl.make_workload(shape, 31, "cuda", extra_pages=200, capacity_pages=110)
    plan = plan_for(shape)
    fd.fd_set_plan(plan)
    out = torch.empty_like(w.q)
    lse = torch.empty(w.q.shape[:3], dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):            # warm-up outside capture
        fd.fd_decode_paged(w.q, w.k_cache, w.v_cache, None, w.page_table, w.cache_seqlens, 1, 4, out, lse)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fd.fd_decode_paged(w.q, w.k_cache, w.v_cache, None, w.page_table, w.cache_seqlens, 1, 4, out, lse)
    rng = np.random.default_rng(4)
    for trial in range(3):
        lens = rng.integers(1, 1600, size=2)
        n_pages = w.k_cache.shape[0]
        new_pt = torch.full_like(w.page_table, -1)
        for b in range(2):
            need = -(-int(lens[b]) // 16)
            new_pt[b, :need] = torch.from_numpy(rng.choice(n_pages, need, replace=False).astype(np.int32))
        w.page_table.copy_(new_pt)
        w.cache_seqlens.copy_(torch.from_numpy(lens.astype(np.int32)))
        w.lengths = lens
        g.replay()
        torch.cuda.synchronize()
        ref_out, ref_lse = decode_ref_inputs(wl.oracle_inputs(w))
        assert_parity(out, lse, ref_out, ref_lse, label=f"graph replay {trial}")


def test_profiled_calls_inside_a_captured_graph():
    """Profiling events captured as graph nodes: timed per call, results unchanged."""
    shape = _shape("bf16", 2, 1, 16, 4, 128, 16, (700, 1500))
    w = wl.make_workload(shape, 33, "cuda")
    plan = plan_for(shape)
    fd.fd_set_plan(plan)
    out = torch.empty_like(w.q)
    lse = torch.empty(w.q.shape[:3], dtype=torch.float32, device="cuda")

    def call():
        fd.fd_decode_paged(w.q, w.k_cache, w.v_cache, None, w.page_table, w.cache_seqlens, 1, 4, out, lse)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    fd.fd_profile_begin(plan)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
            call()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    del g
    calls, s1_ms, s2_ms = fd.fd_profile_end(plan)
    assert calls == 3 and s1_ms > 0 and s2_ms > 0
    ref_out, ref_lse = decode_ref_inputs(wl.oracle_inputs(w))
    assert_parity(out, lse, ref_out, ref_lse, label="profiled graph")


# ---------------------------------------------------------------------------
# full-size workloads, in the launch configuration the bench times, on sampled requests


FULL = ["mixed_bf16", "long_bf16_b64", "int8_lognormal", "int4_mtp"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    shape = wl.CONFIGS[name]
    w = wl.make_workload(shape, wl.CONFIG_SEEDS[name], "cuda")
    plan = plan_for(shape, max_splits=64)
    fd.fd_set_max_seqlen_hint(plan, int(w.lengths.max()))
    out, lse = run(w, 0, plan=plan)                    # num_splits from the plan (bench setting)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(0)
    sample = sorted(set([int(np.argmax(w.lengths)), int(np.argmin(w.lengths))] +
                        rng.choice(shape.batch, 2, replace=False).tolist()))
    inp = wl.oracle_inputs(w, requests=sample)
    ref_out, ref_lse = decode_ref_inputs(inp)
    assert_parity(out, lse, ref_out, ref_lse, requests=sample, label=name)
    del w
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# the long-context sweep at full size: one 32768-key request, and two requests
# of the 16-request batch, against the oracle at every num_splits of the sweep
# (batch 1 at 16 splits runs the one-wave deep variant the tuner picks there),
# plus agreement between split counts on the whole 16-request batch


SWEEP_S = (1, 2, 4, 8, 16, 32, 64)


@pytest.fixture(scope="module")
def long_b1():
    name = "long_bf16_b1"
    w = wl.make_workload(wl.CONFIGS[name], wl.CONFIG_SEEDS[name], "cuda", needles=True)
    inp = wl.oracle_inputs(w)
    ref = decode_ref_inputs(inp)
    yield w, inp, ref
    del w
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def long_b16():
    name = "long_bf16_b16"
    w = wl.make_workload(wl.CONFIGS[name], wl.CONFIG_SEEDS[name], "cuda")
    sample = [3, 12]
    ref = decode_ref_inputs(wl.oracle_inputs(w, requests=sample))
    yield w, sample, ref
    del w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("S", SWEEP_S)
def test_full_size_long_b1_every_split_count(long_b1, S):
    w, inp, (ref_out, ref_lse) = long_b1
    plan = plan_for(w.shape, max_splits=64)
    out32, lse32 = run(w, S, torch.float32, plan=plan)
    assert_parity(out32, lse32, ref_out, ref_lse, label=f"B1 x 32K S={S} fp32 out")
    out, lse = run(w, S, plan=plan)
    assert_parity(out, lse, ref_out, ref_lse, label=f"B1 x 32K S={S} bf16 out", bf16_rounding=True)
    assert_needles(w, out, inp)


@pytest.mark.parametrize("S", SWEEP_S)
def test_full_size_long_b16_every_split_count(long_b16, S):
    w, sample, (ref_out, ref_lse) = long_b16
    plan = plan_for(w.shape, max_splits=64)
    out, lse = run(w, S, plan=plan)
    assert_parity(out, lse, ref_out, ref_lse, requests=sample, label=f"B16 x 32K S={S}")


@pytest.mark.parametrize("policy", ["balanced", "equal"])
def test_full_size_long_b16_split_agreement(long_b16, policy):
    w, _, _ = long_b16
    plan = plan_for(w.shape, max_splits=64)
    fd.fd_plan_set_split_policy(plan, policy)
    try:
        base_f, base_l = run(w, 1, torch.float32, plan=plan)
        for S in SWEEP_S[1:]:
            of, lf = run(w, S, torch.float32, plan=plan)
            assert (of - base_f).abs().max().item() <= SPLIT_ATOL, f"fp32 out S={S}"
            assert (lf - base_l).abs().max().item() <= SPLIT_ATOL, f"lse S={S}"
    finally:
        fd.fd_plan_set_split_policy(plan, "balanced")


# ---------------------------------------------------------------------------
# the startup tuner on the device: both tables, then decode with its pick


def test_autotune_on_device_then_decode(tmp_path):
    import json
    shape = _shape("bf16", 4, 1, 16, 4, 128, 16, (300, 1800, 900, 40))
    w = wl.make_workload(shape, 61, "cuda", poison=True)
    ref_out, ref_lse = decode_ref_inputs(wl.oracle_inputs(w))
    plan = fd.fd_plan_create(0, 4, 1, 16, 4, 128, 16, "bf16", 16)
    try:
        fd.fd_autotune_set_cache_dir(plan, str(tmp_path))
        fd.fd_autotune(plan, [4], 1024, 2048)
        assert fd.fd_autotune_stats(plan) == (4, 0)          # 2 buckets x (equal, mixed lengths)
        entries = json.load(open(next(tmp_path.glob("fd_splits_*.json"))))["entries"]
        assert len(entries) == 4 and sum(e["spread"] for e in entries) == 2
        assert all(1 <= e["num_splits"] <= 16 and e["time"] > 0 for e in entries)
        fd.fd_set_max_seqlen_hint(plan, 1800)
        fd.fd_set_mean_seqlen_hint(plan, 760)
        S = fd.fd_query_splits(plan, 4, 1800)
        assert 1 <= S <= 16
        out, lse = run(w, 0, torch.float32, plan=plan)         # num_splits from the table
        assert_parity(out, lse, ref_out, ref_lse, label=f"tuned S={S}")
        assert fd.fd_read_device_status(plan) == 0
    finally:
        fd.fd_set_plan(None)
        fd.fd_plan_destroy(plan)


# ---------------------------------------------------------------------------
# warmup phases on the device: a decode call in the decode-attention phase
# tunes its batch at the representative length, and the graph captured after
# it uses the tuned value; the rebuild hook sees each tuning key


def test_warmup_decode_call_tunes_then_capture_uses_it(tmp_path, monkeypatch):
    monkeypatch.setenv("FD_AUTOTUNE_SEQ_LEN", "2048")
    shape = _shape("bf16", 3, 1, 16, 4, 128, 16, (5, 9, 2))    # graph-init style short requests
    w = wl.make_workload(shape, 91, "cuda", extra_pages=200, capacity_pages=140)
    plan = fd.fd_plan_create(0, 3, 1, 16, 4, 128, 16, "bf16", 16)
    seen = []
    try:
        fd.fd_autotune_set_cache_dir(plan, str(tmp_path))
        fd.fd_autotune_set_input_hook(plan, lambda b, k, mixed, q, kc, vc, sc: seen.append(
            (b, k, mixed, tuple(q.shape[:4]), tuple(kc.shape[1:4]), sc is None)))
        fd.fd_set_plan(plan)
        out = torch.empty_like(w.q)
        lse = torch.empty(w.q.shape[:3], dtype=torch.float32, device="cuda")
        fd.fd_decode_paged(w.q, w.k_cache, w.v_cache, None, w.page_table, w.cache_seqlens, 1, 0, out, lse)
        torch.cuda.synchronize()
        assert fd.fd_autotune_stats(plan)[0] == 0                 # live phase: no tuning
        with fd.warmup(fd.FD_PHASE_DECODE_ATTENTION):
            fd.fd_decode_paged(w.q, w.k_cache, w.v_cache, None, w.page_table, w.cache_seqlens, 1, 0, out, lse)
        torch.cuda.synchronize()
        assert fd.fd_autotune_stats(plan)[0] == 2                 # (3, 2048): equal and mixed lengths
        assert sorted(x[:3] for x in seen) == [(3, 2048, 0), (3, 2048, 1)]
        assert all(x[3] == (3, 1, 16, 128) and x[4] == (16, 4, 128) and x[5] for x in seen)
        S = fd.fd_query_splits(plan, 3, 9)
        assert 1 <= S <= 16
        # capture with num_splits = 0 after warmup; replay with longer requests
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fd.fd_decode_paged(w.q, w.k_cache, w.v_cache, None, w.page_table, w.cache_seqlens, 1, 0, out, lse)
        rng = np.random.default_rng(8)
        lens = rng.integers(100, 2000, size=3)
        pages = rng.permutation(w.k_cache.shape[0])
        pt = torch.full_like(w.page_table, -1)
        k = 0
        for b in range(3):
            n = -(-int(lens[b]) // 16)
            pt[b, :n] = torch.from_numpy(pages[k:k + n].astype(np.int32))
            k += n
        w.page_table.copy_(pt)
        w.cache_seqlens.copy_(torch.from_numpy(lens.astype(np.int32)))
        w.lengths = lens
        g.replay()
        torch.cuda.synchronize()
        ref_out, ref_lse = decode_ref_inputs(wl.oracle_inputs(w))
        assert_parity(out, lse, ref_out, ref_lse, label="graph after warmup tuning")
        del g
        # a hook that fails aborts the tuning with its status
        fd.fd_autotune_clear(plan)
        fd.fd_autotune_set_input_hook(plan, lambda *a: 1 / 0)
        with pytest.raises(fd.FdError):
            fd.fd_autotune(plan, [3], 1024, 1024)
    finally:
        fd.fd_set_plan(None)
        fd.fd_plan_destroy(plan)
