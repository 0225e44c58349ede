"""Decode metadata from a request-to-token pool: the oracle's pins (CPU), the
C ABI's argument checks (CPU, no launch), and the CUDA kernel against the
oracle, alone and captured with the decode call in one CUDA graph (GPU)."""
import numpy as np
import pytest
import torch

import split_kv_paged_gqa_gb300 as fd
from oracle.graph_metadata_ref import Q_CUMSUM, Q_PRESET, Q_STRIDED, graph_metadata_ref
from split_kv_paged_gqa_gb300 import workloads as wl

# ---------------------------------------------------------------------------
# the oracle, pinned


def _hand_pool():
    # page size 4; pool row 0: one page (5); row 1: pages 2, 7, 0; row 2: page 3,
    # then a page start with no slot; row 3: empty
    P = 4
    pool = np.full((4, 12), -1, dtype=np.int32)
    pool[0, 0:4] = [20, 21, 22, 23]
    pool[1, 0:12] = [8, 9, 10, 11, 28, 29, 30, 31, 0, 1, 2, 3]
    pool[2, 0:4] = [12, 13, 14, 15]
    return pool, P


def test_oracle_hand_worked_example():
    pool, P = _hand_pool()
    idx = np.array([1, -1, 2, 0])          # row 1 is padding
    lens = np.array([10, 99, 6, 4])
    out = graph_metadata_ref(pool, idx, lens, P, 4, Q_CUMSUM, q_in=np.array([1, 5, 4, 2]))
    assert out["page_table"].tolist() == [[2, 7, 0, -1], [-1, -1, -1, -1], [3, -1, -1, -1], [5, -1, -1, -1]]
    assert out["cache_seqlens"].tolist() == [10, 0, 6, 4]
    assert out["cu_seqlens_k"].tolist() == [0, 10, 10, 16, 20]
    assert out["cu_seqlens_q"].tolist() == [0, 1, 1, 5, 7]   # the padding row adds no query tokens
    strided = graph_metadata_ref(pool, idx, lens, P, 4, Q_STRIDED, q_stride=4)
    assert strided["cu_seqlens_q"].tolist() == [0, 4, 8, 12, 16]
    preset = graph_metadata_ref(pool, idx, lens, P, 4, Q_PRESET, q_in=np.array([0, 3, 3, 9, 11]))
    assert preset["cu_seqlens_q"].tolist() == [0, 3, 3, 9, 11]
    narrow = graph_metadata_ref(pool, idx, lens, P, 2, Q_STRIDED, q_stride=1)
    assert narrow["page_table"].tolist() == [[2, 7], [-1, -1], [3, -1], [5, -1]]


@pytest.mark.parametrize("seed", range(6))
def test_oracle_against_token_level_slots(seed):
    """Every visible key's slot, read token by token from the pool, equals
    page_table[b, j // P] * P + j % P; the prefix sums match their definition."""
    rng = np.random.default_rng(seed)
    P = int(rng.choice([1, 2, 4, 16]))
    lens = rng.integers(0, 70, size=int(rng.integers(1, 9)))
    pool, _ = wl.make_token_pool(seed, lens, P, extra_rows=2)
    order = rng.permutation(len(pool))[:len(lens)]             # may pick the empty extra rows
    idx = np.where(rng.random(len(lens)) < 0.2, -1, order)    # -1: padding rows
    row_len = np.concatenate([lens, np.zeros(len(pool) - len(lens), dtype=lens.dtype)])
    seq = np.where(idx >= 0, row_len[np.maximum(idx, 0)], rng.integers(0, 50, size=len(idx)))
    W = int(max(1, (seq.max(initial=1) + P - 1) // P))
    q = rng.integers(0, 5, size=len(idx))
    out = graph_metadata_ref(pool, idx, seq, P, W, Q_CUMSUM, q_in=q)
    for b, r in enumerate(idx):
        if r < 0:
            assert (out["page_table"][b] == -1).all() and out["cache_seqlens"][b] == 0
            continue
        for j in range(int(seq[b])):
            assert pool[r, j] == out["page_table"][b, j // P] * P + j % P
        assert (out["page_table"][b, -(-int(seq[b]) // P):] == -1).all()
    live = idx >= 0
    assert out["cu_seqlens_k"][0] == 0 and (np.diff(out["cu_seqlens_k"]) == out["cache_seqlens"]).all()
    assert (np.diff(out["cu_seqlens_q"]) == np.where(live, q, 0)).all()


# ---------------------------------------------------------------------------
# argument checks of the C ABI (host pointers: nothing is launched)


def _host_args(B=3, W=4, R=5, C=16):
    return dict(req_to_token=torch.zeros(R, C, dtype=torch.int32),
                req_pool_indices=torch.zeros(B, dtype=torch.int64),
                seq_lens=torch.zeros(B, dtype=torch.int32),
                page_table=torch.zeros(B, W, dtype=torch.int32),
                cache_seqlens=torch.zeros(B, dtype=torch.int32),
                cu_seqlens_k=torch.zeros(B + 1, dtype=torch.int32),
                cu_seqlens_q=torch.zeros(B + 1, dtype=torch.int32))


@pytest.mark.parametrize("change,status", [
    (dict(req_to_token=torch.zeros(5, 16, dtype=torch.int64)), fd.FD_ERR_INVALID_ARG),
    (dict(req_pool_indices=torch.zeros(3, dtype=torch.float32)), fd.FD_ERR_INVALID_ARG),
    (dict(seq_lens=torch.zeros(4, dtype=torch.int32)), fd.FD_ERR_INVALID_ARG),
    (dict(page_table=torch.zeros(2, 4, dtype=torch.int32)), fd.FD_ERR_INVALID_ARG),
    (dict(cu_seqlens_k=torch.zeros(3, dtype=torch.int32)), fd.FD_ERR_INVALID_ARG),
    (dict(cu_seqlens_q=torch.zeros(4, dtype=torch.int64)), fd.FD_ERR_INVALID_ARG),
    (dict(page_size=0), fd.FD_ERR_INVALID_ARG),
    (dict(q_mode=7), fd.FD_ERR_INVALID_ARG),
    (dict(q_mode=fd.FD_QMODE_CUMSUM, q_in=torch.zeros(4, dtype=torch.int32)), fd.FD_ERR_INVALID_ARG),
    (dict(q_mode=fd.FD_QMODE_PRESET, q_in=torch.zeros(3, dtype=torch.int32)), fd.FD_ERR_INVALID_ARG),
])
def test_graph_metadata_rejects(change, status):
    fd.load_library()
    args = _host_args()
    kw = dict(page_size=4, q_mode=fd.FD_QMODE_STRIDED, q_in=None, q_stride=1)
    for k, v in change.items():
        (kw if k in kw else args)[k] = v
    with pytest.raises(fd.FdError) as e:
        fd.fd_graph_metadata(args["req_to_token"], args["req_pool_indices"], args["seq_lens"], kw["page_size"],
                             kw["q_mode"], kw["q_in"], kw["q_stride"], args["page_table"], args["cache_seqlens"],
                             args["cu_seqlens_k"], args["cu_seqlens_q"], stream=0)
    assert e.value.status == status


# ---------------------------------------------------------------------------
# the CUDA kernel against the oracle


def _run_gpu(pool, idx, seq, P, W, mode, q_in=None, q_stride=1, idx_dtype=torch.int64):
    dev = "cuda"
    B = len(idx)
    t = dict(rt=torch.from_numpy(pool).to(dev), idx=torch.tensor(idx, dtype=idx_dtype, device=dev),
             seq=torch.tensor(seq, dtype=torch.int32, device=dev))
    qt = None if q_in is None else torch.tensor(q_in, dtype=torch.int32, device=dev)
    pt = torch.full((B, W), 12345, dtype=torch.int32, device=dev)      # stale contents
    cs = torch.full((B,), 777, dtype=torch.int32, device=dev)
    ck = torch.full((B + 1,), -5, dtype=torch.int32, device=dev)
    cq = torch.full((B + 1,), -5, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    fd.fd_graph_metadata(t["rt"], t["idx"], t["seq"], P, mode, qt, q_stride, pt, cs, ck, cq, st)
    torch.cuda.synchronize()
    return dict(page_table=pt.cpu().numpy(), cache_seqlens=cs.cpu().numpy(), cu_seqlens_k=ck.cpu().numpy(),
                cu_seqlens_q=cq.cpu().numpy()), int(st.item())


@pytest.mark.gpu
@pytest.mark.parametrize("B,P", [(1, 16), (7, 1), (33, 16), (300, 64), (64, 4)])
@pytest.mark.parametrize("mode", ["preset", "cumsum", "strided"])
@pytest.mark.parametrize("idx_dtype", [torch.int32, torch.int64])
def test_graph_metadata_matches_oracle(B, P, mode, idx_dtype):
    import __graft_entry__
    __graft_entry__.build()
    rng = np.random.default_rng(B * 131 + P)
    lens = rng.integers(0, 5000, size=B)
    pool, _ = wl.make_token_pool(B + P, lens, P, extra_rows=3, unallocated_frac=0.05)
    idx = rng.permutation(B).astype(np.int64)
    idx[rng.random(B) < 0.1] = -1                      # padding rows
    seq = np.where(idx >= 0, lens[np.maximum(idx, 0)], rng.integers(0, 9, size=B))
    W = int(max(1, (lens.max() + P - 1) // P)) + 2
    q_mode = {"preset": Q_PRESET, "cumsum": Q_CUMSUM, "strided": Q_STRIDED}[mode]
    q_in = None
    if mode == "cumsum":
        q_in = rng.integers(0, 6, size=B)
    elif mode == "preset":
        q_in = np.concatenate([[0], np.cumsum(rng.integers(1, 4, size=B))])
    ref = graph_metadata_ref(pool, idx, seq, P, W, q_mode, q_in=q_in, q_stride=4)
    got, status = _run_gpu(pool, idx, seq, P, W, mode, q_in, 4, idx_dtype)
    for k in ref:
        assert np.array_equal(got[k], ref[k]), k
    assert status == 0


@pytest.mark.gpu
def test_graph_metadata_status_bits():
    pool, _ = wl.make_token_pool(3, [40, 10], 16)
    # pool index past the pool: recorded, row treated as padding
    got, status = _run_gpu(pool, [0, 9], [40, 10], 16, 4, "strided")
    assert status & fd.FD_DEVSTAT_BAD_PAGE and (got["page_table"][1] == -1).all() and got["cache_seqlens"][1] == 0
    # more pages than the table holds: recorded, table truncated
    got, status = _run_gpu(pool, [0, 1], [40, 10], 16, 2, "strided")
    assert status & fd.FD_DEVSTAT_SEQLEN_OVERFLOW and got["page_table"][0].tolist() == (pool[0, [0, 16]] // 16).tolist()


@pytest.mark.gpu
def test_metadata_and_decode_in_one_graph():
    """The step before the path and the path, captured together: each replay
    rebuilds page_table / cache_seqlens from the pool on the device and decodes
    with them; results match the oracle for new pool contents and lengths."""
    from oracle import decode_ref_inputs
    import __graft_entry__
    __graft_entry__.build()
    B, Hq, Hkv, D, P = 4, 16, 4, 128, 16
    max_len = 1500
    shape = wl.DecodeShape("graph", B, Hq, Hkv, D, P, 1, "bf16", "fixed:" + ",".join(["1"] * B))
    n_pages = 4 * B * (-(-max_len // P))
    w = wl.make_workload(shape, 71, "cuda", lengths=[1] * B, extra_pages=n_pages)
    W = -(-max_len // P)
    dev = "cuda"
    rt = torch.full((8, W * P), -1, dtype=torch.int32, device=dev)   # pool of 8 request rows
    idx = torch.zeros(B, dtype=torch.int64, device=dev)
    seq = torch.ones(B, dtype=torch.int32, device=dev)
    pt = torch.full((B, W), -1, dtype=torch.int32, device=dev)
    cs = torch.zeros(B, dtype=torch.int32, device=dev)
    ck = torch.zeros(B + 1, dtype=torch.int32, device=dev)
    cq = torch.zeros(B + 1, dtype=torch.int32, device=dev)
    out = torch.empty_like(w.q)
    lse = torch.empty(w.q.shape[:3], dtype=torch.float32, device=dev)
    plan = fd.fd_plan_create(0, B, 1, Hq, Hkv, D, P, "bf16", 8)
    fd.fd_set_plan(plan)

    def step():
        fd.fd_graph_metadata(rt, idx, seq, P, "strided", None, 1, pt, cs, ck, cq)
        fd.fd_decode_paged(w.q, w.k_cache, w.v_cache, None, pt, cs, 1, 4, out, lse)

    try:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step()
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        rng = np.random.default_rng(5)
        for trial in range(3):
            lens = rng.integers(1, max_len, size=8)
            pool, _ = wl.make_token_pool(100 + trial, lens, P, max_ctx=W * P)
            rows = rng.permutation(8)[:B]
            rt.copy_(torch.from_numpy(pool))
            idx.copy_(torch.from_numpy(rows.astype(np.int64)))
            seq.copy_(torch.from_numpy(lens[rows].astype(np.int32)))
            g.replay()
            torch.cuda.synchronize()
            meta = graph_metadata_ref(pool, rows, lens[rows], P, W, Q_STRIDED, q_stride=1)
            assert np.array_equal(pt.cpu().numpy(), meta["page_table"])
            w.page_table = torch.from_numpy(meta["page_table"]).to(dev)
            w.cache_seqlens = torch.from_numpy(meta["cache_seqlens"]).to(dev)
            w.lengths = meta["cache_seqlens"].astype(np.int64)
            ref_out, ref_lse = decode_ref_inputs(wl.oracle_inputs(w))
            from tests.gpu_common import assert_parity
            assert_parity(out, lse, ref_out, ref_lse, label=f"graph replay {trial}")
        del g
    finally:
        fd.fd_set_plan(None)
        fd.fd_plan_destroy(plan)
