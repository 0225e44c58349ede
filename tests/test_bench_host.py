"""Host-side logic of bench.py (no GPU): algorithmic bytes and the L2 rotation."""
import numpy as np

import pytest

import bench
from split_kv_paged_gqa_gb300 import workloads as wl


def test_algorithmic_bytes_long_context_request():
    # one request of 32768 keys, 8 KV heads x 128 channels of bf16 K and V:
    # 32768 * 8 * 128 * 2 B * 2 = 134,217,728 B of KV, plus q, page ids, length, out, lse
    shape = wl.CONFIGS["long_bf16_b1"]
    s1, call = bench.algorithmic_bytes(shape, np.array([32768]), direct=np.array([False]))
    q = 64 * 128 * 2
    meta = 512 * 4 + 4
    out = 64 * 128 * 2 + 64 * 4
    assert s1 == 134217728 + q + meta
    assert call == s1 + out
    s1_fused, _ = bench.algorithmic_bytes(shape, np.array([32768]), direct=np.array([True]))
    assert s1_fused == call


def _equal_counts(L, P, S):
    """Equal splits per request, written out by hand: chunk = P * ceil(ceil(L/S)/P)."""
    out = []
    for x in L:
        if x <= 0:
            out.append(0)
            continue
        chunk = P * -(-(-(-x // S)) // P)
        out.append(min(S, -(-x // chunk)))
    return np.array(out)


def test_balanced_split_counts_equal_the_equal_policy_on_equal_lengths():
    for L, P in ((32768, 64), (1000, 16), (17, 16), (4096, 8)):
        for S in (1, 2, 3, 7, 16, 19, 64):
            got = bench.split_counts(np.full(6, L), P, S)
            assert (got == _equal_counts([L] * 6, P, S)).all(), (L, P, S)


def test_balanced_split_counts_follow_length_and_stay_bounded():
    rng = np.random.default_rng(3)
    for _ in range(50):
        B = int(rng.integers(2, 70))
        P = int(2 ** rng.integers(3, 9))
        L = rng.integers(0, 40000, size=B)
        L[rng.random(B) < 0.1] = 0
        for S in (1, 2, 5, 16, 64):
            nv = bench.split_counts(L, P, S)
            assert (nv[L == 0] == 0).all() and (nv[L > 0] >= 1).all() and nv.max() <= 64
            assert nv.sum() <= B * (S + 1)                  # the grid's bound
            n = -(-L // P)
            cp = max(1, -(-int(n.sum()) // (B * S)))        # pages per split of the batch
            want = -(-n // cp)
            free = (want <= 64) & (L > 0)
            assert (nv[free] == want[free]).all()           # uncapped: exactly ceil(n / cp) splits
    nv = bench.split_counts(np.array([32768, 1024]), 16, 8, s_cap=4)
    assert nv.tolist() == [4, 1]                            # the cap binds on the long request


def test_launches_per_call():
    assert bench.launches_per_call(1, 1) == 1
    assert bench.launches_per_call(64, 1) == 2              # balanced: long requests may split
    assert bench.launches_per_call(64, 1, balanced=False) == 1
    assert bench.launches_per_call(1, 4) == 2


def test_rotation_copies_span_four_l2():
    l2 = 126 << 20
    assert bench.rotation_copies(9 << 30, l2) == 1          # a batch-64 step is far beyond L2
    assert bench.rotation_copies(4 * l2, l2) == 1
    k = bench.rotation_copies(134217728, l2)               # one 32K request
    assert k * 134217728 >= 4 * l2 and (k - 1) * 134217728 < 4 * l2
    assert bench.rotation_copies(1000, l2, limit=64) == 64


def test_stage1_sha_covers_kernel_sources_only():
    sha = bench.stage1_source_sha()
    assert len(sha) == 16 and all(c in "0123456789abcdef" for c in sha)
    assert "fd_api.cu" not in bench.STAGE1_SOURCES and "stage1.cuh" in bench.STAGE1_SOURCES


def test_batch64_traffic_is_the_batch16_capture_scaled():
    """The 8.6 GB batch-64 workload is not captured with DRAM counters; its
    traffic is the batch-16 capture of the same kernel scaled by the units
    processed (64 / 16)."""
    t64, t16 = bench.profiled_traffic("long_bf16_b64"), bench.profiled_traffic("long_bf16_b16")
    if t64 is None or t16 is None:
        pytest.skip("the committed summaries were taken on another stage-1 source")
    assert t64 == 4 * t16


def test_source_hash_ignores_comments_and_layout_but_not_code():
    src = 'int a = 1; // note\n/* block\n comment */ const char *s = "x // kept /* kept */";\nint  b;'
    assert bench.strip_c_comments(src) == 'int a = 1; const char *s = "x // kept /* kept */"; int b;'
    assert bench.strip_c_comments("a /* x */ b") == bench.strip_c_comments("a   b")
    assert bench.strip_c_comments("x = 1;") != bench.strip_c_comments("x = 2;")
    assert bench.strip_c_comments("c = '\\'';// q") == "c = '\\'';"


def test_nearest_pow2_matches_the_log_midpoint():
    assert [bench.nearest_pow2(v) for v in (1, 2, 3, 5, 6, 5932, 5000, 23000, 23171, 32768)] == \
        [1, 2, 4, 4, 8, 8192, 4096, 16384, 32768, 32768]


def test_cpu_baseline_sample_takes_whole_requests_until_the_budget():
    calls = []

    def fake(b):  # request b takes b + 1 seconds and moves 100 bytes
        calls.append(b)
        return 0.0, float(b + 1), 100

    reqs, secs, nbytes = bench.cpu_baseline_sample(fake, 64, budget_s=10.0)
    assert reqs == [0, 1, 2, 3] and calls == reqs      # 1 + 2 + 3 + 4 = 10 s
    assert secs == 10.0 and nbytes == 400
    reqs, secs, nbytes = bench.cpu_baseline_sample(fake, 2, budget_s=10.0)
    assert reqs == [0, 1] and secs == 3.0            # the whole (small) batch
