"""Host-side logic of bench.py (no GPU): algorithmic bytes and the L2 rotation."""
import numpy as np

import bench
from split_kv_paged_gqa_gb300 import workloads as wl


def test_algorithmic_bytes_long_context_request():
    # one request of 32768 keys, 8 KV heads x 128 channels of bf16 K and V:
    # 32768 * 8 * 128 * 2 B * 2 = 134,217,728 B of KV, plus q, page ids, length, out, lse
    shape = wl.CONFIGS["long_bf16_b1"]
    s1, call = bench.algorithmic_bytes(shape, np.array([32768]), False)
    q = 64 * 128 * 2
    meta = 512 * 4 + 4
    out = 64 * 128 * 2 + 64 * 4
    assert s1 == 134217728 + q + meta
    assert call == s1 + out
    s1_fused, _ = bench.algorithmic_bytes(shape, np.array([32768]), True)
    assert s1_fused == call


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
