"""The C-ABI library on the host: exports, argument validation, autotune table logic.

No test here launches a kernel: plans are host-only (device = -1), so every
call returns before any CUDA work. The library itself is built here with nvcc.
"""
import json
import os
import re
import shutil

import pytest
import torch

import split_kv_paged_gqa_gb300 as fd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fd.h")


@pytest.fixture(scope="module", autouse=True)
def lib():
    if shutil.which("nvcc") is None and not os.path.exists(fd.LIB_PATH):
        pytest.skip("nvcc unavailable and libfd.so not built")
    from split_kv_paged_gqa_gb300 import build
    build.build()
    return fd.load_library()


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^FD_API[^()]*?\b(fd_\w+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "fd_decode_paged" in names and len(names) >= 15
    for n in names:
        assert hasattr(lib, n), f"{n} declared in fd.h but not exported"


def test_status_strings(lib):
    assert fd.fd_status_string(fd.FD_OK) == "FD_OK"
    assert fd.fd_status_string(fd.FD_ERR_CAPTURING) == "FD_ERR_CAPTURING"
    assert fd.fd_status_string(99) == "FD_ERR_UNKNOWN"


@pytest.mark.parametrize("args,status", [
    (dict(head_dim=96), fd.FD_ERR_UNSUPPORTED),
    (dict(page_size=24), fd.FD_ERR_UNSUPPORTED),
    (dict(page_size=4), fd.FD_ERR_UNSUPPORTED),
    (dict(page_size=512), fd.FD_ERR_UNSUPPORTED),
    (dict(num_q_heads=10, num_kv_heads=4), fd.FD_ERR_INVALID_ARG),
    (dict(max_splits=65), fd.FD_ERR_INVALID_ARG),
    (dict(max_batch=0), fd.FD_ERR_INVALID_ARG),
    (dict(kv_dtype=fd.FD_FP32), fd.FD_ERR_UNSUPPORTED),
])
def test_plan_create_rejects(args, status):
    kw = dict(device=-1, max_batch=4, max_q_per_req=1, num_q_heads=8, num_kv_heads=2, head_dim=128,
              page_size=16, kv_dtype="bf16", max_splits=8)
    kw.update(args)
    with pytest.raises(fd.FdError) as e:
        fd.fd_plan_create(**kw)
    assert e.value.status == status


def _host_plan(kind="bf16", B=4, Tq=1, Hq=8, Hkv=2, D=128, P=16, S=8):
    return fd.fd_plan_create(-1, B, Tq, Hq, Hkv, D, P, kind, S)


def _tensors(kind="bf16", B=2, Tq=1, Hq=8, Hkv=2, D=128, P=16, N=10, W=4):
    t = dict(
        q=torch.zeros(B, Tq, Hq, D, dtype=torch.bfloat16),
        page_table=torch.zeros(B, W, dtype=torch.int32),
        cache_seqlens=torch.zeros(B, dtype=torch.int32),
        out=torch.zeros(B, Tq, Hq, D, dtype=torch.bfloat16),
        lse=torch.zeros(B, Tq, Hq, dtype=torch.float32),
    )
    if kind == "bf16":
        t["k_cache"] = torch.zeros(N, P, Hkv, D, dtype=torch.bfloat16)
        t["kv_scales"] = None
    elif kind == "int8":
        t["k_cache"] = torch.zeros(N, P, Hkv, D, dtype=torch.int8)
        t["kv_scales"] = torch.zeros(2, N, P, Hkv, 1, dtype=torch.float32)
    else:
        t["k_cache"] = torch.zeros(N, P, Hkv, D // 2, dtype=torch.uint8)
        t["kv_scales"] = torch.zeros(2, N, P, Hkv, D // 32, dtype=torch.float32)
    t["v_cache"] = t["k_cache"].clone()
    return t


def _call(t, Tq=1, S=2):
    fd.fd_decode_paged(t["q"], t["k_cache"], t["v_cache"], t["kv_scales"], t["page_table"],
                       t["cache_seqlens"], Tq, S, t["out"], t["lse"], stream=0)


def _expect(status, t, **kw):
    with pytest.raises(fd.FdError) as e:
        _call(t, **kw)
    assert e.value.status == status, str(e.value)


@pytest.mark.parametrize("kind", ["bf16", "int8", "int4"])
def test_valid_call_reaches_workspace_check(kind):
    plan = _host_plan(kind)
    try:
        fd.fd_set_plan(plan)
        _expect(fd.FD_ERR_WORKSPACE, _tensors(kind))     # valid descriptors; host-only plan
    finally:
        fd.fd_set_plan(None)
        fd.fd_plan_destroy(plan)


def test_no_plan():
    fd.fd_set_plan(None)
    _expect(fd.FD_ERR_NO_PLAN, _tensors())


def _mut(**changes):
    t = _tensors()
    t.update(changes)
    return t


BAD = [
    ("q dtype", lambda: _mut(q=torch.zeros(2, 1, 8, 128, dtype=torch.float32)), {}, fd.FD_ERR_INVALID_ARG),
    ("q heads", lambda: _mut(q=torch.zeros(2, 1, 6, 128, dtype=torch.bfloat16)), {}, fd.FD_ERR_INVALID_ARG),
    ("q_per_req", lambda: _tensors(), dict(Tq=2), fd.FD_ERR_INVALID_ARG),
    ("batch > max", lambda: _tensors(B=5), {}, fd.FD_ERR_INVALID_ARG),
    ("splits > max", lambda: _tensors(), dict(S=9), fd.FD_ERR_INVALID_ARG),
    ("negative splits", lambda: _tensors(), dict(S=-1), fd.FD_ERR_INVALID_ARG),
    ("cache dtype", lambda: _mut(k_cache=torch.zeros(10, 16, 2, 128, dtype=torch.int8),
                                 v_cache=torch.zeros(10, 16, 2, 128, dtype=torch.int8)), {}, fd.FD_ERR_INVALID_ARG),
    ("page size", lambda: _mut(k_cache=torch.zeros(10, 8, 2, 128, dtype=torch.bfloat16),
                               v_cache=torch.zeros(10, 8, 2, 128, dtype=torch.bfloat16)), {}, fd.FD_ERR_INVALID_ARG),
    ("k/v differ", lambda: _mut(v_cache=torch.zeros(11, 16, 2, 128, dtype=torch.bfloat16)), {}, fd.FD_ERR_INVALID_ARG),
    ("cache strided d", lambda: _mut(k_cache=torch.zeros(10, 16, 2, 256, dtype=torch.bfloat16)[..., ::2],
                                     v_cache=torch.zeros(10, 16, 2, 256, dtype=torch.bfloat16)[..., ::2]),
     {}, fd.FD_ERR_UNSUPPORTED),
    ("scales for bf16", lambda: _mut(kv_scales=torch.zeros(2, 10, 16, 2, 1)), {}, fd.FD_ERR_INVALID_ARG),
    ("page table dtype", lambda: _mut(page_table=torch.zeros(2, 4, dtype=torch.int64)), {}, fd.FD_ERR_INVALID_ARG),
    ("page table batch", lambda: _mut(page_table=torch.zeros(3, 4, dtype=torch.int32)), {}, fd.FD_ERR_INVALID_ARG),
    ("seqlens shape", lambda: _mut(cache_seqlens=torch.zeros(3, dtype=torch.int32)), {}, fd.FD_ERR_INVALID_ARG),
    ("out shape", lambda: _mut(out=torch.zeros(2, 1, 8, 64, dtype=torch.bfloat16)), {}, fd.FD_ERR_INVALID_ARG),
    ("out dtype", lambda: _mut(out=torch.zeros(2, 1, 8, 128, dtype=torch.int32)), {}, fd.FD_ERR_INVALID_ARG),
    ("lse shape", lambda: _mut(lse=torch.zeros(2, 8, dtype=torch.float32)), {}, fd.FD_ERR_INVALID_ARG),
    ("q misaligned", lambda: _mut(q=torch.zeros(2 * 8 * 128 + 1, dtype=torch.bfloat16)[1:].view(2, 1, 8, 128)),
     {}, fd.FD_ERR_UNSUPPORTED),
]


@pytest.mark.parametrize("name,make,kw,status", BAD, ids=[b[0] for b in BAD])
def test_descriptor_validation(name, make, kw, status):
    plan = _host_plan()
    try:
        fd.fd_set_plan(plan)
        _expect(status, make(), **kw)
    finally:
        fd.fd_set_plan(None)
        fd.fd_plan_destroy(plan)


def test_quantised_scale_checks():
    plan = _host_plan("int4")
    try:
        fd.fd_set_plan(plan)
        t = _tensors("int4")
        t["kv_scales"] = None
        _expect(fd.FD_ERR_INVALID_ARG, t)
        t = _tensors("int4")
        t["kv_scales"] = torch.zeros(2, 10, 16, 2, 1)               # n_g must be D/32 = 4
        _expect(fd.FD_ERR_INVALID_ARG, t)
    finally:
        fd.fd_set_plan(None)
        fd.fd_plan_destroy(plan)


# ---------------------------------------------------------------------------
# autotune table logic with a fake timer (no kernel launches)


def _fake_timer(best_for):
    calls = []

    def timer(batch, bucket, S):
        calls.append((batch, bucket, S))
        return abs(S - best_for(batch, bucket)) + 1.0
    return timer, calls


def test_autotune_buckets_nearest_and_persistence(tmp_path, monkeypatch):
    monkeypatch.delenv("FD_FORCE_AUTOTUNE", raising=False)
    # a made-up optimum; the mixed-length inputs (bucket -K) want twice the splits
    best = lambda b, k: min(64, max(1, abs(k) // (256 * b)) * (2 if k < 0 else 1))
    plan = _host_plan(B=64, S=64)
    try:
        fd.fd_autotune_set_cache_dir(plan, str(tmp_path))
        timer, calls = _fake_timer(best)
        fd.fd_autotune_set_timer(plan, timer)
        fd.fd_autotune(plan, [1, 16], 1024, 8192)
        # 4 buckets x (batch 1: equal lengths; batch 16: equal and mixed lengths);
        # every power of two up to 64 is tried for each key, plus split counts
        # that fill one or two waves of the SMs
        assert fd.fd_autotune_stats(plan) == (12, 0)
        per_key = {}
        for b, k, S in calls:
            per_key.setdefault((b, k), []).append(S)
        assert len(per_key) == 12 and sum(1 for b, k in per_key if k < 0) == 4
        assert all(b == 16 for b, k in per_key if k < 0)
        for (b, k), S_list in per_key.items():
            # powers of two whose splits hold at least 128 keys of the bucket
            want = {S for S in (1, 2, 4, 8, 16, 32, 64) if S * 128 <= abs(k)}
            assert want <= set(S_list) and max(S_list) <= min(64, abs(k) // 128)
            assert len(S_list) == len(set(S_list))
        for b in (1, 16):
            for k in (1024, 2048, 4096, 8192):
                assert fd.fd_query_splits(plan, b, k) == best(b, k)
        # bucket of a length is the next power of two; beyond the range, the nearest bucket
        assert fd.fd_query_splits(plan, 1, 1500) == best(1, 2048)
        assert fd.fd_query_splits(plan, 1, 100000) == best(1, 8192)
        assert fd.fd_query_splits(plan, 1, 10) == best(1, 1024)
        # batch: smallest tuned batch >= B, else the largest
        assert fd.fd_query_splits(plan, 8, 4096) == best(16, 4096)
        assert fd.fd_query_splits(plan, 40, 4096) == best(16, 4096)
        # persisted file holds exactly the tuned keys
        files = list(tmp_path.glob("fd_splits_*.json"))
        assert len(files) == 1
        entries = json.load(open(files[0]))["entries"]
        assert len(entries) == 12 and sum(e["spread"] for e in entries) == 4
        assert all(e["bucket"] > 0 for e in entries)
        # hints that show a spread (max >= 1.25 x mean) use the mixed-length table
        fd.fd_set_mean_seqlen_hint(plan, 2000)
        assert fd.fd_query_splits(plan, 16, 8000) == best(16, -2048)
        assert fd.fd_query_splits(plan, 16, 2400) == best(16, 2048)   # max / mean = 1.2
        assert fd.fd_query_splits(plan, 1, 8000) == best(1, 2048)     # one request: no spread
        fd.fd_set_mean_seqlen_hint(plan, 0)
        # a second call is served from the table: no new search
        calls.clear()
        fd.fd_autotune(plan, [1, 16], 1024, 8192)
        assert calls == [] and fd.fd_autotune_stats(plan) == (12, 12)
    finally:
        fd.fd_plan_destroy(plan)

    # a new plan with the same key reloads the persisted table without searching
    plan2 = _host_plan(B=64, S=64)
    try:
        fd.fd_autotune_set_cache_dir(plan2, str(tmp_path))
        assert fd.fd_query_splits(plan2, 16, 2048) == best(16, 2048)
        timer2, calls2 = _fake_timer(best)
        fd.fd_autotune_set_timer(plan2, timer2)
        fd.fd_autotune(plan2, [16], 1024, 8192)
        assert calls2 == [] and fd.fd_autotune_stats(plan2) == (0, 8)
        fd.fd_set_mean_seqlen_hint(plan2, 2000)                      # the mixed table reloads too
        assert fd.fd_query_splits(plan2, 16, 8000) == best(16, -2048)
        # decode attention treats FD_FORCE_AUTOTUNE as adaptive: cached keys are kept
        monkeypatch.setenv("FD_FORCE_AUTOTUNE", "1")
        fd.fd_autotune(plan2, [16], 1024, 1024)
        assert calls2 == []
    finally:
        fd.fd_plan_destroy(plan2)


def test_nearest_match_is_invalidated_when_a_config_is_saved(tmp_path):
    plan = _host_plan(B=64, S=64)
    try:
        fd.fd_autotune_set_cache_dir(plan, str(tmp_path))
        fd.fd_autotune_set_timer(plan, lambda b, k, S: abs(S - 2))
        fd.fd_autotune(plan, [32], 4096, 4096)
        assert fd.fd_query_splits(plan, 8, 4096) == 2      # nearest batch 32, memoised
        fd.fd_autotune_set_timer(plan, lambda b, k, S: abs(S - 16))
        fd.fd_autotune(plan, [8], 4096, 4096)               # saving a new config drops the memo
        assert fd.fd_query_splits(plan, 8, 4096) == 16
    finally:
        fd.fd_plan_destroy(plan)


def test_tuner_keeps_the_fastest_and_breaks_exact_ties_toward_fewer_splits(tmp_path):
    plan = _host_plan(B=64, S=64)
    try:
        fd.fd_autotune_set_cache_dir(plan, str(tmp_path))
        times = {1: 100.0, 2: 99.5, 4: 101.2, 8: 103.0}
        fd.fd_autotune_set_timer(plan, lambda b, k, S: times.get(S, 200.0))
        fd.fd_autotune(plan, [64], 32768, 32768)
        assert fd.fd_query_splits(plan, 64, 32768) == 2    # the argmin, however close
        times2 = {2: 100.0, 4: 100.0, 1: 100.0}
        fd.fd_autotune_set_timer(plan, lambda b, k, S: times2.get(S, 200.0))
        fd.fd_autotune(plan, [16], 32768, 32768)
        assert fd.fd_query_splits(plan, 16, 32768) == 1    # exact tie: fewer splits
    finally:
        fd.fd_plan_destroy(plan)


def test_heuristic_without_table():
    plan = _host_plan(B=64, S=64)
    try:
        fd.fd_autotune_set_cache_dir(plan, None)
        s1 = fd.fd_query_splits(plan, 1, 32768)
        s64 = fd.fd_query_splits(plan, 64, 32768)
        assert 1 <= s64 <= s1 <= 64
        assert fd.fd_query_splits(plan, 1, 300) == 1        # short requests are not split finely
    finally:
        fd.fd_plan_destroy(plan)


def test_autotune_rejects_bad_arguments():
    plan = _host_plan()
    try:
        fd.fd_autotune_set_timer(plan, lambda b, k, S: 1.0)
        for args in ([[0]], [[5]], [[1], 3000, 4096], [[1], 8192, 1024]):
            with pytest.raises(fd.FdError) as e:
                fd.fd_autotune(plan, *args)
            assert e.value.status == fd.FD_ERR_INVALID_ARG
        fd.fd_autotune_set_timer(plan, None)
        with pytest.raises(fd.FdError) as e:                # host-only plan cannot time kernels
            fd.fd_autotune(plan, [1], 1024, 1024, stream=0)
        assert e.value.status == fd.FD_ERR_WORKSPACE
    finally:
        fd.fd_plan_destroy(plan)


def test_split_policy_argument():
    plan = _host_plan()
    try:
        fd.fd_plan_set_split_policy(plan, fd.FD_SPLIT_EQUAL)
        fd.fd_plan_set_split_policy(plan, "balanced")
        with pytest.raises(fd.FdError) as e:
            fd.fd_plan_set_split_policy(plan, 2)
        assert e.value.status == fd.FD_ERR_INVALID_ARG
    finally:
        fd.fd_plan_destroy(plan)
    with pytest.raises(fd.FdError):
        fd.fd_plan_set_split_policy(None, 0)


def test_mean_hint_picks_the_nearest_bucket_under_the_balanced_policy(tmp_path):
    plan = _host_plan(B=64, S=64)
    try:
        fd.fd_autotune_set_cache_dir(plan, str(tmp_path))
        best = {4096: 2, 8192: 4, 16384: 8, 32768: 16}
        best_mixed = {4096: 4, 8192: 8, 16384: 16, 32768: 32}
        fd.fd_autotune_set_timer(plan, lambda b, k, S: abs(S - (best[k] if k > 0 else best_mixed[-k])) + 1.0)
        fd.fd_autotune(plan, [64], 4096, 32768)
        assert fd.fd_query_splits(plan, 64, 30000) == 16          # no mean hint: bucket of the max
        fd.fd_set_mean_seqlen_hint(plan, 5932)                    # nearest power of two: 8192
        assert fd.fd_query_splits(plan, 64, 7000) == 4            # max / mean < 1.25: equal lengths
        assert fd.fd_query_splits(plan, 64, 30000) == 8           # spread: the mixed-length table
        fd.fd_set_mean_seqlen_hint(plan, 5000)                    # below 8192 / sqrt(2): 4096
        assert fd.fd_query_splits(plan, 64, 6000) == 2
        fd.fd_set_mean_seqlen_hint(plan, 23000)                   # 16384 * sqrt(2) = 23170.5: 16384
        assert fd.fd_query_splits(plan, 64, 24000) == 8
        fd.fd_plan_set_split_policy(plan, "equal")                # equal splits: the max decides
        assert fd.fd_query_splits(plan, 64, 30000) == 16
        fd.fd_plan_set_split_policy(plan, "balanced")
        fd.fd_set_mean_seqlen_hint(plan, 0)                       # cleared
        assert fd.fd_query_splits(plan, 64, 30000) == 16
        with pytest.raises(fd.FdError):
            fd.fd_set_mean_seqlen_hint(plan, -1)
    finally:
        fd.fd_plan_destroy(plan)


def test_tuner_skips_splits_shorter_than_128_keys(tmp_path):
    plan = _host_plan(B=64, S=64)
    try:
        fd.fd_autotune_set_cache_dir(plan, str(tmp_path))
        calls = []
        fd.fd_autotune_set_timer(plan, lambda b, k, S: calls.append((abs(k), S)) or float(S))
        fd.fd_autotune(plan, [2], 256, 1024)
        for k, S in calls:
            assert S * 128 <= k or S == 1, (k, S)
        assert {S for k, S in calls if k == 1024} >= {1, 2, 4, 8}
        assert {S for k, S in calls if k == 256} == {1, 2}
    finally:
        fd.fd_plan_destroy(plan)


# ---------------------------------------------------------------------------
# warmup phases: decode attention tunes on its calls only in its own phase


def test_warmup_scopes_nest_and_restore():
    assert fd.fd_warmup_current() == fd.FD_PHASE_NONE
    with fd.warmup(fd.FD_PHASE_DECODE_ATTENTION):
        assert fd.fd_warmup_current() == fd.FD_PHASE_DECODE_ATTENTION
        with fd.warmup(fd.FD_PHASE_GENERAL):
            assert fd.fd_warmup_current() == fd.FD_PHASE_GENERAL
        assert fd.fd_warmup_current() == fd.FD_PHASE_DECODE_ATTENTION
    assert fd.fd_warmup_current() == fd.FD_PHASE_NONE
    with pytest.raises(fd.FdError):
        fd.fd_warmup_enter(9)
    assert fd.fd_warmup_current() == fd.FD_PHASE_NONE


def test_decode_call_tunes_only_inside_the_decode_attention_phase(tmp_path, monkeypatch):
    monkeypatch.delenv("FD_AUTOTUNE_SEQ_LEN", raising=False)
    plan = _host_plan(B=4, S=8)
    calls = []
    try:
        fd.fd_autotune_set_cache_dir(plan, str(tmp_path))
        fd.fd_autotune_set_timer(plan, lambda b, k, S: calls.append((b, k, S)) or abs(S - 4) + 1.0)
        fd.fd_set_plan(plan)
        t = _tensors()                                   # batch 2, valid descriptors
        _expect(fd.FD_ERR_WORKSPACE, t, S=0)                  # live phase: no tuning
        with fd.warmup(fd.FD_PHASE_GENERAL):
            _expect(fd.FD_ERR_WORKSPACE, t, S=0)              # general phase: decode attention does not tune
        assert calls == []
        with fd.warmup(fd.FD_PHASE_DECODE_ATTENTION):
            _expect(fd.FD_ERR_WORKSPACE, t, S=0)              # tunes batch 2 at 32768, then fails on the host plan
            assert {(b, abs(k)) for b, k, S in calls} == {(2, 32768)}
            assert {k for b, k, S in calls} == {32768, -32768}     # equal and mixed lengths
            assert fd.fd_autotune_stats(plan)[0] == 2
            n = len(calls)
            _expect(fd.FD_ERR_WORKSPACE, t, S=0)              # tuned already: adaptive, no new search
            assert len(calls) == n
        assert fd.fd_query_splits(plan, 2, 32768) == 4
        monkeypatch.setenv("FD_AUTOTUNE_SEQ_LEN", "5000")
        with fd.warmup(fd.FD_PHASE_DECODE_ATTENTION):
            _expect(fd.FD_ERR_WORKSPACE, t, S=0)              # representative length 5000: bucket 8192
        assert (2, 8192) in {(b, abs(k)) for b, k, S in calls}
        # an explicit num_splits never tunes
        calls.clear()
        with fd.warmup(fd.FD_PHASE_DECODE_ATTENTION):
            _expect(fd.FD_ERR_WORKSPACE, t, S=2)
        assert calls == []
    finally:
        fd.fd_set_plan(None)
        fd.fd_plan_destroy(plan)


def test_force_is_adaptive_and_clear_searches_afresh(tmp_path, monkeypatch):
    plan = _host_plan(B=64, S=64)
    try:
        fd.fd_autotune_set_cache_dir(plan, str(tmp_path))
        calls = []
        fd.fd_autotune_set_timer(plan, lambda b, k, S: calls.append(S) or float(S))
        fd.fd_autotune(plan, [4], 4096, 4096)
        first = len(calls)
        monkeypatch.setenv("FD_FORCE_AUTOTUNE", "1")     # adaptive for decode attention: no re-search
        fd.fd_autotune(plan, [4], 4096, 4096)
        assert len(calls) == first
        files = list(tmp_path.glob("fd_splits_*.json"))
        assert len(files) == 1
        fd.fd_autotune_clear(plan, remove_file=True)      # a fresh search
        assert not files[0].exists()
        fd.fd_autotune(plan, [4], 4096, 4096)
        assert len(calls) == 2 * first
    finally:
        fd.fd_plan_destroy(plan)


def test_descriptor_reuse_matches_a_fresh_build():
    # the binding reuses a descriptor only for the same pointer, dtype, shape and strides
    t = torch.zeros(6, 4, 3, dtype=torch.bfloat16)
    a, b = fd.make_descriptor(t), fd.make_descriptor(t)
    assert a is b
    v = t[:, 1:3]                                    # a view: other pointer, shape and strides
    d = fd.make_descriptor(v)
    assert d is not a
    assert d.data == v.data_ptr() and d.ndim == 3
    assert list(d.shape)[:3] == [6, 2, 3] and list(d.stride)[:3] == list(v.stride())
    assert fd.make_descriptor(t.view(6, 12)).ndim == 2
    assert fd.make_descriptor(None) is None
