"""Split-KV paged GQA flash decode for GB300: Python binding of libfd.

A thin ctypes layer over the C ABI declared in ``include/fd.h``: every function
here has the name of the C entry point it calls and only marshals arguments
(torch tensors become ``fd_tensor`` descriptors of their device pointer, dtype,
shape and strides; the stream defaults to torch's current stream). All work
runs in the CUDA library; there is no fallback. If ``libfd.so`` has not been
built, every call raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

__all__ = [
    "FdError", "load_library", "fd_plan_create", "fd_plan_destroy", "fd_set_plan", "fd_get_plan",
    "fd_decode_paged", "fd_decode_paged_static", "fd_plan_set_split_policy", "fd_set_max_seqlen_hint",
    "fd_set_mean_seqlen_hint", "fd_graph_metadata", "fd_warmup_enter", "fd_warmup_exit", "fd_warmup_current",
    "warmup", "fd_autotune_set_input_hook", "fd_autotune_clear", "fd_autotune", "fd_query_splits",
    "fd_autotune_set_timer", "fd_autotune_set_cache_dir", "fd_autotune_stats",
    "fd_read_device_status", "fd_selftest_wait_timeout", "fd_plan_workspace_bytes", "fd_profile_begin",
    "fd_profile_end", "fd_probe_hbm_read", "fd_probe_hbm_copy",
    "fd_status_string", "fd_last_error",
    "FD_OK", "FD_ERR_INVALID_ARG", "FD_ERR_UNSUPPORTED", "FD_ERR_WORKSPACE", "FD_ERR_CAPTURING",
    "FD_ERR_CUDA", "FD_ERR_DEVICE_STATUS", "FD_ERR_TIMEOUT", "FD_ERR_NO_PLAN", "FD_ERR_IO",
    "FD_BF16", "FD_FP32", "FD_INT8", "FD_INT4X2", "FD_INT32", "FD_INT64",
    "FD_QMODE_PRESET", "FD_QMODE_CUMSUM", "FD_QMODE_STRIDED",
    "FD_PHASE_NONE", "FD_PHASE_GENERAL", "FD_PHASE_DECODE_ATTENTION",
    "FD_DEVSTAT_BAD_PAGE", "FD_DEVSTAT_SEQLEN_OVERFLOW", "FD_DEVSTAT_WAIT_TIMEOUT",
    "FD_SPLIT_BALANCED", "FD_SPLIT_EQUAL",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfd.so")

(FD_OK, FD_ERR_INVALID_ARG, FD_ERR_UNSUPPORTED, FD_ERR_WORKSPACE, FD_ERR_CAPTURING, FD_ERR_CUDA,
 FD_ERR_DEVICE_STATUS, FD_ERR_TIMEOUT, FD_ERR_NO_PLAN, FD_ERR_IO) = range(10)
FD_BF16, FD_FP32, FD_INT8, FD_INT4X2, FD_INT32, FD_INT64 = range(6)
FD_QMODE_PRESET, FD_QMODE_CUMSUM, FD_QMODE_STRIDED = range(3)
FD_PHASE_NONE, FD_PHASE_GENERAL, FD_PHASE_DECODE_ATTENTION = range(3)
FD_DEVSTAT_BAD_PAGE, FD_DEVSTAT_SEQLEN_OVERFLOW, FD_DEVSTAT_WAIT_TIMEOUT = 1, 2, 4
FD_SPLIT_BALANCED, FD_SPLIT_EQUAL = 0, 1

_KV_NAMES = {"bf16": FD_BF16, "int8": FD_INT8, "int4": FD_INT4X2}


class FdTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 5), ("stride", ctypes.c_int64 * 5)]


TIMER_FN = ctypes.CFUNCTYPE(ctypes.c_double, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int)
INPUTS_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                             ctypes.POINTER(FdTensor), ctypes.POINTER(FdTensor), ctypes.POINTER(FdTensor),
                             ctypes.POINTER(FdTensor), ctypes.c_void_p)


class FdError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


def _status_name(s: int) -> str:
    names = ["FD_OK", "FD_ERR_INVALID_ARG", "FD_ERR_UNSUPPORTED", "FD_ERR_WORKSPACE", "FD_ERR_CAPTURING",
             "FD_ERR_CUDA", "FD_ERR_DEVICE_STATUS", "FD_ERR_TIMEOUT", "FD_ERR_NO_PLAN", "FD_ERR_IO"]
    return names[s] if 0 <= s < len(names) else f"status {s}"


_LIB = None


def load_library(path: Optional[str] = None):
    """Load libfd.so (once) and declare its signatures."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(p)
    P, T, I, F = ctypes.c_void_p, ctypes.POINTER(FdTensor), ctypes.c_int, ctypes.c_float
    sig = {
        "fd_plan_create": (I, [I, I, I, I, I, I, I, I, I, F, ctypes.POINTER(P)]),
        "fd_plan_destroy": (I, [P]),
        "fd_set_plan": (I, [P]),
        "fd_get_plan": (P, []),
        "fd_decode_paged": (I, [T, T, T, T, T, T, I, I, T, T, P]),
        "fd_decode_paged_static": (I, [T, T, T, T, T, T, I, I, F, T, T, P]),
        "fd_plan_set_split_policy": (I, [P, I]),
        "fd_set_max_seqlen_hint": (I, [P, I]),
        "fd_set_mean_seqlen_hint": (I, [P, I]),
        "fd_graph_metadata": (I, [T, T, T, I, I, T, I, T, T, T, T, T, P]),
        "fd_warmup_enter": (I, [I, ctypes.POINTER(I)]),
        "fd_warmup_exit": (I, [I]),
        "fd_warmup_current": (I, []),
        "fd_autotune_set_input_hook": (I, [P, INPUTS_FN, P]),
        "fd_autotune_clear": (I, [P, I]),
        "fd_autotune": (I, [P, ctypes.POINTER(I), I, I, I, P]),
        "fd_query_splits": (I, [P, I, I, ctypes.POINTER(I)]),
        "fd_autotune_set_timer": (I, [P, TIMER_FN, P]),
        "fd_autotune_set_cache_dir": (I, [P, ctypes.c_char_p]),
        "fd_autotune_stats": (I, [P, ctypes.POINTER(I), ctypes.POINTER(I)]),
        "fd_read_device_status": (I, [P, ctypes.POINTER(I)]),
        "fd_selftest_wait_timeout": (I, [P, ctypes.c_uint, P]),
        "fd_plan_workspace_bytes": (I, [P, ctypes.POINTER(ctypes.c_size_t)]),
        "fd_profile_begin": (I, [P]),
        "fd_profile_end": (I, [P, ctypes.POINTER(I), ctypes.POINTER(ctypes.c_double),
                               ctypes.POINTER(ctypes.c_double)]),
        "fd_probe_hbm_read": (I, [P, ctypes.c_size_t, P, P]),
        "fd_probe_hbm_copy": (I, [P, P, ctypes.c_size_t, P]),
        "fd_status_string": (ctypes.c_char_p, [I]),
        "fd_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = lib
    return lib


def _check(status: int):
    if status != FD_OK:
        raise FdError(status, load_library().fd_last_error().decode(errors="replace"))


def fd_status_string(status: int) -> str:
    return load_library().fd_status_string(status).decode()


def fd_last_error() -> str:
    return load_library().fd_last_error().decode(errors="replace")


# ---------------------------------------------------------------------------
# descriptors


def _dtype_code(t) -> int:
    import torch
    m = {torch.bfloat16: FD_BF16, torch.float32: FD_FP32, torch.int8: FD_INT8, torch.uint8: FD_INT4X2,
         torch.int32: FD_INT32, torch.int64: FD_INT64}
    return m.get(t.dtype, -1)      # the library rejects unknown codes


# Descriptors by (pointer, dtype, shape, strides): a serving loop passes the
# same buffers every step, and a descriptor holds nothing but these fields, so
# a cached one is exactly the one that would be built (about 2 us saved per
# tensor per call).
_DESC_CACHE: dict = {}
_DESC_CACHE_MAX = 4096


def make_descriptor(t) -> Optional[FdTensor]:
    """fd_tensor for a torch tensor (or None for None)."""
    if t is None:
        return None
    shape = tuple(t.shape)
    if len(shape) > 5:
        raise ValueError("at most 5 dimensions")
    stride = t.stride()
    key = (t.data_ptr(), t.dtype, shape, stride)
    d = _DESC_CACHE.get(key)
    if d is not None:
        return d
    d = FdTensor()
    d.data = key[0]
    d.dtype = _dtype_code(t)
    d.ndim = len(shape)
    for i, (sz, st) in enumerate(zip(shape, stride)):
        d.shape[i] = sz
        d.stride[i] = st
    if len(_DESC_CACHE) >= _DESC_CACHE_MAX:
        _DESC_CACHE.clear()
    _DESC_CACHE[key] = d
    return d


def _ref(d: Optional[FdTensor]):
    return ctypes.byref(d) if d is not None else None


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _kv_code(kv_dtype) -> int:
    return _KV_NAMES[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype)


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI)


def fd_plan_create(device: int, max_batch: int, max_q_per_req: int, num_q_heads: int, num_kv_heads: int,
                   head_dim: int, page_size: int, kv_dtype, max_splits: int,
                   softmax_scale: float = 0.0) -> int:
    """Create a plan; returns the opaque handle (an int). device=-1: host-only plan."""
    h = ctypes.c_void_p()
    _check(load_library().fd_plan_create(device, max_batch, max_q_per_req, num_q_heads, num_kv_heads, head_dim,
                                         page_size, _kv_code(kv_dtype), max_splits, softmax_scale,
                                         ctypes.byref(h)))
    return h.value


def fd_plan_destroy(plan: int) -> None:
    _check(load_library().fd_plan_destroy(plan))


def fd_set_plan(plan: Optional[int]) -> None:
    _check(load_library().fd_set_plan(plan))


def fd_get_plan() -> Optional[int]:
    return load_library().fd_get_plan()


def fd_decode_paged(q, k_cache, v_cache, kv_scales, page_table, cache_seqlens, q_per_req: int,
                    num_splits: int, out, lse, stream=None) -> None:
    """Enqueue one decode call on ``stream`` (default: torch's current stream)."""
    descs = [make_descriptor(t) for t in (q, k_cache, v_cache, kv_scales, page_table, cache_seqlens, out, lse)]
    _check(load_library().fd_decode_paged(*(_ref(d) for d in descs[:6]), q_per_req, num_splits,
                                          _ref(descs[6]), _ref(descs[7]), _stream_handle(stream)))


def fd_decode_paged_static(q, k_cache, v_cache, kv_scales, page_table, cache_seqlens, q_per_req: int,
                           num_splits: int, softmax_scale: float, out, lse, stream=None) -> None:
    """fd_decode_paged without a plan and without any device allocation.

    For callers that cannot allocate GPU memory. The split workspace is a
    fixed 32 MiB array inside the library; num_splits must be given (1..64).
    The first call on a device does a one-time set-up, so make it before any
    stream capture. Calls that overlap on the GPU race on the shared array.
    """
    descs = [make_descriptor(t) for t in (q, k_cache, v_cache, kv_scales, page_table, cache_seqlens, out, lse)]
    _check(load_library().fd_decode_paged_static(*(_ref(d) for d in descs[:6]), q_per_req, num_splits,
                                                 softmax_scale, _ref(descs[6]), _ref(descs[7]),
                                                 _stream_handle(stream)))


def fd_plan_set_split_policy(plan: int, policy) -> None:
    """FD_SPLIT_BALANCED (default) or FD_SPLIT_EQUAL; also "balanced" / "equal"."""
    if isinstance(policy, str):
        policy = {"balanced": FD_SPLIT_BALANCED, "equal": FD_SPLIT_EQUAL}[policy]
    _check(load_library().fd_plan_set_split_policy(plan, int(policy)))


def fd_set_max_seqlen_hint(plan: int, max_seqlen: int) -> None:
    _check(load_library().fd_set_max_seqlen_hint(plan, max_seqlen))


def fd_set_mean_seqlen_hint(plan: int, mean_seqlen: int) -> None:
    _check(load_library().fd_set_mean_seqlen_hint(plan, int(mean_seqlen)))


def fd_graph_metadata(req_to_token, req_pool_indices, seq_lens, page_size: int, q_mode, q_in, q_stride: int,
                      page_table, cache_seqlens, cu_seqlens_k, cu_seqlens_q, status=None, stream=None) -> None:
    """Enqueue the one-launch rebuild of a decode batch's metadata (page_table,
    cache_seqlens, cu_seqlens_k, cu_seqlens_q) from a request-to-token pool.
    q_mode: FD_QMODE_* or "preset" / "cumsum" / "strided"."""
    if isinstance(q_mode, str):
        q_mode = {"preset": FD_QMODE_PRESET, "cumsum": FD_QMODE_CUMSUM, "strided": FD_QMODE_STRIDED}[q_mode]
    d = [make_descriptor(t) for t in (req_to_token, req_pool_indices, seq_lens, q_in, page_table, cache_seqlens,
                                      cu_seqlens_k, cu_seqlens_q, status)]
    _check(load_library().fd_graph_metadata(_ref(d[0]), _ref(d[1]), _ref(d[2]), page_size, int(q_mode), _ref(d[3]),
                                            q_stride, _ref(d[4]), _ref(d[5]), _ref(d[6]), _ref(d[7]), _ref(d[8]),
                                            _stream_handle(stream)))


def fd_warmup_enter(phase: int) -> int:
    """Enter a warmup phase on this thread; returns the phase to restore."""
    prev = ctypes.c_int()
    _check(load_library().fd_warmup_enter(int(phase), ctypes.byref(prev)))
    return prev.value


def fd_warmup_exit(previous: int) -> None:
    _check(load_library().fd_warmup_exit(int(previous)))


def fd_warmup_current() -> int:
    return load_library().fd_warmup_current()


class warmup:
    """Nestable warmup scope: ``with warmup(FD_PHASE_DECODE_ATTENTION): ...``
    restores the previous phase on exit."""

    def __init__(self, phase: int):
        self.phase = phase
        self.prev = None

    def __enter__(self):
        self.prev = fd_warmup_enter(self.phase)
        return self

    def __exit__(self, *exc):
        fd_warmup_exit(self.prev)
        return False


_input_hooks = {}


def fd_autotune_set_input_hook(plan: int, fn) -> None:
    """Install ``fn(batch, bucket, mixed, q, k_cache, v_cache, kv_scales)``
    (fd_tensor descriptors of the tuner's device buffers; kv_scales is None
    for bf16) that writes representative tuning inputs; None removes it."""
    if fn is None:
        _input_hooks.pop(plan, None)
        _check(load_library().fd_autotune_set_input_hook(plan, INPUTS_FN(), None))
        return

    def hook(user, b, k, mixed, q, kc, vc, sc, stream):
        try:
            fn(b, k, mixed, q.contents, kc.contents, vc.contents, sc.contents if sc else None)
            return FD_OK
        except Exception:
            return FD_ERR_INVALID_ARG
    cb = INPUTS_FN(hook)
    _input_hooks[plan] = cb
    _check(load_library().fd_autotune_set_input_hook(plan, cb, None))


def fd_autotune_clear(plan: int, remove_file: bool = False) -> None:
    _check(load_library().fd_autotune_clear(plan, 1 if remove_file else 0))


def fd_autotune(plan: int, batch_sizes: Sequence[int], min_bucket: int = 0, max_bucket: int = 0,
                stream=None) -> None:
    arr = (ctypes.c_int * len(batch_sizes))(*batch_sizes)
    st = None if plan in _timers else _stream_handle(stream)   # a timer hook launches nothing
    _check(load_library().fd_autotune(plan, arr, len(batch_sizes), min_bucket, max_bucket, st))


def fd_query_splits(plan: int, batch: int, max_seqlen: int) -> int:
    v = ctypes.c_int()
    _check(load_library().fd_query_splits(plan, batch, max_seqlen, ctypes.byref(v)))
    return v.value


_timers = {}


def fd_autotune_set_timer(plan: int, fn) -> None:
    """Install ``fn(batch, bucket, num_splits) -> time`` (None restores CUDA events)."""
    if fn is None:
        _timers.pop(plan, None)
        _check(load_library().fd_autotune_set_timer(plan, TIMER_FN(), None))
        return
    cb = TIMER_FN(lambda user, b, k, s: float(fn(b, k, s)))
    _timers[plan] = cb  # keep the callback alive
    _check(load_library().fd_autotune_set_timer(plan, cb, None))


def fd_autotune_set_cache_dir(plan: int, directory: Optional[str]) -> None:
    _check(load_library().fd_autotune_set_cache_dir(plan, directory.encode() if directory else None))


def fd_autotune_stats(plan: int) -> Tuple[int, int]:
    a, b = ctypes.c_int(), ctypes.c_int()
    _check(load_library().fd_autotune_stats(plan, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def fd_read_device_status(plan: int) -> int:
    """Read and clear the plan's device status word (FD_DEVSTAT_* bits)."""
    v = ctypes.c_int()
    s = load_library().fd_read_device_status(plan, ctypes.byref(v))
    if s not in (FD_OK, FD_ERR_DEVICE_STATUS):
        _check(s)
    return v.value


def fd_selftest_wait_timeout(plan: int, limit_us: int, stream=None) -> None:
    """Enqueue the bounded-wait self-test: a wait that nothing completes gives
    up after limit_us and sets FD_DEVSTAT_WAIT_TIMEOUT in the plan's status."""
    _check(load_library().fd_selftest_wait_timeout(plan, limit_us, _stream_handle(stream)))


def fd_plan_workspace_bytes(plan: int) -> int:
    v = ctypes.c_size_t()
    _check(load_library().fd_plan_workspace_bytes(plan, ctypes.byref(v)))
    return v.value


def fd_profile_begin(plan: int) -> None:
    _check(load_library().fd_profile_begin(plan))


def fd_profile_end(plan: int) -> Tuple[int, float, float]:
    """(calls, summed stage-1 ms, summed stage-2 ms) since fd_profile_begin."""
    n, a, b = ctypes.c_int(), ctypes.c_double(), ctypes.c_double()
    _check(load_library().fd_profile_end(plan, ctypes.byref(n), ctypes.byref(a), ctypes.byref(b)))
    return n.value, a.value, b.value


def fd_probe_hbm_read(src, sink, stream=None) -> None:
    """Enqueue the read-only HBM probe over all of ``src`` (a contiguous device
    tensor of a multiple of 16 bytes); every 16-byte word is XORed into
    ``sink`` (a device tensor of 4 int32 / uint32)."""
    if not src.is_contiguous() or not sink.is_contiguous():
        raise ValueError("src and sink must be contiguous")
    _check(load_library().fd_probe_hbm_read(src.data_ptr(), src.numel() * src.element_size(), sink.data_ptr(),
                                            _stream_handle(stream)))


def fd_probe_hbm_copy(src, dst, stream=None) -> None:
    """Enqueue the HBM copy probe: all bytes of ``src`` into ``dst`` (contiguous
    device tensors of the same byte size)."""
    if not src.is_contiguous() or not dst.is_contiguous():
        raise ValueError("src and dst must be contiguous")
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("src and dst byte sizes differ")
    _check(load_library().fd_probe_hbm_copy(src.data_ptr(), dst.data_ptr(), nbytes, _stream_handle(stream)))
