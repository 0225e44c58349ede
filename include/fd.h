/*
 * fd.h - C ABI of libfd: split-KV grouped-query flash decode over a paged KV
 * cache, for NVIDIA GB300 (sm_103a).
 *
 * What the library computes. For every request b, query token t < Tq and
 * query head h, softmax attention of q[b, t, h, :] over the first
 * L_b - (Tq - 1) + t keys of request b, where L_b = cache_seqlens[b] and key j
 * lives in cache page page_table[b, j / P] at slot j % P, KV head h / G
 * (G = Hq / Hkv). This is the decode attention of the kernels listed in
 * "feat(autotune): separate general and decode attention warmup" (LightLLM
 * PR 1549), section "Covered decode kernels": GQA flash decode stage 1, the
 * stage-2 merge, INT8 and INT4 KV variants, MTP attention with several query
 * tokens per request, and the num_splits knob of FA3 KV-cache decode.
 * Stage 1 computes, per (request, KV head, KV split), a partial output and its
 * log-sum-exp; stage 2 merges the splits by LSE. Split boundaries and
 * per-request metadata are derived on the device from cache_seqlens, so a call
 * reads no device memory on the host, never synchronises, never allocates and
 * can be captured in a CUDA graph (sglang PR 29843 summary, sections
 * "motivation" and "implementation": graph-replayed metadata built from
 * cache_seqlens / page_table with no .item() call).
 *
 * Conventions shared by every entry point:
 *  - Every function returns an fd_status. None aborts, prints or exits.
 *    fd_last_error() returns a thread-local message for the last failure.
 *  - Pointers inside fd_tensor are device pointers unless stated otherwise;
 *    the caller owns every tensor. The library never frees caller memory.
 *  - Work is enqueued on the given stream only (NULL = legacy default stream).
 *  - A plan is not thread-safe: calls that use one plan from several host
 *    threads at once must be serialised by the caller.
 */
#ifndef FD_H_
#define FD_H_

#include <stddef.h>
#include <stdint.h>

#if defined(FD_BUILDING_LIBRARY) && defined(__GNUC__)
#define FD_API __attribute__((visibility("default")))
#else
#define FD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *fd_stream_t;

typedef enum fd_status {
  FD_OK = 0,
  FD_ERR_INVALID_ARG = 1,    /* a descriptor or argument is malformed or inconsistent */
  FD_ERR_UNSUPPORTED = 2,    /* well formed but outside what the kernels implement */
  FD_ERR_WORKSPACE = 3,      /* the plan's workspace is too small or absent (host-only plan) */
  FD_ERR_CAPTURING = 4,      /* refused because the stream is capturing a CUDA graph */
  FD_ERR_CUDA = 5,           /* a CUDA runtime / driver call failed (message has the code) */
  FD_ERR_DEVICE_STATUS = 6,  /* a kernel recorded a problem in the plan's status word */
  FD_ERR_TIMEOUT = 7,        /* a bounded device-side wait gave up */
  FD_ERR_NO_PLAN = 8,        /* no current plan on this thread (see fd_set_plan) */
  FD_ERR_IO = 9              /* autotune cache file could not be read or written */
} fd_status;

typedef enum fd_dtype {
  FD_BF16 = 0,
  FD_FP32 = 1,
  FD_INT8 = 2,
  FD_INT4X2 = 3,  /* two signed 4-bit codes per byte, even channel in the low nibble */
  FD_INT32 = 4,
  FD_INT64 = 5
} fd_dtype;

/* How fd_graph_metadata forms cu_seqlens_q. */
typedef enum fd_q_mode {
  FD_QMODE_PRESET = 0,  /* copied from q_in, int32 [B + 1] */
  FD_QMODE_CUMSUM = 1,  /* exclusive prefix sum of q_in, int32 [B] query tokens per request */
  FD_QMODE_STRIDED = 2  /* b * q_stride: q_stride query tokens per request */
} fd_q_mode;

/* How a call cuts its requests' keys into splits (fd_plan_set_split_policy). */
typedef enum fd_split_policy {
  /* Default. Every split of the batch holds about the same number of pages:
   * the batch's n_total pages (sum of ceil(L_b / P)) are cut into chunks of
   * cp = ceil(n_total / (B * num_splits)) pages, and request b gets
   * min(s_cap, ceil(ceil(L_b / P) / cp)) equal page-aligned splits, where
   * s_cap = min(64, the plan's workspace rows / (B * Tq * Hq)) >= max_splits.
   * A long request gets more splits than a short one, so a mixed-length
   * batch keeps its CTAs evenly loaded; with equal lengths the splits are
   * exactly those of FD_SPLIT_EQUAL. The map is rebuilt on the device from
   * cache_seqlens by every call. */
  FD_SPLIT_BALANCED = 0,
  /* num_splits equal page-aligned chunks of each request's keys:
   * chunk_b = P * ceil(ceil(L_b / num_splits) / P). */
  FD_SPLIT_EQUAL = 1
} fd_split_policy;

/* Bits of the plan's device status word (see fd_read_device_status). */
#define FD_DEVSTAT_BAD_PAGE 1u         /* a visible key's page id was outside [0, num_pages) */
#define FD_DEVSTAT_SEQLEN_OVERFLOW 2u  /* cache_seqlens[b] > page_table width * page size, or < 0 */
#define FD_DEVSTAT_WAIT_TIMEOUT 4u     /* a pipeline wait gave up; results of that call are garbage */

/*
 * A strided tensor descriptor. shape/stride have ndim valid entries (ndim <=
 * 5), outermost first; strides are in elements (for FD_INT4X2, in bytes).
 * data is a device pointer (host pointer only where an entry point says so).
 */
typedef struct fd_tensor {
  void *data;
  int32_t dtype; /* an fd_dtype */
  int32_t ndim;
  int64_t shape[5];
  int64_t stride[5];
} fd_tensor;

/* Opaque plan: problem geometry, device workspace, status word and the
 * num_splits autotune table. */
typedef struct fd_plan fd_plan;

/*
 * fd_plan_create - build a plan for one decode geometry, OUTSIDE graph capture.
 * No passage defines it (plain reading): the pages' kernels need split
 * scratch, and a captured call cannot allocate it ("sglang PR 29843"
 * summary, section 实现拆解 and its test: a captured decode graph reads
 * metadata buffers prepared per batch size before capture), so it is
 * allocated once here, with the tuning table beside it.
 *
 *  device          CUDA device ordinal; -1 makes a host-only plan that holds a
 *                  tuning table and validates descriptors but cannot decode
 *                  (fd_decode_paged then returns FD_ERR_WORKSPACE).
 *  max_batch       largest B any call will use (>= 1).
 *  max_q_per_req   largest Tq (query tokens per request, MTP) any call will use.
 *  num_q_heads     Hq; num_kv_heads Hkv; Hq % Hkv == 0.
 *  head_dim        D, 64 or 128.
 *  page_size       P, a power of two in [8, 256] (a page's rows are moved as
 *                  whole 8-row TMA swizzle atoms).
 *  kv_dtype        FD_BF16, FD_INT8 or FD_INT4X2.
 *  max_splits      largest num_splits any call will use, 1..64.
 *  softmax_scale   > 0, or 0 for 1/sqrt(D).
 *  plan            out: the new plan.
 *
 * Allocates the split workspace (fp32 partial outputs and LSE, sized for
 * max_batch * max_q_per_req * Hq * max_splits rows of D) and a status word on
 * the device. Reads, at creation:
 *  - FD_AUTOTUNE_CACHE_DIR: the tuning cache directory;
 *  - FD_MERGE=fused: merge splits in stage 1 (last split CTA of a tile)
 *    instead of the stage-2 kernel (equal split policy only);
 *  - FD_QUANT_KERNEL=tc: run INT8 / INT4 caches with head_dim 128 on the
 *    tcgen05 stage-1 kernel (tensor-memory accumulators) instead of the
 *    register (mma.sync) kernel. Same results within rounding; slower on
 *    GB300 at the time of writing.
 */
FD_API fd_status fd_plan_create(int device, int max_batch, int max_q_per_req, int num_q_heads,
                         int num_kv_heads, int head_dim, int page_size, fd_dtype kv_dtype,
                         int max_splits, float softmax_scale, fd_plan **plan);

/* fd_plan_destroy - free a plan and its device memory (NULL is a no-op).
 * The caller must make sure no enqueued call still uses it. */
FD_API fd_status fd_plan_destroy(fd_plan *plan);

/* fd_set_plan - make plan the current plan of the calling thread (NULL
 * clears it). fd_decode_paged uses the current plan. */
FD_API fd_status fd_set_plan(fd_plan *plan);

/* fd_get_plan - the calling thread's current plan, or NULL. */
FD_API fd_plan *fd_get_plan(void);

/*
 * fd_plan_set_split_policy - choose how calls on this plan place their split
 * boundaries (an fd_split_policy; default FD_SPLIT_BALANCED). Results do not
 * depend on it beyond rounding. Host only; takes effect from the next call.
 * The balanced policy is this library's own: the pages describe per-request
 * num_splits only (FA3's knob in "Covered decode kernels" of "feat(autotune):
 * separate general and decode attention warmup").
 */
FD_API fd_status fd_plan_set_split_policy(fd_plan *plan, int policy);

/*
 * fd_decode_paged - one decode attention call (stage 1 and, when any request
 * is split, stage 2), enqueued on stream.
 *
 *  q             bf16 [B, Tq, Hq, D], innermost stride 1.
 *  k_cache       [num_pages, P, Hkv, D] bf16 or int8, or [num_pages, P, Hkv, D/2]
 *                int4x2; innermost stride 1, every other stride a multiple of
 *                16 bytes, base 16-byte aligned (the cache is read with TMA).
 *  v_cache       same dtype, shape and strides as k_cache.
 *  kv_scales     fp32 [2, num_pages, P, Hkv, n_g] (index 0 = K scales, 1 = V
 *                scales; n_g = 1 for int8, D/32 for int4; innermost stride 1,
 *                n_g * 4 bytes aligned). NULL for bf16. The scale of a cache
 *                row sits at the row's (page, slot, head) index:
 *                value = code * scale[group of the channel].
 *  page_table    int32 [B, W], innermost stride 1. Entries past a request's
 *                last page (the -1 sentinel) are never read.
 *  cache_seqlens int32 [B] (device): L_b, the keys request b owns. Must be
 *                <= W * P; rows with L_b - (Tq-1) + t <= 0 keys get out = 0,
 *                lse = -inf.
 *  q_per_req     Tq, equal to q.shape[1] and <= the plan's max_q_per_req.
 *                Query token t sees keys [0, L_b - (Tq-1) + t) (causal MTP).
 *  num_splits    1..plan max_splits, or 0 to use the autotuned value for
 *                (B, bucket of the max-seqlen hint) (see fd_set_max_seqlen_hint).
 *                Splits per request: on average over the batch under the
 *                balanced policy, exactly under the equal one (see
 *                fd_split_policy). Results do not depend on it beyond
 *                rounding. A request with a single non-empty split gets its
 *                outputs from stage 1 directly.
 *  out           [B, Tq, Hq, D] bf16 (round to nearest even) or fp32,
 *                innermost stride 1.
 *  lse           fp32 [B, Tq, Hq] natural-log LSE of the scaled scores, or NULL.
 *  stream        stream to enqueue on.
 *
 * Kernels record bad metadata (page id out of range, L_b over capacity) in
 * the plan's status word instead of faulting; read it with
 * fd_read_device_status. Calls on one plan that overlap on the device race on
 * its workspace: serialise them on one stream.
 */
FD_API fd_status fd_decode_paged(const fd_tensor *q, const fd_tensor *k_cache, const fd_tensor *v_cache,
                          const fd_tensor *kv_scales, const fd_tensor *page_table,
                          const fd_tensor *cache_seqlens, int q_per_req, int num_splits,
                          fd_tensor *out, fd_tensor *lse, fd_stream_t stream);

/*
 * fd_decode_paged_static - fd_decode_paged for callers that cannot allocate
 * device memory. The reference pages have no counterpart; it exists because
 * some callers cannot call cudaMalloc: a serving engine that has already
 * reserved all GPU memory for its own pool, or a plugin inside a process
 * that forbids foreign device allocations. It needs no plan and allocates
 * nothing.
 *
 * The split workspace is a fixed 32 MiB array inside the library, held on
 * every GPU that loads it until the process exits. A call needing more,
 * B*Tq*Hq*num_splits*(D+1)*4 bytes when num_splits > 1, fails with
 * FD_ERR_WORKSPACE.
 *
 * Arguments are those of fd_decode_paged, with these differences:
 *  - num_splits must be 1..64 (there is no tuning table), and splits are
 *    always FD_SPLIT_EQUAL, merged by the stage-2 kernel;
 *  - softmax_scale is explicit (0 = 1/sqrt(D));
 *  - Hq is at most 4096;
 *  - the device is the current one (compute capability 10.x or later, else
 *    FD_ERR_UNSUPPORTED).
 *
 * The first call on a device does a one-time set-up: it looks up the array's
 * address, reads the device's SM count and compute capability, and raises
 * the kernels' shared-memory limit.
 *
 * All calls share the array. Calls that overlap on the GPU race on it, so
 * serialise them on one stream. Kernel status bits go to an internal word
 * that this entry point does not report.
 */
FD_API fd_status fd_decode_paged_static(const fd_tensor *q, const fd_tensor *k_cache,
                                        const fd_tensor *v_cache, const fd_tensor *kv_scales,
                                        const fd_tensor *page_table, const fd_tensor *cache_seqlens,
                                        int q_per_req, int num_splits, float softmax_scale,
                                        fd_tensor *out, fd_tensor *lse, fd_stream_t stream);

/*
 * fd_graph_metadata - the per-step metadata of a decode batch, built on the
 * device in one launch from a serving engine's request-to-token pool: the
 * step before fd_decode_paged in a graph-replayed decode loop ("sglang PR
 * 29843" summary, section 实现拆解 item 1: one program per batch row builds
 * cache_seqlens, cu_seqlens_k / cu_seqlens_q and page_table, three q modes
 * and a -1 sentinel guard, replacing about 25 host-dispatched operations that
 * cost 0.7-1.0 ms per replay, section 功能与动机).
 *
 *  req_to_token     int32 [R, C] (device): KV slot of token position c of
 *                   pool request r, slot = page * P + offset; < 0 = no slot.
 *                   A request's pages start on page boundaries.
 *  req_pool_indices int32 or int64 [B]: pool row of batch row b; < 0 marks a
 *                   padding row (all outputs of the row empty).
 *  seq_lens         int32 [B]: keys of each request.
 *  page_size        P >= 1.
 *  q_mode           an fd_q_mode; q_in and q_stride as the mode says
 *                   (q_in may be NULL for FD_QMODE_STRIDED).
 *  page_table       int32 [B, W] out: entry j = req_to_token[r, j * P] / P
 *                   for j < ceil(L_b / P), else -1 (also for an unallocated
 *                   slot and on padding rows).
 *  cache_seqlens    int32 [B] out: seq_lens (0 on padding rows).
 *  cu_seqlens_k     int32 [B + 1] out: exclusive prefix sum of cache_seqlens.
 *  cu_seqlens_q     int32 [B + 1] out.
 *  status           int32 [1] (device) or NULL: FD_DEVSTAT_BAD_PAGE for a
 *                   pool index >= R or a page past column C, and
 *                   FD_DEVSTAT_SEQLEN_OVERFLOW for more than W pages, ORed in.
 *  stream           stream to enqueue on.
 *
 * Reads no device memory on the host, never synchronises or allocates: the
 * call can be captured in a CUDA graph together with fd_decode_paged, whose
 * page_table and cache_seqlens it fills. Sums must fit in int32.
 */
FD_API fd_status fd_graph_metadata(const fd_tensor *req_to_token, const fd_tensor *req_pool_indices,
                                   const fd_tensor *seq_lens, int page_size, int q_mode, const fd_tensor *q_in,
                                   int q_stride, fd_tensor *page_table, fd_tensor *cache_seqlens,
                                   fd_tensor *cu_seqlens_k, fd_tensor *cu_seqlens_q, fd_tensor *status,
                                   fd_stream_t stream);

/* fd_set_max_seqlen_hint - host-known upper bound of cache_seqlens for the
 * next calls with num_splits = 0; picks the KV-length bucket of the tuning
 * table without reading device memory ("feat(autotune): ...", section
 * "Covered decode kernels": run keys bucketed by KV length while execution
 * uses the real length). 0 clears the hint (the longest bucket is used). */
FD_API fd_status fd_set_max_seqlen_hint(fd_plan *plan, int max_seqlen);

/* fd_set_mean_seqlen_hint - host-known mean of cache_seqlens for the next
 * calls with num_splits = 0 under the balanced split policy: the tuning table
 * is then looked up at the power of two nearest the mean (log scale) instead
 * of the bucket of the max. Balanced splits give a mixed-length batch of mean
 * m the per-CTA work of an equal-length batch of length m, which is what the
 * table was tuned on. If the max hint is also set and at least 1.25 x the
 * mean, the table tuned on mixed lengths is used (when it has entries).
 * 0 clears the hint. Host only. */
FD_API fd_status fd_set_mean_seqlen_hint(fd_plan *plan, int mean_seqlen);

/*
 * fd_autotune - pick num_splits per (batch, KV-length bucket) by timing
 * (same page, sections "Changes" and "Covered decode kernels": decode
 * attention tuned at startup on representative inputs, outside graph capture,
 * at a representative length, default 32768; configs persisted and reused).
 *
 *  batch_sizes / n_batch  batch sizes to tune (each 1..max_batch).
 *  min_bucket, max_bucket KV-length buckets: powers of two from min_bucket to
 *                         max_bucket (0, 0 = 1024 .. FD_AUTOTUNE_SEQ_LEN or 32768).
 *  stream                 stream whose queued work the timing launches follow
 *                         (an argument of this library's own: the page tunes
 *                         inside the engine's process and names no stream).
 *
 * Candidates are num_splits in {1, 2, 3, 4, 6, 8, 12, 16, 32, 64} (up to
 * max_splits), plus the counts
 * that fill one or two waves of one CTA per SM, none cutting the bucket into
 * splits of fewer than 128 keys. For each key not already in
 * the table (loaded from the cache directory), synthetic inputs of the bucket
 * length are timed as a decode loop runs them: a CUDA graph of consecutive
 * calls, each on pages of its own (together at least 4x L2 where memory
 * allows), replayed back to back, median of five timed blocks. The fastest
 * candidate is stored (an exact tie goes to fewer splits) and the table
 * saved. Each (batch, bucket K) is tuned twice: with every request K keys
 * long, and (batches of 2 or more) with lengths spread evenly over
 * [K/8, 15K/8] (mean K), the table that calls whose hints show a spread use
 * (see fd_set_mean_seqlen_hint). Refuses with FD_ERR_CAPTURING while
 * the stream is capturing. Keys already in the table (tuned earlier or loaded
 * from the cache) are not searched again; see fd_autotune_clear.
 * Allocates temporary device buffers and a private stream (freed before
 * return); the timing runs on that stream after the work of `stream`.
 */
FD_API fd_status fd_autotune(fd_plan *plan, const int *batch_sizes, int n_batch, int min_bucket,
                      int max_bucket, fd_stream_t stream);

/* fd_query_splits - the num_splits a num_splits = 0 call would use for
 * (batch, max_seqlen) and the plan's mean-length hint: the tuned entry of the
 * nearest tuned batch and the lookup bucket (see fd_set_mean_seqlen_hint),
 * else the built-in heuristic. Host only. No passage defines it (plain
 * reading): it exposes the lookup that fd_decode_paged makes. */
FD_API fd_status fd_query_splits(fd_plan *plan, int batch, int max_seqlen, int *num_splits);

/* Timer hook for fd_autotune: returns the time of one call with num_splits
 * for (batch, bucket), in any unit; bucket is negative (-K) for the
 * mixed-length inputs of bucket K. NULL restores CUDA-event timing. With a
 * hook installed fd_autotune launches nothing, so its table logic can be
 * exercised on a host-only plan. */
typedef double (*fd_timer_fn)(void *user, int batch, int bucket, int num_splits);
FD_API fd_status fd_autotune_set_timer(fd_plan *plan, fd_timer_fn fn, void *user);

/*
 * Warmup phases ("feat(autotune): separate general and decode attention
 * warmup", section "Changes"): tuning is split into a GENERAL and a
 * DECODE_ATTENTION warmup phase, entered through a nestable scope that
 * restores the previous phase. Only decode-attention kernels search inside
 * the decode-attention phase; nothing searches outside warmup (live
 * requests). In this library: an fd_decode_paged call with num_splits = 0,
 * made inside FD_PHASE_DECODE_ATTENTION on a stream that is not capturing,
 * first tunes its batch at the representative KV length
 * (FD_AUTOTUNE_SEQ_LEN, default 32768) if the plan's table has no entry for
 * it, then runs with the tuned value; the same call in any other phase, or
 * under capture, only looks the table up. A serving engine runs one such
 * decode before capturing each decode graph, and the capture then uses the
 * tuned value. fd_autotune itself (explicit start-up tuning) runs in any
 * phase. The phase is per host thread.
 */
typedef enum fd_warmup_phase {
  FD_PHASE_NONE = 0,              /* live requests: no tuning */
  FD_PHASE_GENERAL = 1,           /* general (prefill) kernels may tune; decode attention does not */
  FD_PHASE_DECODE_ATTENTION = 2   /* decode attention tunes on its calls */
} fd_warmup_phase;

/* fd_warmup_enter - make phase current on this thread; *previous (may be
 * NULL) receives the phase to restore. fd_warmup_exit - restore it. Scopes
 * nest: exit with the value the matching enter returned. */
FD_API fd_status fd_warmup_enter(int phase, int *previous);
FD_API fd_status fd_warmup_exit(int previous);
/* fd_warmup_current - the calling thread's current phase. */
FD_API int fd_warmup_current(void);

/* Hook that writes representative tuning inputs (the page's
 * rebuild_input_func): called by fd_autotune once per (batch, bucket,
 * spread) key, outside capture, before that key is timed, with the tuner's
 * own buffers: q [batch, Tq, Hq, D], k_cache / v_cache [N, P, Hkv, *] and
 * kv_scales (NULL for bf16). It may overwrite their contents (for example
 * with values drawn like the engine's); the page placement and the lengths
 * stay the tuner's (bucket length, or spread over [K/8, 15K/8] when mixed is
 * 1). A non-FD_OK return aborts the tuning with that status. */
typedef fd_status (*fd_tune_inputs_fn)(void *user, int batch, int bucket, int mixed, fd_tensor *q,
                                       fd_tensor *k_cache, fd_tensor *v_cache, fd_tensor *kv_scales,
                                       fd_stream_t stream);
FD_API fd_status fd_autotune_set_input_hook(fd_plan *plan, fd_tune_inputs_fn fn, void *user);

/* fd_autotune_clear - forget every tuned entry of the plan (and, when
 * remove_file is nonzero, delete its persisted table), so the next tuning
 * searches afresh. Decode attention treats FD_FORCE_AUTOTUNE as adaptive
 * (same page, section "Changes"): cached entries are reused, so that the many
 * layers sharing a geometry never retune; a fresh search needs this call or
 * the cache file removed. */
FD_API fd_status fd_autotune_clear(fd_plan *plan, int remove_file);

/* fd_autotune_set_cache_dir - directory of the persisted tuning table (NULL
 * or "" disables persistence). Default: $FD_AUTOTUNE_CACHE_DIR if set. */
FD_API fd_status fd_autotune_set_cache_dir(fd_plan *plan, const char *dir);

/* fd_autotune_stats - number of (batch, bucket) searches run and cache hits
 * served by fd_autotune on this plan. */
FD_API fd_status fd_autotune_stats(fd_plan *plan, int *searches, int *cache_hits);

/* fd_read_device_status - copy the plan's status word (FD_DEVSTAT_* bits) to
 * *code and clear it. Synchronises the plan's device; not for use inside
 * graph capture. Returns FD_ERR_DEVICE_STATUS when any bit was set. No
 * passage defines it (plain reading): the kernels record bad page ids and
 * lengths instead of faulting, and this reads the record. */
FD_API fd_status fd_read_device_status(fd_plan *plan, int *code);

/* fd_selftest_wait_timeout - run the decode kernels' bounded-wait failure
 * path on purpose. The pages have no counterpart: this checks this library's
 * own guard against a pipeline that never delivers. One CTA of one warp
 * waits, with the decode kernels' wait routine, on a fresh mbarrier that
 * nothing arrives on, and gives up after limit_us microseconds of
 * %globaltimer time (1 .. 2,000,000; the decode kernels use 2 s). It records
 * FD_DEVSTAT_WAIT_TIMEOUT in the plan's status word and returns. No fault, no
 * trap, and the context stays usable. The launch is asynchronous on `stream`;
 * fd_read_device_status reports the bit. Returns FD_ERR_INVALID_ARG for a
 * NULL plan or a limit outside the range, FD_ERR_WORKSPACE for a plan without
 * a device, FD_ERR_CUDA if the launch fails. */
FD_API fd_status fd_selftest_wait_timeout(fd_plan *plan, unsigned limit_us, fd_stream_t stream);

/* fd_plan_workspace_bytes - device bytes the plan's split workspace holds.
 * No passage defines it (plain reading): introspection of fd_plan_create's
 * allocation. */
FD_API fd_status fd_plan_workspace_bytes(fd_plan *plan, size_t *bytes);

/* fd_profile_begin / fd_profile_end - per-stage device time of decode calls.
 * Between begin and end, every fd_decode_paged on this plan records CUDA
 * events on its stream before stage 1, between the stages and after stage 2.
 * Calls made while a stream is being captured record the events as timed
 * event nodes of the graph; replay the graph (once) before fd_profile_end,
 * and destroy it before or right after: fd_profile_end destroys the events.
 * The merge kernel of a profiled call is launched without programmatic
 * dependent launch (the event between the stages separates them anyway).
 * fd_profile_end synchronises on those events and returns the number of
 * calls and the summed stage-1 and stage-2 milliseconds (stage 2 is 0 for
 * calls that launch no merge). fd_profile_end itself is not for use inside
 * graph capture. */
FD_API fd_status fd_profile_begin(fd_plan *plan);
FD_API fd_status fd_profile_end(fd_plan *plan, int *calls, double *stage1_ms, double *stage2_ms);

/*
 * fd_probe_hbm_read / fd_probe_hbm_copy - HBM bandwidth probes. No passage
 * defines them: they measure, on the same GPU and in the same process, the
 * denominator of the decode kernels' roofline (the path is bound by HBM
 * bandwidth on the KV bytes). The read probe reads as the decode kernels do:
 * bulk copies (TMA) of 32 KiB chunks into a six-stage shared-memory ring per
 * SM, each CTA streaming one run of consecutive chunks, folded by the CTA's
 * other warps. The copy probe moves 16-byte vectors, eight loads in flight
 * per thread, four 512-thread CTAs per SM.
 *
 *  fd_probe_hbm_read  reads bytes from src (device) and XORs every 16-byte
 *                     word of it into sink (device, uint32 [4], 16-byte
 *                     aligned), so sink ^= XOR of all words: zero sink first
 *                     to read back the XOR of the buffer.
 *  fd_probe_hbm_copy  copies bytes from src to dst (device, not overlapping).
 *
 * Pointers must be 16-byte aligned and bytes a multiple of 16
 * (FD_ERR_UNSUPPORTED otherwise); NULL pointers give FD_ERR_INVALID_ARG.
 * Enqueued on stream on the current device; no allocation, no sync. Time them
 * with CUDA events over a buffer much larger than L2. */
FD_API fd_status fd_probe_hbm_read(const void *src, size_t bytes, uint32_t *sink, fd_stream_t stream);
FD_API fd_status fd_probe_hbm_copy(const void *src, void *dst, size_t bytes, fd_stream_t stream);

/* Static strings; never NULL. */
FD_API const char *fd_status_string(fd_status status);
FD_API const char *fd_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FD_H_ */
