/*
 * fp8_mqa_logits.h -- C ABI of the GB300 (sm_103a) prefill FP8 MQA indexer-logits library.
 *
 * The operation (ROCm/aiter PR #7183 "[HIP] [JIT] Add gfx950 prefill FP8 MQA logits",
 * section "Motivation", the displayed formula):
 *
 *     out[m, n] = kv_scale[n] * sum_{h < H} relu( Q[m,h,:] . K[n,:] ) * w[m,h]
 *                 for n in [ks[m], ke[m]),   -inf elsewhere (clean_logits = 1).
 *
 * Operator contract (same page, "PR-specific question" and "Motivation"): H = 32 heads,
 * D = 128 head dimension, FP8 Q/K, float32 kv_scale / w / out, int32 row bounds, all
 * contiguous row-major.  FP8 here means OCP E4M3 ("e4m3fn", largest finite value 448).
 *
 * Conventions shared by every entry point below:
 *   - All tensor pointers are DEVICE pointers (cudaMalloc / torch CUDA memory) owned by
 *     the caller, unless an entry point says otherwise.  The library never frees them.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Compute entry
 *     points are asynchronous and stream-ordered: they return after enqueueing work.
 *   - Return value: FP8MQA_OK (0) or a negative fp8mqa_status.  Argument errors are
 *     detected on the host BEFORE anything is enqueued; the library never aborts or
 *     exits the process and throws no exceptions.
 *   - The library keeps one small device buffer per device (about 260 KB: scheduler
 *     slots and a status word), allocated on the first compute call on that device and
 *     kept until process exit.  That first call therefore must not be made while the
 *     stream is being captured into a CUDA graph.
 *   - Scheduler slots.  Each launch's work queue lives in a slot of that buffer.  Direct
 *     launches take slots from a ring of 256 in turn, so more than 256 launches running
 *     at the same moment (on many streams) would share slots and produce wrong output.
 *     A launch made while its stream is being captured into a CUDA graph gets a slot of
 *     its own that no other launch ever uses (a graph's kernel keeps its slot for every
 *     replay); up to 16384 launches can be captured per device and process, after which
 *     capturing returns FP8MQA_ERR_CAPACITY.  Replays of one instantiated graph are
 *     ordered by CUDA; two instantiations of the same captured graph must not run at
 *     the same time.
 */
#ifndef FP8_MQA_LOGITS_H
#define FP8_MQA_LOGITS_H

#include <stdint.h>

#if defined(__GNUC__)
#define FP8MQA_API __attribute__((visibility("default")))
#else
#define FP8MQA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum fp8mqa_status {
    FP8MQA_OK = 0,
    FP8MQA_ERR_INVALID_ARG = -1,       /* null pointer, negative size, bad flag, bad split_n */
    FP8MQA_ERR_UNSUPPORTED_SHAPE = -2, /* H != 32, D != 128, or a size beyond the limits   */
    FP8MQA_ERR_MISALIGNED = -3,        /* q/k/w/kv_scale not 16-byte aligned, out/ks/ke not 4 */
    FP8MQA_ERR_ARCH = -4,              /* current device is not compute capability 10.3     */
    FP8MQA_ERR_LAUNCH = -5,            /* the kernel could not be configured or launched    */
    FP8MQA_ERR_TIMEOUT = -6,           /* a bounded on-device wait gave up (see check_error) */
    FP8MQA_ERR_CUDA = -7,              /* a CUDA runtime call failed                        */
    FP8MQA_ERR_BOUNDS = -8,            /* a bounds-checking build found a bad access        */
    FP8MQA_ERR_CAPACITY = -9           /* no scheduler slot left for another captured launch */
};

/*
 * fp8_mqa_logits -- the logits of every query row against its key window.
 *
 *   q_fp8     [M, H, D] E4M3 bytes, row-major (query row m, head h, dim d at
 *             (m*H + h)*D + d).  16-byte aligned.
 *   k_fp8     [N, D] E4M3 bytes, row-major.  16-byte aligned.
 *   kv_scale  [N] float32, per-key scale, applied after the head sum.  16-byte aligned.
 *   w         [M, H] float32, per-(row, head) weight, applied after relu.  16-byte aligned.
 *   ks, ke    [M] int32: row m attends keys n with ks[m] <= n < ke[m].  Bounds are
 *             clamped to [0, N); ks[m] >= ke[m] is an empty row.  4-byte aligned.
 *   out       [M, N] float32, row-major, 4-byte aligned.  In-window entries are always
 *             written.  clean_logits = 1: every out-of-window entry is written with -inf
 *             (IEEE 0xff800000), so the whole matrix is defined.  clean_logits = 0:
 *             out-of-window entries are not written at all (they keep whatever the
 *             caller put there; "caller-managed output masks", page section
 *             "PR Self-Review / Behavior and intent").
 *   M, N      query rows and keys (>= 0).  M = 0 or N = 0 enqueues nothing and returns OK.
 *             Limits: M*H < 2^31, N < 2^31.
 *   H, D      must be 32 and 128 (FP8MQA_ERR_UNSUPPORTED_SHAPE otherwise).
 *   split_n   0 = automatic; > 0 = split each row block's key range into that many
 *             chunks scheduled independently (the page's "SplitN", section "Design /
 *             Grid choice" and "Known limitations").  Values above ceil(N/128) are
 *             clamped.  The result is bit-identical for every split_n.
 *   stream    cudaStream_t to enqueue on.
 *
 * Numerics: the dot products are exact (FP8 products accumulate in fp32 on the tensor
 * cores); relu, the w-weighted head sum and the kv_scale multiply are fp32.
 * Asynchronous device-side failures (a bounded wait that gave up) are reported by
 * fp8_mqa_logits_check_error.
 */
FP8MQA_API int fp8_mqa_logits(const uint8_t* q_fp8, const uint8_t* k_fp8, const float* kv_scale,
                   const float* w, const int32_t* ks, const int32_t* ke, float* out,
                   int64_t M, int64_t N, int32_t H, int32_t D, int32_t clean_logits,
                   int32_t split_n, void* stream);

/*
 * fp8_mqa_logits_is_supported -- 1 if (M, N, H, D) is inside this library's contract
 * (H = 32, D = 128, M >= 0, N >= 0, M*H < 2^31, N < 2^31) and, for device >= 0, CUDA
 * device `device` exists and has compute capability 10.3; else 0 (the page's
 * is_supported(), section "Motivation").  With device < 0 it is pure host arithmetic and
 * may be called without a GPU; with device >= 0 it only queries device attributes (it
 * launches and allocates nothing).
 */
FP8MQA_API int fp8_mqa_logits_is_supported(int64_t M, int64_t N, int32_t H, int32_t D,
                                           int32_t device);

/*
 * fp8_mqa_logits_default_split -- the split_n that split_n = 0 selects for an
 * (M, N) problem on a GPU with `num_sms` multiprocessors.  Host arithmetic only.
 */
FP8MQA_API int fp8_mqa_logits_default_split(int64_t M, int64_t N, int32_t num_sms);

/*
 * fp8_mqa_logits_check_error -- synchronizes `stream`, then reads and clears the
 * current device's status words: the one of fp8_mqa_logits / fp8_mqa_logits_host and the
 * one of fp8_mqa_logits_noalloc (each only if a call has set it up; this call allocates
 * nothing).  Returns FP8MQA_ERR_TIMEOUT if a launch since the last check had a bounded
 * on-device wait give up (its output is then incomplete), FP8MQA_ERR_BOUNDS if a
 * bounds-checking build of the library recorded an out-of-range access,
 * FP8MQA_ERR_CUDA if the synchronization or a read failed, else FP8MQA_OK.
 */
FP8MQA_API int fp8_mqa_logits_check_error(void* stream);

/*
 * fp8_mqa_logits_set_wait_limit_ns -- sets how long one on-device pipeline wait may last
 * before the kernel gives up (FP8MQA_ERR_TIMEOUT, reported by check_error), for launches
 * enqueued after the call; 0 restores the default of 1 s.  Returns the previous limit.
 * A kernel that gives up still waits for its own copies and tensor-core work in flight
 * (for up to 1 s more) before it frees its resources and exits; the next launch is
 * unaffected.  Meant for diagnostics and for testing that failure path; a limit far
 * below a call's duration makes every call fail.  Host only; process-wide.
 */
FP8MQA_API uint64_t fp8_mqa_logits_set_wait_limit_ns(uint64_t ns);

/*
 * fp8_mqa_logits_host_workspace_bytes -- size of the device workspace that
 * fp8_mqa_logits_host needs for an (M, N) problem (H = 32, D = 128), or 0 for a
 * shape outside the contract.
 */
FP8MQA_API uint64_t fp8_mqa_logits_host_workspace_bytes(int64_t M, int64_t N, int32_t H, int32_t D);

/*
 * fp8_mqa_logits_host -- the same operation on HOST buffers.  Enqueues host->device
 * copies of q, k, kv_scale, w, ks, ke into `workspace`, the kernel, and device->host
 * copies of all of out, ordered after the work already on `stream`; work enqueued on
 * `stream` after the call runs after all of it.  The rows go in chunks of about 32 MB of
 * logits (at most 8): the inputs travel on a library stream, the chunks' kernels run on
 * `stream`, and each chunk's logits go back on a second library stream as soon as its
 * kernel is done, so the copies in both directions and the kernels overlap.  The two
 * library streams and their events are created on a device's first call and live until
 * the process exits; calls on one device enqueue one at a time, and their copies share
 * the library streams.  The call can be captured into a CUDA graph (the library streams
 * fork from `stream` by an event and join it again).  Host buffers should be pinned
 * (cudaHostAlloc) for the copies to be asynchronous; pageable memory works but the
 * copies then block.  The call returns after enqueueing; synchronize `stream` before
 * reading `out`.  With clean_logits = 0, the device copy of out is first filled from the
 * host `out`, so untouched entries come back unchanged.
 *   workspace        device pointer, 256-byte aligned, at least
 *                    fp8_mqa_logits_host_workspace_bytes(M, N, H, D) bytes, caller-owned.
 *   workspace_bytes  its size.
 * Other arguments as for fp8_mqa_logits.
 */
FP8MQA_API int fp8_mqa_logits_host(const uint8_t* q_fp8, const uint8_t* k_fp8, const float* kv_scale,
                        const float* w, const int32_t* ks, const int32_t* ke, float* out,
                        int64_t M, int64_t N, int32_t H, int32_t D, int32_t clean_logits,
                        int32_t split_n, void* workspace, uint64_t workspace_bytes,
                        void* stream);

/*
 * fp8_mqa_logits_noalloc -- fp8_mqa_logits for callers that cannot allocate device
 * memory.  The pages this library follows have no counterpart: it exists for hosts such
 * as serving engines that reserve nearly all HBM for their own pools up front and forbid
 * allocations outside them, plug-in interfaces of inference runtimes whose contract bars
 * a plug-in from allocating, and latency-critical loops where a cudaMalloc (which can
 * synchronize the device) or a first-call allocation is not acceptable.
 *
 * Arguments, layouts, results and errors are those of fp8_mqa_logits; the output is the
 * same bit for bit.  Differences:
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.  Its scratch (the
 *     scheduler's work counters and a status word) is a 256-byte device array compiled
 *     into the library, which every GPU that loads the library holds until process exit.
 *     The scratch a call needs does not depend on M or N; a call that needed more than
 *     the array holds would be refused with FP8MQA_ERR_UNSUPPORTED_SHAPE.
 *   - The first call on a device looks up the array's device address (once per device,
 *     with that device current); make that first call before any stream capture.
 *   - Every call shares the one array.  Each call clears the work counters on `stream`
 *     before its kernel, so calls that overlap on the GPU (for example on two streams
 *     at once) race on them and may produce wrong output: order such calls on one
 *     stream or with events.
 *   - A bounded on-device wait that gives up is recorded in the array's status word;
 *     fp8_mqa_logits_check_error reads and clears it (and allocates nothing).
 */
FP8MQA_API int fp8_mqa_logits_noalloc(const uint8_t* q_fp8, const uint8_t* k_fp8,
                                      const float* kv_scale, const float* w, const int32_t* ks,
                                      const int32_t* ke, float* out, int64_t M, int64_t N,
                                      int32_t H, int32_t D, int32_t clean_logits,
                                      int32_t split_n, void* stream);

/*
 * fp8_mqa_topk -- per-row top-k over a logits matrix, the step that consumes the indexer
 * logits (ROCm/aiter PR #7183 "[HIP] [JIT] Add gfx950 prefill FP8 MQA logits", "Test plan":
 * top-512 selections compared end to end; ROCm/aiter PR #6159 "[Triton/Gluon] GFX950 sparse
 * mla optimizations", "Technical Details": sparse MLA with top-k 512).  The pages fix no tie
 * rule or padding; this library reads the step as:
 *   - only finite entries are eligible (-inf, a key outside the row's window, never is);
 *   - row m's result lists its k largest eligible entries by value, descending, and equal
 *     values by index, ascending (-0.0 equals +0.0);
 *   - slots past the row's eligible entries hold index -1 and value -inf.
 * The result is therefore unique.
 *
 *   logits   DEVICE float32, row m at logits + m * ld (ld >= N), 4-byte aligned; typically
 *            the `out` of fp8_mqa_logits with clean_logits = 1.  Not modified.
 *   M, N     rows and entries per row (M >= 0, 0 <= N <= 2^30).  M = 0 enqueues nothing.
 *   k        1 <= k <= 2048.
 *   indices  DEVICE int32 [M, k], row-major, 4-byte aligned, written.
 *   values   DEVICE float32 [M, k] or NULL; when given, the selected logits (their exact
 *            bits), -inf in padded slots.
 *   stream   cudaStream_t; asynchronous.
 * Errors: FP8MQA_ERR_INVALID_ARG (sizes, k, null pointers), FP8MQA_ERR_UNSUPPORTED_SHAPE
 * (N too large), FP8MQA_ERR_MISALIGNED, FP8MQA_ERR_ARCH, FP8MQA_ERR_LAUNCH.  The first call on
 * a device sets up the same per-device state as fp8_mqa_logits.
 */
FP8MQA_API int fp8_mqa_topk(const float* logits, int64_t M, int64_t N, int64_t ld, int32_t k,
                            int32_t* indices, float* values, void* stream);

/*
 * fp8_mqa_topk_windowed -- fp8_mqa_topk restricted to each row's key window: row m's result
 * is the top-k of logits[m, n] for n in [ks[m], ke[m]) (clamped to [0, N); empty when
 * ks[m] >= ke[m]), with the same order, tie rule and padding.  Entries outside the window are
 * never read, so the logits may come from fp8_mqa_logits with clean_logits = 0 (whatever lies
 * outside the windows is ignored), and only the windows' bytes are read.  With the windows that
 * made the logits, the result equals fp8_mqa_topk's on the clean_logits = 1 output.  The page
 * has no such entry; it is this library's way to let the consumer skip the -inf fill.
 *
 *   ks, ke   DEVICE int32 [M], 4-byte aligned, the same windows as fp8_mqa_logits takes; both
 *            null gives fp8_mqa_topk.  Not modified.
 *   the other arguments and the errors are fp8_mqa_topk's; ks without ke (or the reverse) is
 *   FP8MQA_ERR_INVALID_ARG.
 */
FP8MQA_API int fp8_mqa_topk_windowed(const float* logits, int64_t M, int64_t N, int64_t ld,
                                     const int32_t* ks, const int32_t* ke, int32_t k,
                                     int32_t* indices, float* values, void* stream);

/*
 * fp8_mqa_topk_ex -- fp8_mqa_topk_windowed with flags.
 *
 *   flags    0, or FP8MQA_TOPK_UNSORTED: each row's result holds the same entries (the same
 *            set of indices, each with its exact value), in an unspecified order that may differ
 *            between calls; the padding still follows the selected entries.  This skips the
 *            winners' sort, for consumers that take the indices as a set (sparse attention
 *            gathers them).  Any other bit is FP8MQA_ERR_INVALID_ARG.
 *   the other arguments and the errors are fp8_mqa_topk_windowed's.
 */
#define FP8MQA_TOPK_UNSORTED 1
FP8MQA_API int fp8_mqa_topk_ex(const float* logits, int64_t M, int64_t N, int64_t ld,
                               const int32_t* ks, const int32_t* ke, int32_t k, int32_t flags,
                               int32_t* indices, float* values, void* stream);

/* fp8_mqa_logits_strerror -- a static, human-readable name for a status code. */
FP8MQA_API const char* fp8_mqa_logits_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* FP8_MQA_LOGITS_H */
