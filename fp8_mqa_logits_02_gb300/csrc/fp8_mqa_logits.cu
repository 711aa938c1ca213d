// Host side of the C ABI declared in include/fp8_mqa_logits.h: argument validation,
// per-device state (scheduler slots, status word), TMA tensor maps, split choice and
// the launch.  The device code is in logits_kernel.cuh.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <functional>
#include <mutex>

#include "../../include/fp8_mqa_logits.h"
#include "logits_kernel.cuh"
#include "topk_kernel.cuh"

namespace fp8mqa {
namespace {

constexpr int kMaxDevices = 64;
// Scheduler slots: a ring for direct launches (a slot is reused every kSchedSlots launches)
// and one slot of its own for every launch captured into a CUDA graph (never reused, since a
// graph's kernel keeps its slot for every replay).
constexpr uint32_t kSchedSlots = 256;
constexpr uint32_t kGraphSlots = 16384;
constexpr uint64_t kDefaultWaitNs = 1000000000ull;  // bounded device waits give up after 1 s
constexpr uint64_t kDrainNs = 1000000000ull;        // bound of the drain before a CTA exits
constexpr uint64_t kHintedWaitNs = 100000ull;       // shorter limits also bound each suspension
constexpr size_t kStatusBytes = 256;                // status word + first bounds violation

std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};

struct DeviceState {
    std::once_flag once;
    int init_status = FP8MQA_OK;
    std::atomic<bool> ready{false};
    int sm_count = 0;
    SchedSlot* sched = nullptr;  // kSchedSlots ring slots, then kGraphSlots graph slots, zeroed
    int32_t* status = nullptr;   // status word (+ bounds record)
    std::atomic<uint32_t> seq{0};
    std::atomic<uint32_t> graph_seq{0};
};

DeviceState g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode()
{
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
}


// Every top-k kernel's dynamic shared memory limit, for the whole-row (kWin = false) and the
// windowed instantiations.
template <bool kWin>
bool topk_set_smem()
{
    const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
    return cudaFuncSetAttribute(topk_kernel<TopkSmemOne, kWin, 12>, attr,
                                int(sizeof(TopkSmemOne))) == cudaSuccess &&
           cudaFuncSetAttribute(topk_kernel<TopkSmemPair, kWin, 11>, attr,
                                int(2 * sizeof(TopkSmemPair))) == cudaSuccess &&
           cudaFuncSetAttribute(topk_kernel<TopkSmemPair, kWin, 12>, attr,
                                int(2 * sizeof(TopkSmemPair))) == cudaSuccess &&
           cudaFuncSetAttribute(topk_kernel<TopkSmemPairWide, kWin, 11>, attr,
                                int(2 * sizeof(TopkSmemPairWide))) == cudaSuccess &&
           cudaFuncSetAttribute(topk_kernel<TopkSmemPairWide, kWin, 12>, attr,
                                int(2 * sizeof(TopkSmemPairWide))) == cudaSuccess &&
           cudaFuncSetAttribute(topk_reg_kernel<kWin>, attr,
                                int(kTopkRegRows * sizeof(TopkRegSmem))) == cudaSuccess;
}

// One launch of the top-k for rows of N keys: the staged-row kernel for rows of up to 8192 keys
// at k <= 1024; two rows per CTA up to 65536 keys at k <= 512 and up to 32768 keys at larger k;
// one row per CTA beyond.  At most one CTA per SM, each walking rows (the rows in flight stay
// resident in L2 for the select's re-reads).  Two rows per SM overlap one row's selection with
// the other's reads; for longer rows one row per SM wins, as 1024 rows of 131072 keys fill
// 304 row slots unevenly and a wider k crowds the shared per-two-warp histograms.
template <bool kWin>
void topk_launch(const TopkParams& p, int64_t M, int64_t N, int32_t k, int sm_count, cudaStream_t s)
{
    const int64_t pair_grid = (M + 1) / 2 < sm_count ? (M + 1) / 2 : sm_count;
    if (N <= kTopkRegKeys && k <= kTopkRegMaxK) {
        const int64_t rows = (M + kTopkRegRows - 1) / kTopkRegRows;
        const int64_t grid = rows < sm_count ? rows : sm_count;
        topk_reg_kernel<kWin><<<dim3(uint32_t(grid)), kTopkThreads,
                                kTopkRegRows * sizeof(TopkRegSmem), s>>>(p);
    } else if (N <= 65536 && k <= 512) {
        // rows over 32768 keys sample into the finer histogram: a tighter threshold, fewer kept
        if (N > 32768)
            topk_kernel<TopkSmemPair, kWin, 12><<<dim3(uint32_t(pair_grid)), kTopkThreads,
                                                  2 * sizeof(TopkSmemPair), s>>>(p);
        else
            topk_kernel<TopkSmemPair, kWin, 11><<<dim3(uint32_t(pair_grid)), kTopkThreads,
                                                  2 * sizeof(TopkSmemPair), s>>>(p);
    } else if (N <= 32768) {
        // the finer sample histogram pays at k > 1024 once rows are longer than 8192 keys
        if (k > 1024 && N > 8192)
            topk_kernel<TopkSmemPairWide, kWin, 12><<<dim3(uint32_t(pair_grid)), kTopkThreads,
                                                      2 * sizeof(TopkSmemPairWide), s>>>(p);
        else
            topk_kernel<TopkSmemPairWide, kWin, 11><<<dim3(uint32_t(pair_grid)), kTopkThreads,
                                                      2 * sizeof(TopkSmemPairWide), s>>>(p);
    } else {
        const int64_t grid = M < sm_count ? M : sm_count;
        topk_kernel<TopkSmemOne, kWin, 12><<<dim3(uint32_t(grid)), kTopkThreads,
                                             sizeof(TopkSmemOne), s>>>(p);
    }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// One-time per-device setup: architecture check, kernel attributes, library buffers.
void init_device(int dev, DeviceState& st)
{
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        st.init_status = FP8MQA_ERR_CUDA;
        return;
    }
    if (major != 10 || minor != 3) {
        st.init_status = FP8MQA_ERR_ARCH;
        return;
    }
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, fp8_mqa_logits_kernel) != cudaSuccess) {
        st.init_status = FP8MQA_ERR_LAUNCH;
        return;
    }
    // setmaxnreg redistributes exactly the launch allocation; any other register count
    // would make the epilogue's request unsatisfiable, so refuse to launch.
    if (uint32_t(fa.numRegs) != kLaunchRegs) {
        st.init_status = FP8MQA_ERR_LAUNCH;
        return;
    }
    if (cudaFuncSetAttribute(fp8_mqa_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSmemBytes)) != cudaSuccess ||
        !topk_set_smem<false>() || !topk_set_smem<true>()) {
        st.init_status = FP8MQA_ERR_LAUNCH;
        return;
    }
    void* buf = nullptr;
    const size_t bytes = size_t(kSchedSlots + kGraphSlots) * sizeof(SchedSlot) + kStatusBytes;
    if (cudaMalloc(&buf, bytes) != cudaSuccess) {
        st.init_status = FP8MQA_ERR_CUDA;
        return;
    }
    if (cudaMemset(buf, 0, bytes) != cudaSuccess) {
        cudaFree(buf);
        st.init_status = FP8MQA_ERR_CUDA;
        return;
    }
    st.sched = static_cast<SchedSlot*>(buf);
    st.status = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(buf) +
                                           size_t(kSchedSlots + kGraphSlots) * sizeof(SchedSlot));
    std::call_once(g_encode_once, load_encode);
    if (!g_encode) {
        st.init_status = FP8MQA_ERR_CUDA;
        return;
    }
    st.ready.store(true, std::memory_order_release);
}

DeviceState* device_state(int* err)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        *err = FP8MQA_ERR_CUDA;
        return nullptr;
    }
    DeviceState& st = g_dev[dev];
    std::call_once(st.once, init_device, dev, std::ref(st));
    if (st.init_status != FP8MQA_OK) {
        *err = st.init_status;
        return nullptr;
    }
    *err = FP8MQA_OK;
    return &st;
}

bool encode(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base,
            const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
            CUtensorMapSwizzle swizzle)
{
    const cuuint32_t elem_strides[2] = {1, 1};
    return g_encode(map, dtype, rank, const_cast<void*>(base), dims, strides, box, elem_strides,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int check_args(const uint8_t* q, const uint8_t* k, const float* kv, const float* w,
               const int32_t* ks, const int32_t* ke, const float* out, int64_t M, int64_t N,
               int32_t H, int32_t D, int32_t clean, int32_t split_n)
{
    if (M < 0 || N < 0 || split_n < 0 || (clean != 0 && clean != 1))
        return FP8MQA_ERR_INVALID_ARG;
    if (!fp8_mqa_logits_is_supported(M, N, H, D, -1)) return FP8MQA_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || N == 0) return FP8MQA_OK;
    if (!q || !k || !kv || !w || !ks || !ke || !out) return FP8MQA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(kv, 16) || !aligned(w, 16) ||
        !aligned(ks, 4) || !aligned(ke, 4) || !aligned(out, 4))
        return FP8MQA_ERR_MISALIGNED;
    return FP8MQA_OK;
}

// Builds the tensor maps and parameters and launches the persistent kernel.  `sched` and
// `status` are the caller's scratch; with `clear_sched` the scheduler counters are zeroed
// on `stream` first.
int enqueue(SchedSlot* sched, int32_t* status, int sm_count, bool clear_sched,
            const uint8_t* q, const uint8_t* k, const float* kv, const float* w,
            const int32_t* ks, const int32_t* ke, float* out, int64_t M, int64_t N,
            int32_t clean, int32_t split_n, cudaStream_t stream)
{
    const int32_t num_tiles = int32_t((N + kTileKeys - 1) / kTileKeys);
    int32_t split = split_n > 0 ? split_n : fp8_mqa_logits_default_split(M, N, sm_count);
    if (split > num_tiles) split = num_tiles;
    if (split < 1) split = 1;
    const int32_t tpc = (num_tiles + split - 1) / split;
    split = (num_tiles + tpc - 1) / tpc;  // drop chunks that would be empty
    const int64_t num_blocks = (M + kRows - 1) / kRows;
    const int64_t num_units = num_blocks * split;
    if (num_units > INT32_MAX) return FP8MQA_ERR_UNSUPPORTED_SHAPE;

    CUtensorMap tm_q, tm_k, tm_w;
    {
        const cuuint64_t dims[2] = {cuuint64_t(kDim), cuuint64_t(M) * kHeads};
        const cuuint64_t strides[1] = {cuuint64_t(kDim)};
        const cuuint32_t box[2] = {kDim, kUmmaN};
        if (!encode(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, q, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
            return FP8MQA_ERR_LAUNCH;
    }
    {
        const cuuint64_t dims[2] = {cuuint64_t(kDim), cuuint64_t(N)};
        const cuuint64_t strides[1] = {cuuint64_t(kDim)};
        const cuuint32_t box[2] = {kDim, kTileKeys};
        if (!encode(&tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, k, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
            return FP8MQA_ERR_LAUNCH;
    }
    {
        const cuuint64_t dims[2] = {cuuint64_t(kHeads), cuuint64_t(M)};
        const cuuint64_t strides[1] = {cuuint64_t(kHeads) * 4};
        const cuuint32_t box[2] = {kHeads, kRows};
        if (!encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, w, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
            return FP8MQA_ERR_LAUNCH;
    }
    Params p;
    p.kv_scale = kv;
    p.ks = ks;
    p.ke = ke;
    p.out = out;
    p.M = M;
    p.N = N;
    p.num_tiles = num_tiles;
    p.tiles_per_chunk = tpc;
    p.split = split;
    p.num_blocks = int32_t(num_blocks);
    p.num_units = int32_t(num_units);
    p.clean = clean;
    p.sched = sched;
    p.status = status;
    p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    p.drain_ns = kDrainNs;
    p.suspend_ns = p.wait_ns < kHintedWaitNs ? uint32_t(p.wait_ns > 32 ? p.wait_ns : 32) : 0u;

    if (clear_sched && cudaMemsetAsync(sched, 0, sizeof(SchedSlot), stream) != cudaSuccess)
        return FP8MQA_ERR_CUDA;
    const int64_t grid = num_units < sm_count ? num_units : sm_count;
    fp8_mqa_logits_kernel<<<unsigned(grid), kThreads, kSmemBytes, stream>>>(tm_q, tm_k, tm_w, p);
    if (cudaGetLastError() != cudaSuccess) return FP8MQA_ERR_LAUNCH;
    return FP8MQA_OK;
}

int launch(const uint8_t* q, const uint8_t* k, const float* kv, const float* w,
           const int32_t* ks, const int32_t* ke, float* out, int64_t M, int64_t N,
           int32_t clean, int32_t split_n, cudaStream_t stream)
{
    int err = FP8MQA_OK;
    DeviceState* st = device_state(&err);
    if (!st) return err;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        cudaGetLastError();
        return FP8MQA_ERR_CUDA;
    }
    SchedSlot* slot;
    if (cap == cudaStreamCaptureStatusNone) {
        slot = st->sched + (st->seq.fetch_add(1, std::memory_order_relaxed) % kSchedSlots);
    } else {
        // a captured launch keeps its slot for every replay of the graph: give it one that
        // no other launch uses
        const uint32_t i = st->graph_seq.fetch_add(1, std::memory_order_relaxed);
        if (i >= kGraphSlots) return FP8MQA_ERR_CAPACITY;
        slot = st->sched + kSchedSlots + i;
    }
    return enqueue(slot, st->status, st->sm_count, false, q, k, kv, w, ks, ke, out, M, N, clean,
                   split_n, stream);
}

uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

// ---------------------------------------------------------------------------------------
// Host-buffer entry (fp8_mqa_logits_host): the rows go in chunks, so that the copies in
// both directions and the kernels overlap.  Inputs travel on one library stream, the
// chunks' kernels run on the caller's stream, and each chunk's logits go back on a second
// library stream as soon as its kernel is done.  Events fork the two streams from the
// caller's stream at the start of a call and join them back at its end.
constexpr int kHostChunksMax = 8;
constexpr uint64_t kHostChunkBytes = uint64_t(32) << 20;  // logits per chunk, about

struct HostPipe {
    std::mutex mu;  // one call enqueues at a time per device
    bool ready = false;
    int init_status = FP8MQA_OK;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t in_ev[kHostChunksMax] = {}, k_ev[kHostChunksMax] = {};
};

HostPipe g_pipe[kMaxDevices];

// Creates the pipeline's streams and events on first use (under the device's lock); they
// live until the process exits.
int host_pipe_init(HostPipe& hp)
{
    if (hp.ready) return hp.init_status;
    hp.ready = true;
    const unsigned ev_flags = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.start, ev_flags) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.done, ev_flags) == cudaSuccess;
    for (int c = 0; ok && c < kHostChunksMax; ++c)
        ok = cudaEventCreateWithFlags(&hp.in_ev[c], ev_flags) == cudaSuccess &&
             cudaEventCreateWithFlags(&hp.k_ev[c], ev_flags) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        hp.init_status = FP8MQA_ERR_CUDA;
    }
    return hp.init_status;
}

// ---------------------------------------------------------------------------------------
// Allocation-free variant (fp8_mqa_logits_noalloc).  Its scratch -- the scheduler's work
// counters and a status word -- lives in the file-scope array below instead of memory
// from cudaMalloc.  Host code may not pass the array's name to a kernel (on the host it
// is only a stand-in for the symbol), so set-up looks up its device address once per
// device with cudaGetSymbolAddress, with that device current.
constexpr size_t kNoAllocScratchBytes = 256;  // the array's fixed size
constexpr size_t kNoAllocStatusOffset = 128;  // status word after the scheduler slot

struct NoAllocState {
    std::once_flag once;
    int init_status = FP8MQA_OK;
    std::atomic<bool> ready{false};
    int sm_count = 0;
    uint8_t* scratch = nullptr;  // device address of no_alloc_scratch on this device
};

NoAllocState g_noalloc[kMaxDevices];

}  // namespace
}  // namespace fp8mqa

static __device__ __align__(256) uint8_t no_alloc_scratch[fp8mqa::kNoAllocScratchBytes];

namespace fp8mqa {
namespace {

// Bytes of the array one call uses: a scheduler slot, the status word and its bounds record.
// The need does not grow with M or N; the check below guards the layout against the array size.
constexpr size_t kNoAllocNeed = kNoAllocStatusOffset + 16;
static_assert(sizeof(SchedSlot) <= kNoAllocStatusOffset, "scratch layout");
static_assert(kNoAllocNeed <= kNoAllocScratchBytes, "scratch array too small");

void init_noalloc(int dev, NoAllocState& st)
{
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        st.init_status = FP8MQA_ERR_CUDA;
        return;
    }
    if (major != 10 || minor != 3) {
        st.init_status = FP8MQA_ERR_ARCH;
        return;
    }
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, fp8_mqa_logits_kernel) != cudaSuccess ||
        uint32_t(fa.numRegs) != kLaunchRegs ||
        cudaFuncSetAttribute(fp8_mqa_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSmemBytes)) != cudaSuccess) {
        st.init_status = FP8MQA_ERR_LAUNCH;
        return;
    }
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, no_alloc_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        st.init_status = FP8MQA_ERR_CUDA;
        return;
    }
    st.scratch = static_cast<uint8_t*>(ptr);
    std::call_once(g_encode_once, load_encode);
    if (!g_encode) {
        st.init_status = FP8MQA_ERR_CUDA;
        return;
    }
    st.ready.store(true, std::memory_order_release);
}

// Reads and clears a status word and its bounds record (16 bytes of device memory) after
// the caller has synchronized; ORs the flags into *flags.  A bounds record (written only by
// the bounds-checking build) is also reported on stderr.  Allocates nothing.
bool take_status(int32_t* dev_status, int32_t* flags)
{
    uint32_t word[4] = {0, 0, 0, 0};
    if (cudaMemcpy(word, dev_status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return false;
    if (word[0] != 0 || word[2] != 0 || word[3] != 0) {
        const uint64_t rec = uint64_t(word[2]) | (uint64_t(word[3]) << 32);
        if (rec != 0)
            std::fprintf(stderr,
                         "fp8mqa: bounds violation recorded: kind %u, index %lld "
                         "(kinds: 1 store, 2 kv_scale, 3 -inf span, 4 K tile, 5 Q block, "
                         "6 window row, 7 TMEM column)\n",
                         unsigned(rec >> 48), static_cast<long long>(rec & 0xFFFFFFFFFFFFull));
        const int32_t zero[4] = {0, 0, 0, 0};
        if (cudaMemcpy(dev_status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return false;
    }
    *flags |= int32_t(word[0]);
    return true;
}

int launch_noalloc(const uint8_t* q, const uint8_t* k, const float* kv, const float* w,
                   const int32_t* ks, const int32_t* ke, float* out, int64_t M, int64_t N,
                   int32_t clean, int32_t split_n, cudaStream_t stream)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return FP8MQA_ERR_CUDA;
    }
    NoAllocState& st = g_noalloc[dev];
    std::call_once(st.once, init_noalloc, dev, std::ref(st));
    if (st.init_status != FP8MQA_OK) return st.init_status;
    if (kNoAllocNeed > kNoAllocScratchBytes) return FP8MQA_ERR_UNSUPPORTED_SHAPE;
    // The work counters must start at zero; the array keeps whatever the last call left.
    return enqueue(reinterpret_cast<SchedSlot*>(st.scratch),
                   reinterpret_cast<int32_t*>(st.scratch + kNoAllocStatusOffset), st.sm_count,
                   true, q, k, kv, w, ks, ke, out, M, N, clean, split_n, stream);
}

}  // namespace
}  // namespace fp8mqa

extern "C" {

int fp8_mqa_logits_is_supported(int64_t M, int64_t N, int32_t H, int32_t D, int32_t device)
{
    if (H != fp8mqa::kHeads || D != fp8mqa::kDim) return 0;
    if (M < 0 || N < 0) return 0;
    if (M * int64_t(H) >= (int64_t(1) << 31)) return 0;
    if (N >= (int64_t(1) << 31)) return 0;
    if (device >= 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) !=
                cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        if (major != 10 || minor != 3) return 0;
    }
    return 1;
}

int fp8_mqa_logits_default_split(int64_t M, int64_t N, int32_t num_sms)
{
    // Larger problems (below): enough units for the dynamic scheduler to balance the tail,
    // and no more, since every unit costs a claim, a Q load and a pipeline restart.  About 4
    // units per SM when there are four or more row blocks per SM (heaviest-first order then
    // balances whole blocks), 20 with two to four blocks per SM, and 16 under two (every
    // block is then split into many chunks of equal work and the last chunks decide the
    // finish).  Chunks keep at least 8 key tiles; the kernel splits a block with narrow
    // windows along its own tile range.
    if (M <= 0 || N <= 0) return 1;
    if (num_sms < 1) num_sms = 1;
    const int64_t tiles = (N + fp8mqa::kTileKeys - 1) / fp8mqa::kTileKeys;
    const int64_t blocks = (M + fp8mqa::kRows - 1) / fp8mqa::kRows;
    const int64_t sms = num_sms;
    if (blocks * tiles <= 128 * sms) {
        // Small problems (128 key tiles per SM or fewer): launch and set-up weigh, so take
        // the split with the least estimated time.  Units run in rounds of one per SM, and
        // a unit costs its tiles plus a fixed set-up of about 3.3 tiles (its claim, Q load
        // and pipeline fill: about 2 us against about 0.6 us per tile, measured on GB300).
        constexpr double kUnitSetupTiles = 3.3;
        const int64_t s_max = std::min<int64_t>(tiles, 4 * sms / blocks + 1);
        int64_t best = 1;
        double best_cost = 0;
        for (int64_t s = 1; s <= s_max; ++s) {
            const int64_t tpc = (tiles + s - 1) / s;
            const int64_t units = blocks * ((tiles + tpc - 1) / tpc);
            const double cost = double((units + sms - 1) / sms) * (kUnitSetupTiles + double(tpc));
            if (s == 1 || cost < best_cost) {
                best = s;
                best_cost = cost;
            }
        }
        return int(best);
    }
    const int64_t per_sm = blocks < 2 * sms ? 16 : (blocks < 4 * sms ? 20 : 4);
    const int64_t target = per_sm * sms;
    int64_t s = (target + blocks - 1) / blocks;
    const int64_t cap = tiles / 8 > 1 ? tiles / 8 : 1;
    if (s > cap) s = cap;
    if (s < 1) s = 1;
    return int(s);
}

int fp8_mqa_logits(const uint8_t* q_fp8, const uint8_t* k_fp8, const float* kv_scale,
                   const float* w, const int32_t* ks, const int32_t* ke, float* out, int64_t M,
                   int64_t N, int32_t H, int32_t D, int32_t clean_logits, int32_t split_n,
                   void* stream)
{
    const int rc =
        fp8mqa::check_args(q_fp8, k_fp8, kv_scale, w, ks, ke, out, M, N, H, D, clean_logits,
                           split_n);
    if (rc != FP8MQA_OK || M == 0 || N == 0) return rc;
    return fp8mqa::launch(q_fp8, k_fp8, kv_scale, w, ks, ke, out, M, N, clean_logits, split_n,
                          static_cast<cudaStream_t>(stream));
}

int fp8_mqa_logits_check_error(void* stream)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= fp8mqa::kMaxDevices) {
        cudaGetLastError();
        return FP8MQA_ERR_CUDA;
    }
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return FP8MQA_ERR_CUDA;
    }
    // Only state that earlier calls set up is read: this call allocates nothing.
    int32_t flags = 0;
    fp8mqa::DeviceState& st = fp8mqa::g_dev[dev];
    if (st.ready.load(std::memory_order_acquire) && !fp8mqa::take_status(st.status, &flags))
        return FP8MQA_ERR_CUDA;
    fp8mqa::NoAllocState& na = fp8mqa::g_noalloc[dev];
    if (na.ready.load(std::memory_order_acquire) &&
        !fp8mqa::take_status(reinterpret_cast<int32_t*>(na.scratch + fp8mqa::kNoAllocStatusOffset),
                             &flags))
        return FP8MQA_ERR_CUDA;
    if (flags & fp8mqa::kStatusBounds) return FP8MQA_ERR_BOUNDS;
    if (flags & fp8mqa::kStatusTimeout) return FP8MQA_ERR_TIMEOUT;
    return FP8MQA_OK;
}

uint64_t fp8_mqa_logits_set_wait_limit_ns(uint64_t ns)
{
    return fp8mqa::g_wait_ns.exchange(ns ? ns : fp8mqa::kDefaultWaitNs);
}

uint64_t fp8_mqa_logits_host_workspace_bytes(int64_t M, int64_t N, int32_t H, int32_t D)
{
    if (!fp8_mqa_logits_is_supported(M, N, H, D, -1)) return 0;
    using fp8mqa::align256;
    const uint64_t m = uint64_t(M), n = uint64_t(N);
    return align256(m * H * D) + align256(n * D) + align256(n * 4) + align256(m * H * 4) +
           align256(m * 4) * 2 + align256(m * n * 4);
}

int fp8_mqa_logits_host(const uint8_t* q_fp8, const uint8_t* k_fp8, const float* kv_scale,
                        const float* w, const int32_t* ks, const int32_t* ke, float* out,
                        int64_t M, int64_t N, int32_t H, int32_t D, int32_t clean_logits,
                        int32_t split_n, void* workspace, uint64_t workspace_bytes,
                        void* stream)
{
    int rc = fp8mqa::check_args(q_fp8, k_fp8, kv_scale, w, ks, ke, out, M, N, H, D,
                                clean_logits, split_n);
    if (rc != FP8MQA_OK || M == 0 || N == 0) return rc;
    if (!workspace) return FP8MQA_ERR_INVALID_ARG;
    if (!fp8mqa::aligned(workspace, 256)) return FP8MQA_ERR_MISALIGNED;
    if (workspace_bytes < fp8_mqa_logits_host_workspace_bytes(M, N, H, D))
        return FP8MQA_ERR_INVALID_ARG;
    using fp8mqa::align256;
    const uint64_t m = uint64_t(M), n = uint64_t(N);
    uint8_t* base = static_cast<uint8_t*>(workspace);
    uint8_t* dq = base;
    uint8_t* dk = dq + align256(m * H * D);
    float* dkv = reinterpret_cast<float*>(dk + align256(n * D));
    float* dw = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(dkv) + align256(n * 4));
    int32_t* dks = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(dw) + align256(m * H * 4));
    int32_t* dke = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(dks) + align256(m * 4));
    float* dout = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(dke) + align256(m * 4));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= fp8mqa::kMaxDevices) {
        cudaGetLastError();
        return FP8MQA_ERR_CUDA;
    }
    int err = FP8MQA_OK;
    if (!fp8mqa::device_state(&err)) return err;
    fp8mqa::HostPipe& hp = fp8mqa::g_pipe[dev];
    std::lock_guard<std::mutex> lock(hp.mu);
    rc = fp8mqa::host_pipe_init(hp);
    if (rc != FP8MQA_OK) return rc;

    // chunks of whole 8-row blocks, about kHostChunkBytes of logits each
    int64_t chunks = int64_t((m * n * 4) / fp8mqa::kHostChunkBytes);
    chunks = std::max<int64_t>(1, std::min<int64_t>(chunks, fp8mqa::kHostChunksMax));
    int64_t rows = (M + chunks - 1) / chunks;
    rows = (rows + fp8mqa::kRows - 1) / fp8mqa::kRows * fp8mqa::kRows;
    chunks = (M + rows - 1) / rows;

    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
    bool ok = cudaEventRecord(hp.start, s) == cudaSuccess &&
              cudaStreamWaitEvent(hp.in, hp.start, 0) == cudaSuccess &&
              cudaStreamWaitEvent(hp.out, hp.start, 0) == cudaSuccess &&
              cudaMemcpyAsync(dk, k_fp8, n * D, h2d, hp.in) == cudaSuccess &&
              cudaMemcpyAsync(dkv, kv_scale, n * 4, h2d, hp.in) == cudaSuccess;
    for (int64_t c = 0; ok && c < chunks; ++c) {
        const uint64_t r0 = uint64_t(c * rows), mr = uint64_t(std::min<int64_t>(rows, M - c * rows));
        ok = cudaMemcpyAsync(dq + r0 * H * D, q_fp8 + r0 * H * D, mr * H * D, h2d, hp.in) == cudaSuccess &&
             cudaMemcpyAsync(dw + r0 * H, w + r0 * H, mr * H * 4, h2d, hp.in) == cudaSuccess &&
             cudaMemcpyAsync(dks + r0, ks + r0, mr * 4, h2d, hp.in) == cudaSuccess &&
             cudaMemcpyAsync(dke + r0, ke + r0, mr * 4, h2d, hp.in) == cudaSuccess &&
             (clean_logits ||
              cudaMemcpyAsync(dout + r0 * n, out + r0 * n, mr * n * 4, h2d, hp.in) == cudaSuccess) &&
             cudaEventRecord(hp.in_ev[c], hp.in) == cudaSuccess &&
             cudaStreamWaitEvent(s, hp.in_ev[c], 0) == cudaSuccess;
        if (!ok) break;
        rc = fp8mqa::launch(dq + r0 * H * D, dk, dkv, dw + r0 * H, dks + r0, dke + r0, dout + r0 * n,
                            int64_t(mr), N, clean_logits, split_n, s);
        if (rc != FP8MQA_OK) break;
        ok = cudaEventRecord(hp.k_ev[c], s) == cudaSuccess &&
             cudaStreamWaitEvent(hp.out, hp.k_ev[c], 0) == cudaSuccess &&
             cudaMemcpyAsync(out + r0 * n, dout + r0 * n, mr * n * 4, d2h, hp.out) == cudaSuccess;
    }
    // join: later work on the caller's stream sees every copy of this call
    const bool joined = cudaEventRecord(hp.done, hp.out) == cudaSuccess &&
                        cudaStreamWaitEvent(s, hp.done, 0) == cudaSuccess;
    if (rc != FP8MQA_OK) return rc;
    if (!ok || !joined) {
        cudaGetLastError();
        return FP8MQA_ERR_CUDA;
    }
    return FP8MQA_OK;
}

int fp8_mqa_logits_noalloc(const uint8_t* q_fp8, const uint8_t* k_fp8, const float* kv_scale,
                           const float* w, const int32_t* ks, const int32_t* ke, float* out,
                           int64_t M, int64_t N, int32_t H, int32_t D, int32_t clean_logits,
                           int32_t split_n, void* stream)
{
    const int rc = fp8mqa::check_args(q_fp8, k_fp8, kv_scale, w, ks, ke, out, M, N, H, D,
                                      clean_logits, split_n);
    if (rc != FP8MQA_OK || M == 0 || N == 0) return rc;
    return fp8mqa::launch_noalloc(q_fp8, k_fp8, kv_scale, w, ks, ke, out, M, N, clean_logits,
                                  split_n, static_cast<cudaStream_t>(stream));
}

int fp8_mqa_topk(const float* logits, int64_t M, int64_t N, int64_t ld, int32_t k,
                 int32_t* indices, float* values, void* stream)
{
    return fp8_mqa_topk_windowed(logits, M, N, ld, nullptr, nullptr, k, indices, values, stream);
}

int fp8_mqa_topk_windowed(const float* logits, int64_t M, int64_t N, int64_t ld,
                          const int32_t* ks, const int32_t* ke, int32_t k, int32_t* indices,
                          float* values, void* stream)
{
    return fp8_mqa_topk_ex(logits, M, N, ld, ks, ke, k, 0, indices, values, stream);
}

int fp8_mqa_topk_ex(const float* logits, int64_t M, int64_t N, int64_t ld, const int32_t* ks,
                    const int32_t* ke, int32_t k, int32_t flags, int32_t* indices, float* values,
                    void* stream)
{
    if (M < 0 || N < 0 || ld < N || k < 1 || k > fp8mqa::kTopkMaxK) return FP8MQA_ERR_INVALID_ARG;
    if ((flags & ~int32_t(FP8MQA_TOPK_UNSORTED)) != 0) return FP8MQA_ERR_INVALID_ARG;
    if (N > (int64_t(1) << 30)) return FP8MQA_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return FP8MQA_OK;
    if (!indices || (N > 0 && !logits) || (ks == nullptr) != (ke == nullptr))
        return FP8MQA_ERR_INVALID_ARG;
    if (!fp8mqa::aligned(logits, 4) || !fp8mqa::aligned(indices, 4) ||
        (values && !fp8mqa::aligned(values, 4)) || (ks && !fp8mqa::aligned(ks, 4)) ||
        (ke && !fp8mqa::aligned(ke, 4)))
        return FP8MQA_ERR_MISALIGNED;
    int err = FP8MQA_OK;
    fp8mqa::DeviceState* st = fp8mqa::device_state(&err);
    if (!st) return err;
    fp8mqa::TopkParams p;
    p.logits = logits;
    p.M = M;
    p.N = N;
    p.ld = ld;
    p.k = k;
    p.indices = indices;
    p.values = values;
    p.ks = ks;
    p.ke = ke;
    p.sorted = (flags & FP8MQA_TOPK_UNSORTED) ? 0 : 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (ks)
        fp8mqa::topk_launch<true>(p, M, N, k, st->sm_count, s);
    else
        fp8mqa::topk_launch<false>(p, M, N, k, st->sm_count, s);
    if (cudaGetLastError() != cudaSuccess) return FP8MQA_ERR_LAUNCH;
    return FP8MQA_OK;
}

const char* fp8_mqa_logits_strerror(int status)
{
    switch (status) {
        case FP8MQA_OK: return "FP8MQA_OK";
        case FP8MQA_ERR_INVALID_ARG: return "FP8MQA_ERR_INVALID_ARG: invalid argument";
        case FP8MQA_ERR_UNSUPPORTED_SHAPE:
            return "FP8MQA_ERR_UNSUPPORTED_SHAPE: needs H=32, D=128 and sizes within limits";
        case FP8MQA_ERR_MISALIGNED: return "FP8MQA_ERR_MISALIGNED: pointer alignment";
        case FP8MQA_ERR_ARCH: return "FP8MQA_ERR_ARCH: device is not compute capability 10.3";
        case FP8MQA_ERR_LAUNCH: return "FP8MQA_ERR_LAUNCH: kernel configuration or launch failed";
        case FP8MQA_ERR_TIMEOUT: return "FP8MQA_ERR_TIMEOUT: a bounded device wait gave up";
        case FP8MQA_ERR_CUDA: return "FP8MQA_ERR_CUDA: CUDA runtime error";
        case FP8MQA_ERR_BOUNDS:
            return "FP8MQA_ERR_BOUNDS: a bounds-checking build found an out-of-range access";
        case FP8MQA_ERR_CAPACITY:
            return "FP8MQA_ERR_CAPACITY: no scheduler slot left for another captured launch";
        default: return "FP8MQA: unknown status";
    }
}

}  // extern "C"
