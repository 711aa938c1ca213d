// The prefill FP8 MQA indexer-logits kernel for GB300 (sm_103a).
//
//   out[m, n] = kv_scale[n] * sum_h relu(Q[m,h,:] . K[n,:]) * w[m,h],  n in [ks[m], ke[m])
//
// (ROCm/aiter PR #7183 "[HIP] [JIT] Add gfx950 prefill FP8 MQA logits", "Motivation".)
//
// Work unit = (row block of kRows = 8 query rows, key chunk).  A persistent grid of one
// CTA per SM pulls units from a global counter, heaviest row blocks first (the page's
// "reverse_rows", section "Design / Grid choice"); key chunks are the page's SplitN.  A
// block whose windows cover under half of the keys is chunked along its own tile range
// instead (the page's layout-aware split for multi-request chunks, "Known limitations").
//
// Warp roles in a 640-thread CTA:
//   warp 0      producer: claims units, computes each unit's key-tile range from the
//               window union of its rows, and streams Q+w (once per unit) and K tiles
//               (once per unit) into shared memory with TMA (page: "K is read once per 32
//               rows", section "Design").
//   warps 1, 3  MMA issuers (warp 1 also owns TMEM): per 128-key tile, 4 tcgen05.mma (K = 32
//               each) of A = K tile [128 keys x 128] by B = Q block [8 rows x 32 heads =
//               256 x 128], accumulating S[key, (row, head)] in fp32 in TMEM; warp 1 issues
//               the even tiles into buffer 0, warp 3 the odd tiles into buffer 1.
//   warp 2      -inf writer (clean_logits = 1): fills every out-of-window span outside the
//               computed tile range, on its own light-first unit order so the writes
//               overlap the compute-heavy units (page: "With clean_logits the kernel writes
//               -inf itself").  The spans go out as bulk copies from a shared-memory -inf
//               buffer, so the TMA engine, not the issue slots the epilogue needs, does them.
//   warps 4-19  epilogue, four warps per SM sub-partition, two query rows per warp:
//               thread = one key (TMEM lane), so one tcgen05.ld gives it the 64 values
//               (row, head) of its two rows; relu, times w, head sum in registers (no
//               cross-lane reduction), times kv_scale once per (m, n), then a coalesced
//               store.  Tiles inside both rows' windows store without compare/select;
//               boundary tiles are masked (page: "clean stages" vs "masked boundary
//               stages").  kv_scale comes through the read-only path, one tile ahead.
//
// Keys sit on the MMA M axis (TMEM lanes) and (row, head) on the N axis: this transposes
// the page's layout (query heads on the matrix rows) so that the head reduction is a sum
// inside one thread instead of a cross-lane permutation.
//
// Every mbarrier wait is bounded (globaltimer, Params::wait_ns): on expiry the CTA raises a
// shared abort flag and a global status bit, drains its in-flight TMA, MMA and bulk copies
// (bounded separately by Params::drain_ns), frees TMEM and returns.
//
// Built with FP8MQA_DEBUG_BOUNDS, every global access and TMA coordinate is checked first;
// a violation is recorded in the status word and the access skipped.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "sm103_ptx.cuh"

namespace fp8mqa {

constexpr int kHeads = 32;
constexpr int kDim = 128;
constexpr int kRows = 8;                  // query rows per unit: kRows x 32 heads is the MMA N
constexpr int kTileKeys = 128;            // keys per tile (MMA M)
constexpr int kUmmaN = kRows * kHeads;    // 256 (MMA N)
constexpr int kUmmaK = 32;                // FP8 K per tcgen05.mma
constexpr int kStages = 6;                // K ring depth
constexpr int kQSlots = 3;
constexpr int kUnitSlots = 4;
constexpr int kClaimAhead = 4;           // K tiles of a unit left to issue when the next is claimed
constexpr int kAccBufs = 2;
constexpr uint32_t kAccStride = 256;      // TMEM columns between accumulator buffers
constexpr uint32_t kTmemCols = kAccBufs * kAccStride;  // 512 (a power of two)
constexpr int kRowsPerEpiWarp = 2;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = kRows * 4 / kRowsPerEpiWarp;  // 16: four TMEM sub-partitions
constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;  // 640
constexpr int kMmaWarp0 = 1;              // issues the even tiles (accumulator buffer 0)
constexpr int kMmaWarp1 = 3;              // issues the odd tiles (accumulator buffer 1)
constexpr int kFillWarp = 2;

constexpr uint32_t kQBytes = kRows * kHeads * kDim;   // 32768
constexpr uint32_t kWBytes = kRows * kHeads * 4;      // 1024
constexpr uint32_t kKBytes = kTileKeys * kDim;        // 16384
constexpr uint32_t kFillBytes = 16384;                // -inf source for bulk stores

// Shared-memory layout, offsets from a 1024-byte aligned base.
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQSlots * kQBytes;
constexpr uint32_t kOffW = kOffK + kStages * kKBytes;
constexpr uint32_t kOffFill = kOffW + kQSlots * kWBytes;
constexpr uint32_t kOffBar = kOffFill + kFillBytes;

constexpr int kBarKFull = 0;
constexpr int kBarKEmpty = kBarKFull + kStages;
constexpr int kBarQFull = kBarKEmpty + kStages;
constexpr int kBarQEmpty = kBarQFull + kQSlots;
constexpr int kBarAccFull = kBarQEmpty + kQSlots;
constexpr int kBarAccEmpty = kBarAccFull + kAccBufs;
constexpr int kBarUnitFull = kBarAccEmpty + kAccBufs;
constexpr int kBarUnitEmpty = kBarUnitFull + kUnitSlots;
constexpr int kBarDrain = kBarUnitEmpty + kUnitSlots;
constexpr int kNumBars = kBarDrain + 1;

struct UnitInfo {
    int32_t m0;      // first query row
    int32_t t0, t1;  // key tiles [t0, t1) computed by MMA + epilogue
    int32_t flags;   // kUnitTerminate
    int32_t lo[kRows], hi[kRows];  // each row's window clamped to [0, N); rows past M: empty
};
constexpr int32_t kUnitTerminate = 1;

constexpr uint32_t kOffUnits = kOffBar + kNumBars * 8;
constexpr uint32_t kOffMisc = kOffUnits + kUnitSlots * sizeof(UnitInfo);
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for aligning the base
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kUmmaN <= int(kAccStride), "accumulator buffer width");
static_assert(kQBytes % 1024 == 0 && kWBytes % 128 == 0, "shared-memory alignment");

// Per-role register budgets (setmaxnreg): the control warpgroup gives registers to the
// epilogue warpgroups; the total must stay within the launch allocation (threads x the
// per-thread count the kernel is compiled to, which fills the register file).
constexpr uint32_t kLaunchRegs = (65536u / kThreads) & ~7u;  // 96
constexpr uint32_t kCtlRegs = 32u;
constexpr uint32_t kEpiRegs = ((kLaunchRegs * kThreads - 128u * kCtlRegs) / (kEpiWarps * 32u)) & ~7u;
static_assert(128 * kCtlRegs + kEpiWarps * 32 * kEpiRegs <= kThreads * kLaunchRegs,
              "register split");

// Status word bits (status[0]); status[2..3] hold the first bounds violation (debug builds).
constexpr int32_t kStatusTimeout = 1;
constexpr int32_t kStatusBounds = 2;

#ifdef FP8MQA_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif

// Kinds of bounds violation a debug build records.
enum BoundsKind : uint32_t {
    kBoundsStore = 1,     // epilogue logit store outside [0, M) x [0, N)
    kBoundsKvScale = 2,   // kv_scale read outside [0, N)
    kBoundsFill = 3,      // -inf span outside its row's [0, N)
    kBoundsKTile = 4,     // K tile coordinate outside [0, ceil(N / 128))
    kBoundsQBlock = 5,    // Q / w row block outside [0, M)
    kBoundsWindow = 6,    // ks / ke read outside [0, M)
    kBoundsTmem = 7,      // TMEM column outside the allocation
};

// Scheduler slot in global memory: work counters that the last CTA resets.
struct SchedSlot {
    uint32_t next_unit;
    uint32_t next_fill;
    uint32_t done_ctas;
    uint32_t pad;
};

struct Params {
    const float* kv_scale;
    const int32_t* ks;
    const int32_t* ke;
    float* out;
    int64_t M;
    int64_t N;
    int32_t num_tiles;        // ceil(N / 128)
    int32_t tiles_per_chunk;  // ceil(num_tiles / split)
    int32_t split;            // key chunks per row block
    int32_t num_blocks;       // ceil(M / 8)
    int32_t num_units;        // num_blocks * split
    int32_t clean;
    SchedSlot* sched;
    int32_t* status;          // status[0]: flags; status[2..3]: first bounds violation
    uint64_t wait_ns;         // a pipeline wait gives up (abort) after this long
    uint64_t drain_ns;        // bound of the waits for in-flight work before exit
    uint32_t suspend_ns;      // 0: waits suspend for the hardware's own time; else at most this
};

// True when the access may go ahead: always in normal builds.  In debug builds, only when
// `ok`; otherwise the first violation's (kind, index) goes to status[2..3] (the host's
// check_error reports it) and kStatusBounds is set.
__device__ __forceinline__ bool in_bounds(bool ok, int32_t* status, uint32_t kind, int64_t index)
{
    if (!kDebugBounds || ok) return true;
    const unsigned long long v =
        (static_cast<unsigned long long>(kind) << 48) |
        (static_cast<unsigned long long>(index) & 0xFFFFFFFFFFFFull);
    atomicCAS(reinterpret_cast<unsigned long long*>(status + 2), 0ull, v);
    atomicOr(status, kStatusBounds);
    return false;
}

// tcgen05 instruction descriptor: D f32, A = B = E4M3, both K-major, M = 128, N = 256.
constexpr uint32_t kIdesc = (1u << 4)                          // D format: f32
                            | (0u << 7) | (0u << 10)           // A, B format: E4M3
                            | (uint32_t(kUmmaN >> 3) << 17)    // N / 8
                            | (uint32_t(kTileKeys >> 4) << 24);  // M / 16

// Shared-memory matrix descriptor for a K-major operand whose rows are exactly 128 bytes,
// stored with the 128-byte swizzle (8-row atoms of 1024 bytes, as TMA writes them).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFF);  // start address
    d |= uint64_t(1) << 16;                // leading byte offset (unused with this swizzle)
    d |= uint64_t(1024 >> 4) << 32;        // stride byte offset: next 8-row atom
    d |= uint64_t(1) << 46;                // descriptor version
    d |= uint64_t(2) << 61;                // 128-byte swizzle
    return d;
}

template <bool B>
struct BoolTag {
    static constexpr bool value = B;
};

template <int V>
struct IntTag {
    static constexpr int value = V;
};

// What a wait needs: the CTA's abort flag (shared memory) and the kernel parameters (read
// from the constant bank only on a wait's slow path, so they hold no registers).
struct Ctl {
    volatile int32_t* abort;
    const Params& p;
};

// One poll of a wait's slow path.  By default try_wait suspends the thread in hardware until
// the phase completes or a system-dependent time passes; a short wait limit also bounds the
// suspension, so that the limit is checked in time.
__device__ __forceinline__ bool poll_bar(uint32_t bar, uint32_t parity, const Ctl& c)
{
    return c.p.suspend_ns ? ptx::mbar_try_wait_sleep(bar, parity, c.p.suspend_ns)
                          : ptx::mbar_try_wait(bar, parity);
}

__device__ __forceinline__ void raise_timeout(const Ctl& c)
{
    *c.abort = 1;
    atomicOr(c.p.status, kStatusTimeout);
}

// Bounded single-thread wait.  try_wait suspends the thread in hardware for a while when the
// phase is still open, so the loop issues few instructions.  Returns false when the CTA is
// aborting or this wait ran out (which starts the abort).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
        if (poll_bar(bar, parity, c)) return true;
        if (*c.abort) return false;
        if (ptx::globaltimer_ns() - t0 > c.p.wait_ns) {
            raise_timeout(c);
            return false;
        }
    }
}

// Bounded wait for a whole warp: lane 0 waits, then every lane observes the completed
// phase itself (immediate) so each lane has acquired the barrier's data.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const Ctl& c)
{
    const int lane = threadIdx.x & 31;
    int ok = 1;
    if (lane == 0) ok = wait_bar(bar, parity, c) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
        for (uint32_t i = 0; i < (1u << 20) && !ptx::mbar_try_wait(bar, parity); ++i) {
        }
    }
    return ok != 0;
}

// Bounded wait by every lane of a warp: all lanes poll and a warp vote decides, so the warp
// stays converged.  Returns false (for the whole warp) when the CTA is aborting or the wait
// ran out.
__device__ __forceinline__ bool wait_bar_all(uint32_t bar, uint32_t parity, const Ctl& c)
{
    if (__all_sync(0xffffffffu, ptx::mbar_try_wait(bar, parity))) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
        if (__all_sync(0xffffffffu, poll_bar(bar, parity, c))) return true;
        int stop = *c.abort ? 1 : 0;
        if ((threadIdx.x & 31) == 0 && !stop && ptx::globaltimer_ns() - t0 > c.p.wait_ns) {
            raise_timeout(c);
            stop = 1;
        }
        if (__any_sync(0xffffffffu, stop)) return false;
    }
}

// Drain: wait for a phase without looking at the abort flag (bounded by drain_ns).
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, uint64_t drain_ns)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > drain_ns) break;
    }
}

__device__ __forceinline__ int64_t clamp64(int64_t v, int64_t lo, int64_t hi)
{
    return v < lo ? lo : (v > hi ? hi : v);
}

// Unit geometry shared by the producer and the -inf writers: row block b, chunk c.
// Key tiles [t0, t1) are those of chunk c that meet the union of the block's windows.
struct Geometry {
    int32_t m0, t0, t1, ct0, ct1;
    int32_t ut0, ut1;  // key tiles meeting the union of the block's windows (empty: ut0 >= ut1)
    int32_t skip;      // compute claims: chunks of this block before `skip` hold nothing more
    int32_t lo, hi;  // lane r < kRows: row m0 + r's window clamped to [0, N) (empty past M)
};

__device__ __forceinline__ Geometry unit_geometry(const Params& p, int32_t b, int32_t c,
                                                  bool compute = false)
{
    const int lane = threadIdx.x & 31;
    Geometry g;
    g.m0 = b * kRows;
    int64_t lo = INT64_MAX, hi = INT64_MIN;
    g.lo = 0;
    g.hi = 0;
    if (lane < kRows && g.m0 + lane < p.M) {
        const int64_t m = g.m0 + lane;
        if (in_bounds(m >= 0 && m < p.M, p.status, kBoundsWindow, m)) {
            const int64_t s = clamp64(p.ks[m], 0, p.N);
            const int64_t e = clamp64(p.ke[m], 0, p.N);
            g.lo = int32_t(s);
            g.hi = int32_t(e);
            if (s < e) {
                lo = s;
                hi = e;
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const int64_t olo = __shfl_xor_sync(0xffffffffu, lo, off);
        const int64_t ohi = __shfl_xor_sync(0xffffffffu, hi, off);
        lo = olo < lo ? olo : lo;
        hi = ohi > hi ? ohi : hi;
    }
    g.ct0 = c * p.tiles_per_chunk;
    g.ct1 = min(g.ct0 + p.tiles_per_chunk, p.num_tiles);
    g.t0 = g.ct0;
    g.t1 = g.ct0;
    g.ut0 = 0;
    g.ut1 = 0;
    g.skip = p.split;  // no tiles: every chunk of the block is empty
    if (lo < hi) {
        g.ut0 = int32_t(lo / kTileKeys);
        g.ut1 = int32_t((hi + kTileKeys - 1) / kTileKeys);
        const int32_t len = g.ut1 - g.ut0;
        if (compute && 2 * len < p.num_tiles) {
            // A block whose windows cover under half of the keys (a request of a
            // multi-request chunk, say) is split along its own tile range into equal chunks
            // of at least 8 tiles, so it yields `split` units of work instead of mostly empty
            // fixed chunks.
            int32_t L = (len + p.split - 1) / p.split;
            if (L < 8) L = len < 8 ? len : 8;
            const int32_t nchunks = (len + L - 1) / L;
            g.t0 = g.ut0 + min(c, nchunks) * L;
            g.t1 = c < nchunks ? min(g.t0 + L, g.ut1) : g.t0;
            g.skip = c >= nchunks - 1 ? p.split : 0;
        } else {
            // fixed key chunks: chunk c's share of the block's tile range
            if (g.ct0 < g.ct1) {
                g.t0 = max(g.ct0, g.ut0);
                g.t1 = min(g.ct1, g.ut1);
                if (g.t1 < g.t0) g.t1 = g.t0;
            }
            const int32_t c_lo = g.ut0 / p.tiles_per_chunk;
            const int32_t c_hi = (g.ut1 - 1) / p.tiles_per_chunk;
            g.skip = c < c_lo ? c_lo : (c >= c_hi ? p.split : 0);
        }
    }
    return g;
}

// Warp-cooperative -inf fill of row[a, e): the 16-byte aligned middle goes out as bulk
// copies (TMA engine) of up to kFillBytes from the shared-memory -inf buffer at `src`, issued
// by lane 0; the ragged ends (under 4 floats each) are plain stores.
__device__ __forceinline__ void fill_neg_inf(const Params& p, int64_t m, int64_t a, int64_t e,
                                             uint32_t src)
{
    if (a >= e) return;
    if (!in_bounds(m >= 0 && m < p.M && a >= 0 && e <= p.N, p.status, kBoundsFill,
                   m * p.N + (a < 0 || a >= p.N ? a : e)))
        return;
    float* row = p.out + m * p.N;
    const int lane = threadIdx.x & 31;
    const float ninf = __int_as_float(0xff800000u);
    const uintptr_t addr = reinterpret_cast<uintptr_t>(row + a);
    int64_t a4 = a + int64_t(((16u - (addr & 15u)) & 15u) >> 2);
    if (a4 > e) a4 = e;
    const int64_t e4 = a4 + ((e - a4) & ~int64_t(3));
    if (lane < a4 - a) __stcs(row + a + lane, ninf);
    if (lane < e - e4) __stcs(row + e4 + lane, ninf);
    if (lane == 0) {
        constexpr int64_t kChunk = kFillBytes / 4;
        for (int64_t x = a4; x < e4; x += kChunk) {
            const int64_t c = e4 - x < kChunk ? e4 - x : kChunk;
            ptx::bulk_store(row + x, src, uint32_t(c) * 4u);
        }
    }
}

// Head quads (4 heads) whose relu runs on the FMA pipe instead of the ALU: for those the
// sum takes s*w + |s|*w = 2 relu(s) w, in a chain halved at the end.  Splitting the relu
// between the ALU (max, half rate) and the FMA pipe (|x| operands are free) balances the
// two pipes.  Any mask is valid; the default was chosen by measurement.
#ifndef FP8MQA_ABS_QUADS
#define FP8MQA_ABS_QUADS 0xA4u
#endif
constexpr uint32_t kAbsQuads = FP8MQA_ABS_QUADS;

__device__ __forceinline__ float2 abs2(float2 v) { return make_float2(fabsf(v.x), fabsf(v.y)); }
__device__ __forceinline__ float2 relu2(float2 v)
{
    return make_float2(fmaxf(v.x, 0.f), fmaxf(v.y, 0.f));
}
__device__ __forceinline__ float2 f2(uint32_t a, uint32_t b)
{
    return make_float2(__uint_as_float(a), __uint_as_float(b));
}

// sum_h relu(S[h]) * w[h] for two query rows: s[0..31] row a, s[32..63] row b; w of row a in
// wsm[0..7] and of row b in wsm[8..15] (shared memory, 4 heads per float4).  Two accumulator
// chains per row (ALU-relu heads and FMA-relu heads), joined once at the end.
__device__ __forceinline__ void relu_dot_2rows(const uint32_t (&s)[64], const float4* wsm,
                                               float& va, float& vb)
{
    float2 xa = make_float2(0.f, 0.f), xb = xa, ya = xa, yb = xa;  // x: ALU relu, y: FMA relu
    bool x_init = false, y_init = false;
#pragma unroll
    for (int j = 0; j < kHeads / 4; ++j) {
        const float4 u = wsm[j];
        const float4 v = wsm[kHeads / 4 + j];
        const float2 wa0 = make_float2(u.x, u.y), wa1 = make_float2(u.z, u.w);
        const float2 wb0 = make_float2(v.x, v.y), wb1 = make_float2(v.z, v.w);
        const float2 sa0 = f2(s[4 * j], s[4 * j + 1]), sa1 = f2(s[4 * j + 2], s[4 * j + 3]);
        const float2 sb0 = f2(s[32 + 4 * j], s[32 + 4 * j + 1]);
        const float2 sb1 = f2(s[32 + 4 * j + 2], s[32 + 4 * j + 3]);
        if (kAbsQuads & (1u << j)) {
            if (!y_init) {
                ya = __fmul2_rn(sa0, wa0);
                yb = __fmul2_rn(sb0, wb0);
                y_init = true;
            } else {
                ya = __ffma2_rn(sa0, wa0, ya);
                yb = __ffma2_rn(sb0, wb0, yb);
            }
            ya = __ffma2_rn(abs2(sa0), wa0, ya);
            yb = __ffma2_rn(abs2(sb0), wb0, yb);
            ya = __ffma2_rn(sa1, wa1, ya);
            yb = __ffma2_rn(sb1, wb1, yb);
            ya = __ffma2_rn(abs2(sa1), wa1, ya);
            yb = __ffma2_rn(abs2(sb1), wb1, yb);
        } else {
            if (!x_init) {
                xa = __fmul2_rn(relu2(sa0), wa0);
                xb = __fmul2_rn(relu2(sb0), wb0);
                x_init = true;
            } else {
                xa = __ffma2_rn(relu2(sa0), wa0, xa);
                xb = __ffma2_rn(relu2(sb0), wb0, xb);
            }
            xa = __ffma2_rn(relu2(sa1), wa1, xa);
            xb = __ffma2_rn(relu2(sb1), wb1, xb);
        }
    }
    const float2 half = make_float2(0.5f, 0.5f);
    float2 ra = xa, rb = xb;
    if (y_init) {
        ra = x_init ? __ffma2_rn(ya, half, xa) : __fmul2_rn(ya, half);
        rb = x_init ? __ffma2_rn(yb, half, xb) : __fmul2_rn(yb, half);
    }
    va = ra.x + ra.y;
    vb = rb.x + rb.y;
}

__global__ void __launch_bounds__(kThreads, 1)
    fp8_mqa_logits_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_w, const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = ptx::smem_addr(smem_raw);
    const uint32_t pad = ((raw_base + 1023u) & ~1023u) - raw_base;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw_base + pad;

    // warp-uniform role index (the shuffle tells the compiler it is uniform, so addresses
    // derived from it can live in uniform registers)
    const int warp = __shfl_sync(0xffffffffu, int(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;

    auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * uint32_t(i); };
    UnitInfo* units = reinterpret_cast<UnitInfo*>(smem + kOffUnits);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc);
    volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + kOffMisc + 4);
    const Ctl ctl{abort_flag, p};

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(bar(kBarKFull + i), 1);
            ptx::mbar_init(bar(kBarKEmpty + i), 1);
        }
        for (int i = 0; i < kQSlots; ++i) {
            ptx::mbar_init(bar(kBarQFull + i), 1);
            ptx::mbar_init(bar(kBarQEmpty + i), 2 + kEpiWarps);
        }
        for (int i = 0; i < kAccBufs; ++i) {
            ptx::mbar_init(bar(kBarAccFull + i), 1);
            ptx::mbar_init(bar(kBarAccEmpty + i), kEpiWarps * 32);  // every epilogue lane
        }
        for (int i = 0; i < kUnitSlots; ++i) {
            ptx::mbar_init(bar(kBarUnitFull + i), 1);
            ptx::mbar_init(bar(kBarUnitEmpty + i), 2 + kEpiWarps);
        }
        ptx::mbar_init(bar(kBarDrain), 2);
        *abort_flag = 0;
        ptx::mbar_init_fence();
        // Each CTA's first unit is its own index (no shared counter): its Q + w load starts
        // now, before the set-up barrier, and overlaps the reads of the unit's windows.
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_w);
        const int32_t b0 = p.num_blocks - 1 - int32_t(blockIdx.x / uint32_t(p.split));
        if (in_bounds(b0 >= 0 && int64_t(b0) * kRows < p.M, p.status, kBoundsQBlock, b0)) {
            ptx::mbar_arrive_expect_tx(bar(kBarQFull), kQBytes + kWBytes);
            ptx::tma_load_2d_hint(sbase + kOffQ, &tm_q, bar(kBarQFull), 0, b0 * kRows * kHeads,
                                  ptx::policy_evict_first());
            ptx::tma_load_2d(sbase + kOffW, &tm_w, bar(kBarQFull), 0, b0 * kRows);
        } else {
            ptx::mbar_arrive(bar(kBarQFull));
        }
        ptx::prefetch_tensormap(&tm_k);
    }
    if (warp == kFillWarp) {
        // The first unit's window words and its chunk's first two K tiles head for L2 now, so
        // the producer's window reads and first K loads after the set-up barrier find them
        // there (prefetches only: nothing waits on them).
        const int32_t b0 = p.num_blocks - 1 - int32_t(blockIdx.x / uint32_t(p.split));
        const int32_t c0 = int32_t(blockIdx.x % uint32_t(p.split));
        if (lane < 2 && b0 >= 0 && int64_t(b0) * kRows < p.M)
            ptx::prefetch_l2((lane ? p.ke : p.ks) + int64_t(b0) * kRows);
        const int32_t ct0 = c0 * p.tiles_per_chunk;
        const int32_t ct1 = min(ct0 + p.tiles_per_chunk, p.num_tiles);
        const int32_t t = ct0 + lane - 2;
        if (lane >= 2 && lane < 4 && t < ct1) ptx::tma_prefetch_2d(&tm_k, 0, t * kTileKeys);
    }
    if (warp == kMmaWarp0) {
        ptx::tmem_alloc(sbase + kOffMisc, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = __shfl_sync(0xffffffffu, *tmem_slot, 0);

    if (warp < kEpiWarp0) ptx::regs_dec<kCtlRegs>();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const uint64_t pol_k = ptx::policy_evict_last();
        const uint64_t pol_q = ptx::policy_evict_first();
        uint32_t ui = 0, g = 0, qi = 0;
        // Claim the next unit with key tiles (empty units are skipped here, never published);
        // every lane returns the same unit, lane r < kRows also its row's window.  Units below
        // gridDim.x are the CTAs' static first units; the shared counter hands out the rest.
        // When every unit is a first unit, the counter is never touched.
        const bool dynamic = uint32_t(p.num_units) > gridDim.x;
        auto claim = [&]() -> Geometry {
            while (true) {
                uint32_t u = 0;
                int stop = 0;
                if (lane == 0) {
                    u = dynamic ? gridDim.x + atomicAdd(&p.sched->next_unit, 1u) : uint32_t(p.num_units);
                    stop = (u >= uint32_t(p.num_units) || *abort_flag) ? 1 : 0;
                }
                u = __shfl_sync(0xffffffffu, u, 0);
                if (__shfl_sync(0xffffffffu, stop, 0)) {
                    Geometry none{};
                    none.m0 = -1;
                    return none;
                }
                const int32_t b = p.num_blocks - 1 - int32_t(u / uint32_t(p.split));
                const int32_t c = int32_t(u % uint32_t(p.split));
                const Geometry geo = unit_geometry(p, b, c, true);
                // Move the shared counter past the chunks of this block that this claim has
                // shown to be empty, so no CTA spends a claim on them (a hint: a unit that is
                // claimed anyway is found empty).
                const uint32_t next_useful = u - uint32_t(c) + uint32_t(geo.skip);
                if (lane == 0 && geo.skip > 0 && next_useful > gridDim.x)
                    atomicMax(&p.sched->next_unit, next_useful - gridDim.x);
                if (geo.t1 > geo.t0) return geo;
            }
        };
        // Publish a unit to the consumers (m0 < 0: the terminate marker) and start its Q + w
        // load.  Returns false when the CTA is aborting.
        auto publish = [&](const Geometry& geo, bool q_requested) -> bool {
            const uint32_t slot = ui % kUnitSlots;
            int ok = 1;
            if (lane == 0) ok = wait_bar(bar(kBarUnitEmpty + slot), ((ui / kUnitSlots) & 1u) ^ 1u, ctl);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) return false;
            UnitInfo& dst = units[slot];
            if (lane < kRows) {
                dst.lo[lane] = geo.lo;
                dst.hi[lane] = geo.hi;
            }
            if (lane == 0) {
                dst.m0 = geo.m0;
                dst.t0 = geo.t0;
                dst.t1 = geo.t1;
                dst.flags = geo.m0 < 0 ? kUnitTerminate : 0;
            }
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(bar(kBarUnitFull + slot));
                if (geo.m0 >= 0 && q_requested) {
                    ++qi;
                } else if (geo.m0 >= 0) {
                    const uint32_t qs = qi % kQSlots;
                    ok = wait_bar(bar(kBarQEmpty + qs), ((qi / kQSlots) & 1u) ^ 1u, ctl);
                    if (ok) {
                        const uint32_t fb = bar(kBarQFull + qs);
                        if (in_bounds(geo.m0 >= 0 && geo.m0 < p.M, p.status, kBoundsQBlock,
                                      geo.m0)) {
                            ptx::mbar_arrive_expect_tx(fb, kQBytes + kWBytes);
                            ptx::tma_load_2d_hint(sbase + kOffQ + qs * kQBytes, &tm_q, fb, 0,
                                                  geo.m0 * kHeads, pol_q);
                            ptx::tma_load_2d(sbase + kOffW + qs * kWBytes, &tm_w, fb, 0,
                                             geo.m0);
                        } else {
                            ptx::mbar_arrive(fb);
                        }
                        ++qi;
                    }
                }
            }
            ++ui;
            return __shfl_sync(0xffffffffu, ok, 0) != 0;
        };
        // One unit of lookahead: the next unit is claimed, published and its Q requested
        // while the current unit's last kClaimAhead K tiles are still to be issued (plus the
        // kStages in the ring), so the claim's global round trips and the Q load hide behind
        // them.  Claiming earlier would hold units back from CTAs that finish first.
        // The static first unit is published even when it has no key tiles (its Q is already
        // on the way); the consumers then skip it.
        Geometry cur = unit_geometry(p, p.num_blocks - 1 - int32_t(blockIdx.x / uint32_t(p.split)),
                                     int32_t(blockIdx.x % uint32_t(p.split)), true);
        if (lane == 0 && cur.skip > 0) {
            const uint32_t next_useful = blockIdx.x - blockIdx.x % uint32_t(p.split) + uint32_t(cur.skip);
            if (dynamic && next_useful > gridDim.x)
                atomicMax(&p.sched->next_unit, next_useful - gridDim.x);
        }
        bool ok = publish(cur, true);
        while (ok && cur.m0 >= 0) {
            Geometry nxt{};
            bool have_nxt = false;
            const int32_t claim_at = max(cur.t0, cur.t1 - kClaimAhead);
            for (int32_t t = cur.t0; ok && t < cur.t1; ++t) {
                if (t == claim_at) {
                    nxt = claim();
                    ok = publish(nxt, false);
                    have_nxt = true;
                    if (!ok) break;
                }
                int issued = 1;
                if (lane == 0) {
                    const uint32_t st = g % kStages;
                    issued = wait_bar(bar(kBarKEmpty + st), ((g / kStages) & 1u) ^ 1u, ctl) ? 1 : 0;
                    if (issued) {
                        const uint32_t fb = bar(kBarKFull + st);
                        if (in_bounds(t >= 0 && t < p.num_tiles, p.status, kBoundsKTile, t)) {
                            ptx::mbar_arrive_expect_tx(fb, kKBytes);
                            ptx::tma_load_2d_hint(sbase + kOffK + st * kKBytes, &tm_k, fb, 0,
                                                  t * kTileKeys, pol_k);
                        } else {
                            ptx::mbar_arrive(fb);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, issued, 0) != 0;
                if (ok) ++g;
            }
            if (ok && !have_nxt) {
                nxt = claim();
                ok = publish(nxt, false);
            }
            cur = nxt;
        }
        if (lane == 0) {
            // Wait for any TMA load still in flight before the CTA can exit: only the last
            // kStages K loads and the last kQSlots Q loads can be outstanding.
            for (uint32_t j = (g > kStages ? g - kStages : 0); j < g; ++j)
                drain_bar(bar(kBarKFull + j % kStages), (j / kStages) & 1u, p.drain_ns);
            for (uint32_t j = (qi > kQSlots ? qi - kQSlots : 0); j < qi; ++j)
                drain_bar(bar(kBarQFull + j % kQSlots), (j / kQSlots) & 1u, p.drain_ns);
        }
    } else if (warp == kMmaWarp0 || warp == kMmaWarp1) {
        // ------------------------------------------------------------ MMA issuers
        // Two issuers on different SM sub-partitions take alternate tiles, so each owns one
        // accumulator buffer; issuing tcgen05.mma slows the issuing sub-partition's other
        // warps, and splitting it keeps any one set of epilogue warps from falling behind.
        if (lane == 0) {
            const uint32_t par = warp == kMmaWarp1 ? 1u : 0u;
            uint32_t ui = 0, g = 0, qi = 0;
            bool ok = true;
            while (ok) {
                const uint32_t slot = ui % kUnitSlots;
                if (!wait_bar(bar(kBarUnitFull + slot), (ui / kUnitSlots) & 1u, ctl)) break;
                const int32_t flags = units[slot].flags;
                const int32_t ut0 = units[slot].t0, ut1 = units[slot].t1;
                ptx::mbar_arrive(bar(kBarUnitEmpty + slot));
                ++ui;
                if (flags & kUnitTerminate) break;
                const uint32_t qs = qi % kQSlots;
                if (!wait_bar(bar(kBarQFull + qs), (qi / kQSlots) & 1u, ctl)) break;
                ++qi;
                const uint64_t bdesc = sw128_desc(sbase + kOffQ + qs * kQBytes);
                for (int32_t t = ut0; t < ut1; ++t) {
                    const uint32_t st = g % kStages;
                    const uint32_t ab = g & 1u;
                    if (ab != par) {  // the other issuer's tile
                        ++g;
                        continue;
                    }
                    if (!wait_bar(bar(kBarKFull + st), (g / kStages) & 1u, ctl)) {
                        ok = false;
                        break;
                    }
                    if (!wait_bar(bar(kBarAccEmpty + ab), ((g >> 1) & 1u) ^ 1u, ctl)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint64_t adesc = sw128_desc(sbase + kOffK + st * kKBytes);
                    const uint32_t d = tmem_base + ab * kAccStride;
#pragma unroll
                    for (int k = 0; k < kDim / kUmmaK; ++k) {
                        // advance 32 bytes along K inside the swizzle atom
                        ptx::mma_f8f6f4(d, adesc + 2ull * k, bdesc + 2ull * k, kIdesc,
                                        k > 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(bar(kBarKEmpty + st));
                    ptx::mma_commit(bar(kBarAccFull + ab));
                    ++g;
                }
                if (!ok) break;
                ptx::mma_commit(bar(kBarQEmpty + qs));
            }
            // all MMAs issued by this thread complete before TMEM can be released
            ptx::mma_commit(bar(kBarDrain));
            drain_bar(bar(kBarDrain), 0, p.drain_ns);
        }
        __syncwarp();
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------------------ -inf writer
        if (p.clean) {
            const uint32_t src = sbase + kOffFill;
            {
                float4* f = reinterpret_cast<float4*>(smem + kOffFill);
                const float ninf = __int_as_float(0xff800000u);
                for (int i = lane; i < int(kFillBytes / 16); i += 32)
                    f[i] = make_float4(ninf, ninf, ninf, ninf);
                ptx::fence_proxy_async_smem();  // visible to the bulk copies
                __syncwarp();
            }
            // the CTA's own index first, then the shared counter (untouched when every unit is
            // a first unit)
            const bool dynamic = uint32_t(p.num_units) > gridDim.x;
            for (bool first = true;; first = false) {
                uint32_t u = 0;
                int stop = 0;
                if (lane == 0) {
                    u = first ? blockIdx.x
                              : (dynamic ? gridDim.x + atomicAdd(&p.sched->next_fill, 1u)
                                         : uint32_t(p.num_units));
                    stop = (u >= uint32_t(p.num_units) || *abort_flag) ? 1 : 0;
                }
                u = __shfl_sync(0xffffffffu, u, 0);
                if (__shfl_sync(0xffffffffu, stop, 0)) break;
                // light-first order: the blocks with the most -inf first
                const int32_t b = int32_t(u / uint32_t(p.split));
                const int32_t c = int32_t(u % uint32_t(p.split));
                const Geometry geo = unit_geometry(p, b, c);
                const int64_t col_lo = int64_t(geo.ct0) * kTileKeys;
                const int64_t col_hi = min(int64_t(geo.ct1) * kTileKeys, p.N);
                const bool any = geo.t1 > geo.t0;
                const int64_t left_end = any ? int64_t(geo.t0) * kTileKeys : col_hi;
                const int64_t right_beg = any ? min(int64_t(geo.t1) * kTileKeys, p.N) : col_hi;
                for (int r = 0; r < kRows; ++r) {
                    const int64_t m = int64_t(geo.m0) + r;
                    if (m >= p.M) break;
                    fill_neg_inf(p, m, col_lo, left_end, src);
                    fill_neg_inf(p, m, right_beg, col_hi, src);
                }
                if (lane == 0) {
                    // keep at most a few units' bulk copies queued
                    ptx::bulk_commit();
                    ptx::bulk_wait_read<4>();
                }
                __syncwarp();
            }
            // every bulk copy has landed before the CTA (and its shared memory) goes away
            if (lane == 0) ptx::bulk_wait_all();
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ epilogue
        ptx::regs_inc<kEpiRegs>();
        const int sp = warp & 3;                                // TMEM sub-partition
        const int grp = (warp - kEpiWarp0) >> 2;               // rows 2 grp, 2 grp + 1 of the 8
        const uint32_t tcol = uint32_t(grp * kRowsPerEpiWarp * kHeads);
        const uint32_t tm_warp = tmem_base + (uint32_t(sp * 32) << 16) + tcol;
        const uint32_t full0 = bar(kBarAccFull), empty0 = bar(kBarAccEmpty);
        const float ninf = __int_as_float(0xff800000u);
        if (!in_bounds(tcol + kAccStride + kRowsPerEpiWarp * kHeads <= kTmemCols, p.status,
                       kBoundsTmem, tcol))
            ctl.abort[0] = 1;
        uint32_t ui = 0, g = 0, qi = 0;
        bool ok = true;
        while (ok) {
            const uint32_t slot = ui % kUnitSlots;
            if (!wait_bar_warp(bar(kBarUnitFull + slot), (ui / kUnitSlots) & 1u, ctl)) break;
            // the unit and this warp's rows' windows, copied out before the slot is released
            const UnitInfo& src = units[slot];
            const int32_t flags = src.flags, m0 = src.m0, t0 = src.t0, t1 = src.t1;
            const int32_t lo_a = src.lo[2 * grp], hi_a = src.hi[2 * grp];
            const int32_t lo_b = src.lo[2 * grp + 1], hi_b = src.hi[2 * grp + 1];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kBarUnitEmpty + slot));
            ++ui;
            if (flags & kUnitTerminate) break;

            const uint32_t qs = qi % kQSlots;
            if (!wait_bar_warp(bar(kBarQFull + qs), (qi / kQSlots) & 1u, ctl)) break;
            ++qi;
            // w of this warp's rows stays in shared memory for the whole unit; every lane
            // reads the same address (a broadcast), 4 heads per 16-byte load
            const float4* wsm = reinterpret_cast<const float4*>(
                smem + kOffW + qs * kWBytes + grp * kRowsPerEpiWarp * kHeads * 4);

            // This warp's rows, and the key tiles that lie inside both rows' windows (stored
            // without compare/select).  Rows past M have empty windows.
            const int64_t ma = int64_t(m0) + 2 * grp;
            const bool ok_a = ma < p.M, ok_b = ma + 1 < p.M;
            int32_t cs = max((lo_a + kTileKeys - 1) / kTileKeys, (lo_b + kTileKeys - 1) / kTileKeys);
            int32_t ce = min(hi_a / kTileKeys, hi_b / kTileKeys);
            if (!ok_b) ce = 0;
            cs = max(t0, min(cs, t1));
            ce = max(cs, min(ce, t1));

            // this lane's key, and its rows' starts (row b's is row a's plus N, formed per tile:
            // fewer live registers than two running pointers)
            int32_t n = t0 * kTileKeys + sp * 32 + lane;
            float* const row_a = p.out + (ok_a ? ma : 0) * p.N;
            uint32_t ph = (g >> 1) & 1u;
            // kv_scale one tile ahead; past the end the index is clamped (the value is unused)
            float kv_next = __ldg(p.kv_scale + min(n, int32_t(p.N) - 1));

            // One tile.  kClean: inside both rows' windows (no compare/select).  kAB: the
            // accumulator buffer when known at compile time (the clean middle runs in buffer
            // pairs), -1 when it comes from the tile count.
            auto tile = [&](auto clean_tag, auto ab_tag) -> bool {
                constexpr bool kClean = decltype(clean_tag)::value;
                constexpr int kAB = decltype(ab_tag)::value;
                const uint32_t ab = kAB >= 0 ? uint32_t(kAB) : (g & 1u);
                if (!wait_bar_all(full0 + 8u * ab, ph, ctl)) return false;
                ptx::tc_fence_after();
                // Copy this warp's accumulators out of TMEM and release the buffer at once,
                // so the MMA can refill it while this warp does the arithmetic.
                uint32_t s[64];
                ptx::tmem_ld_32x32b_x64_sync(tm_warp + ab * kAccStride, s);
                ptx::tc_fence_before();
                ptx::mbar_arrive(empty0 + 8u * ab);  // all 32 lanes arrive
                const float kv = kv_next;
                const int32_t n_kv = min(n + kTileKeys, int32_t(p.N) - 1);
                if (in_bounds(n_kv >= 0 && n_kv < p.N, p.status, kBoundsKvScale, n_kv))
                    kv_next = __ldg(p.kv_scale + n_kv);
                float va, vb;
                relu_dot_2rows(s, wsm, va, vb);
                float* const pa = row_a + n;
                float* const pb = pa + p.N;
                if (kClean) {
                    // inside both rows' windows, so n < N and both rows exist
                    if (in_bounds(n < p.N && ok_b, p.status, kBoundsStore, n)) {
                        __stcs(pa, va * kv);
                        __stcs(pb, vb * kv);
                    }
                } else if (n < p.N) {
                    if (ok_a && in_bounds(ma < p.M, p.status, kBoundsStore, n)) {
                        if (n >= lo_a && n < hi_a)
                            __stcs(pa, va * kv);
                        else if (p.clean)
                            __stcs(pa, ninf);
                    }
                    if (ok_b && in_bounds(ma + 1 < p.M, p.status, kBoundsStore, n)) {
                        if (n >= lo_b && n < hi_b)
                            __stcs(pb, vb * kv);
                        else if (p.clean)
                            __stcs(pb, ninf);
                    }
                }
                n += kTileKeys;
                ph ^= ab;
                ++g;
                return true;
            };
            // masked head, clean middle (in buffer pairs), masked tail
            int32_t t = t0;
            for (; ok && t < cs; ++t) ok = tile(BoolTag<false>{}, IntTag<-1>{});
            if (ok && t < ce && (g & 1u)) {
                ok = tile(BoolTag<true>{}, IntTag<-1>{});
                ++t;
            }
            for (; ok && t + 1 < ce; t += 2) {
                ok = tile(BoolTag<true>{}, IntTag<0>{});
                if (ok) ok = tile(BoolTag<true>{}, IntTag<1>{});
            }
            if (ok && t < ce) {
                ok = tile(BoolTag<true>{}, IntTag<-1>{});
                ++t;
            }
            for (; ok && t < t1; ++t) ok = tile(BoolTag<false>{}, IntTag<-1>{});
            if (!ok) break;
            // this warp is done with the unit's w
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kBarQEmpty + qs));
        }
    }

    // ---------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
    if (threadIdx.x == 0 && uint32_t(p.num_units) > gridDim.x) {
        // the shared counters were used: the last CTA out resets them for the slot's next launch
        __threadfence();
        const uint32_t prev = atomicAdd(&p.sched->done_ctas, 1u);
        if (prev == gridDim.x - 1) {
            // last CTA out: every producer and writer has stopped claiming work
            p.sched->next_unit = 0;
            p.sched->next_fill = 0;
            p.sched->done_ctas = 0;
            __threadfence();
        }
    }
}

}  // namespace fp8mqa
