// Per-row top-k over indexer logits for GB300 (sm_103a): the step that consumes the logits
// (ROCm/aiter PR #7183 "[HIP] [JIT] Add gfx950 prefill FP8 MQA logits", "Test plan":
// top-512 selections; ROCm/aiter PR #6159 "[Triton/Gluon] GFX950 sparse mla optimizations",
// "Technical Details": sparse MLA with top-k 512).
//
// For every row: the k largest finite logits (-inf, outside the row's window, is never
// selected), ordered by value descending and, for equal values, by index ascending (-0.0
// equals +0.0); slots past the row's finite entries get index -1 and value -inf.  An unsorted
// call (TopkParams::sorted = 0) writes the same entries in selection order, without the sort.
//
// Every kernel takes an optional window per row (fp8_mqa_topk_windowed): only entries inside
// it are candidates, and nothing outside it is read.  Rows of up to 8192 keys at k <= 1024 go
// to the staged-row kernel at the end of this file.  For the others, a persistent grid of at
// most one CTA per SM walks the rows: rows of up to 65536 keys at k <= 512, and of up to
// 32768 keys at larger k, two at a time, 256 threads each on a named barrier of their own, so
// one row's barrier waits overlap the other's work; longer rows one at a time with all 512
// threads.
//
// Each row first tries a sampled threshold.  A histogram of one 32-byte sector in eight of the
// window (over the top 11 or 12 key bits, a template choice) gives G; one pass keeps the
// entries >= G in a buffer, and a radix cut over their composites (key, index) picks the k
// winners.  That pass keeps the next chunk's loads in flight while it examines the current
// one, tests each float4 by its largest entry and lets a passing lane claim slots for its kept
// entries with one shared-memory atomic; once it ends, the next row's sample sectors are
// prefetched into L2.  When the threshold misses (fewer than k kept, or more than the buffer
// holds), the row takes the full radix select on an order-preserving 32-bit key (its second
// read of the row comes from L2):
//   1. read the row, histogram the top 11 key bits (a private histogram per warp, so hot
//      bins do not serialise the whole block);
//   2. the bin b0 holding the k-th largest is found from the top;
//   3. read the row again and append the keys of b0 and above to a shared-memory buffer
//      (one append per key); those above b0 are winners, and two more radix passes (key
//      bits 20..10 and 9..0) over those of b0 pick the rest, equal keys taken by index;
//   4. the winners (at most 2048) are sorted (each warp sorts a run in registers, then the
//      runs are merged pairwise) and written.
// When b0 and the bins above hold more entries than the buffer, the remaining 21 key bits
// of b0 are resolved by two more histogram passes over the row and a collect pass that
// takes the ties in index order.
#pragma once

#include <cstdint>

namespace fp8mqa {

constexpr int kTopkThreads = 512;  // threads per CTA
constexpr int kTopkMaxK = 2048;
constexpr int kTopkBins = 2048;      // 11-bit digits

struct TopkParams {
    const float* logits;
    int64_t M, N, ld;  // row m at logits + m * ld
    int32_t k;
    int32_t* indices;  // [M, k]
    float* values;     // [M, k] or null
    const int32_t* ks;  // row m's window [ks[m], ke[m]) clamped to [0, N); null: the whole row
    const int32_t* ke;
    int32_t sorted;     // 1: each row's winners by value descending; 0: in selection order
};

// Row m's window, clamped to [0, N) (an empty window when ks >= ke).
__device__ __forceinline__ void topk_window(const TopkParams& p, int64_t m, int& lo, int& hi)
{
    lo = 0;
    hi = int(p.N);
    if (p.ks) {
        const int64_t a = p.ks[m], b = p.ke[m];
        lo = int(a < 0 ? 0 : (a > p.N ? p.N : a));
        hi = int(b < lo ? lo : (b > p.N ? p.N : b));
    }
}

// A CTA works on kTopkThreads / NT rows at once, NT threads each, a row's threads
// synchronising on a named barrier of their own (the whole CTA's barrier when NT is the
// CTA).  One row's shared memory; TIE entries of the threshold bin (and the bins above it)
// are selected in it; its warps share HW first-pass histograms.
template <int NT, int TIE, int HW = NT / 32>
struct TopkSmem {
    static constexpr int kNT = NT;
    static constexpr int kTie = TIE;
    static constexpr int kHW = HW;
    uint32_t whist[HW][kTopkBins];  // first-pass histograms, later the spare buffer
    uint32_t hist[kTopkBins];
    unsigned long long cand[kTopkMaxK];
    unsigned long long tbuf[TIE];
    uint32_t scratch[NT / 32];
    uint32_t sel_bin, sel_above, sel_count, n_cand, n_tie, tie_base, n_spare, pad;
};
// Two rows per CTA, 256 threads each: rows of up to 65536 keys at k <= 512 with a 2048-entry
// threshold-bin buffer and a histogram per warp; rows of up to 32768 keys at larger k with a
// 4096-entry buffer and a histogram per two warps.  Longer rows go one per CTA with the
// 8192-entry buffer.
using TopkSmemPair = TopkSmem<256, 2048>;
using TopkSmemPairWide = TopkSmem<256, 4096, 4>;
using TopkSmemOne = TopkSmem<512, 8192>;
static_assert(sizeof(TopkSmemOne) <= 232448 && 2 * sizeof(TopkSmemPair) <= 232448 &&
                  2 * sizeof(TopkSmemPairWide) <= 232448,
              "top-k shared memory");
static_assert(sizeof(TopkSmemPair) % 16 == 0 && sizeof(TopkSmemPairWide) % 16 == 0,
              "row slices stay 16-byte aligned");
static_assert(TopkSmemPair::kTie <= TopkSmemPair::kHW * kTopkBins / 2 &&
                  TopkSmemPairWide::kTie <= TopkSmemPairWide::kHW * kTopkBins / 2 &&
                  TopkSmemOne::kTie <= TopkSmemOne::kHW * kTopkBins / 2,
              "the spare buffer holds the threshold-bin buffer");

// This thread's index among its row's NT threads, and the row's barrier.
template <int NT>
__device__ __forceinline__ int topk_tid()
{
    return NT == kTopkThreads ? int(threadIdx.x) : int(threadIdx.x) % NT;
}

template <int NT>
__device__ __forceinline__ void topk_sync()
{
    if constexpr (NT == kTopkThreads)
        __syncthreads();
    else
        asm volatile("bar.sync %0, %1;" ::"r"(1 + int(threadIdx.x) / NT), "n"(NT) : "memory");
}

// Order-preserving key of a finite float (larger value, larger key; -0.0 and +0.0 equal).
__device__ __forceinline__ uint32_t topk_key(float x)
{
    uint32_t u = __float_as_uint(x);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ bool topk_eligible(float x)
{
    return (__float_as_uint(x) & 0x7F800000u) != 0x7F800000u;  // finite
}

// Ask for the 32-byte sector at p to be brought into L2 (no register is written).
__device__ __forceinline__ void topk_prefetch_l2(const float* p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Winners sort by this value, descending: key first, then the lower index.
__device__ __forceinline__ unsigned long long topk_composite(uint32_t key, int i)
{
    return (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - uint32_t(i));
}

// Inclusive sum over a row's NT threads in index order; `scratch` holds NT / 32 words.
template <int NT>
__device__ __forceinline__ uint32_t topk_block_scan(uint32_t v, uint32_t* scratch, uint32_t& total)
{
    const int lane = threadIdx.x & 31, warp = topk_tid<NT>() >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) scratch[warp] = v;
    topk_sync<NT>();
    uint32_t before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        const uint32_t s = scratch[w];
        if (w < warp) before += s;
        total += s;
    }
    topk_sync<NT>();
    return v + before;
}

// Visit every element of the row's window [lo, hi) once, in chunks whose trip count is uniform
// over the row's threads (so warp votes inside `fn` see every lane): fn(index, value, valid);
// nothing outside the window is read.  16-byte aligned rows are read four floats per thread
// per chunk (from lo rounded down to a multiple of 4) unless kInOrder asks for one element per
// thread per call, so that successive calls cover the window in index order.  kWin = false:
// the window is the whole row [0, hi) (lo is not looked at).
template <int NT, bool kInOrder = false, bool kWin = true, typename Fn>
__device__ __forceinline__ void topk_for_row(const float* x, int lo, int hi, Fn&& fn)
{
    const int tid = topk_tid<NT>();
    if (!kWin) lo = 0;
    auto in = [&](int i) { return (!kWin || i >= lo) && i < hi; };
    if (!kInOrder && (reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
        // four 16-byte loads in flight per thread before any is used
        constexpr int kU = 4;
        for (int c0 = lo & ~3; c0 < hi; c0 += 4 * kU * NT) {
            float4 v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = c0 + 4 * (u * NT + tid);
                v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if ((!kWin || i >= lo) && i + 3 < hi) {
                    v[u] = __ldg(reinterpret_cast<const float4*>(x + i));
                } else {
                    if (in(i)) v[u].x = __ldg(x + i);
                    if (in(i + 1)) v[u].y = __ldg(x + i + 1);
                    if (in(i + 2)) v[u].z = __ldg(x + i + 2);
                    if (in(i + 3)) v[u].w = __ldg(x + i + 3);
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = c0 + 4 * (u * NT + tid);
                fn(i, v[u].x, in(i));
                fn(i + 1, v[u].y, in(i + 1));
                fn(i + 2, v[u].z, in(i + 2));
                fn(i + 3, v[u].w, in(i + 3));
            }
        }
    } else {
        for (int c0 = lo; c0 < hi; c0 += NT) {
            const int i = c0 + tid;
            fn(i, i < hi ? __ldg(x + i) : 0.f, i < hi);
        }
    }
}

// Add one to hist[bin] for every lane with `in`.
__device__ __forceinline__ void topk_hist_add(uint32_t* hist, uint32_t bin, bool in)
{
    if (in) atomicAdd(&hist[bin], 1u);
}

// Append `v` for every lane with `take` to buf[*count...], one atomic per warp.
__device__ __forceinline__ void topk_append(unsigned long long* buf, uint32_t* count,
                                            unsigned long long v, bool take)
{
    const uint32_t mask = __ballot_sync(0xffffffffu, take);
    if (mask == 0) return;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(mask) - 1;
    uint32_t base = 0;
    if (lane == leader) base = atomicAdd(count, uint32_t(__popc(mask)));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (take) buf[base + __popc(mask & ((1u << lane) - 1u))] = v;
}

// The bin holding the kk-th largest entry, scanning hist[0, nb) from the top; writes
// sel_bin, sel_above (entries in higher bins) and sel_count (entries in the bin).  Returns
// the total count.  Uniform over the row's threads.
template <typename S>
__device__ __forceinline__ uint32_t topk_find_bin(S& s, const uint32_t* hist, uint32_t nb,
                                                  uint32_t kk)
{
    constexpr int NT = S::kNT;
    const int tid = topk_tid<NT>();
    const int per = int(nb) / NT;
    uint32_t run = 0;
    if (per >= 4) {
        // the thread's bins as 16-byte reads, rotated so that the eight lanes of each
        // quarter warp read distinct bank groups (a plain walk would put all lanes' reads on
        // two banks); the sum does not depend on the order (hist: 16-byte aligned)
        const int nv = per >> 2;
        const int rot = 5 - (__ffs(per) - 1);
        const uint32_t* base = hist + (int(nb) - per * (tid + 1));
        for (int v = 0; v < nv; ++v) {
            const uint4 h = *reinterpret_cast<const uint4*>(base + 4 * ((v + (tid >> rot)) & (nv - 1)));
            run += h.x + h.y + h.z + h.w;
        }
    } else {
        for (int j = 0; j < per; ++j) run += hist[nb - 1 - (tid * per + j)];
    }
    uint32_t total = 0;
    const uint32_t incl = topk_block_scan<NT>(run, s.scratch, total);
    const uint32_t excl = incl - run;
    if (kk <= total && excl < kk && incl >= kk) {
        uint32_t above = excl;
        for (int j = 0; j < per; ++j) {
            const uint32_t b = nb - 1 - (tid * per + j);
            const uint32_t h = hist[b];
            if (above + h >= kk) {
                s.sel_bin = b;
                s.sel_above = above;
                s.sel_count = h;
                break;
            }
            above += h;
        }
    }
    topk_sync<NT>();
    return total;
}

// Descending sort of buf[0, n), fastest network for n.
template <int NT>
__device__ __forceinline__ void topk_sort_any(unsigned long long* buf, int n);

// Move the kk largest composites of buf[0, n) (all with the same top 11 key bits) to the
// winners.  Two radix passes over the buffer, on key bits 20..10 and 9..0, narrow it to the
// entries whose key equals the kk-th largest key; of those, the ones with the lowest index
// are taken (a sort of just these ties when the cut falls inside them).  `spare` holds at
// least n composites.
template <typename S>
__device__ __forceinline__ void topk_select_buffer(S& s, unsigned long long* buf,
                                                   unsigned long long* spare, uint32_t n,
                                                   uint32_t kk)
{
    constexpr int NT = S::kNT;
    const int tid = topk_tid<NT>();
    topk_sync<NT>();  // every thread holds its arguments (n may be a count reset below)
    for (int pass = 0; pass < 2; ++pass) {
        const int shift = pass == 0 ? 10 : 0;
        const uint32_t nb = pass == 0 ? 2048u : 1024u;
        for (uint32_t b = tid; b < nb; b += NT) s.hist[b] = 0;
        if (tid == 0) s.n_tie = 0;
        topk_sync<NT>();
        for (uint32_t j = tid; j < n; j += NT)
            atomicAdd(&s.hist[uint32_t(buf[j] >> (32 + shift)) & (nb - 1)], 1u);
        topk_sync<NT>();
        topk_find_bin(s, s.hist, nb, kk);
        const uint32_t b = s.sel_bin;
        kk -= s.sel_above;
        // entries above the bin are winners; the bin's entries move on to the next pass
        const uint32_t rounds = (n + NT - 1) / NT;
        for (uint32_t r = 0; r < rounds; ++r) {
            const uint32_t j = r * NT + tid;
            const unsigned long long c = j < n ? buf[j] : 0ull;
            const uint32_t d = uint32_t(c >> (32 + shift)) & (nb - 1);
            topk_append(s.cand, &s.n_cand, c, j < n && d > b);
            topk_append(spare, &s.n_tie, c, j < n && d == b);
        }
        topk_sync<NT>();
        n = s.n_tie;
        unsigned long long* t = buf;
        buf = spare;
        spare = t;
        topk_sync<NT>();  // every thread has read n before the next pass resets the count
    }
    // buf[0, n) now holds the entries equal to the kk-th largest key; take kk by index
    if (kk < n) topk_sort_any<NT>(buf, int(n));
    for (uint32_t j = tid; j < kk; j += NT) {
        // the composite orders equal keys by index, so after the sort these are the lowest
        s.cand[s.n_cand + j] = buf[j];
    }
    topk_sync<NT>();
    if (tid == 0) s.n_cand += kk;
    topk_sync<NT>();
}

// Bitonic sort of buf[0, n) descending (padding with zeros up to the next power of two,
// which the buffer must hold).
template <int NT>
__device__ __forceinline__ void topk_sort_desc(unsigned long long* buf, int n)
{
    const int tid = topk_tid<NT>();
    int P = 1;
    while (P < n) P <<= 1;
    for (int i = n + tid; i < P; i += NT) buf[i] = 0ull;
    topk_sync<NT>();
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = tid; t < P / 2; t += NT) {
                const int lo = (t / stride) * stride * 2 + (t % stride);
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const unsigned long long a = buf[lo], b = buf[hi];
                if ((a < b) == desc) {
                    buf[lo] = b;
                    buf[hi] = a;
                }
            }
            topk_sync<NT>();
        }
    }
}

// One compare-exchange step at stride S < E between a thread's own elements (S fixed at
// compile time so the elements stay in registers).
template <int E, int S>
__device__ __forceinline__ void topk_sort_in_thread(unsigned long long (&v)[E], int tid, int size)
{
    if constexpr (S < E) {
#pragma unroll
        for (int j = 0; j < E; ++j) {
            if (j & S) continue;
            // size >= E: the direction is the thread's (the same for all its entries)
            const bool desc = size >= E ? ((tid * E) & size) == 0 : (j & size) == 0;
            const unsigned long long a = v[j], b = v[j | S];
            if ((a < b) == desc) {
                v[j] = b;
                v[j | S] = a;
            }
        }
    }
}

// Bitonic sort of buf[0, n) descending for n <= NT * E, with thread t holding elements
// t*E .. t*E+E-1 in registers: compare-exchanges at strides below E stay in the thread, at
// strides below 32*E use warp shuffles, and only the wider ones go through shared memory
// (two barriers each; the buffer holds NT * E entries).
template <int NT, int E>
__device__ __forceinline__ void topk_sort_desc_reg(unsigned long long* buf, int n)
{
    constexpr int P = NT * E;
    const int tid = topk_tid<NT>();
    unsigned long long v[E];
#pragma unroll
    for (int j = 0; j < E; ++j) {
        const int e = tid * E + j;
        v[j] = e < n ? buf[e] : 0ull;
    }
    topk_sync<NT>();
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride >= 32 * E) {
#pragma unroll
                for (int j = 0; j < E; ++j) buf[tid * E + j] = v[j];
                topk_sync<NT>();
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    const int e = tid * E + j;
                    const unsigned long long o = buf[e ^ stride];
                    const bool desc = (e & size) == 0, lo = (e & stride) == 0;
                    const bool keep_max = desc == lo;
                    v[j] = (o > v[j]) == keep_max ? o : v[j];  // composites differ, but for padding zeros
                }
                topk_sync<NT>();
            } else if (stride >= E) {
                const int lanes = stride / E;
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    const int e = tid * E + j;
                    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v[j], lanes);
                    const bool desc = (e & size) == 0, lo = (e & stride) == 0;
                    const bool keep_max = desc == lo;
                    v[j] = (o > v[j]) == keep_max ? o : v[j];  // composites differ, but for padding zeros
                }
            } else if (stride == 1) {
                topk_sort_in_thread<E, 1>(v, tid, size);
            } else if (stride == 2) {
                topk_sort_in_thread<E, 2>(v, tid, size);
            } else {
                topk_sort_in_thread<E, 4>(v, tid, size);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < E; ++j) {
        const int e = tid * E + j;
        if (e < n) buf[e] = v[j];
    }
    topk_sync<NT>();
}

// Descending sort of buf[0, n): in registers up to 2048 entries, else in shared memory.
template <int NT>
__device__ __forceinline__ void topk_sort_any(unsigned long long* buf, int n)
{
    if (n <= NT)
        topk_sort_desc_reg<NT, 1>(buf, n);
    else if (n <= 2 * NT)
        topk_sort_desc_reg<NT, 2>(buf, n);
    else if (n <= 4 * NT)
        topk_sort_desc_reg<NT, 4>(buf, n);
    else if constexpr (NT * 8 <= kTopkMaxK) {
        // a row of fewer threads holds up to eight entries each (its buffers hold 2048)
        if (n <= 8 * NT)
            topk_sort_desc_reg<NT, 8>(buf, n);
        else
            topk_sort_desc<NT>(buf, n);
    } else {
        topk_sort_desc<NT>(buf, n);
    }
}

// Sort of the winners buf[0, n) descending, NT < n <= NT * E, through tmp (NT * E entries):
// each warp sorts its run of 32 * E entries in registers (strides below E in the thread, the
// rest by shuffles, no barrier), then the runs are merged pairwise: every thread finds where
// its E outputs start on its merge diagonal by binary search and merges them in sequence.
// Buffers ping-pong between buf and tmp, the result ends in buf; zeros pad past n.
template <int NT, int E>
__device__ __forceinline__ void topk_sort_merge(unsigned long long* buf, unsigned long long* tmp,
                                                int n)
{
    constexpr int R = 32 * E;  // one warp's run
    constexpr int P = NT * E;
    const int tid = topk_tid<NT>();
    const int lane = tid & 31, warp = tid >> 5;
    {
        unsigned long long v[E];
#pragma unroll
        for (int j = 0; j < E; ++j) {
            const int e = warp * R + lane * E + j;
            v[j] = e < n ? buf[e] : 0ull;
        }
#pragma unroll
        for (int size = 2; size <= R; size <<= 1) {
#pragma unroll
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                if (stride >= E) {
                    // the lane's direction and side, the same for all its entries
                    const int le = lane * E;
                    const bool keep_max = ((le & size) == 0) == ((le & stride) == 0);
#pragma unroll
                    for (int j = 0; j < E; ++j) {
                        const unsigned long long o = __shfl_xor_sync(0xffffffffu, v[j], stride / E);
                        v[j] = (o > v[j]) == keep_max ? o : v[j];
                    }
                } else if (stride == 1) {
                    topk_sort_in_thread<E, 1>(v, lane, size);
                } else if (stride == 2) {
                    topk_sort_in_thread<E, 2>(v, lane, size);
                } else {
                    topk_sort_in_thread<E, 4>(v, lane, size);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < E; ++j) buf[warp * R + lane * E + j] = v[j];
    }
    topk_sync<NT>();
    unsigned long long* src = buf;
    unsigned long long* dst = tmp;
    for (int L = R; L < P; L <<= 1) {
        // runs [base, base + L) and [base + L, base + 2L) merge into dst[base, base + 2L)
        const int o0 = tid * E;
        const int base = o0 & ~(2 * L - 1);
        const int d = o0 - base;
        const unsigned long long* A = src + base;
        const unsigned long long* B = src + base + L;
        int lo = d > L ? d - L : 0, hi = d < L ? d : L;
        while (lo < hi) {  // how many of the first d outputs come from A
            const int mid = (lo + hi) >> 1;
            if (A[mid] > B[d - 1 - mid])
                lo = mid + 1;
            else
                hi = mid;
        }
        int i = lo, j = d - lo;
        // the heads of both runs stay in registers; only the consumed one is reloaded
        unsigned long long a = i < L ? A[i] : 0ull, b = j < L ? B[j] : 0ull;
#pragma unroll
        for (int q = 0; q < E; ++q) {
            const bool take_a = j >= L || (i < L && a > b);
            dst[o0 + q] = take_a ? a : b;
            if (q + 1 < E) {
                if (take_a) {
                    ++i;
                    a = i < L ? A[i] : 0ull;
                } else {
                    ++j;
                    b = j < L ? B[j] : 0ull;
                }
            }
        }
        topk_sync<NT>();
        unsigned long long* t = src;
        src = dst;
        dst = t;
    }
    if (src != buf) {
        for (int e = tid; e < n; e += NT) buf[e] = src[e];
        topk_sync<NT>();
    }
}

// The winners' sort: in registers for up to NT entries, by runs and merges beyond.
template <int NT>
__device__ __forceinline__ void topk_sort_winners(unsigned long long* buf, unsigned long long* tmp,
                                                  int n)
{
    if (n <= NT)
        topk_sort_desc_reg<NT, 1>(buf, n);
    else if (n <= 2 * NT)
        topk_sort_merge<NT, 2>(buf, tmp, n);
    else if (n <= 4 * NT)
        topk_sort_merge<NT, 4>(buf, tmp, n);
    else if constexpr (NT * 8 <= kTopkMaxK) {
        if (n <= 8 * NT)
            topk_sort_merge<NT, 8>(buf, tmp, n);
        else
            topk_sort_desc<NT>(buf, n);
    } else {
        topk_sort_desc<NT>(buf, n);
    }
}

// Composite of an element (0 when it is not eligible: 0 sorts below every eligible entry).
__device__ __forceinline__ unsigned long long topk_reg_comp(float v, int i)
{
    return topk_eligible(v) ? topk_composite(topk_key(v), i) : 0ull;
}

// topk_append with a capacity: an entry past `cap` is dropped (the selection hands over at
// most `cap` winners, so none is; the guard keeps a wrong count inside the buffer).
__device__ __forceinline__ void topk_append_capped(unsigned long long* buf, uint32_t* count,
                                                   unsigned long long v, bool take, uint32_t cap)
{
    const uint32_t mask = __ballot_sync(0xffffffffu, take);
    if (mask == 0) return;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(mask) - 1;
    uint32_t base = 0;
    if (lane == leader) base = atomicAdd(count, uint32_t(__popc(mask)));
    base = __shfl_sync(0xffffffffu, base, leader);
    const uint32_t at = base + uint32_t(__popc(mask & ((1u << lane) - 1u)));
    if (take && at < cap) buf[at] = v;
}

// Bytes of the index part that can differ between entries of a row of n keys: the index part
// is 0xFFFFFFFF - index, so for every index below 2^(8 b) its bytes above the low b are all
// ones.
__device__ __forceinline__ int topk_index_bytes(int64_t n)
{
    return n <= (int64_t(1) << 16) ? 2 : n <= (int64_t(1) << 24) ? 3 : 4;
}

// The cut: the largest value such that exactly min(k, n) of the row's nonzero composites are
// >= it (n: how many there are); 1 when n <= k.  Radix passes of 8 bits over the composite's
// key (bits 63..32), then over the low `idx_bytes` bytes of the index part
// (topk_index_bytes of the row length); the index part's higher bytes are all ones, so they
// join the prefix before the index passes.  A pass whose selected bin is taken whole ends the
// search.
// `src(fn)` calls fn(composite) for each of this thread's composites, with a trip count that
// may differ between threads.  Uniform over the row's threads.
template <typename S, typename Src>
__device__ __forceinline__ unsigned long long topk_reg_cut(S& s, uint32_t k, int idx_bytes,
                                                           Src&& src)
{
    constexpr int NT = S::kNT;
    constexpr uint32_t kBins = 256u < uint32_t(NT) ? uint32_t(NT) : 256u;  // scanned (>= NT)
    const int tid = topk_tid<NT>();
    unsigned long long prefix = 0ull, mask = 0ull;
    uint32_t need = k;
    const int passes = 4 + idx_bytes;
#pragma unroll 1
    for (int pass = 0; pass < passes; ++pass) {
        const int sh = pass < 4 ? 56 - 8 * pass : 8 * (passes - 1 - pass);
        if (pass == 4 && idx_bytes < 4) {
            const unsigned long long ones = (0xFFFFFFFFull << (8 * idx_bytes)) & 0xFFFFFFFFull;
            prefix |= ones;
            mask |= ones;
        }
        for (uint32_t b = tid; b < kBins; b += NT) s.hist[b] = 0u;
        topk_sync<NT>();
        src([&](unsigned long long c) {
            if (c != 0ull && (c & mask) == prefix) atomicAdd(&s.hist[uint32_t(c >> sh) & 255u], 1u);
        });
        topk_sync<NT>();
        const uint32_t total = topk_find_bin(s, s.hist, kBins, need);
        if (pass == 0 && total <= need) return 1ull;
        const uint32_t d = s.sel_bin, above = s.sel_above, cnt = s.sel_count;
        topk_sync<NT>();
        prefix |= static_cast<unsigned long long>(d) << sh;
        mask |= 0xFFull << sh;
        need -= above;
        if (cnt == need) break;  // the whole bin is taken: every composite >= prefix wins
    }
    return prefix;
}

// The sampled threshold's pass: append the composite of every finite entry >= g of the
// window [lo, hi) to s.tbuf (the first S::kTie of them; s.n_tie counts them).  g is finite, so
// NaN and -inf never pass.  A 16-byte aligned row streams in chunks of kU float4 per thread,
// the next chunk's loads issued before the current chunk is examined; a float4 is first tested
// by its largest entry, and only a lane whose float4 passes looks at its four entries, claiming
// slots for the ones it keeps with one shared-memory atomic (kept entries are a few per warp
// and chunk, so this beats warp-wide ballots).  Entries outside the window load as -inf, so
// interior chunks carry no bounds test.  Once more than S::kTie entries are kept the threshold
// has failed (the caller then selects over the whole row), and the pass stops at the next
// chunk; n_tie then only has to exceed S::kTie.
template <typename S, bool kWin, int kU>
__device__ __forceinline__ void topk_keep_above(S& s, const float* x, int lo, int hi, float g)
{
    constexpr int NT = S::kNT;
    const int tid = topk_tid<NT>();
    const float ninf = __int_as_float(0xff800000u);
    if (!kWin) lo = 0;
    auto keep = [&](int i, float v) {
        if (v >= g && topk_eligible(v)) {
            const uint32_t at = atomicAdd(&s.n_tie, 1u);
            if (at < uint32_t(S::kTie)) s.tbuf[at] = topk_composite(topk_key(v), i);
        }
    };
    auto over = [&]() {
        return *reinterpret_cast<volatile uint32_t*>(&s.n_tie) > uint32_t(S::kTie);
    };
    if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0) {
        for (int c0 = lo; c0 < hi && !over(); c0 += NT) {
            const int i = c0 + tid;
            if (i < hi) keep(i, __ldg(x + i));
        }
        return;
    }
    constexpr int kChunk = 4 * kU * NT;
    auto load = [&](float4 (&v)[kU], int c0) {
        if ((!kWin || c0 >= lo) && c0 + kChunk <= hi) {
#pragma unroll
            for (int u = 0; u < kU; ++u)
                v[u] = __ldg(reinterpret_cast<const float4*>(x + c0 + 4 * (u * NT + tid)));
        } else {
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = c0 + 4 * (u * NT + tid);
                if (i >= lo && i + 3 < hi) {
                    v[u] = __ldg(reinterpret_cast<const float4*>(x + i));
                } else {
                    v[u].x = i >= lo && i < hi ? __ldg(x + i) : ninf;
                    v[u].y = i + 1 >= lo && i + 1 < hi ? __ldg(x + i + 1) : ninf;
                    v[u].z = i + 2 >= lo && i + 2 < hi ? __ldg(x + i + 2) : ninf;
                    v[u].w = i + 3 >= lo && i + 3 < hi ? __ldg(x + i + 3) : ninf;
                }
            }
        }
    };
    const int c_begin = lo & ~3;
    float4 v[kU], nv[kU];
    if (c_begin < hi) load(v, c_begin);
    for (int c0 = c_begin; c0 < hi && !over(); c0 += kChunk) {
        if (c0 + kChunk < hi) load(nv, c0 + kChunk);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const float mx = fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w));
            if (mx >= g) {
                // one slot claim for the lane's kept entries of this float4
                const int i = c0 + 4 * (u * NT + tid);
                const bool t0 = v[u].x >= g && topk_eligible(v[u].x);
                const bool t1 = v[u].y >= g && topk_eligible(v[u].y);
                const bool t2 = v[u].z >= g && topk_eligible(v[u].z);
                const bool t3 = v[u].w >= g && topk_eligible(v[u].w);
                const uint32_t n = uint32_t(t0) + uint32_t(t1) + uint32_t(t2) + uint32_t(t3);
                if (n != 0u) {
                    uint32_t at = atomicAdd(&s.n_tie, n);
                    auto put = [&](bool t, float f, int e) {
                        if (t) {
                            if (at < uint32_t(S::kTie)) s.tbuf[at] = topk_composite(topk_key(f), e);
                            ++at;
                        }
                    };
                    put(t0, v[u].x, i);
                    put(t1, v[u].y, i + 1);
                    put(t2, v[u].z, i + 2);
                    put(t3, v[u].w, i + 3);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) v[u] = nv[u];
    }
}

// kSBits: key bits of the sample's histogram (11: a quarter octave per bin; 12: an eighth).
template <typename S, bool kWin, int kSBits>
__global__ void __launch_bounds__(kTopkThreads, 1) topk_kernel(const TopkParams p)
{
    constexpr int NT = S::kNT;
    constexpr int kRowsPerCta = kTopkThreads / NT;
    extern __shared__ __align__(16) uint8_t topk_smem_raw[];
    const int slot = int(threadIdx.x) / NT;  // which of the CTA's rows this thread works on
    S& s = reinterpret_cast<S*>(topk_smem_raw)[slot];
    const int tid = topk_tid<NT>(), warp = tid >> 5;
    const int N = int(p.N);
    const int k = p.k;
    uint32_t* const my_hist = s.whist[warp % S::kHW];

    for (int64_t row = int64_t(blockIdx.x) * kRowsPerCta + slot; row < p.M;
         row += int64_t(gridDim.x) * kRowsPerCta) {
        const float* x = p.logits + row * p.ld;
        int lo = 0, hi = N;
        if (kWin) topk_window(p, row, lo, hi);

        // ---- 0. a threshold G from a sample of the window (8 of every 64 elements: one
        // 32-byte sector in eight, so the sample reads an eighth of the row), then one pass
        // that keeps the entries >= G in the buffer (the rest of the row is read once, here)
        if (tid == 0) {
            s.n_cand = 0;
            s.n_tie = 0;
        }
        // the sample's histogram over the top kSBits key bits; beyond 11 bits it takes the
        // per-warp histograms' space, free until the full select
        static_assert(kSBits == 11 || kSBits == 12, "sample histogram bits");
        static_assert(S::kHW * kTopkBins >= (1 << kSBits), "the sample histogram fits");
        constexpr uint32_t n_sb = 1u << kSBits;
        constexpr int s_shift = 32 - kSBits;
        uint32_t* const shist = kSBits == 11 ? s.hist : &s.whist[0][0];
        for (int b = tid; b < int(n_sb); b += NT) shist[b] = 0u;
        topk_sync<NT>();
        {
            const bool aligned = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
            for (int gi = (lo >> 6) + tid; gi < ((hi + 63) >> 6); gi += NT) {
                const int e = gi << 6;
                float v[8];
                if (aligned && e >= lo && e + 7 < hi) {
                    const float4 a = __ldg(reinterpret_cast<const float4*>(x + e));
                    const float4 c = __ldg(reinterpret_cast<const float4*>(x + e + 4));
                    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
                    v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        v[c] = e + c >= lo && e + c < hi ? __ldg(x + e + c) : __int_as_float(0xff800000u);
                }
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    if (topk_eligible(v[c])) atomicAdd(&shist[topk_key(v[c]) >> s_shift], 1u);
            }
        }
        topk_sync<NT>();
        // sampled keys needed above the threshold: an eighth of k plus about two standard
        // deviations of the sampled count
        const uint32_t r = (uint32_t(k) >> 3) + (uint32_t(k) >> 5) + 6u;
        const bool lowest = topk_find_bin(s, shist, n_sb, r) < r;
        float g = -3.402823466e38f;
        if (!lowest) {
            const uint32_t kt = s.sel_bin << s_shift;  // a finite key: non-finite bins were not counted
            g = __uint_as_float((kt & 0x80000000u) ? (kt & 0x7FFFFFFFu) : ~kt);
        }
        topk_keep_above<S, kWin, 4>(s, x, lo, hi, g);
        topk_sync<NT>();
        {
            // the next row's sample sectors go to L2 now, while this row's selection runs,
            // so that row's sample pass finds them there
            const int64_t nrow = row + int64_t(gridDim.x) * kRowsPerCta;
            if (nrow < p.M) {
                int nlo = 0, nhi = N;
                if (kWin) topk_window(p, nrow, nlo, nhi);
                const float* nx = p.logits + nrow * p.ld;
                for (int gi = (nlo >> 6) + tid; gi < ((nhi + 63) >> 6); gi += NT) {
                    const int e = max(gi << 6, nlo);
                    if (e < nhi) topk_prefetch_l2(nx + e);
                }
            }
        }
        const uint32_t n_kept = s.n_tie;
        const bool sampled = n_kept <= uint32_t(S::kTie) && (n_kept >= uint32_t(k) || lowest);
        if (sampled) {
            // the cut over the kept entries' composites, and the winners
            const int nc = int(n_kept);
            const unsigned long long cut =
                topk_reg_cut(s, uint32_t(k), topk_index_bytes(N), [&](auto&& fn) {
                    for (int i = tid; i < nc; i += NT) fn(s.tbuf[i]);
                });
            for (int i0 = 0; i0 < nc; i0 += NT) {
                const int i = i0 + tid;
                const unsigned long long c = i < nc ? s.tbuf[i] : 0ull;
                topk_append_capped(s.cand, &s.n_cand, c, c != 0ull && c >= cut, uint32_t(k));
            }
            topk_sync<NT>();
        } else {

        // ---- 1. top 11 key bits, one histogram per warp, then their sum
        if constexpr (S::kHW == NT / 32) {
            for (int b = tid & 31; b < kTopkBins; b += 32) my_hist[b] = 0;
            __syncwarp();
        } else {
            // warps share histograms: all of them are cleared before any warp counts
            for (int b = tid; b < S::kHW * kTopkBins; b += NT) (&s.whist[0][0])[b] = 0;
            topk_sync<NT>();
        }
        topk_for_row<NT, false, kWin>(x, lo, hi, [&](int, float v, bool valid) {
            const bool in = valid && topk_eligible(v);
            topk_hist_add(my_hist, in ? (topk_key(v) >> 21) : 0u, in);
        });
        topk_sync<NT>();
        for (int b = tid; b < kTopkBins; b += NT) {
            uint32_t h = 0;
#pragma unroll
            for (int w = 0; w < S::kHW; ++w) h += s.whist[w][b];
            s.hist[b] = h;
        }
        if (tid == 0) {
            s.n_cand = 0;
            s.n_tie = 0;
            s.tie_base = 0;
        }
        topk_sync<NT>();

        // ---- 2. the bin of the k-th largest
        const uint32_t total = topk_find_bin(s, s.hist, kTopkBins, uint32_t(k));
        const bool take_all = total <= uint32_t(k);
        const uint32_t b0 = s.sel_bin, above0 = s.sel_above, count0 = s.sel_count;
        const bool fast = take_all || above0 + count0 <= uint32_t(S::kTie);

        if (fast) {
            // ---- 3. one append per entry: every finite entry when all are winners, else
            // the entries of b0 and above into the buffer
            unsigned long long* const spare = reinterpret_cast<unsigned long long*>(&s.whist[0][0]);
            unsigned long long* const dst = take_all ? s.cand : s.tbuf;
            uint32_t* const cnt = take_all ? &s.n_cand : &s.n_tie;
            topk_for_row<NT, false, kWin>(x, lo, hi, [&](int i, float v, bool valid) {
                const bool in = valid && topk_eligible(v);
                const uint32_t key = in ? topk_key(v) : 0u;
                topk_append(dst, cnt, topk_composite(key, i), in && (take_all || (key >> 21) >= b0));
            });
            topk_sync<NT>();
            if (!take_all) {
                // split the buffer: entries above b0 are winners, those of b0 go to the
                // spare buffer (the per-warp histograms, free now), where the kk largest of
                // them are selected with ties by index
                const uint32_t n = s.n_tie;
                const uint32_t rounds = (n + NT - 1) / NT;
                if (tid == 0) s.n_spare = 0;
                topk_sync<NT>();
                for (uint32_t r = 0; r < rounds; ++r) {
                    const uint32_t j = r * NT + tid;
                    const unsigned long long c = j < n ? s.tbuf[j] : 0ull;
                    const uint32_t d = uint32_t(c >> 53);
                    topk_append(s.cand, &s.n_cand, c, j < n && d > b0);
                    topk_append(spare, &s.n_spare, c, j < n && d == b0);
                }
                topk_sync<NT>();
                topk_select_buffer(s, spare, s.tbuf, s.n_spare, uint32_t(k) - above0);
            }
        } else {
            // ---- 3'. b0 and the bins above hold more entries than the buffer: resolve the
            // other 21 key bits of b0 with two more histogram passes (11 and 10 bits)
            uint32_t prefix = b0 << 21, pmask = 0x7FFu << 21;
            uint32_t kk = uint32_t(k) - above0;
            uint32_t tie_total = count0;
            for (int pass = 1; pass < 3; ++pass) {
                const int shift = pass == 1 ? 10 : 0;
                const uint32_t nb = pass == 1 ? 2048u : 1024u;
                for (uint32_t b = tid; b < nb; b += NT) s.hist[b] = 0;
                topk_sync<NT>();
                topk_for_row<NT, false, kWin>(x, lo, hi, [&](int, float v, bool valid) {
                    bool in = valid && topk_eligible(v);
                    const uint32_t key = in ? topk_key(v) : 0u;
                    in = in && (key & pmask) == prefix;
                    topk_hist_add(s.hist, (key >> shift) & (nb - 1), in);
                });
                topk_sync<NT>();
                topk_find_bin(s, s.hist, nb, kk);
                kk -= s.sel_above;
                prefix |= s.sel_bin << shift;
                pmask |= (nb - 1) << shift;
                tie_total = s.sel_count;
                topk_sync<NT>();
            }
            const uint32_t T = prefix;  // the k-th largest key; kk of the entries equal to it
            const bool ordered_ties = kk < tie_total;
            auto collect = [&](int i, float v, bool valid) {
                const bool in = valid && topk_eligible(v);
                const uint32_t key = in ? topk_key(v) : 0u;
                const bool greater = in && key > T;
                const bool tie = in && key == T;
                bool take = greater || (tie && !ordered_ties);
                if (ordered_ties) {
                    // rank of this tie among the row's ties, in index order (the in-order
                    // visit gives one element per thread per call, threads in index order)
                    uint32_t step_ties = 0;
                    const uint32_t incl = topk_block_scan<NT>(tie ? 1u : 0u, s.scratch, step_ties);
                    const uint32_t rank = s.tie_base + incl - (tie ? 1u : 0u);
                    take = greater || (tie && rank < kk);
                    topk_sync<NT>();
                    if (tid == 0) s.tie_base += step_ties;
                }
                topk_append(s.cand, &s.n_cand, topk_composite(key, i), take);
            };
            if (ordered_ties)
                topk_for_row<NT, true, kWin>(x, lo, hi, collect);
            else
                topk_for_row<NT, false, kWin>(x, lo, hi, collect);
            topk_sync<NT>();
        }
        }  // the sample's threshold missed

        // ---- 4. order the winners and write the row
        const int n_sel = int(min(s.n_cand, uint32_t(k)));
        if (p.sorted)
            topk_sort_winners<NT>(s.cand, reinterpret_cast<unsigned long long*>(&s.whist[0][0]), n_sel);
        int32_t* oi = p.indices + row * int64_t(k);
        float* ov = p.values ? p.values + row * int64_t(k) : nullptr;
        for (int j = tid; j < k; j += NT) {
            int32_t idx = -1;
            float val = __int_as_float(0xff800000);
            if (j < n_sel) {
                const unsigned long long cv = s.cand[j];
                idx = int32_t(0xFFFFFFFFu - uint32_t(cv & 0xFFFFFFFFull));
                const uint32_t key = uint32_t(cv >> 32);
                if (key == 0x80000000u) {
                    // a zero: the key folded its sign away, so read it back (every composite
                    // carries an index below N; the guard keeps the read in bounds)
                    val = uint32_t(idx) < uint32_t(N) ? x[idx] : __int_as_float(0x7fc00000);
                } else {
                    // the key's inverse: the value itself, with no dependent global read
                    val = __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
                }
            }
            oi[j] = idx;
            if (ov) ov[j] = val;
        }
        topk_sync<NT>();
    }
}

// ---------------------------------------------------------------------------------------
// Rows of up to kTopkRegKeys keys and k <= kTopkRegMaxK: the row is staged in shared memory.
//
// Four rows per 512-thread CTA, 128 threads per row on a named barrier of their own.  A row
// arrives in shared memory by asynchronous copies (thread t copies elements 512 q + 4 t .. +3,
// q < 16: each warp's copy reads 512 contiguous bytes).  Per row:
//   1. A histogram of the top 11 key bits over every eighth element of the row gives a
//      threshold G a little below where the k-th largest key is expected.
//   2. One compare per key and a warp ballot mark the keys >= G (the candidates); the ballot
//      words give each candidate's slot, and the candidates' composites go to a buffer.
//   3. A radix select over the candidates' 64-bit composites (key, then index) finds the cut:
//      exactly min(k, eligible) composites are >= it.  The composites are unique, so the cut
//      resolves ties at the k-th value by index without a separate tie step.
//   4. The winners are sorted and written.
// When the threshold misses (fewer than k eligible candidates, or more than the buffer holds),
// step 3 runs over the whole staged row instead.  The next row's copies are issued as soon as
// the staged row is no longer read, so they land during the selection and the sort.
constexpr int kTopkRegThreads = 128;                  // threads per row
constexpr int kTopkRegRows = kTopkThreads / kTopkRegThreads;
constexpr int kTopkRegPerThread = 64;                 // keys per thread
constexpr int kTopkRegKeys = kTopkRegThreads * kTopkRegPerThread;  // 8192
constexpr int kTopkRegMaxK = 1024;
constexpr int kTopkRegCap = 2048;                     // candidate buffer (composites)

struct TopkRegSmem {
    static constexpr int kNT = kTopkRegThreads;
    float row[kTopkRegKeys];
    // the candidates; the winners' sort uses its first kTopkRegMaxK entries as scratch once
    // the candidates are spent
    unsigned long long cand[kTopkRegCap];
    // the winners; before them the same bytes hold the sample histogram, then the ballots,
    // then the cut's histograms
    union {
        unsigned long long win[kTopkRegMaxK];
        uint32_t hist[kTopkBins];
        uint32_t ballots[kTopkRegThreads / 32][kTopkRegPerThread];
    };
    uint32_t scratch[kTopkRegThreads / 32];
    uint32_t sel_bin, sel_above, sel_count, n_win, n_bad, pad[3];
};
static_assert(kTopkRegRows * sizeof(TopkRegSmem) <= 232448, "top-k shared memory");
static_assert(sizeof(TopkRegSmem) % 16 == 0, "row slices stay 16-byte aligned");
static_assert(kTopkRegMaxK <= kTopkRegCap, "the sort's scratch fits in the candidate buffer");

// The row element in key slot j of thread tid.
__device__ __forceinline__ int topk_reg_elem(int tid, int j)
{
    return 512 * (j >> 2) + 4 * tid + (j & 3);
}

// The 512-element chunks of a row that meet its window [lo, hi): [q_lo, q_hi).
__device__ __forceinline__ int topk_reg_qlo(int lo) { return lo >> 9; }
__device__ __forceinline__ int topk_reg_qhi(int lo, int hi) { return hi > lo ? (hi + 511) >> 9 : lo >> 9; }

// Start the asynchronous copy of a row's window [lo, hi) to `dst`: the chunks that meet the
// window, with -inf in their slots outside it (chunks outside the window are left as they
// are and never read).  16-byte copies where a slot group lies inside the window and the row
// is 16-byte aligned, else 4-byte ones.
// kWin = false: the window is the whole row [0, hi), and every chunk is written.
template <bool kWin>
__device__ __forceinline__ void topk_reg_stage(float* dst, const float* x, int lo, int hi, int tid)
{
    const bool aligned = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
    if (!kWin) lo = 0;
    const int q_lo = topk_reg_qlo(lo), q_hi = topk_reg_qhi(lo, hi);
#pragma unroll 4
    for (int q = 0; q < kTopkRegPerThread / 4; ++q) {
        if (kWin && (q < q_lo || q >= q_hi)) continue;
        const int e = topk_reg_elem(tid, 4 * q);
        const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst + e));
        if (aligned && (!kWin || e >= lo) && e + 3 < hi) {
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(x + e)
                         : "memory");
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if ((!kWin || e + c >= lo) && e + c < hi)
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d + 4u * c),
                                 "l"(x + e + c)
                                 : "memory");
                else
                    dst[e + c] = __int_as_float(0xff800000u);
            }
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait for this thread's staged copies (a hardware wait: no spin).
__device__ __forceinline__ void topk_reg_stage_wait()
{
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

template <bool kWin>
__global__ void __launch_bounds__(kTopkThreads, 1) topk_reg_kernel(const TopkParams p)
{
    constexpr int NT = kTopkRegThreads;
    constexpr int E = kTopkRegPerThread;
    extern __shared__ __align__(16) uint8_t topk_smem_raw[];
    const int slot = int(threadIdx.x) / NT;
    TopkRegSmem& s = reinterpret_cast<TopkRegSmem*>(topk_smem_raw)[slot];
    const int tid = topk_tid<NT>();
    const int lane = tid & 31, warp = tid >> 5;
    const int N = int(p.N);
    const uint32_t k = uint32_t(p.k);
    const int64_t row_step = int64_t(gridDim.x) * kTopkRegRows;
    // sampled keys needed above the threshold: an eighth of k plus a margin of about two
    // standard deviations of the sampled count
    const uint32_t r = (k >> 3) + (k >> 5) + 6u;

    int64_t row = int64_t(blockIdx.x) * kTopkRegRows + slot;
    int lo = 0, hi = N;  // the row's window
    if (row < p.M) {
        if (kWin) topk_window(p, row, lo, hi);
        topk_reg_stage<kWin>(s.row, p.logits + row * p.ld, lo, hi, tid);
    }
    for (; row < p.M; row += row_step) {
        const float* x = p.logits + row * p.ld;
        const int q_lo = topk_reg_qlo(lo), q_hi = topk_reg_qhi(lo, hi);
        for (int b = tid; b < kTopkBins; b += NT) s.hist[b] = 0u;
        if (tid == 0) {
            s.n_win = 0u;
            s.n_bad = 0u;
        }
        topk_reg_stage_wait();
        topk_sync<NT>();  // the staged row and the cleared histogram, for every thread

        // ---- 1. the threshold G from the sampled keys: every eighth element, so any window
        // of the row is sampled evenly
#pragma unroll
        for (int i = 0; i < kTopkRegKeys / (8 * NT); ++i) {
            const int e = 8 * (tid + NT * i);
            const float f = !kWin || (e >= lo && e < hi) ? s.row[e] : __int_as_float(0xff800000u);
            if (topk_eligible(f)) atomicAdd(&s.hist[topk_key(f) >> 21], 1u);
        }
        topk_sync<NT>();
        const uint32_t sampled = topk_find_bin(s, s.hist, uint32_t(kTopkBins), r);
        const bool lowest = sampled < r;  // few eligible keys: every one is a candidate
        float g = -3.402823466e38f;
        if (!lowest) {
            // the lowest value of the selected bin (finite: bins below 4 hold only -inf and
            // -NaN, and those keys were not counted)
            const uint32_t kt = s.sel_bin << 21;
            g = __uint_as_float((kt & 0x80000000u) ? (kt & 0x7FFFFFFFu) : ~kt);
        }
        topk_sync<NT>();  // the histogram's bytes become the ballots

        // ---- 2. candidates: one ballot per key slot (+inf passes the compare and is dropped
        // below; NaN and -inf fail it)
#pragma unroll
        for (int q = 0; q < E / 4; ++q) {
            if (kWin && (q < q_lo || q >= q_hi)) {  // outside the window: no candidates
                if (lane == 0)
                    *reinterpret_cast<uint4*>(&s.ballots[warp][4 * q]) = make_uint4(0u, 0u, 0u, 0u);
                continue;
            }
            const float4 f = *reinterpret_cast<const float4*>(&s.row[topk_reg_elem(tid, 4 * q)]);
            const uint32_t m0 = __ballot_sync(0xffffffffu, f.x >= g);
            const uint32_t m1 = __ballot_sync(0xffffffffu, f.y >= g);
            const uint32_t m2 = __ballot_sync(0xffffffffu, f.z >= g);
            const uint32_t m3 = __ballot_sync(0xffffffffu, f.w >= g);
            if (lane == 0)
                *reinterpret_cast<uint4*>(&s.ballots[warp][4 * q]) = make_uint4(m0, m1, m2, m3);
        }
        __syncwarp();
        const uint32_t b0 = s.ballots[warp][lane], b1 = s.ballots[warp][lane + 32];
        const uint32_t n_mine = uint32_t(__popc(b0) + __popc(b1));
        uint32_t n_cand = 0;
        uint32_t pos = topk_block_scan<NT>(n_mine, s.scratch, n_cand) - n_mine;
        bool fast = n_cand <= uint32_t(kTopkRegCap) && (n_cand >= k || lowest);

        unsigned long long cut = 1ull;
        if (fast) {
            // this lane writes the candidates of key slots `lane` and `lane + 32` of its
            // warp: bit b of a slot's ballot is that slot's element in lane b
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = lane + 32 * h;
                uint32_t bits = h ? b1 : b0;
                while (bits) {
                    const int b = __ffs(bits) - 1;
                    bits &= bits - 1u;
                    const int i = topk_reg_elem(32 * warp + b, j);
                    const unsigned long long c = topk_reg_comp(s.row[i], i);
                    if (c == 0ull) atomicAdd(&s.n_bad, 1u);  // +inf
                    s.cand[pos++] = c;
                }
            }
            topk_sync<NT>();
            // a threshold above the k-th eligible key (the candidates held +inf entries)
            if (!lowest && n_cand - s.n_bad < k) fast = false;
        }
        if (!fast) {
            // the threshold missed: select over the whole staged window
            cut = topk_reg_cut(s, k, 2, [&](auto&& fn) {  // rows of at most 8192 keys
                for (int i = lo + tid; i < hi; i += NT) fn(topk_reg_comp(s.row[i], i));
            });
            for (int i0 = lo; i0 < hi; i0 += NT) {
                const int i = i0 + tid;
                const unsigned long long c = i < hi ? topk_reg_comp(s.row[i], i) : 0ull;
                topk_append_capped(s.win, &s.n_win, c, c != 0ull && c >= cut, k);
            }
        }
        topk_sync<NT>();  // every read of the staged row is done

        // ---- the next row's copies go out now
        const int64_t next = row + row_step;
        int next_lo = 0, next_hi = N;
        if (next < p.M) {
            if (kWin) topk_window(p, next, next_lo, next_hi);
            topk_reg_stage<kWin>(s.row, p.logits + next * p.ld, next_lo, next_hi, tid);
        }

        // ---- 3. the cut over the candidates, and the winners
        if (fast) {
            const int nc = int(n_cand);
            cut = topk_reg_cut(s, k, 2, [&](auto&& fn) {
                for (int i = tid; i < nc; i += NT) fn(s.cand[i]);
            });
            for (int i0 = 0; i0 < nc; i0 += NT) {
                const int i = i0 + tid;
                const unsigned long long c = i < nc ? s.cand[i] : 0ull;
                topk_append_capped(s.win, &s.n_win, c, c != 0ull && c >= cut, k);
            }
            topk_sync<NT>();
        }
        const int n_sel = int(min(s.n_win, k));

        // ---- 4. order the winners and write the row
        if (p.sorted) topk_sort_winners<NT>(s.win, s.cand, n_sel);
        int32_t* oi = p.indices + row * int64_t(k);
        float* ov = p.values ? p.values + row * int64_t(k) : nullptr;
        for (int j = tid; j < int(k); j += NT) {
            int32_t idx = -1;
            float val = __int_as_float(0xff800000);
            if (j < n_sel) {
                const unsigned long long cv = s.win[j];
                idx = int32_t(0xFFFFFFFFu - uint32_t(cv & 0xFFFFFFFFull));
                const uint32_t kj = uint32_t(cv >> 32);
                if (kj == 0x80000000u) {
                    // a zero: the key folded its sign away, so read it back (the guard keeps
                    // the read in bounds)
                    val = uint32_t(idx) < uint32_t(N) ? x[idx] : __int_as_float(0x7fc00000);
                } else {
                    val = __uint_as_float((kj & 0x80000000u) ? (kj & 0x7FFFFFFFu) : ~kj);
                }
            }
            oi[j] = idx;
            if (ov) ov[j] = val;
        }
        topk_sync<NT>();
        lo = next_lo;
        hi = next_hi;
    }
}

}  // namespace fp8mqa
