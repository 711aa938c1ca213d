// Per-row top-k over indexer logits for GB300 (sm_103a): the step that consumes the logits
// (ROCm/aiter PR #7183 "[HIP] [JIT] Add gfx950 prefill FP8 MQA logits", "Test plan":
// top-512 selections; ROCm/aiter PR #6159 "[Triton/Gluon] GFX950 sparse mla optimizations",
// "Technical Details": sparse MLA with top-k 512).
//
// For every row: the k largest finite logits (-inf, outside the row's window, is never
// selected), ordered by value descending and, for equal values, by index ascending (-0.0
// equals +0.0); slots past the row's finite entries get index -1 and value -inf.
//
// One CTA per row at a time (persistent grid of one CTA per SM, so a row's re-reads come
// from L2).  Radix select on an order-preserving 32-bit key: three histogram passes of
// 11, 11 and 10 bits find the exact k-th key T and how many of the entries equal to T are
// taken; a collect pass gathers the entries above T and, in index order, the needed ties;
// a bitonic sort in shared memory orders the (at most 2048) winners.
#pragma once

#include <cstdint>

namespace fp8mqa {

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkMaxK = 2048;
constexpr int kTopkBins = 2048;  // 11-bit digits

struct TopkParams {
    const float* logits;
    int64_t M, N, ld;  // row m at logits + m * ld
    int32_t k;
    int32_t* indices;  // [M, k]
    float* values;     // [M, k] or null
};

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

// Block-wide inclusive sum over threads in index order; `scratch` holds kTopkWarps words.
__device__ __forceinline__ uint32_t topk_block_scan(uint32_t v, uint32_t* scratch, uint32_t& total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) scratch[warp] = v;
    __syncthreads();
    uint32_t before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < kTopkWarps; ++w) {
        const uint32_t s = scratch[w];
        if (w < warp) before += s;
        total += s;
    }
    __syncthreads();
    return v + before;
}

__global__ void __launch_bounds__(kTopkThreads, 1) topk_kernel(const TopkParams p)
{
    __shared__ uint32_t hist[kTopkBins];
    __shared__ unsigned long long cand[kTopkMaxK];
    __shared__ uint32_t scratch[kTopkWarps];
    __shared__ uint32_t sel_bin, sel_above, n_cand, tie_base;

    const int tid = threadIdx.x, lane = tid & 31;
    const int N = int(p.N);
    const int k = p.k;

    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
        const float* x = p.logits + row * p.ld;

        // ---- radix select: find the k-th largest key T and how many entries equal to T
        uint32_t prefix = 0, pmask = 0;
        int kk = k;              // entries still to take among those matching the prefix
        uint32_t tie_total = 0;  // entries equal to T
        bool take_all = false;   // fewer than k eligible entries: take every one
        for (int pass = 0; pass < 3; ++pass) {
            const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
            const int width = pass < 2 ? 11 : 10;
            const uint32_t nb = 1u << width;
            for (uint32_t b = tid; b < nb; b += kTopkThreads) hist[b] = 0;
            __syncthreads();
            // a trip count uniform over the block, so the warp votes below see every lane
            for (int c0 = 0; c0 < N; c0 += kTopkThreads) {
                const int i = c0 + tid;
                const float v = i < N ? x[i] : __int_as_float(0xff800000);
                bool in = topk_eligible(v);
                uint32_t bin = 0;
                if (in) {
                    const uint32_t key = topk_key(v);
                    in = (key & pmask) == prefix;
                    bin = (key >> shift) & (nb - 1);
                }
                // one shared-memory atomic per distinct bin in the warp
                const uint32_t act = __ballot_sync(0xffffffffu, in);
                if (in) {
                    const uint32_t peers = __match_any_sync(act, bin);
                    if (lane == __ffs(peers) - 1) atomicAdd(&hist[bin], uint32_t(__popc(peers)));
                }
            }
            __syncthreads();
            // the bin holding the kk-th largest, scanning from the top: each thread owns a
            // run of nb / kTopkThreads bins, highest bins at thread 0
            const int per = int(nb) / kTopkThreads;
            uint32_t run = 0;
            for (int j = 0; j < per; ++j) run += hist[nb - 1 - (tid * per + j)];
            uint32_t total = 0;
            const uint32_t incl = topk_block_scan(run, scratch, total);
            if (pass == 0 && total <= uint32_t(k)) {
                take_all = true;
                break;
            }
            const uint32_t excl = incl - run;
            if (excl < uint32_t(kk) && incl >= uint32_t(kk)) {
                uint32_t above = excl;
                for (int j = 0; j < per; ++j) {
                    const uint32_t b = nb - 1 - (tid * per + j);
                    const uint32_t h = hist[b];
                    if (above + h >= uint32_t(kk)) {
                        sel_bin = b;
                        sel_above = above;
                        tie_base = h;
                        break;
                    }
                    above += h;
                }
            }
            __syncthreads();
            kk -= int(sel_above);
            prefix |= sel_bin << shift;
            pmask |= (nb - 1) << shift;
            tie_total = tie_base;
            __syncthreads();
        }
        const uint32_t T = prefix;
        // ties need index order only when the cut falls inside them
        const bool ordered_ties = !take_all && uint32_t(kk) < tie_total;

        // ---- collect the winners (unordered), ties in index order when needed
        if (tid == 0) {
            n_cand = 0;
            tie_base = 0;
        }
        __syncthreads();
        for (int c0 = 0; c0 < N; c0 += kTopkThreads) {
            const int i = c0 + tid;
            bool greater = false, tie = false;
            uint32_t key = 0;
            if (i < N) {
                const float v = x[i];
                if (topk_eligible(v)) {
                    key = topk_key(v);
                    greater = take_all || key > T;
                    tie = !take_all && key == T;
                }
            }
            bool take = greater || (tie && !ordered_ties);
            if (ordered_ties) {
                // rank of this tie among all ties of the row, in index order
                uint32_t chunk_ties = 0;
                const uint32_t incl = topk_block_scan(tie ? 1u : 0u, scratch, chunk_ties);
                const uint32_t rank = tie_base + incl - (tie ? 1u : 0u);
                take = greater || (tie && rank < uint32_t(kk));
                __syncthreads();
                if (tid == 0) tie_base += chunk_ties;
            }
            if (take) {
                const uint32_t slot = atomicAdd(&n_cand, 1u);
                cand[slot] = (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - uint32_t(i));
            }
        }
        __syncthreads();
        const int n_sel = int(n_cand);

        // ---- bitonic sort, descending on (key, -index)
        int P = 1;
        while (P < n_sel) P <<= 1;
        for (int i = n_sel + tid; i < P; i += kTopkThreads) cand[i] = 0ull;
        __syncthreads();
        for (int size = 2; size <= P; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int t = tid; t < P / 2; t += kTopkThreads) {
                    const int lo = (t / stride) * stride * 2 + (t % stride);
                    const int hi = lo + stride;
                    const bool desc = (lo & size) == 0;
                    const unsigned long long a = cand[lo], b = cand[hi];
                    if ((a < b) == desc) {
                        cand[lo] = b;
                        cand[hi] = a;
                    }
                }
                __syncthreads();
            }
        }

        // ---- write the row
        int32_t* oi = p.indices + row * int64_t(k);
        float* ov = p.values ? p.values + row * int64_t(k) : nullptr;
        for (int j = tid; j < k; j += kTopkThreads) {
            int32_t idx = -1;
            float val = __int_as_float(0xff800000);
            if (j < n_sel) {
                idx = int32_t(0xFFFFFFFFu - uint32_t(cand[j] & 0xFFFFFFFFull));
                val = x[idx];
            }
            oi[j] = idx;
            if (ov) ov[j] = val;
        }
        __syncthreads();
    }
}

}  // namespace fp8mqa
