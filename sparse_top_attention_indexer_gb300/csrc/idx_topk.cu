// idx_topk.cu -- sliding-window indices and the Indexer's top-k selection.
//
// DeepSeek V4.1, attention "attend/selected" page:
//   get_window_topk_idxs   which window-KV rows each query sees (prefill band / decode ring)
//   Indexer.forward        topk = min(index_topk, visible); indices re-sorted into position
//                          order; unreachable -> -1, the rest shifted by offset
//
// Top-k is a radix select, never a sort of the row: scores become order-preserving 32-bit keys,
// three histogram passes (11, 11 and 10 bits, warp-aggregated shared-memory atomics) find the
// exact key tau of the k-th largest visible score, and one ordered compaction emits every
// position with key > tau plus the lowest-positioned keys == tau until k are taken -- already
// in ascending position order, which is the order the page's `.sort()` produces.
#include <cuda_runtime.h>

#include "sti_internal.h"
#include "sti_ptx.cuh"

namespace sti {
namespace {

constexpr int kTopkThreads = 512;
constexpr int kWarps = kTopkThreads / 32;
constexpr int kBins = 2048;
constexpr int kSmemKeyCap = 32768;   // rows up to this many visible positions are staged in shared memory
constexpr int kCandCap = 4096;       // threshold-bin members kept for passes 2 and 3
constexpr uint32_t kFull = 0xFFFFFFFFu;

__global__ void window_idx_kernel(const int32_t* __restrict__ start_pos, int B, int s, int W, int width,
                                  int32_t* __restrict__ idxs, int64_t row_stride, uint32_t* status) {
    const int64_t total = (int64_t)B * s * width;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = e / width;
        const int i = (int)(e - row * width);
        const int b = (int)(row / s), t = (int)(row - (int64_t)b * s);
        const int sp = __ldg(start_pos + b);
        int v;
        if (s > 1) {
            // prefill band: starts at max(0, t-W+1); slots past t hold nothing
            if (sp != 0) {
                if (i == 0 && status) atomicOr(status, 4u /* STI_FLAG_CHUNKED */);
                v = -1;
            } else {
                const int idx = max(0, t - W + 1) + i;
                v = idx > t ? -1 : idx;
            }
        } else {
            // decode ring, oldest first: slots (sp%W)+1 .. W-1, then 0 .. sp%W
            const int oldest = sp % W + 1;
            const int idx = i < W - oldest ? oldest + i : i - (W - oldest);
            v = idx > sp ? -1 : idx;
        }
        idxs[row * row_stride + i] = v;
    }
}

// Block-wide exclusive prefix sum over the 512 threads; also returns the total.
__device__ __forceinline__ int block_excl_scan(int v, int* warp_tot, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += x;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    int wpre = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const int x = warp_tot[w];
        wpre += w < warp ? x : 0;
        tot += x;
    }
    __syncthreads();
    total = tot;
    return wpre + inc - v;
}

// Value of window slot i for query (b, t) (get_window_topk_idxs): prefill band when s > 1,
// decode ring otherwise; -1 for slots that hold nothing.
__device__ __forceinline__ int window_slot(int s, int t, int sp, int W, int i) {
    if (s > 1) {
        const int idx = max(0, t - W + 1) + i;
        return (sp != 0 || idx > t) ? -1 : idx;
    }
    const int oldest = sp % W + 1;
    const int idx = i < W - oldest ? oldest + i : i - (W - oldest);
    return idx > sp ? -1 : idx;
}

// Histogram of digit (key >> shift) & mask over the n keys from `src` whose bits above
// hi_shift equal `prefix`, then the bin d* where the count from the top first reaches
// `remaining`: returns d* and the number of matching keys in higher bins (via *above).
template <typename Src>
__device__ __forceinline__ int radix_pass(Src src, int n, int hi_shift, int shift, int bits, uint32_t prefix,
                                          int remaining, uint32_t* hist, int* warp_tot, int* misc, int* above_out,
                                          bool hist_ready) {
    const int tid = threadIdx.x, lane = tid & 31;
    const uint32_t mask = (1u << bits) - 1u;
    if (!hist_ready) {
        for (int i = tid; i < kBins; i += kTopkThreads) hist[i] = 0;
        __syncthreads();
        for (int base = 0; base < n; base += kTopkThreads) {
            const int j = base + tid;
            bool m = false;
            uint32_t dig = 0xFFFFFFFFu;
            if (j < n) {
                const uint32_t key = src(j);
                m = hi_shift >= 32 ? true : ((key >> hi_shift) == prefix);
                if (m) dig = (key >> shift) & mask;
            }
            const unsigned peers = __match_any_sync(kFull, dig);
            if (m && lane == __ffs(peers) - 1) atomicAdd(&hist[dig], (uint32_t)__popc(peers));
        }
        __syncthreads();
    }
    int local = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) local += (int)hist[4 * tid + i];
    int total;
    const int excl = block_excl_scan(local, warp_tot, total);
    int above = total - excl - local;   // matching keys in bins above this thread's 4 bins
#pragma unroll
    for (int i = 3; i >= 0; --i) {
        const int bin = 4 * tid + i;
        const int c = (int)hist[bin];
        if (above < remaining && above + c >= remaining) {
            misc[0] = bin;
            misc[1] = above;
        }
        above += c;
    }
    __syncthreads();
    const int d = misc[0];
    *above_out = misc[1];
    __syncthreads();
    return d;
}

template <bool HAS_HIST>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const TopkParams p, int use_smem) {
    extern __shared__ uint32_t sm[];
    uint32_t* hist = sm;                                      // [kBins]
    int* warp_tot = reinterpret_cast<int*>(sm + kBins);       // [kWarps]
    int* misc = warp_tot + kWarps;                            // [8]
    uint32_t* cand = sm + kBins + kWarps + 8;                 // [kCandCap] keys of the threshold bin
    uint32_t* keys = cand + kCandCap;                         // [vis] when staged

    const int row = blockIdx.x;
    const int b = row / p.s, t = row - b * p.s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sp = __ldg(p.start_pos + b);
    if (p.win_out != nullptr) {
        int32_t* wrow = p.win_out + (int64_t)row * p.row_stride;
        for (int i = tid; i < p.win_width; i += kTopkThreads) wrow[i] = window_slot(p.s, t, sp, p.win_W, i);
        if (tid == 0 && p.s > 1 && sp != 0 && p.status) atomicOr(p.status, 4u /* STI_FLAG_CHUNKED */);
    }
    int vis = (sp + t + 1) / p.ratio;
    vis = max(0, min(vis, p.n_cols));
    int32_t* out = p.idxs + (int64_t)row * p.row_stride;
    uint32_t* ghist = HAS_HIST ? p.hist + (size_t)row * kBins : nullptr;

    if (vis <= p.k) {  // every visible position is selected
        for (int i = tid; i < p.k; i += kTopkThreads) out[i] = i < vis ? i + p.offset : -1;
        if (HAS_HIST)
            for (int i = tid; i < kBins; i += kTopkThreads) ghist[i] = 0;
        return;
    }

    const float* src = p.scores + (int64_t)row * p.n_cols;
    if (use_smem) {
        for (int j = tid; j < vis; j += kTopkThreads) keys[j] = float_key(__ldg(src + j));
    }
    if (HAS_HIST) {
        for (int i = tid; i < kBins; i += kTopkThreads) {
            hist[i] = ghist[i];
            ghist[i] = 0;   // ready for the next call
        }
    }
    __syncthreads();
    auto key_at = [&](int j) -> uint32_t { return use_smem ? keys[j] : float_key(__ldg(src + j)); };

    // pass 1: top 11 bits over the whole row (histogram precomputed by the scores kernel, or here)
    int above;
    const int d1 = radix_pass(key_at, vis, 32, 21, 11, 0u, p.k, hist, warp_tot, misc, &above, HAS_HIST);
    int remaining = p.k - above;
    uint32_t prefix = (uint32_t)d1;
    const int c1 = (int)hist[d1];
    __syncthreads();
    if (c1 <= kCandCap) {
        // passes 2 and 3 only look at the keys of bin d1: gather them first
        if (tid == 0) misc[2] = 0;
        __syncthreads();
        for (int base = 0; base < vis; base += kTopkThreads) {
            const int j = base + tid;
            const uint32_t key = j < vis ? key_at(j) : 0u;
            const bool m = j < vis && (key >> 21) == (uint32_t)d1;
            const unsigned bal = __ballot_sync(kFull, m);
            int wbase = 0;
            if (lane == 0 && bal) wbase = atomicAdd(&misc[2], __popc(bal));
            wbase = __shfl_sync(kFull, wbase, 0);
            const int at = wbase + __popc(bal & ((1u << lane) - 1u));
            if (m && at < kCandCap) cand[at] = key;
        }
        __syncthreads();
    }
    if (c1 <= kCandCap && misc[2] == c1) {
        auto cand_at = [&](int j) -> uint32_t { return cand[j]; };
        const int d2 = radix_pass(cand_at, c1, 21, 10, 11, prefix, remaining, hist, warp_tot, misc, &above, false);
        remaining -= above;
        prefix = (prefix << 11) | (uint32_t)d2;
        const int d3 = radix_pass(cand_at, c1, 10, 0, 10, prefix, remaining, hist, warp_tot, misc, &above, false);
        remaining -= above;
        prefix = (prefix << 10) | (uint32_t)d3;
    } else {
        const int d2 = radix_pass(key_at, vis, 21, 10, 11, prefix, remaining, hist, warp_tot, misc, &above, false);
        remaining -= above;
        prefix = (prefix << 11) | (uint32_t)d2;
        const int d3 = radix_pass(key_at, vis, 10, 0, 10, prefix, remaining, hist, warp_tot, misc, &above, false);
        remaining -= above;
        prefix = (prefix << 10) | (uint32_t)d3;
    }
    const uint32_t tau = prefix;
    const int need_eq = remaining;   // >= 1 keys equal to tau are taken, lowest positions first

    // ordered compaction: warp w owns the contiguous segment [w*seg, (w+1)*seg)
    const int seg = ((vis + kWarps - 1) / kWarps + 31) & ~31;
    const int lo = min(vis, warp * seg), hi = min(vis, lo + seg);
    int n_gt = 0, n_eq = 0;
    for (int j0 = lo; j0 < hi; j0 += 32) {
        const int j = j0 + lane;
        const uint32_t key = j < hi ? key_at(j) : 0u;
        n_gt += __popc(__ballot_sync(kFull, j < hi && key > tau));
        n_eq += __popc(__ballot_sync(kFull, j < hi && key == tau));
    }
    if (lane == 0) warp_tot[warp] = n_eq;
    __syncthreads();
    int eq_before = 0;
    for (int w = 0; w < warp; ++w) eq_before += warp_tot[w];
    const int eq_take = max(0, min(n_eq, need_eq - eq_before));
    __syncthreads();
    if (lane == 0) warp_tot[warp] = n_gt + eq_take;
    __syncthreads();
    int pos = 0;
    for (int w = 0; w < warp; ++w) pos += warp_tot[w];
    int eq_seen = 0;
    for (int j0 = lo; j0 < hi; j0 += 32) {
        const int j = j0 + lane;
        const uint32_t key = j < hi ? key_at(j) : 0u;
        const bool gt = j < hi && key > tau;
        const bool eq = j < hi && key == tau;
        const unsigned eq_mask = __ballot_sync(kFull, eq);
        const int eq_rank = eq_seen + __popc(eq_mask & ((1u << lane) - 1u));
        const bool take = gt || (eq && eq_rank < eq_take);
        const unsigned take_mask = __ballot_sync(kFull, take);
        const int at = pos + __popc(take_mask & ((1u << lane) - 1u));
        if (take && at < p.k) out[at] = j + p.offset;
        pos += __popc(take_mask);
        eq_seen += __popc(eq_mask);
    }
    // vis > k here, so exactly k entries were written; nothing to pad
}

}  // namespace

cudaError_t launch_window_idxs(const int32_t* start_pos, int B, int s, int W, int width, int32_t* idxs,
                               int64_t row_stride, uint32_t* status, cudaStream_t stream) {
    const int64_t total = (int64_t)B * s * width;
    if (total == 0) return cudaSuccess;
    int blocks = (int)((total + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    window_idx_kernel<<<blocks, 256, 0, stream>>>(start_pos, B, s, W, width, idxs, row_stride, status);
    return cudaGetLastError();
}

cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream) {
    const int rows = p.B * p.s;
    if (rows == 0) return cudaSuccess;
    const int use_smem = p.n_cols <= kSmemKeyCap ? 1 : 0;
    const size_t smem = (size_t)(kBins + kWarps + 8 + kCandCap + (use_smem ? p.n_cols : 0)) * 4;
    auto kern = p.hist != nullptr ? topk_kernel<true> : topk_kernel<false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    kern<<<rows, kTopkThreads, smem, stream>>>(p, use_smem);
    return cudaGetLastError();
}

}  // namespace sti
