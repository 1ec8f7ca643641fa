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

__global__ void __launch_bounds__(kTopkThreads)
    topk_kernel(const float* __restrict__ scores, const int32_t* __restrict__ start_pos, int s, int n_cols,
                int ratio, int k, int32_t offset, int32_t* __restrict__ idxs, int64_t row_stride, int use_smem) {
    extern __shared__ uint32_t sm[];
    uint32_t* hist = sm;                                      // [kBins]
    int* warp_tot = reinterpret_cast<int*>(sm + kBins);       // [kWarps]
    int* misc = warp_tot + kWarps;                            // [8]
    uint32_t* keys = sm + kBins + kWarps + 8;                 // [vis] when staged

    const int row = blockIdx.x;
    const int b = row / s, t = row - b * s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int vis = (__ldg(start_pos + b) + t + 1) / ratio;
    vis = max(0, min(vis, n_cols));
    int32_t* out = idxs + (int64_t)row * row_stride;

    if (vis <= k) {  // every visible position is selected
        for (int i = tid; i < k; i += kTopkThreads) out[i] = i < vis ? i + offset : -1;
        return;
    }

    const float* src = scores + (int64_t)row * n_cols;
    if (use_smem) {
        for (int j = tid; j < vis; j += kTopkThreads) keys[j] = float_key(__ldg(src + j));
        __syncthreads();
    }
    auto key_at = [&](int j) -> uint32_t { return use_smem ? keys[j] : float_key(__ldg(src + j)); };

    uint32_t prefix = 0;
    int remaining = k;   // how many still to take at or below the current prefix
    int shift = 32;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int bits = pass < 2 ? 11 : 10;
        const int hi_shift = shift;   // bits above the digit are already fixed in `prefix`
        shift -= bits;
        const uint32_t mask = (1u << bits) - 1u;
        for (int i = tid; i < kBins; i += kTopkThreads) hist[i] = 0;
        __syncthreads();
        for (int base = 0; base < vis; base += kTopkThreads) {
            const int j = base + tid;
            bool m = false;
            uint32_t dig = 0xFFFFFFFFu;
            if (j < vis) {
                const uint32_t key = key_at(j);
                m = hi_shift >= 32 ? true : ((key >> hi_shift) == prefix);
                if (m) dig = (key >> shift) & mask;
            }
            const unsigned peers = __match_any_sync(kFull, dig);
            if (m && lane == __ffs(peers) - 1) atomicAdd(&hist[dig], (uint32_t)__popc(peers));
        }
        __syncthreads();
        // bins owned by this thread: 4*tid .. 4*tid+3; entries above them = total - inclusive
        int local = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) local += (int)hist[4 * tid + i];
        int total;
        const int excl = block_excl_scan(local, warp_tot, total);
        int above = total - excl - local;
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
        const int dstar = misc[0];
        remaining -= misc[1];
        prefix = (prefix << bits) | (uint32_t)dstar;
        __syncthreads();
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
        if (take) out[pos + __popc(take_mask & ((1u << lane) - 1u))] = j + offset;
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

cudaError_t launch_topk(const float* scores, const int32_t* start_pos, int B, int s, int n_cols, int ratio, int k,
                        int32_t offset, int32_t* idxs, int64_t row_stride, uint32_t* /*status*/,
                        cudaStream_t stream) {
    const int rows = B * s;
    if (rows == 0) return cudaSuccess;
    const int use_smem = n_cols <= kSmemKeyCap ? 1 : 0;
    const size_t smem = (size_t)(kBins + kWarps + 8 + (use_smem ? n_cols : 0)) * 4;
    cudaError_t err = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    topk_kernel<<<rows, kTopkThreads, smem, stream>>>(scores, start_pos, s, n_cols, ratio, k, offset, idxs,
                                                       row_stride, use_smem);
    return cudaGetLastError();
}

}  // namespace sti
