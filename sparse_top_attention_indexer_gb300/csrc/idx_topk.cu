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
                                  int32_t* __restrict__ idxs, int64_t row_stride, uint32_t* status, int chunked) {
    const int64_t total = (int64_t)B * s * width;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = e / width;
        const int i = (int)(e - row * width);
        const int b = (int)(row / s), t = (int)(row - (int64_t)b * s);
        const int sp = __ldg(start_pos + b);
        int v;
        if (chunked) {
            // a chunk continuing its sequence: the prefill band at position P = sp + t over the
            // source [ring before the chunk (W rows) ; the chunk's rows]; position p lives in
            // chunk row W + (p - sp) or, before the chunk, in ring slot p % W
            const int P = sp + t;
            const int p = max(0, P - W + 1) + i;
            v = p > P ? -1 : (p >= sp ? W + (p - sp) : p % W);
        } else if (s > 1) {
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
    griddep_launch_dependents();
    const int sp = __ldg(p.start_pos + b);
    if (p.win_out != nullptr) {
        int32_t* wrow = p.win_out + (int64_t)row * p.row_stride;
        for (int i = tid; i < p.win_width; i += kTopkThreads) wrow[i] = window_slot(p.s, t, sp, p.win_W, i);
        if (tid == 0 && p.s > 1 && sp != 0 && p.status) atomicOr(p.status, 4u /* STI_FLAG_CHUNKED */);
    }
    griddep_wait();   // the scores (and histogram) are complete from here on
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

// ---------------------------------------------------------------------------------------------
// Warp top-k for rows of at most 2048 columns (prefill): one warp per row, its 64 keys a lane in
// registers (lane l holds positions 32 i + l), a first radix pass over the top 11 bits into the
// warp's own 2048-bin histogram, the threshold bin's keys listed and three passes of 7 bits over
// them, then the ordered compaction by ballots -- no block barrier anywhere, so the many short
// rows of a prefill are not bound by block-wide synchronisation.

constexpr int kWarpRowCap = 2048;             // visible positions a warp holds (64 a lane)
constexpr int kWtThreads = 512;               // 16 rows per CTA
constexpr int kWtRows = kWtThreads / 32;
constexpr int kWtCandCap = 512;               // keys of the first pass's threshold bin listed per row
constexpr int kWarpRowsMin = 4096;            // fewer rows take the CTA-per-row kernel

// The digit d of a 128-bin histogram where the count of keys from the top first reaches
// `remaining` (1 <= remaining <= total), and in *above the keys in higher bins.  Lane l holds
// bins [4 l, 4 l + 4); the same d and *above come back in every lane.
__device__ __forceinline__ int warp_select128(const uint32_t* hist, int remaining, int lane, int* above_out) {
    const uint4 c4 = reinterpret_cast<const uint4*>(hist)[lane];
    const int c[4] = {(int)c4.x, (int)c4.y, (int)c4.z, (int)c4.w};
    const int local = c[0] + c[1] + c[2] + c[3];
    int inc = local;   // suffix sum: this lane's bins and every higher lane's
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_down_sync(kFull, inc, o);
        if (lane + o < 32) inc += x;
    }
    int above = inc - local, d = -1, ab = 0;
#pragma unroll
    for (int i = 3; i >= 0; --i) {
        if (above < remaining && above + c[i] >= remaining) {
            d = 4 * lane + i;
            ab = above;
        }
        above += c[i];
    }
    const unsigned m = __ballot_sync(kFull, d >= 0);
    const int from = m ? __ffs(m) - 1 : 0;
    *above_out = __shfl_sync(kFull, ab, from);
    return __shfl_sync(kFull, d, from);
}

template <bool HAS_WIN>
__global__ void __launch_bounds__(kWtThreads) topk_warp_kernel(const TopkParams p) {
    extern __shared__ __align__(16) uint32_t wt_smem[];
    uint32_t (*hist_s)[kBins] = reinterpret_cast<uint32_t (*)[kBins]>(wt_smem);                  // per warp
    uint32_t (*cand_s)[kWtCandCap] = reinterpret_cast<uint32_t (*)[kWtCandCap]>(wt_smem + kWtRows * kBins);
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int row = blockIdx.x * kWtRows + wib;
    griddep_launch_dependents();
    if (row >= p.B * p.s) return;
    const int b = row / p.s, t = row - b * p.s;
    const int sp = __ldg(p.start_pos + b);
    if (HAS_WIN) {
        int32_t* wrow = p.win_out + (int64_t)row * p.row_stride;
        for (int i = lane; i < p.win_width; i += 32) wrow[i] = window_slot(p.s, t, sp, p.win_W, i);
        if (lane == 0 && p.s > 1 && sp != 0 && p.status) atomicOr(p.status, 4u /* STI_FLAG_CHUNKED */);
    }
    griddep_wait();   // the scores are complete from here on
    int vis = (sp + t + 1) / p.ratio;
    vis = max(0, min(vis, p.n_cols));
    int32_t* out = p.idxs + (int64_t)row * p.row_stride;
    if (vis <= p.k) {   // every visible position is selected
        for (int i = lane; i < p.k; i += 32) out[i] = i < vis ? i + p.offset : -1;
        return;
    }
    const float* src = p.scores + (int64_t)row * p.n_cols;
    uint32_t key[kWarpRowCap / 32];
#pragma unroll
    for (int i = 0; i < kWarpRowCap / 32; ++i) {
        const int j = 32 * i + lane;
        key[i] = j < vis ? float_key(__ldg(src + j)) : 0u;
    }
    // pass 1 over the top 11 bits (a float key's sign, exponent and two mantissa bits) into the
    // warp's 2048-bin histogram, lane l owning bins [64 l, 64 l + 64) for the selection
    uint32_t* h = hist_s[wib];
    uint32_t* cand = cand_s[wib];
    uint32_t prefix = 0u;
    int remaining = p.k;
    {
        uint4* h4 = reinterpret_cast<uint4*>(h);
#pragma unroll
        for (int i = 0; i < 16; ++i) h4[32 * i + lane] = make_uint4(0u, 0u, 0u, 0u);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < kWarpRowCap / 32; ++i)
            if (32 * i + lane < vis) atomicAdd(&h[key[i] >> 21], 1u);
        __syncwarp();
        // the threshold bin: suffix sums of the lanes' 64-bin totals, then a walk down one lane's bins
        int local = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint4 c = h4[16 * lane + i];
            local += (int)(c.x + c.y + c.z + c.w);
        }
        int inc = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_down_sync(kFull, inc, o);
            if (lane + o < 32) inc += x;
        }
        int above = inc - local, d = -1, ab = 0;
        if (above < remaining && inc >= remaining) {
            for (int bin = 64 * lane + 63; bin >= 64 * lane; --bin) {
                const int c = (int)h[bin];
                if (above + c >= remaining) {
                    d = bin;
                    ab = above;
                    break;
                }
                above += c;
            }
        }
        const unsigned m = __ballot_sync(kFull, d >= 0);
        const int from = m ? __ffs(m) - 1 : 0;
        d = __shfl_sync(kFull, d, from);
        ab = __shfl_sync(kFull, ab, from);
        remaining -= ab;
        prefix = (uint32_t)d;
    }
    // the bin's keys, listed (ascending position; up to kWtCandCap of them)
    const int c1 = (int)h[prefix];
    if (c1 <= kWtCandCap) {
        int n = 0;
#pragma unroll
        for (int i = 0; i < kWarpRowCap / 32; ++i) {
            const bool mm = 32 * i + lane < vis && (key[i] >> 21) == prefix;
            const unsigned bal = __ballot_sync(kFull, mm);
            if (mm) cand[n + __popc(bal & ((1u << lane) - 1u))] = key[i];
            n += __popc(bal);
        }
        __syncwarp();
        // passes 2..4 over the listed keys: 7 bits each into a 128-bin histogram (four bins a lane)
#pragma unroll 1
        for (int pass = 0; pass < 3; ++pass) {
            const int shift = 14 - 7 * pass;
            reinterpret_cast<uint4*>(h)[lane] = make_uint4(0u, 0u, 0u, 0u);
            __syncwarp();
            for (int j = lane; j < c1; j += 32) {
                const uint32_t kj = cand[j];
                if ((kj >> (shift + 7)) == prefix) atomicAdd(&h[(kj >> shift) & 127u], 1u);
            }
            __syncwarp();
            const uint4 c = reinterpret_cast<const uint4*>(h)[lane];
            const int cs[4] = {(int)c.x, (int)c.y, (int)c.z, (int)c.w};
            const int local = cs[0] + cs[1] + cs[2] + cs[3];
            int inc = local;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int x = __shfl_down_sync(kFull, inc, o);
                if (lane + o < 32) inc += x;
            }
            int above = inc - local, d = -1, ab = 0;
#pragma unroll
            for (int i = 3; i >= 0; --i) {
                if (above < remaining && above + cs[i] >= remaining) {
                    d = 4 * lane + i;
                    ab = above;
                }
                above += cs[i];
            }
            const unsigned m = __ballot_sync(kFull, d >= 0);
            const int from = m ? __ffs(m) - 1 : 0;
            remaining -= __shfl_sync(kFull, ab, from);
            prefix = (prefix << 7) | (uint32_t)__shfl_sync(kFull, d, from);
            __syncwarp();   // every lane has read the histogram before the next pass clears it
        }
    } else {
        // a threshold bin too large to list (rows of many equal scores): passes of 7 bits over the
        // keys in registers
#pragma unroll 1
        for (int pass = 0; pass < 3; ++pass) {
            const int shift = 14 - 7 * pass;
            reinterpret_cast<uint4*>(h)[lane] = make_uint4(0u, 0u, 0u, 0u);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < kWarpRowCap / 32; ++i)
                if (32 * i + lane < vis && (key[i] >> (shift + 7)) == prefix)
                    atomicAdd(&h[(key[i] >> shift) & 127u], 1u);
            __syncwarp();
            int above;
            const int d = warp_select128(h, remaining, lane, &above);
            remaining -= above;
            prefix = (prefix << 7) | (uint32_t)d;
            __syncwarp();
        }
    }
    const uint32_t tau = prefix;
    const int need_eq = remaining;   // >= 1 keys equal to tau are taken, lowest positions first
    // ordered compaction: keys above tau, and the first need_eq keys equal to tau, by position
    const unsigned below = (1u << lane) - 1u;
    int pos = 0, eq_seen = 0;
#pragma unroll
    for (int i = 0; i < kWarpRowCap / 32; ++i) {
        const int j = 32 * i + lane;
        const bool v = j < vis;
        const bool gt = v && key[i] > tau, eq = v && key[i] == tau;
        const unsigned em = __ballot_sync(kFull, eq);
        const bool take = gt || (eq && eq_seen + __popc(em & below) < need_eq);
        const unsigned tm = __ballot_sync(kFull, take);
        const int at = pos + __popc(tm & below);
        if (take && at < p.k) out[at] = j + p.offset;
        pos += __popc(tm);
        eq_seen += __popc(em);
    }
    // vis > k here, so exactly k entries were written
}

// ---------------------------------------------------------------------------------------------
// Cluster top-k for few long rows (decode): the CR CTAs of a cluster split one row into
// contiguous chunks.  The first radix pass comes precomputed from the scores kernel, so every
// CTA knows the threshold bin d1 without talking; rank 0 collects the bin's members (a few
// hundred keys) from the cluster's shared memory and finishes the exact select (passes 2 and
// 3); the CTAs then exchange their counts of selected keys and each writes its chunk's
// positions at its offset, in ascending position order.

#ifdef STI_TOPK_TIMING
__device__ unsigned long long g_topk_t[2048][17];
#define STI_KSTAMP(i)                                                                                  \
    do {                                                                                               \
        if (threadIdx.x == 0 && blockIdx.x < 2048) g_topk_t[blockIdx.x][i] = clock64();                \
    } while (0)
#define STI_KGSTAMP(i)                                                                                 \
    do {                                                                                               \
        if (threadIdx.x == 0 && blockIdx.x < 2048) g_topk_t[blockIdx.x][i] = global_timer_ns();        \
    } while (0)
#else
#define STI_KSTAMP(i) \
    do {              \
    } while (0)
#define STI_KGSTAMP(i) \
    do {               \
    } while (0)
#endif

constexpr int kClThreads = 256;
constexpr int kClWarps = kClThreads / 32;
constexpr int kClCandCap = 2048;   // threshold-bin members a CTA holds (rank 0: of the whole row)

struct __align__(16) ClusterTopkSmem {
    uint32_t hist[kBins];
    int warp_tot[kClWarps];
    int misc[8];
    int n_cand;                 // this CTA's threshold-bin members
    int pub_gt, pub_eq;         // this CTA's keys > tau and == tau
    uint32_t pub_tau;           // (rank 0) the exact k-th key and how many keys == tau to take
    int pub_need;
    int pub_ok;                 // (rank 0) 1 if the candidates fitted and tau is valid
    int n_above;                // this CTA's keys whose first digit is above the threshold bin
    int n_sel;                  // this CTA's threshold-bin members that are selected
    int warp_above[kClWarps];   // per warp segment: keys above the bin
    int warp_sel[kClWarps];     // per warp segment: selected members of the bin
};

constexpr int kRankCap = 1024;  // threshold-bin members every CTA ranks itself

// 256-thread block scan (exclusive) with total.
__device__ __forceinline__ int block_excl_scan256(int v, int* warp_tot, int& total) {
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
    for (int w = 0; w < kClWarps; ++w) {
        const int x = warp_tot[w];
        wpre += w < warp ? x : 0;
        tot += x;
    }
    __syncthreads();
    total = tot;
    return wpre + inc - v;
}

// Bin d* of `hist` (kBins bins, counts of matching keys) where the count from the top first
// reaches `remaining`; *above = count in higher bins.  256 threads, 8 bins each.
__device__ __forceinline__ int select_bin256(const uint32_t* hist, int remaining, int* warp_tot, int* misc,
                                             int* above_out) {
    const int tid = threadIdx.x;
    int local = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) local += (int)hist[8 * tid + i];
    int total;
    const int excl = block_excl_scan256(local, warp_tot, total);
    int above = total - excl - local;
#pragma unroll
    for (int i = 7; i >= 0; --i) {
        const int bin = 8 * tid + i;
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

// Histogram over n keys from src (keys whose bits above hi_shift equal prefix), then select_bin256.
template <typename Src>
__device__ __forceinline__ int radix_pass256(Src src, int n, int hi_shift, int shift, int bits, uint32_t prefix,
                                             int remaining, uint32_t* hist, int* warp_tot, int* misc,
                                             int* above_out) {
    const int tid = threadIdx.x, lane = tid & 31;
    const uint32_t mask = (1u << bits) - 1u;
    for (int i = tid; i < kBins; i += kClThreads) hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < n; base += kClThreads) {
        const int j = base + tid;
        bool m = false;
        uint32_t dig = 0xFFFFFFFFu;
        if (j < n) {
            const uint32_t key = src(j);
            m = (key >> hi_shift) == prefix;
            if (m) dig = (key >> shift) & mask;
        }
        const unsigned peers = __match_any_sync(kFull, dig);
        if (m && lane == __ffs(peers) - 1) atomicAdd(&hist[dig], (uint32_t)__popc(peers));
    }
    __syncthreads();
    return select_bin256(hist, remaining, warp_tot, misc, above_out);
}

template <int CR>
__global__ void __launch_bounds__(kClThreads, 1) topk_cluster_kernel(const TopkParams p, int chunk_cap) {
    extern __shared__ __align__(16) uint8_t cl_smem[];
    ClusterTopkSmem* sm = reinterpret_cast<ClusterTopkSmem*>(cl_smem);
    uint32_t* keys = reinterpret_cast<uint32_t*>(sm + 1);            // [chunk_cap] this CTA's chunk
    uint32_t* cand = keys + chunk_cap;                               // [kClCandCap] (rank 0: all members)
    int* cand_pos = reinterpret_cast<int*>(cand + kClCandCap);       // [kClCandCap] their positions
    // every rank's members as (key << 32 | ~position): a larger value ranks first
    unsigned long long* all_comb = reinterpret_cast<unsigned long long*>(cand_pos + kClCandCap);   // [kRankCap]
    int* rank_part = reinterpret_cast<int*>(all_comb + kRankCap);            // [kRankCap] own members' ranks
    uint32_t* sel_bits = reinterpret_cast<uint32_t*>(rank_part + kRankCap);  // [chunk_cap / 32]

    const int row = blockIdx.x / CR, rank = blockIdx.x - (blockIdx.x / CR) * CR;
    const int b = row / p.s, t = row - b * p.s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t* ghist = p.hist + (size_t)row * kBins;
    STI_KGSTAMP(14);
    STI_KSTAMP(0);
    griddep_launch_dependents();
    // start_pos and the window indices depend on no earlier kernel of the step
    const int sp = __ldg(p.start_pos + b);
    if (p.win_out != nullptr && rank == 0) {
        int32_t* wrow = p.win_out + (int64_t)row * p.row_stride;
        for (int i = tid; i < p.win_width; i += kClThreads) wrow[i] = window_slot(p.s, t, sp, p.win_W, i);
        if (tid == 0 && p.s > 1 && sp != 0 && p.status) atomicOr(p.status, 4u /* STI_FLAG_CHUNKED */);
    }
    STI_KSTAMP(1);
    griddep_wait();   // the scores and the histogram are complete from here on
    STI_KSTAMP(2);
    STI_KGSTAMP(16);
    uint32_t hreg[kBins / kClThreads];
#pragma unroll
    for (int i = 0; i < kBins / kClThreads; ++i) hreg[i] = __ldg(ghist + i * kClThreads + tid);
    int vis = (sp + t + 1) / p.ratio;
    vis = max(0, min(vis, p.n_cols));
    int32_t* out = p.idxs + (int64_t)row * p.row_stride;

    if (vis <= p.k) {   // every visible position is selected (row-uniform: the whole cluster returns)
        if (rank == 0) {
            for (int i = tid; i < p.k; i += kClThreads) out[i] = i < vis ? i + p.offset : -1;
            for (int i = tid; i < kBins; i += kClThreads) ghist[i] = 0;
        }
        return;
    }

    // this CTA's chunk [lo, hi): whole warps of 32
    const int chunk = (((vis + CR - 1) / CR) + 31) & ~31;
    const int lo = min(vis, rank * chunk), hi = min(vis, lo + chunk);
    const int n_mine = hi - lo;
    const float* src = p.scores + (int64_t)row * p.n_cols;
#pragma unroll
    for (int i = 0; i < kBins / kClThreads; ++i) sm->hist[i * kClThreads + tid] = hreg[i];
    // the chunk, eight loads in flight per thread
    for (int base = 0; base < n_mine; base += 8 * kClThreads) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int j = base + u * kClThreads + tid;
            v[u] = j < n_mine ? __ldg(src + lo + j) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int j = base + u * kClThreads + tid;
            if (j < n_mine) keys[j] = float_key(v[u]);
        }
    }
    for (int i = tid; i < chunk_cap / 32; i += kClThreads) sel_bits[i] = 0u;
    for (int i = tid; i < kRankCap; i += kClThreads) rank_part[i] = 0;
    if (tid == 0) {
        sm->n_cand = 0;
        sm->n_above = 0;
        sm->n_sel = 0;
    }
    if (tid < kClWarps) sm->warp_sel[tid] = 0;
    __syncthreads();
    STI_KSTAMP(3);

    // pass 1 from the precomputed histogram: the same d1 in every CTA
    int above;
    const int d1 = select_bin256(sm->hist, p.k, sm->warp_tot, sm->misc, &above);
    const int remaining1 = p.k - above;
    const int c1 = (int)sm->hist[d1];
    STI_KSTAMP(4);
    // this CTA's members of bin d1 (key and position) and, per warp segment, its keys above the
    // bin; warp w owns chunk positions [w*seg, w*seg + seg), its lanes consecutive positions
    const int seg = ((n_mine + kClWarps - 1) / kClWarps + 31) & ~31;
    const int wlo = min(n_mine, warp * seg), whi = min(n_mine, wlo + seg);
    int above_mine = 0;
    for (int j0 = wlo; j0 < whi; j0 += 32) {
        const int j = j0 + lane;
        const uint32_t key = j < whi ? keys[j] : 0u;
        const bool m = j < whi && (key >> 21) == (uint32_t)d1;
        above_mine += __popc(__ballot_sync(kFull, j < whi && (key >> 21) > (uint32_t)d1));
        const unsigned bal = __ballot_sync(kFull, m);
        if (bal == 0u) continue;
        int wbase = 0;
        if (lane == 0) wbase = atomicAdd(&sm->n_cand, __popc(bal));
        wbase = __shfl_sync(kFull, wbase, 0);
        const int at = wbase + __popc(bal & ((1u << lane) - 1u));
        if (m && at < kClCandCap) {
            cand[at] = key;
            cand_pos[at] = lo + j;
        }
    }
    if (lane == 0) {
        sm->warp_above[warp] = above_mine;
        atomicAdd(&sm->n_above, above_mine);
    }
    __syncthreads();
    STI_KSTAMP(5);
    cluster_sync();   // #1: every CTA's members are in its shared memory; every CTA read the histogram

    // lane r of every warp reads rank r's member count; prefix over ranks and total
    static_assert(CR <= kClWarps && CR <= 32, "one warp per cluster rank");
    const int cnt_r = lane < CR ? ld_dsmem_s32(dsmem_addr(&sm->n_cand, (uint32_t)lane)) : 0;
    int cnt_incl = cnt_r;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(kFull, cnt_incl, o);
        if (lane >= o) cnt_incl += x;
    }
    const int tot = __shfl_sync(kFull, cnt_incl, 31);
    STI_KSTAMP(6);
    if (tot == c1 && tot <= kRankCap) {
        // ---- every CTA ranks its own members among all of them: (score desc, position asc)
        if (warp < CR) {   // warp w copies rank w's members
            const int n_w = __shfl_sync(kFull, cnt_r, warp);
            const int at = __shfl_sync(kFull, cnt_incl - cnt_r, warp);
            for (int i0 = 0; i0 < n_w; i0 += 32) {
                const int i = i0 + lane;
                if (i < n_w) {
                    const uint32_t k_ = ld_dsmem_u32(dsmem_addr(cand + i, (uint32_t)warp));
                    const uint32_t p_ = ld_dsmem_u32(dsmem_addr(cand_pos + i, (uint32_t)warp));
                    all_comb[at + i] = ((unsigned long long)k_ << 32) | (unsigned long long)(~p_);
                }
            }
        }
        // keys above the bin in lower ranks' chunks (lane r < rank reads rank r)
        int ab = lane < rank ? ld_dsmem_s32(dsmem_addr(&sm->n_above, (uint32_t)lane)) : 0;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) ab += __shfl_xor_sync(kFull, ab, o);
        __syncthreads();
        STI_KSTAMP(7);
        const int n_own = __shfl_sync(kFull, cnt_r, rank);
        const int own_at = __shfl_sync(kFull, cnt_incl - cnt_r, rank);
#ifdef STI_TOPK_TIMING
        if (tid == 0 && blockIdx.x < 2048) g_topk_t[blockIdx.x][11] = (unsigned long long)tot | ((unsigned long long)n_own << 20) | ((unsigned long long)n_mine << 40);
#endif
        // rank of own member c = how many members rank before it; warp w counts over its eighth
        // of all members, lane l over own members l, l+32, ... (the members read are broadcast)
        {
            const int f_lo = (int)((long long)warp * tot / kClWarps), f_hi = (int)((long long)(warp + 1) * tot / kClWarps);
            for (int c0 = 0; c0 < n_own; c0 += 32) {
                const int c = c0 + lane;
                const unsigned long long me = c < n_own ? all_comb[own_at + c] : ~0ull;
                int r = 0;
#pragma unroll 4
                for (int f = f_lo; f < f_hi; ++f) r += all_comb[f] > me ? 1 : 0;
                if (c < n_own && r > 0) atomicAdd(&rank_part[c], r);
            }
        }
        __syncthreads();
        for (int c = tid; c < n_own; c += kClThreads) {
            if (rank_part[c] < remaining1) {
                const int pos = (int)(~(uint32_t)(all_comb[own_at + c] & 0xFFFFFFFFull));
                atomicOr(&sel_bits[(pos - lo) >> 5], 1u << ((pos - lo) & 31));
                atomicAdd(&sm->n_sel, 1);
                atomicAdd(&sm->warp_sel[(pos - lo) / seg], 1);
            }
        }
        __syncthreads();
        STI_KSTAMP(8);
        cluster_sync();   // #2: every rank's selected count is published
        STI_KSTAMP(9);
        int sl = lane < rank ? ld_dsmem_s32(dsmem_addr(&sm->n_sel, (uint32_t)lane)) : 0;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) sl += __shfl_xor_sync(kFull, sl, o);
        cluster_arrive();   // this CTA reads no partner's shared memory any more
        const int base_sel = ab + sl;   // selected positions before this chunk
        // ordered compaction: keys above the bin, and the bin's selected members
        const uint32_t kb = smem_u32(keys), sb = smem_u32(sel_bits);
        auto take_at = [kb, sb, whi, d1](int j) -> bool {
            if (j >= whi) return false;
            const uint32_t dig = lds_u32(kb + 4u * (uint32_t)j) >> 21;
            return dig > (uint32_t)d1 || (dig == (uint32_t)d1 && ((lds_u32(sb + 4u * (uint32_t)(j >> 5)) >> (j & 31)) & 1u));
        };
        STI_KSTAMP(10);
        int pos = base_sel;   // + the selected positions of lower warp segments
        for (int w = 0; w < warp; ++w) pos += sm->warp_above[w] + sm->warp_sel[w];
        for (int j0 = wlo; j0 < whi; j0 += 32) {
            const int j = j0 + lane;
            const bool take = take_at(j);
            const unsigned tm = __ballot_sync(kFull, take);
            const int at = pos + __popc(tm & ((1u << lane) - 1u));
            if (take && at < p.k) out[at] = lo + j + p.offset;
            pos += __popc(tm);
        }
        if (rank == 0)
            for (int i = tid; i < kBins; i += kClThreads) ghist[i] = 0;   // ready for the next call
        STI_KSTAMP(12);
        cluster_wait();   // no partner still reads this CTA's shared memory
        STI_KSTAMP(13);
        STI_KGSTAMP(15);
        return;
    }
    // ---- otherwise (too many members of one bin): rank 0 finishes the select alone
    STI_KSTAMP(6);

    if (rank == 0) {
        for (int i = tid; i < kBins; i += kClThreads) ghist[i] = 0;   // ready for the next call
        // gather the members of the whole row (total c1) behind this CTA's own
        // lane r of every warp reads rank r's count; warp w then copies rank w's members
        const int my_cnt = lane < CR ? ld_dsmem_s32(dsmem_addr(&sm->n_cand, (uint32_t)lane)) : 0;
        int incl = my_cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += x;
        }
        const int tot = __shfl_sync(kFull, incl, 31);
        const bool fits = tot == c1 && tot <= kClCandCap;
        if (fits && warp >= 1 && warp < CR) {
            const int n_w = __shfl_sync(kFull, my_cnt, warp);
            const int at = __shfl_sync(kFull, incl - my_cnt, warp);
            for (int i0 = 0; i0 < n_w; i0 += 64) {   // two remote loads in flight per lane
                const int i1 = i0 + lane, i2 = i0 + 32 + lane;
                const uint32_t a1 = i1 < n_w ? ld_dsmem_u32(dsmem_addr(cand + i1, (uint32_t)warp)) : 0u;
                const uint32_t a2 = i2 < n_w ? ld_dsmem_u32(dsmem_addr(cand + i2, (uint32_t)warp)) : 0u;
                if (i1 < n_w) cand[at + i1] = a1;
                if (i2 < n_w) cand[at + i2] = a2;
            }
        }
        __syncthreads();
        STI_KSTAMP(7);
        uint32_t prefix = (uint32_t)d1;
        int remaining = remaining1;
        if (fits) {
            auto cand_at = [&](int j) -> uint32_t { return cand[j]; };
            const int d2 = radix_pass256(cand_at, c1, 21, 10, 11, prefix, remaining, sm->hist, sm->warp_tot,
                                         sm->misc, &above);
            remaining -= above;
            prefix = (prefix << 11) | (uint32_t)d2;
            const int d3 = radix_pass256(cand_at, c1, 10, 0, 10, prefix, remaining, sm->hist, sm->warp_tot,
                                         sm->misc, &above);
            remaining -= above;
            prefix = (prefix << 10) | (uint32_t)d3;
        } else {
            // too many members of one bin (heavy ties): passes 2 and 3 over the whole row
            auto row_at = [&](int j) -> uint32_t { return float_key(__ldg(src + j)); };
            const int d2 = radix_pass256(row_at, vis, 21, 10, 11, prefix, remaining, sm->hist, sm->warp_tot,
                                         sm->misc, &above);
            remaining -= above;
            prefix = (prefix << 11) | (uint32_t)d2;
            const int d3 = radix_pass256(row_at, vis, 10, 0, 10, prefix, remaining, sm->hist, sm->warp_tot,
                                         sm->misc, &above);
            remaining -= above;
            prefix = (prefix << 10) | (uint32_t)d3;
        }
        if (tid == 0) {
            sm->pub_tau = prefix;
            sm->pub_need = remaining;
        }
    }
    STI_KSTAMP(8);
    cluster_sync();   // #2: tau published
    STI_KSTAMP(9);
    const uint32_t tau = ld_dsmem_u32(dsmem_addr(&sm->pub_tau, 0u));
    const int need_eq = ld_dsmem_s32(dsmem_addr(&sm->pub_need, 0u));

    // counts of this CTA's chunk, per warp segment (ordered compaction as in the one-CTA kernel)
    int n_gt = 0, n_eq = 0;
    for (int j0 = wlo; j0 < whi; j0 += 32) {
        const int j = j0 + lane;
        const uint32_t key = j < whi ? keys[j] : 0u;
        n_gt += __popc(__ballot_sync(kFull, j < whi && key > tau));
        n_eq += __popc(__ballot_sync(kFull, j < whi && key == tau));
    }
    if (lane == 0) {
        sm->warp_tot[warp] = n_gt;
        sm->misc[warp] = n_eq;   // misc has 8 slots = kClWarps
    }
    __syncthreads();
    if (tid == 0) {
        int g = 0, e = 0;
        for (int w = 0; w < kClWarps; ++w) {
            g += sm->warp_tot[w];
            e += sm->misc[w];
        }
        sm->pub_gt = g;
        sm->pub_eq = e;
    }
    __syncthreads();
    STI_KSTAMP(10);
    cluster_sync();   // #3: every CTA's counts published
    STI_KSTAMP(11);
    // offset of this CTA = keys selected by lower ranks; equal keys go to the lowest positions
    // (lane r < rank reads rank r's counts; prefix over lanes gives the keys == tau before r)
    int g_l = 0, e_l = 0;
    if (lane < rank) {
        g_l = ld_dsmem_s32(dsmem_addr(&sm->pub_gt, (uint32_t)lane));
        e_l = ld_dsmem_s32(dsmem_addr(&sm->pub_eq, (uint32_t)lane));
    }
    int e_incl = e_l;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(kFull, e_incl, o);
        if (lane >= o) e_incl += x;
    }
    int taken = g_l + max(0, min(e_l, need_eq - (e_incl - e_l)));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) taken += __shfl_xor_sync(kFull, taken, o);
    const int base_out = taken;
    const int eq_before = __shfl_sync(kFull, e_incl, 31);
    // within the CTA: warp w's offset and equal-key budget
    int w_gt_before = 0, w_eq_before = 0;
    for (int w = 0; w < warp; ++w) {
        w_gt_before += sm->warp_tot[w];
        w_eq_before += sm->misc[w];
    }
    // keys == tau are taken in position order: lower ranks first, then lower warps
    int pos = base_out + w_gt_before + max(0, min(w_eq_before, need_eq - eq_before));
    int eq_seen = eq_before + w_eq_before;
    for (int j0 = wlo; j0 < whi; j0 += 32) {
        const int j = j0 + lane;
        const uint32_t key = j < whi ? keys[j] : 0u;
        const bool gt = j < whi && key > tau;
        const bool eq = j < whi && key == tau;
        const unsigned eq_mask = __ballot_sync(kFull, eq);
        const int eq_rank = eq_seen + __popc(eq_mask & ((1u << lane) - 1u));
        const bool take = gt || (eq && eq_rank < need_eq);
        const unsigned take_mask = __ballot_sync(kFull, take);
        const int at = pos + __popc(take_mask & ((1u << lane) - 1u));
        if (take && at < p.k) out[at] = lo + j + p.offset;
        pos += __popc(take_mask);
        eq_seen += __popc(eq_mask);
    }
    STI_KSTAMP(12);
    cluster_sync();   // #4: no partner still reads this CTA's shared memory
    STI_KSTAMP(13);
    STI_KGSTAMP(15);
}

}  // namespace

cudaError_t launch_window_idxs(const int32_t* start_pos, int B, int s, int W, int width, int32_t* idxs,
                               int64_t row_stride, uint32_t* status, cudaStream_t stream, bool chunked) {
    const int64_t total = (int64_t)B * s * width;
    if (total == 0) return cudaSuccess;
    int blocks = (int)((total + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    window_idx_kernel<<<blocks, 256, 0, stream>>>(start_pos, B, s, W, width, idxs, row_stride, status,
                                                  chunked ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream) {
    const int rows = p.B * p.s;
    if (rows == 0) return cudaSuccess;
    constexpr int CR = 8;
    if (p.hist != nullptr && rows * CR <= 8 * device_num_sms() && p.n_cols <= CR * 8192) {
        // few long rows with the first pass precomputed: one cluster of CR CTAs per row
        const int chunk_cap = ((((p.n_cols + CR - 1) / CR) + 31) & ~31);
        const size_t smem = sizeof(ClusterTopkSmem) +
                            (size_t)(chunk_cap + 2 * kClCandCap + 3 * kRankCap + chunk_cap / 32) * 4;
        cudaError_t err =
            cudaFuncSetAttribute(topk_cluster_kernel<CR>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(rows * CR));
        cfg.blockDim = dim3(kClThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CR;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = p.pdl ? 2 : 1;
        err = cudaLaunchKernelEx(&cfg, topk_cluster_kernel<CR>, p, chunk_cap);
        return err != cudaSuccess ? err : cudaGetLastError();
    }
    if (p.hist == nullptr && p.n_cols <= kWarpRowCap && rows >= kWarpRowsMin) {
        // many short rows without a precomputed first pass (prefill): one warp per row.  A warp
        // takes longer over a row than a 512-thread CTA but holds 16 rows per SM at once, so it
        // wins only when there are rows enough to fill the GPU several times over
        const size_t wsmem = (size_t)kWtRows * (kBins + kWtCandCap) * 4;
        cudaError_t e0 = cudaFuncSetAttribute(topk_warp_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wsmem);
        if (e0 == cudaSuccess)
            e0 = cudaFuncSetAttribute(topk_warp_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wsmem);
        if (e0 != cudaSuccess) return e0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((rows + kWtRows - 1) / kWtRows));
        cfg.blockDim = dim3(kWtThreads);
        cfg.dynamicSmemBytes = wsmem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = p.pdl ? 1 : 0;
        const cudaError_t err = p.win_out != nullptr ? cudaLaunchKernelEx(&cfg, topk_warp_kernel<true>, p)
                                                     : cudaLaunchKernelEx(&cfg, topk_warp_kernel<false>, p);
        return err != cudaSuccess ? err : cudaGetLastError();
    }
    const int use_smem = p.n_cols <= kSmemKeyCap ? 1 : 0;
    const size_t smem = (size_t)(kBins + kWarps + 8 + kCandCap + (use_smem ? p.n_cols : 0)) * 4;
    auto kern = p.hist != nullptr ? topk_kernel<true> : topk_kernel<false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows);
    cfg.blockDim = dim3(kTopkThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.pdl ? 1 : 0;
    err = cudaLaunchKernelEx(&cfg, kern, p, use_smem);
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace sti

#ifdef STI_TOPK_TIMING
// profiling builds only: per-CTA clock64 stamps of the cluster top-k phases
extern "C" int sti_dbg_topk_times(unsigned long long* host, int n_blocks) {
    return (int)cudaMemcpyFromSymbol(host, sti::g_topk_t, sizeof(unsigned long long) * 17 * (size_t)n_blocks);
}
#endif
