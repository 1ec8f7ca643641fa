// sti_attn_util.cuh -- device helpers shared by the attention kernels: a bounded barrier wait
// that every thread of a CTA abandons once one of them timed out, a warp reduce-scatter of
// per-lane value arrays, and TMEM loads/stores sized by a template width.
#pragma once
#include "sti_ptx.cuh"

namespace sti {

constexpr uint32_t kWarpFull = 0xFFFFFFFFu;

// Bounded wait that also gives up when another thread of the CTA already timed out.
__device__ __forceinline__ bool attn_wait(uint64_t* bar, uint32_t parity, uint32_t* status, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > STI_WAIT_TIMEOUT_NS) {
            if (status) atomicOr(status, 2u /* STI_FLAG_TIMEOUT */);
            *abort = 1;
            return false;
        }
    }
}

// The same, acquiring at cluster scope (for barriers that other CTAs of the cluster arrive on
// after writing shared memory this thread then reads).
__device__ __forceinline__ bool attn_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t* status,
                                                  volatile int* abort) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > STI_WAIT_TIMEOUT_NS) {
            if (status) atomicOr(status, 2u /* STI_FLAG_TIMEOUT */);
            *abort = 1;
            return false;
        }
    }
}

// Reduce N values per lane over the warp's 32 lanes, scattering the results: afterwards v[0] of
// lane l is the reduction of value l >> (5 - log2 N) (each held by 32/N adjacent lanes).
template <int N, bool IS_MAX>
__device__ __forceinline__ void warp_reduce_scatter_n(float (&v)[N]) {
    const int lane = threadIdx.x & 31;
    int off = 16;
#pragma unroll
    for (int half = N / 2; half >= 1; half >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float lo = v[i], hi = v[i + half];
            const float send = upper ? lo : hi;
            const float keep = upper ? hi : lo;
            const float recv = __shfl_xor_sync(kWarpFull, send, off);
            v[i] = IS_MAX ? fmaxf(keep, recv) : keep + recv;
        }
    }
#pragma unroll
    for (; off >= 1; off >>= 1) {
        const float recv = __shfl_xor_sync(kWarpFull, v[0], off);
        v[0] = IS_MAX ? fmaxf(v[0], recv) : v[0] + recv;
    }
}

template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N]) {
    if constexpr (N == 16) tmem_ld16(taddr, r);
    else tmem_ld32(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t (&r)[N]) {
    if constexpr (N == 16) tmem_st16(taddr, r);
    else tmem_st32(taddr, r);
}
// The output's inverse rotary rotation on values held as O^T rows: this lane holds dimension dd
// of N heads' outputs and lane^1 holds dimension dd^1 of the same heads.  Dims [d - rd, d) form
// rd/2 interleaved pairs (x, y) rotated back by their angle: x' = x c + y s, y' = y c - x s, with
// (c, s) = cs[2i], cs[2i+1] for pair i.  Every lane of the warp must call it (shuffles).
template <int N>
__device__ __forceinline__ void rope_inverse_pairs(float (&v)[N], int dd, int d, int rd, const float* cs) {
    const bool in = dd < d && dd >= d - rd;
    float c = 1.f, s = 0.f;
    if (in) {
        const int i = (dd - (d - rd)) >> 1;
        c = cs[2 * i];       // (shared or global memory)
        s = cs[2 * i + 1];
    }
    const bool odd = (dd & 1) != 0;
#pragma unroll
    for (int j = 0; j < N; ++j) {
        const float pv = __shfl_xor_sync(kWarpFull, v[j], 1);
        if (in) v[j] = odd ? v[j] * c - pv * s : v[j] * c + pv * s;
    }
}

}  // namespace sti
