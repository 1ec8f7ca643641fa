// sparse_attn.cu -- sparse multi-head attention with an attention sink over gathered rows of one
// shared latent KV.
//
// DeepSeek V4.1, attention "attend/selected" page, sparse_attn_kernel / sparse_attn:
//   for every query and head, over the slots i whose index is not -1:
//     s_i = softmax_scale * q . kv[idx_i];  o = sum_i e^{s_i} kv[idx_i] / (sum_i e^{s_i} + e^{sink_h})
//   the same row serving as key and value; a query with no valid slot gets 0.
//
// GB300 design (not the page's kernel, which puts the heads in the MMA M dimension):
//   * One CTA handles one query and a range of 128-row KV tiles.  The rows of a tile are gathered
//     with 16-byte cp.async straight into the 128-byte-swizzled UMMA layout (column blocks of
//     128 rows x 128 bytes); masked slots are zero-filled and get score -inf.
//   * S^T = KV_tile . Q^T runs as tcgen05 M=128 (rows) x N=64 (heads, zero-padded) x K=d, so the
//     MMA uses the full 128-lane datapath even though a query has only 64 heads.  The tile is the
//     K-major A operand; Q (resident, zero-padded to 64 heads) the K-major B operand.
//   * Online softmax in fp32 on the TMEM tile: thread r owns row r; per-head maxima and sums across
//     the 128 rows are warp reduce-scatters plus a 4-warp combine in shared memory.  P^T is
//     written as bf16 (the page also rounds P to bf16 before the PV product).
//   * O^T += V^T . P^T runs as tcgen05 M=128 (d block) x N=64 x K=128 rows, reading the SAME
//     shared-memory tile as an MN-major A operand -- K and V are one row, fetched once.
//     O^T lives in TMEM (d/128 blocks of 128 lanes x 64 columns); rescaling when a head's
//     running max grows is a TMEM load-scale-store by the owning thread.
//   * Few queries (decode) split a query's index slots over a thread-block cluster of up to 8
//     CTAs (one wave on the GPU).  Each CTA runs the online softmax over its slots; the cluster
//     then exchanges running maxima and sums through distributed shared memory, every CTA scales
//     its O^T by 2^(m_cta - M) / (sum_c l_c 2^(m_c - M) + 2^(sink - M)) into its own shared
//     memory, and each CTA sums a slice of d across the cluster and writes it -- no partials in
//     global memory and no second kernel.  Many queries use one CTA per query.
#include <cuda_bf16.h>
#include <math.h>

#include <mutex>
#include <vector>

#include "sti_internal.h"
#include "sti_kvfp4.h"
#include "sti_ptx.cuh"
#include "sti_attn_util.cuh"

namespace sti {
namespace {

constexpr int kThreads = 256;  // 8 warps: warps w and w+4 share TMEM lanes, split the 64 head columns
constexpr int kRows = 128;        // KV rows per tile (MMA M)
constexpr int kHp = 64;           // heads padded (MMA N)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr uint32_t kFull = 0xFFFFFFFFu;

struct __align__(8) AttnSmemTail {
    uint64_t mma_bar;
    uint64_t q_bar;        // Q tile landed (TMA)
    uint64_t gather_bar;   // this tile's rows landed (TMA)
    uint64_t recv_bar;     // cluster partners' O slices landed (bulk copies)
    uint32_t tmem_base;
    int rescale;           // some head's running max moved in this tile
    float m_run[kHp];     // running max, log2 domain
    float l_run[kHp];     // running sum of 2^(x - m)
    float alpha[kHp];     // rescale factor of this tile
    float red[4][kHp];    // per-warp partial reductions
    const uint16_t* row_src[kRows];
    int row_valid[kRows];
    int row_coord[kRows];  // row in its source viewed as [B*rows, d]
    int row_srcid[kRows];  // 0: kv, 1: kv2, -1: masked
};

// Swizzled byte offset of 16-byte chunk `ch` (of 8 bf16) of row `r` in a tile of `rows` rows
// stored as column blocks of rows x 128 bytes (128-byte swizzle: chunk ^= row % 8).
__device__ __forceinline__ uint32_t sw128_offset(int r, int ch, int rows) {
    return (uint32_t)(ch >> 3) * (uint32_t)rows * 128u + (uint32_t)r * 128u + (uint32_t)(((ch & 7) ^ (r & 7)) << 4);
}

// Reduce-scatter of 32 per-lane values over the 32 lanes of a warp: afterwards lane l holds in
// v[0] the reduction over the warp's 32 rows of value l.
template <bool IS_MAX>
__device__ __forceinline__ void warp_reduce_scatter32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        const int half = 16 >> step;          // values still held: 2*half
        const int off = 16 >> step;           // partner lane distance
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float lo = v[i], hi = v[i + half];
            const float send = upper ? lo : hi;
            const float keep = upper ? hi : lo;
            const float recv = __shfl_xor_sync(kFull, send, off);
            v[i] = IS_MAX ? fmaxf(keep, recv) : keep + recv;
        }
    }
}

#ifdef STI_ATTN_TIMING
__device__ unsigned long long g_attn_t[2048][16];
#define STI_TSTAMP(i)                                                                                  \
    do {                                                                                               \
        if (threadIdx.x == 0 && blockIdx.x < 2048) g_attn_t[blockIdx.x][i] = clock64();               \
    } while (0)
#else
#define STI_TSTAMP(i) \
    do {              \
    } while (0)
#endif

__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv1,
                       const __grid_constant__ CUtensorMap tm_kv2, const AttnParams p, const KvFp4 f) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned start, offset from the __shared__ array itself so every derived pointer
    // stays a known shared-memory pointer (ld/st.shared, not generic accesses)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* q_s = smem;                                 // [64 heads] x d_pad, K-major SW128
    uint8_t* kv_s = q_s + (size_t)kHp * p.d_pad * 2;     // [128 rows] x d_pad, SW128
    uint8_t* p_s = kv_s + (size_t)kRows * p.d_pad * 2;   // [128 rows] x 64 heads bf16, SW128
    AttnSmemTail* tl = reinterpret_cast<AttnSmemTail*>(p_s + kRows * 128);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = tid & (kRows - 1);       // TMEM lane / KV row this thread owns
    const int hg = tid >> 7;                 // head group: columns [32*hg, 32*hg + 32)
    const int C = p.cluster;
    const int query = blockIdx.x / C, rank = blockIdx.x - (blockIdx.x / C) * C;   // rank in the cluster
    const int b = query / p.s;
    const int slot_begin = min(p.k, rank * p.rows_per_cta);
    const int slot_end = min(p.k, slot_begin + p.rows_per_cta);
    const int tile_begin = 0;
    const int tile_end = (slot_end - slot_begin + kRows - 1) / kRows;
    STI_TSTAMP(0);

    if (warp == 0) {
        tmem_alloc(&tl->tmem_base, 512);
        tmem_relinquish();
    }
    const int ncb_real = p.d / 64;        // column blocks holding data; the rest stay zero
    const int ncb = p.d_pad / 64;
    if (tid == 0) {
        mbar_init(&tl->mma_bar, 1);
        mbar_init(&tl->q_bar, 1);
        mbar_init(&tl->gather_bar, 1);
        mbar_init(&tl->recv_bar, 1);
        fence_mbar_init();
    }
    if (tid < kHp) {
        tl->m_run[tid] = -INFINITY;
        tl->l_run[tid] = 0.f;
    }
    if (p.use_tma) {
        // zero what no copy writes: Q rows >= h, and every padded column block of Q and the tile
        for (int cb = 0; cb < ncb; ++cb) {
            const int r0 = cb < ncb_real ? p.h : 0;
            uint4* q_blk = reinterpret_cast<uint4*>(q_s + (size_t)cb * kHp * 128);
            for (int i = r0 * 8 + tid; i < kHp * 8; i += kThreads) q_blk[i] = make_uint4(0, 0, 0, 0);
            if (cb >= ncb_real) {
                uint4* kv_blk = reinterpret_cast<uint4*>(kv_s + (size_t)cb * kRows * 128);
                for (int i = tid; i < kRows * 8; i += kThreads) kv_blk[i] = make_uint4(0, 0, 0, 0);
            }
        }
        __syncthreads();   // barrier initialisation visible before the copies use it
        if (tid == 0) {
            tma_prefetch_desc(&tm_kv1);
            tma_prefetch_desc(&tm_kv2);
            mbar_arrive_expect_tx(&tl->q_bar, (uint32_t)(ncb_real * p.h * 128));
            for (int cb = 0; cb < ncb_real; ++cb)
                tma_load_2d(q_s + (size_t)cb * kHp * 128, &tm_q, &tl->q_bar, cb * 64, query * p.h);
        }
    } else {
        // Q -> shared memory (heads >= h and columns >= d are zero)
        const uint16_t* qrow = p.q + (size_t)query * p.h * p.d;
        const int chunks_per_row = p.d_pad / 8;
        for (int c = tid; c < kHp * chunks_per_row; c += kThreads) {
            const int hr = c / chunks_per_row, ch = c - hr * chunks_per_row;
            const bool ok = hr < p.h && ch * 8 < p.d;
            const uint16_t* src = ok ? qrow + (size_t)hr * p.d + ch * 8 : p.q;
            cp_async_16(smem_u32(q_s) + sw128_offset(hr, ch, kHp), src, ok ? 16u : 0u);
        }
        cp_async_commit();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tl->tmem_base;
    STI_TSTAMP(1);
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;   // this warp's TMEM lane quarter
    const uint32_t tm_s = tmem;              // S^T: columns [0, 64)
    const uint32_t tm_o = tmem + 64;         // O^T block m: columns [64 + 64m, 128 + 64m)
    const int nmb = p.d_pad / 128;           // d blocks of 128
    uint32_t mma_phase = 0, gather_phase = 0;
    bool dead = false;

    const uint32_t idesc_qk = idesc_bf16_f32(128, kHp, false, false);
    const uint32_t idesc_pv = idesc_bf16_f32(128, kHp, true, true);
    const int32_t* idx_row = p.idx + (size_t)query * p.idx_stride;
    const int n_rows = p.n1 + p.n2;
    griddep_wait();   // the indices are complete from here on (Q, KV and the sink come from the caller)

    for (int tile = tile_begin; tile < tile_end; ++tile) {
        // ---- gather: thread r < 128 resolves slot r of the tile
        if (tid == 0) tl->rescale = 0;
        if (tid < kRows) {
            const int slot = slot_begin + tile * kRows + tid;
            int idx = slot < slot_end ? __ldg(idx_row + slot) : -1;
            if (idx < -1 || idx >= n_rows) {
                atomicOr(p.status, 1u /* STI_FLAG_INDEX_RANGE */);
                idx = -1;
            }
            const int srcid = idx < 0 ? -1 : (idx < p.n1 ? 0 : 1);
            // fp4 rows of the second source: coord is the row within its batch element, decoded below
            const bool fp4_row = srcid == 1 && f.on;
            const int64_t coord = srcid < 0 ? 0
                                  : (srcid == 0 ? b * p.rows1 + idx : (fp4_row ? idx - p.n1 : b * p.rows2 + (idx - p.n1)));
            const uint16_t* src = (srcid < 0 || fp4_row) ? nullptr : (srcid == 0 ? p.kv : p.kv2) + coord * p.d;
            tl->row_src[tid] = src;
            tl->row_valid[tid] = idx >= 0;
            tl->row_coord[tid] = (int)coord;
            tl->row_srcid[tid] = srcid;
            // the next tile's row goes to L2 now, so its gather does not wait on HBM
            const int nslot = slot + kRows;
            if (tile + 1 < tile_end && nslot < slot_end) {
                const int nidx = __ldg(idx_row + nslot);
                if (nidx >= 0 && nidx < n_rows && nidx >= p.n1 && f.on) {
                    const size_t r2 = (size_t)(nidx - p.n1);
                    prefetch_l2_bulk(f.codes + (size_t)b * f.codes_bstride + r2 * (p.d / 2), (uint32_t)p.d / 2);
                    if ((p.d / 16) % 16 == 0)
                        prefetch_l2_bulk(f.scales + (size_t)b * f.scales_bstride + r2 * (p.d / 16), (uint32_t)p.d / 16);
                } else if (nidx >= 0 && nidx < n_rows) {
                    const uint16_t* nsrc = nidx < p.n1 ? p.kv + (size_t)b * p.kv_bstride + (size_t)nidx * p.d
                                                       : p.kv2 + (size_t)b * p.kv2_bstride + (size_t)(nidx - p.n1) * p.d;
                    prefetch_l2_bulk(nsrc, (uint32_t)p.d * 2);
                }
            }
        }
        __syncthreads();
        const uint32_t kv_base = smem_u32(kv_s);
        const int chunks_per_row = p.d_pad / 8;
        if (p.use_tma) {
            // warp 0: lane g gathers rows 4g..4g+3, one 4-row TMA per 128-byte column block.  Masked
            // slots load a real row of the same source (their score is -inf, so P = 0); a group whose
            // rows come from both sources is copied with cp.async instead.
            if (tid < kRows) {   // rows of 4-row groups with no valid slot get no copy: zero them here
                const int g0 = tid & ~3;
                const bool all_masked = tl->row_srcid[g0] < 0 && tl->row_srcid[g0 + 1] < 0 &&
                                        tl->row_srcid[g0 + 2] < 0 && tl->row_srcid[g0 + 3] < 0;
                if (all_masked)
                    for (int cb = 0; cb < ncb_real; ++cb) {
                        uint4* row = reinterpret_cast<uint4*>(kv_s + (size_t)cb * kRows * 128 + (size_t)tid * 128);
#pragma unroll
                        for (int c = 0; c < 8; ++c) row[c] = make_uint4(0, 0, 0, 0);
                    }
            }
            {   // warp w issues column block w (one issue stream per warp)
                const int g = lane;
                int sid[4], crd[4];
                int S = -1, fc = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    sid[i] = tl->row_srcid[4 * g + i];
                    crd[i] = tl->row_coord[4 * g + i];
                    if (sid[i] >= 0 && S < 0) {
                        S = sid[i];
                        fc = crd[i];
                    }
                }
                bool mixed = false;
#pragma unroll
                for (int i = 0; i < 4; ++i) mixed = mixed || (sid[i] >= 0 && sid[i] != S);
                const bool empty = S < 0;   // zero-filled above

#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (sid[i] != S) crd[i] = fc;
                const unsigned tma_groups = __ballot_sync(kFull, !mixed && !empty);
                if (warp == 0 && lane == 0 && !dead)
                    mbar_arrive_expect_tx(&tl->gather_bar, (uint32_t)(__popc(tma_groups) * ncb_real * 512));
                __syncwarp();
                if (!dead && !empty) {
                    if (!mixed) {
                        const void* map = S == 0 ? (const void*)&tm_kv1 : (const void*)&tm_kv2;
                        for (int cb = warp; cb < ncb_real; cb += kThreads / 32)
                            tma_gather4(kv_s + (size_t)cb * kRows * 128 + (size_t)g * 512, map, &tl->gather_bar,
                                        cb * 64, crd[0], crd[1], crd[2], crd[3]);
                    } else if (warp == 0) {
                        for (int i = 0; i < 4; ++i) {
                            const int r = 4 * g + i;
                            const uint16_t* rs = tl->row_src[r];
                            for (int ch = 0; ch < chunks_per_row; ++ch) {
                                const bool ok = rs != nullptr && ch * 8 < p.d;
                                cp_async_16(kv_base + sw128_offset(r, ch, kRows), ok ? rs + ch * 8 : p.q,
                                            ok ? 16u : 0u);
                            }
                        }
                    }
                }
                cp_async_commit();
                cp_async_wait<0>();
            }
            if (tile == tile_begin && !dead) dead = !mbar_wait(&tl->q_bar, 0, p.status);
            if (!dead) dead = !mbar_wait(&tl->gather_bar, gather_phase, p.status);
            gather_phase ^= 1u;
        } else {
            for (int c = tid; c < kRows * chunks_per_row; c += kThreads) {
                const int r = c / chunks_per_row, ch = c - r * chunks_per_row;
                if (f.on && tl->row_srcid[r] == 1) {
                    // fp4 row: 4 code bytes and the E4M3 scale of their 16-element group -> 8 bf16
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (ch * 8 < p.d) {
                        const size_t r2 = (size_t)tl->row_coord[r];
                        const uint32_t cw = __ldg(reinterpret_cast<const uint32_t*>(
                                                      f.codes + (size_t)b * f.codes_bstride + r2 * (p.d / 2)) + ch);
                        const uint32_t sb = __ldg(f.scales + (size_t)b * f.scales_bstride + r2 * (p.d / 16) + (ch >> 1));
                        v = kvfp4_decode8(cw, e4m3_to_float(sb));
                    }
                    *reinterpret_cast<uint4*>(kv_s + sw128_offset(r, ch, kRows)) = v;
                    continue;
                }
                const uint16_t* rs = tl->row_src[r];
                const bool ok = rs != nullptr && ch * 8 < p.d;
                cp_async_16(kv_base + sw128_offset(r, ch, kRows), ok ? rs + ch * 8 : p.q, ok ? 16u : 0u);
            }
            cp_async_commit();
            cp_async_wait<0>();
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---- S^T = KV . Q^T
        if (tile < 2) STI_TSTAMP(2 + 4 * tile);
        if (tid == 0 && !dead) {
            tc_fence_after();
            const uint32_t a0 = smem_u32(kv_s), b0 = smem_u32(q_s);
            for (int kk = 0; kk < p.d_pad / 16; ++kk) {
                const uint32_t cb = (uint32_t)(kk >> 2), ko = (uint32_t)(kk & 3) * 32u;
                umma_bf16(tm_s, sdesc(a0 + cb * kRows * 128u + ko, 16, 1024, kLayoutSW128),
                          sdesc(b0 + cb * kHp * 128u + ko, 16, 1024, kLayoutSW128), idesc_qk, kk > 0 ? 1u : 0u);
            }
            umma_commit(&tl->mma_bar);
        }
        if (!dead) dead = !mbar_wait(&tl->mma_bar, mma_phase, p.status);
        mma_phase ^= 1u;
        tc_fence_after();

        // ---- online softmax (thread = row, 64 heads in registers)
        if (tile < 2) STI_TSTAMP(3 + 4 * tile);
        float x[32];   // this thread's row, heads [32*hg, 32*hg + 32)
        {
            uint32_t r0[32];
            tmem_ld32(tm_s + lane_base + (uint32_t)(32 * hg), r0);
            tmem_ld_wait();
            const bool valid = tl->row_valid[row] != 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = valid ? __uint_as_float(r0[i]) * p.scale_log2 : -INFINITY;
        }
        {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = x[i];
            warp_reduce_scatter32<true>(v);
            tl->red[warp & 3][32 * hg + lane] = v[0];
        }
        __syncthreads();
        if (tid < kHp) {
            const float mt = fmaxf(fmaxf(tl->red[0][tid], tl->red[1][tid]), fmaxf(tl->red[2][tid], tl->red[3][tid]));
            const float m_old = tl->m_run[tid];
            // keep the running max unless this tile's max passes it by more than 8 (log2 units):
            // every P stays <= 2^8, and O and l are rescaled only when some head's max moves
            const float m_new = (m_old == -INFINITY || mt > m_old + 8.f) ? fmaxf(m_old, mt) : m_old;
            const float a = (m_new == -INFINITY) ? 1.f : exp2f(m_old - m_new);
            tl->alpha[tid] = a;
            tl->m_run[tid] = m_new;
            if (a != 1.f) tl->rescale = 1;
        }
        __syncthreads();
        {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float m = tl->m_run[32 * hg + i];
                x[i] = (m == -INFINITY) ? 0.f : exp2f(x[i] - m);
                v[i] = x[i];
            }
            // P^T row: heads [32*hg, 32*hg+32) as bf16 = 16-byte chunks 4*hg .. 4*hg+3, swizzled
            uint8_t* prow = p_s + row * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint4 pk;
                pk.x = pack_bf16x2(x[8 * c + 0], x[8 * c + 1]);
                pk.y = pack_bf16x2(x[8 * c + 2], x[8 * c + 3]);
                pk.z = pack_bf16x2(x[8 * c + 4], x[8 * c + 5]);
                pk.w = pack_bf16x2(x[8 * c + 6], x[8 * c + 7]);
                *reinterpret_cast<uint4*>(prow + (((4 * hg + c) ^ (row & 7)) << 4)) = pk;
            }
            warp_reduce_scatter32<false>(v);
            tl->red[warp & 3][32 * hg + lane] = v[0];   // every read of the maxima preceded the last barrier
        }
        __syncthreads();
        if (tid < kHp)
            tl->l_run[tid] = tl->l_run[tid] * tl->alpha[tid] + (tl->red[0][tid] + tl->red[1][tid]) +
                             (tl->red[2][tid] + tl->red[3][tid]);
        // rescale the running O^T (lane = d within a block, column = head) when some max moved
        if (tile > tile_begin && !dead && tl->rescale) {
            for (int m = 0; m < nmb; ++m) {
                uint32_t r[32];
                const uint32_t ta = tm_o + lane_base + (uint32_t)(64 * m + 32 * hg);
                tmem_ld32(ta, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * tl->alpha[32 * hg + i]);
                tmem_st32(ta, r);
            }
            tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- O^T += V^T . P^T  (A = the same KV tile, MN-major; B = P^T, MN-major)
        if (tile < 2) STI_TSTAMP(4 + 4 * tile);
        if (tid == 0 && !dead) {
            tc_fence_after();
            const uint32_t a0 = smem_u32(kv_s), b0 = smem_u32(p_s);
            const uint32_t lbo_a = kRows * 128u;      // next 64-column block of the tile
            for (int m = 0; m < nmb; ++m)
                for (int kk = 0; kk < kRows / 16; ++kk)
                    umma_bf16(tm_o + (uint32_t)(64 * m),
                              sdesc(a0 + (uint32_t)(2 * m) * lbo_a + (uint32_t)kk * 2048u, lbo_a, 1024, kLayoutSW128),
                              sdesc(b0 + (uint32_t)kk * 2048u, kRows * 128u, 1024, kLayoutSW128), idesc_pv,
                              (tile > tile_begin || kk > 0) ? 1u : 0u);
            umma_commit(&tl->mma_bar);
        }
        if (!dead) dead = !mbar_wait(&tl->mma_bar, mma_phase, p.status);
        mma_phase ^= 1u;
        tc_fence_after();
        if (tile < 2) STI_TSTAMP(5 + 4 * tile);
    }

    STI_TSTAMP(10);
    // ---- epilogue: O^T (lane = d, column = head) -> output or split partial
    cp_async_wait<0>();   // Q's copy when this CTA had no tile
    if (p.use_tma && tile_begin == tile_end) mbar_wait(&tl->q_bar, 0, p.status);
    __syncthreads();
    const bool has_tiles = tile_begin < tile_end && !dead;
    if (C == 1) {
        // final: o = O / (l + 2^(sink*log2e - m)); empty rows (m = -inf) give 0
        if (tid < kHp) {
            const float m = tl->m_run[tid];
            float inv = 0.f, lse = -INFINITY;
            if (m != -INFINITY && tid < p.h) {
                const float den = tl->l_run[tid] + exp2f(__ldg(p.sink + tid) * kLog2e - m);
                inv = 1.f / den;
                lse = (m + log2f(den)) * kLn2;
            }
            tl->alpha[tid] = inv;
            if (p.lse && tid < p.h) p.lse[(size_t)query * p.h + tid] = lse;
        }
        __syncthreads();
        // the query's [h][d] bf16 output, staged in the free Q buffer, leaves in one bulk store
        uint16_t* stage = reinterpret_cast<uint16_t*>(q_s);
        for (int m = 0; m < nmb; ++m) {
            const int dd = 128 * m + row;
            {
                const int half = hg;   // this thread's 32 head columns
                uint32_t r[32];
                if (has_tiles) {
                    tmem_ld32(tm_o + lane_base + (uint32_t)(64 * m + 32 * half), r);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = 0u;
                }
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * tl->alpha[32 * half + i];
                if (p.rope_dims > 0 && 128 * m + 128 > p.d - p.rope_dims)   // the output's inverse rotation
                    rope_inverse_pairs<32>(v, dd, p.d, p.rope_dims, p.rope_cs + (size_t)query * p.rope_dims);
                if (dd < p.d) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int hh = 32 * half + i;
                        if (hh < p.h) stage[(size_t)hh * p.d + dd] = __bfloat16_as_ushort(__float2bfloat16_rn(v[i]));
                    }
                }
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            bulk_store(p.out + (size_t)query * p.h * p.d, stage, (uint32_t)(p.h * p.d * 2));
            bulk_commit();
            bulk_wait_read_all();   // the stage may be released; the writes complete with the grid
        }
    } else {
        // ---- split query.  The CTAs of the cluster exchange their (m, l) in distributed shared
        // memory; each scales its O^T by 2^(m_cta - M) / L and adds it into the query's fp32
        // accumulator in global memory with bulk reductions (performed at L2).  After a cluster
        // barrier rank r converts columns [r*dper, (r+1)*dper) of every head to bf16 and zeroes
        // them again for the next call.
        if (!has_tiles && tid < kHp) tl->m_run[tid] = -INFINITY;   // nothing valid here
        const int dper = p.d / C;                  // multiple of 32 (host choice)
        cluster_sync();                            // every CTA's m, l are final
        STI_TSTAMP(11);
        if (tid < kHp) {
            float mr[8], lr[8];                    // every partner's (m, l) in flight at once
#pragma unroll
            for (int r = 0; r < 8; ++r)
                if (r < C) {
                    mr[r] = ld_dsmem_f32(dsmem_addr(&tl->m_run[tid], (uint32_t)r));
                    lr[r] = ld_dsmem_f32(dsmem_addr(&tl->l_run[tid], (uint32_t)r));
                }
            float M = -INFINITY;
#pragma unroll
            for (int r = 0; r < 8; ++r)
                if (r < C) M = fmaxf(M, mr[r]);
            float L = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    if (r < C && mr[r] != -INFINITY) L += lr[r] * exp2f(mr[r] - M);
                if (tid < p.h) L += exp2f(__ldg(p.sink + tid) * kLog2e - M);
            }
            const float mo = tl->m_run[tid];
            tl->alpha[tid] = (M == -INFINITY || mo == -INFINITY || L == 0.f) ? 0.f : exp2f(mo - M) / L;
            if (rank == 0 && p.lse && tid < p.h)
                p.lse[(size_t)query * p.h + tid] = (M == -INFINITY) ? -INFINITY : (M + log2f(L)) * kLn2;
        }
        __syncthreads();
        float* acc_q = p.acc + (size_t)query * p.h * p.d;
        if (has_tiles) {
            // scaled O^T -> [h][d] fp32 in the freed KV tile (h*d*4 <= 64*d_pad*4 bytes), one
            // bulk reduction per head row
            float* stage = reinterpret_cast<float*>(kv_s);
            for (int m = 0; m < nmb; ++m) {
                const int dd = 128 * m + row;
                uint32_t v[32];
                tmem_ld32(tm_o + lane_base + (uint32_t)(64 * m + 32 * hg), v);
                tmem_ld_wait();
                if (dd < p.d) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int hh = 32 * hg + i;
                        if (hh < p.h) stage[(size_t)hh * p.d + dd] = __uint_as_float(v[i]) * tl->alpha[hh];
                    }
                }
            }
            fence_proxy_async_smem();              // the bulk-copy engine reads these writes
            __syncthreads();
            if (tid < p.h) {
                bulk_reduce_add_f32(acc_q + (size_t)tid * p.d, stage + (size_t)tid * p.d, (uint32_t)p.d * 4u);
                bulk_commit();
                bulk_wait_all();                   // the additions are performed
            }
            fence_proxy_async_global();
        }
        cluster_sync();                            // every partial is in the accumulator
        STI_TSTAMP(12);
        // this rank's columns: fp32 sums -> bf16 output, accumulator back to zero
        const int q4 = dper / 4;                   // float4 per head row of this rank's slice
        uint16_t* orow = p.out + (size_t)query * p.h * p.d + (size_t)rank * dper;
        float* arow = acc_q + (size_t)rank * dper;
        for (int e0 = 0; e0 < p.h * q4; e0 += 4 * kThreads) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = e0 + u * kThreads + tid;
                if (e < p.h * q4) {
                    const int hh = e / q4, c4 = e - (e / q4) * q4;
                    v[u] = __ldcg(reinterpret_cast<const float4*>(arow + (size_t)hh * p.d) + c4);
                }
            }
            if (p.rope_dims > 0) {   // the output's inverse rotation: pairs (x, y), (z, w) of each float4
                const float* cs = p.rope_cs + (size_t)query * p.rope_dims;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int e = e0 + u * kThreads + tid;
                    if (e < p.h * q4) {
                        const int c4 = e - (e / q4) * q4;
                        const int dd = rank * dper + 4 * c4;
                        float* f = reinterpret_cast<float*>(&v[u]);
#pragma unroll
                        for (int pr = 0; pr < 2; ++pr) {
                            const int dp = dd + 2 * pr;
                            if (dp >= p.d - p.rope_dims) {
                                const int i = (dp - (p.d - p.rope_dims)) >> 1;
                                const float c = __ldg(cs + 2 * i), sn = __ldg(cs + 2 * i + 1);
                                const float x = f[2 * pr], y = f[2 * pr + 1];
                                f[2 * pr] = x * c + y * sn;
                                f[2 * pr + 1] = y * c - x * sn;
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = e0 + u * kThreads + tid;
                if (e < p.h * q4) {
                    const int hh = e / q4, c4 = e - (e / q4) * q4;
                    uint2 o;
                    o.x = pack_bf16x2(v[u].x, v[u].y);
                    o.y = pack_bf16x2(v[u].z, v[u].w);
                    *reinterpret_cast<uint2*>(orow + (size_t)hh * p.d + 4 * c4) = o;
                    __stcg(reinterpret_cast<float4*>(arow + (size_t)hh * p.d) + c4, make_float4(0.f, 0.f, 0.f, 0.f));
                }
            }
        }
        STI_TSTAMP(13);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    STI_TSTAMP(14);
}

size_t attn_smem_bytes(int d_pad) {
    return 1024 + (size_t)kHp * d_pad * 2 + (size_t)kRows * d_pad * 2 + kRows * 128 + sizeof(AttnSmemTail);
}

}  // namespace

static int attn_pick_cluster_uncached(int n_queries, int k, int d) {
    const int num_sms = device_num_sms();
    const int max_c = (k + 63) / 64;          // at least 64 slots per CTA
    int c = n_queries > 0 ? num_sms / n_queries : 1;
    if (c > max_c) c = max_c;
    // 2, 4 or 8 CTAs (portable cluster sizes); after the reduction each converts a slice of
    // d/c columns, d a multiple of 128 and the slice a multiple of 32
    c = c >= 8 ? 8 : (c >= 4 ? 4 : (c >= 2 ? 2 : 1));
    if (d % 128 != 0) c = 1;
    while (c > 1 && (d / c) % 32 != 0) c /= 2;
    if (c <= 1) return 1;
    // shrink the cluster until all queries' clusters are resident at once
    const size_t smem = attn_smem_bytes(512);
    cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    for (; c > 1; c /= 2) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(n_queries * c));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)c;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, sparse_attn_kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (active >= n_queries) return c;
    }
    return 1;
}

int attn_pick_cluster(int n_queries, int k, int d) {
    struct Entry {
        int dev, n_queries, k, d, c;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> g(mu);
        for (const Entry& e : cache)
            if (e.dev == dev && e.n_queries == n_queries && e.k == k && e.d == d) return e.c;
    }
    const int c = attn_pick_cluster_uncached(n_queries, k, d);
    std::lock_guard<std::mutex> g(mu);
    if (cache.size() < 4096) cache.push_back({dev, n_queries, k, d, c});
    return c;
}

cudaError_t launch_sparse_attn(const CUtensorMap& tm_q, const CUtensorMap& tm_kv1, const CUtensorMap& tm_kv2,
                               const AttnParams& p, cudaStream_t stream) {
    KvFp4 none{};
    return launch_sparse_attn_kvfp4(tm_q, tm_kv1, tm_kv2, p, none, stream);
}

cudaError_t launch_sparse_attn_kvfp4(const CUtensorMap& tm_q, const CUtensorMap& tm_kv1, const CUtensorMap& tm_kv2,
                                     const AttnParams& p, const KvFp4& f, cudaStream_t stream) {
    if (f.on && p.use_tma) return cudaErrorInvalidValue;
    const int n_queries = p.B * p.s;
    if (n_queries == 0) return cudaSuccess;
    const size_t smem = attn_smem_bytes(p.d_pad);
    cudaError_t err =
        cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_queries * p.cluster));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (p.cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)p.cluster;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (p.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (unsigned)na;
    err = cudaLaunchKernelEx(&cfg, sparse_attn_kernel, tm_q, tm_kv1, tm_kv2, p, f);
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace sti

#ifdef STI_ATTN_TIMING
// profiling builds only: per-CTA clock64 stamps of the attention phases
extern "C" int sti_dbg_attn_times(unsigned long long* host, int n_blocks) {
    return (int)cudaMemcpyFromSymbol(host, sti::g_attn_t, sizeof(unsigned long long) * 16 * (size_t)n_blocks);
}
#endif
