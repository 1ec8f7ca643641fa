// sparse_attn_hs.cu -- sparse multi-head attention with an attention sink for few queries
// (decode): a thread-block cluster per query splits the query's HEADS, and every KV tile is
// gathered once into the shared memory of all CTAs of the cluster.
//
// DeepSeek V4.1, attention "attend/selected" page, sparse_attn_kernel / sparse_attn:
//   for every query and head, over the slots i whose index is not -1:
//     s_i = softmax_scale * q . kv[idx_i];  o = sum_i e^{s_i} kv[idx_i] / (sum_i e^{s_i} + e^{sink_h})
//   the same row serving as key and value; a query with no valid slot gets 0.
//
// Why a head split: the heads of a query share every KV row, so a partial output over some rows
// is as large as all heads' outputs (h x d fp32 = 128 KB for 64 x 512) -- splitting a query's
// rows over CTAs makes them add up partials larger than the rows they read.  Splitting the heads
// needs no reduction at all, provided each row is fetched once for the whole cluster:
//   * cluster of C CTAs per query, CTA r owning heads [r*HC, (r+1)*HC) (HC = 16 or 32);
//   * a tile = 128 KV rows = d/64 column blocks of 128 rows x 128 bytes (128-byte swizzle), held
//     in a ring of S column-block slots.  CTA r gathers the tile's four-row groups g = r (mod C)
//     with one TMA gather4 per column block, multicast to every CTA of the cluster, so each CTA
//     receives the whole tile while issuing 1/C of it;
//   * a slot is refilled only when all C CTAs have finished the PV product reading it: each CTA's
//     MMA completion arrives on that slot's "empty" barrier in every CTA (multicast commit);
//   * warp 0 resolves slots and issues the gathers, warp 1 allocates TMEM and issues the MMAs,
//     warps 2-5 run the online softmax (thread = KV row) and the epilogue;
//   * S^T = KV_tile . Q_r^T (tcgen05, M=128 rows x N=HC x K=d) accumulates column block by column
//     block as the blocks land; O^T += V^T . P^T (M=128 d-block x N=HC x K=128 rows) reads the same
//     tile as an MN-major operand, P^T being K-major bf16 [HC][128];
//   * the output of the CTA's heads ([HC][d] bf16, contiguous) leaves in one bulk store.
// Four-row groups with no valid slot are not fetched (their rows keep finite earlier contents,
// the ring starting zeroed, and get probability 0); masked slots inside a group repeat one of
// the group's valid rows; a group with rows of both sources fetches row by row.
#include <cuda_bf16.h>
#include <cstddef>
#include <math.h>

#include <mutex>
#include <vector>

#include "sti_internal.h"
#include "sti_ptx.cuh"
#include "sti_attn_util.cuh"

namespace sti {
namespace {

#ifdef STI_ATTN_TIMING
__device__ unsigned long long g_hs_p[2048][40];   // producer: per tile and column block, empty wait done
__device__ unsigned long long g_hs_e[2048][8];    // row-split merge phases
#define STI_ESTAMP(i)                                                                                  \
    do {                                                                                               \
        if (blockIdx.x < 2048) g_hs_e[blockIdx.x][i] = clock64();                                      \
    } while (0)
#else
#define STI_ESTAMP(i) \
    do {              \
    } while (0)
#endif
#ifdef STI_ATTN_TIMING
__device__ unsigned long long g_hs_t[2048][32];
#define STI_HSTAMP(i)                                                                                  \
    do {                                                                                               \
        if (blockIdx.x < 2048) g_hs_t[blockIdx.x][i] = clock64();                                      \
    } while (0)
#else
#define STI_HSTAMP(i) \
    do {              \
    } while (0)
#endif

constexpr int kHsThreads = 416;   // warps 0, 6, 7, 8 produce, 1 issues MMAs, 2-5 and 9-12 run the softmax
constexpr int kProducers = 4;
constexpr int kHsRows = 128;
constexpr int kHsMaxSlots = 12;
constexpr uint32_t kSlotBytes = kHsRows * 128;   // one column block of a tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr uint32_t kFull = 0xFFFFFFFFu;

struct __align__(16) HsTail {
    uint64_t full[kHsMaxSlots];    // slot filled (1 local arrival + the tile's bytes)
    uint64_t empty[kHsMaxSlots];   // slot read by every CTA of the cluster (C arrivals)
    uint64_t s_full[2];            // S^T of a tile in TMEM (double buffer)
    uint64_t p_full;               // P^T written, O^T rescaled
    uint64_t o_done;               // PV product of a tile complete
    uint64_t q_bar;                // Q rows of this CTA's heads landed
    uint64_t recv_bar;             // row-split merge: the partner's partial and (m, l) landed
    uint64_t ready_bar;            // row-split merge: the partner's ring is free to receive
    uint64_t rope_bar;             // the output-rotation table landed in rope_cs
    float peer_ml[64][2];          // row-split merge: the partner's (m, l) per head
    uint32_t tmem_base;
    int abort;                     // a wait of this CTA timed out: the others stop waiting
    float m_run[64];               // running max per head, log2 domain
    float l_run[64];               // running sum of 2^(x - m)
    float alpha[64];               // rescale factor of this tile / final 1 / denominator
    float red_max[4][64];          // per-warp partial maxima
    float red_sum[4][64];          // per-warp partial sums
    alignas(16) float rope_cs[128];   // the query's output-rotation table (rope_dims <= 128): a bulk
                                      // copy's destination, 16-byte aligned
};
static_assert(offsetof(HsTail, rope_cs) % 16 == 0, "bulk-copy destination must be 16-byte aligned");

// S^T double buffer (2 x hc columns) and O^T (d/128 blocks of hc columns, d <= 512)
__host__ __device__ constexpr uint32_t hs_tmem_cols(int hc) { return hc == 16 ? 128u : (hc == 32 ? 256u : 512u); }

__host__ __device__ constexpr size_t hs_smem_bytes(int hc, int d, int slots) {
    return 1024 + (size_t)slots * kSlotBytes + (size_t)hc * d * 2 + (size_t)hc * 256 + sizeof(HsTail);
}

template <int HC>
__global__ void __launch_bounds__(kHsThreads, 1)
    sparse_attn_hs_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv1,
                          const __grid_constant__ CUtensorMap tm_kv2, const __grid_constant__ CUtensorMap tm_win,
                          const AttnParams p, int n_slots) {
    static_assert(HC == 16 || HC == 32 || HC == 64, "16, 32 or 64 heads per CTA");
    constexpr int kSets = HC >= 32 ? 2 : 1;   // softmax warp groups, each over NH heads of every row
    constexpr int NH = HC / kSets;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int S = n_slots;                                      // even, >= 2
    uint8_t* ring = smem;                                       // S x [128 rows x 128 B], SW128
    uint8_t* q_s = ring + (size_t)S * kSlotBytes;               // [d/64] x [HC x 128 B], SW128 K-major
    uint8_t* p_s = q_s + (size_t)HC * p.d * 2;                  // P^T: [2] x [HC x 128 B], SW128 K-major
    HsTail* tl = reinterpret_cast<HsTail*>(p_s + HC * 256);
    volatile int* abort = &tl->abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C = p.cluster;                  // CTAs per query = CH head groups x CR row groups
    const int CR = p.hs_rows, CH = p.cluster / p.hs_rows;
    const int query = blockIdx.x / C, rank = blockIdx.x - (blockIdx.x / C) * C;
    const int hg = rank % CH, rg = rank / CH;   // this CTA's heads [hg*HC, +HC) and row group
    const int b = query / p.s;
    const int ncb = p.d / 64;                 // column blocks per tile
    const int nmb = p.d / 128;                // d blocks of the PV product
    // the row group's slots [r0, r1) of the query's index row, in tiles of 128.  With a window
    // ring the first group also takes the ring tile, which it runs before the indices exist, so
    // the groups split the remaining slots evenly in whole tiles
    const int pre = (p.win_ring == kHsRows && CR == 2 && p.k > kHsRows) ? kHsRows : 0;
    const int rows_rg = pre + (((p.k - pre + CR - 1) / CR + kHsRows - 1) / kHsRows) * kHsRows;
    const int r0 = rg == 0 ? 0 : min(p.k, rows_rg), r1 = rg == 0 ? min(p.k, rows_rg) : p.k;
    const int n_tiles = (r1 - r0 + kHsRows - 1) / kHsRows;
    // the CTAs that share this row group's tiles (multicast targets, slot releases)
    const uint16_t cta_mask = (uint16_t)(((1u << CH) - 1u) << (rg * CH));
    const int n_rows = p.n1 + p.n2;
    const int32_t* idx_row = p.idx + (size_t)query * p.idx_stride;
    // a full window ring is tile 0, loaded as one block in ring-row order (the attention does not
    // depend on slot order); it needs no index, so it runs before the indices are complete
    const bool ring_tile = p.win_ring == kHsRows && r0 == 0 && r1 - r0 >= kHsRows &&
                           __ldg(p.start_pos + b) >= kHsRows - 1;
    if (tid == 0) STI_HSTAMP(0);
#ifdef STI_ATTN_TIMING
    if (tid == 0 && blockIdx.x < 2048) g_hs_t[blockIdx.x][30] = global_timer_ns();
#endif

    if (warp == 1) {
        tmem_alloc(&tl->tmem_base, hs_tmem_cols(HC));
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&tl->full[i], 1);
            mbar_init(&tl->empty[i], (uint32_t)CH);
        }
        mbar_init(&tl->s_full[0], 1);
        mbar_init(&tl->s_full[1], 1);
        mbar_init(&tl->p_full, (uint32_t)kSets);
        mbar_init(&tl->o_done, 1);
        mbar_init(&tl->q_bar, 1);
        mbar_init(&tl->recv_bar, 1);
        mbar_init(&tl->ready_bar, 1);
        mbar_init(&tl->rope_bar, 1);
        // row-split merge: the partner's half of d for this CTA's heads, [d/2][HC] fp32, and (m, l)
        if (CR == 2) mbar_arrive_expect_tx(&tl->recv_bar, (uint32_t)(p.d / 2 * HC * 4 + HC * 8));
        tl->abort = 0;
        fence_mbar_init();
    }
    if (tid < HC) {
        tl->m_run[tid] = -INFINITY;
        tl->l_run[tid] = 0.f;
    }
    // the output rotation's table is an input of the call (no earlier kernel writes it): one bulk
    // copy into shared memory now, waited for in the epilogue, keeps its latency off the path
    // (a row of 16-byte multiple, at most 128 values; otherwise the epilogue reads global memory)
    const bool rope_smem = p.rope_dims > 0 && p.rope_dims <= 128 && p.rope_dims % 4 == 0;
    const float* rope_tab = rope_smem ? tl->rope_cs : p.rope_cs + (size_t)query * p.rope_dims;
    {   // rows that no gather writes keep finite contents
        uint4* r4 = reinterpret_cast<uint4*>(ring);
        const int n16 = S * (int)kSlotBytes / 16;
        for (int i = tid; i < n16; i += kHsThreads) r4[i] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    cluster_sync();   // every CTA's barriers initialised and ring zeroed before any multicast
    tc_fence_after();
    const uint32_t tmem = tl->tmem_base;
    if (tid == 0) STI_HSTAMP(1);
    if (rope_smem && tid == 0) {
        mbar_arrive_expect_tx(&tl->rope_bar, (uint32_t)p.rope_dims * 4u);
        bulk_load(tl->rope_cs, p.rope_cs + (size_t)query * p.rope_dims, (uint32_t)p.rope_dims * 4u, &tl->rope_bar);
    }

    if (warp == 0 || (warp >= 6 && warp <= 8)) {
        // ------------------------------------------------------------ producers
        // producer pi owns the ring slots = pi (mod 4): it waits, arms and fills only those, so
        // four issue streams of TMA gathers run side by side
        const int pi = warp == 0 ? 0 : warp - 5;
        if (warp == 0 && lane == 0) {
            tma_prefetch_desc(&tm_kv1);
            tma_prefetch_desc(&tm_kv2);
            mbar_arrive_expect_tx(&tl->q_bar, (uint32_t)(HC * p.d * 2));
            for (int cb = 0; cb < ncb; ++cb)
                tma_load_2d(q_s + (size_t)cb * HC * 128, &tm_q, &tl->q_bar, cb * 64, query * p.h + hg * HC);
        }
        bool dead = false;
        const bool mine = (lane % CH) == hg;   // four-row group g = lane is this CTA's to fetch
        int t_first = 0;
        if (ring_tile) {   // slots 0..ncb-1 are free on first use: no wait
            if (lane == 0) {
                for (int j = pi; j < ncb; j += kProducers) {   // tile 0: column block j in slot j
                    mbar_arrive_expect_tx(&tl->full[j], kSlotBytes);
                    if (CH == 1)
                        tma_load_2d(ring + (size_t)j * kSlotBytes, &tm_win, &tl->full[j], j * 64, b * (int)p.rows1);
                    else if (hg == 0)
                        tma_load_2d_mc(ring + (size_t)j * kSlotBytes, &tm_win, &tl->full[j], j * 64, b * (int)p.rows1,
                                       cta_mask);
                }
            }
            __syncwarp();
            t_first = 1;
        }
        griddep_wait();   // the indices are complete from here on
#ifdef STI_ATTN_TIMING
        if (pi == 0 && lane == 0 && blockIdx.x < 2048) g_hs_e[blockIdx.x][5] = global_timer_ns();
#endif
        for (int t = t_first; t < n_tiles && !dead; ++t) {
            int sid[4], crd[4];
            int first_s = -1, first_c = 0, n_valid = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int slot = r0 + t * kHsRows + 4 * lane + i;
                int idx = slot < r1 ? __ldg(idx_row + slot) : -1;
                if (idx < -1 || idx >= n_rows) {
                    if (rank == 0 && pi == 0) atomicOr(p.status, 1u /* STI_FLAG_INDEX_RANGE */);
                    idx = -1;
                }
                sid[i] = idx < 0 ? -1 : (idx < p.n1 ? 0 : 1);
                crd[i] = sid[i] < 0 ? 0 : (sid[i] == 0 ? b * (int)p.rows1 + idx : b * (int)p.rows2 + (idx - p.n1));
                if (sid[i] >= 0) {
                    ++n_valid;
                    if (first_s < 0) {
                        first_s = sid[i];
                        first_c = crd[i];
                    }
                }
            }
            bool mixed = false;
#pragma unroll
            for (int i = 0; i < 4; ++i) mixed = mixed || (sid[i] >= 0 && sid[i] != first_s);
            const bool empty = first_s < 0;
            uint32_t tbytes = empty ? 0u : (mixed ? 128u * (uint32_t)n_valid : 512u);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) tbytes += __shfl_xor_sync(kFull, tbytes, o);
            const void* map = first_s == 1 ? (const void*)&tm_kv2 : (const void*)&tm_kv1;
            // the next tile's rows go to L2 now (this CTA's groups, split over the producers), so its
            // gathers -- issued when PV of this tile frees their slots -- do not wait on HBM
            if (t + 1 < n_tiles && (lane % CH) == hg && ((lane / CH) % kProducers) == pi) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int slot = r0 + (t + 1) * kHsRows + 4 * lane + i;
                    const int idx = slot < r1 ? __ldg(idx_row + slot) : -1;
                    if (idx >= 0 && idx < n_rows) {
                        const uint16_t* row_ptr = idx < p.n1 ? p.kv + (size_t)b * p.kv_bstride + (size_t)idx * p.d
                                                             : p.kv2 + (size_t)b * p.kv2_bstride + (size_t)(idx - p.n1) * p.d;
                        prefetch_l2_bulk(row_ptr, (uint32_t)p.d * 2u);
                    }
                }
            }
            for (int j = 0; j < ncb; ++j) {
                const int G = t * ncb + j, slot = G % S, use = G / S;
                if (slot % kProducers != pi) continue;
                if (use > 0 && !dead) dead = !attn_wait(&tl->empty[slot], (uint32_t)((use - 1) & 1), p.status, abort);
#ifdef STI_ATTN_TIMING
                (void)0;
#endif
                dead = __any_sync(kFull, dead);
                if (dead) break;
                uint8_t* dst = ring + (size_t)slot * kSlotBytes;
                if (lane == 0) mbar_arrive_expect_tx(&tl->full[slot], tbytes);
                if (mine && !empty) {
                    if (!mixed) {
                        // masked rows of the group repeat its first valid row
                        const int y0 = sid[0] >= 0 ? crd[0] : first_c, y1 = sid[1] >= 0 ? crd[1] : first_c;
                        const int y2 = sid[2] >= 0 ? crd[2] : first_c, y3 = sid[3] >= 0 ? crd[3] : first_c;
                        if (CH == 1)
                            tma_gather4(dst + lane * 512, map, &tl->full[slot], j * 64, y0, y1, y2, y3);
                        else
                            tma_gather4_mc(dst + lane * 512, map, &tl->full[slot], j * 64, y0, y1, y2, y3, cta_mask);
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (sid[i] >= 0) {
                                const void* m = sid[i] == 1 ? (const void*)&tm_kv2 : (const void*)&tm_kv1;
                                if (CH == 1)
                                    tma_load_2d(dst + (4 * lane + i) * 128, m, &tl->full[slot], j * 64, crd[i]);
                                else
                                    tma_load_2d_mc(dst + (4 * lane + i) * 128, m, &tl->full[slot], j * 64, crd[i],
                                                   cta_mask);
                            }
                    }
                }
            }
            if (pi == 0 && lane == 0 && t < 5) STI_HSTAMP(2 + t);
        }
        // every arrival the cluster makes on this CTA's barriers has landed before it may exit
        const int total = n_tiles * ncb;
        for (int s2 = pi; s2 < S && s2 < total && !dead; s2 += kProducers) {
            const int uses = (total - s2 + S - 1) / S;
            dead = !attn_wait(&tl->empty[s2], (uint32_t)((uses - 1) & 1), p.status, abort);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            bool dead = !attn_wait(&tl->q_bar, 0, p.status, abort);
            const uint32_t idesc_qk = idesc_bf16_f32(kHsRows, HC, false, false);
            const uint32_t idesc_pv = idesc_bf16_f32(128, HC, true, false);
            const uint32_t q0 = smem_u32(q_s), p0 = smem_u32(p_s), r0 = smem_u32(ring);
            // descriptors advance by their 16-byte address units: +2 per 32-byte K step
            const uint64_t qd0 = sdesc(q0, 16, 1024, kLayoutSW128);
            const uint64_t pd0 = sdesc(p0, 16, 1024, kLayoutSW128);
            const uint64_t kd0 = sdesc(r0, 16, 1024, kLayoutSW128);               // K-major tile
            const uint64_t vd0 = sdesc(r0, kSlotBytes, 1024, kLayoutSW128);       // MN-major tile
            int qk_t = 0, qk_j = 0;   // next QK column block to issue
            // QK for column block (qk_t, qk_j); `block`: wait for its data, else only if landed
            auto issue_qk = [&](bool block) -> bool {
                const int G = qk_t * ncb + qk_j, slot = G % S, use = G / S;
                if (block) {
                    if (!attn_wait(&tl->full[slot], (uint32_t)(use & 1), p.status, abort)) return false;
                } else if (!mbar_test_wait(&tl->full[slot], (uint32_t)(use & 1))) {
                    return false;
                }
                tc_fence_after();
                const uint32_t ts = tmem + (uint32_t)((qk_t & 1) * HC);
                const uint64_t a = kd0 + (uint64_t)((uint32_t)slot * (kSlotBytes >> 4));
                const uint64_t bq = qd0 + (uint64_t)((uint32_t)(qk_j * HC * 128) >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(ts, a + 2 * kk, bq + 2 * kk, idesc_qk, (qk_j > 0 || kk > 0) ? 1u : 0u);
                if (++qk_j == ncb) {
                    if (qk_t < 5) STI_HSTAMP(7 + qk_t);
                    umma_commit(&tl->s_full[qk_t & 1]);
                    qk_j = 0;
                    ++qk_t;
                }
                return true;
            };
            for (int t = 0; t < n_tiles && !dead; ++t) {
                while (qk_t == t && !dead) dead = !issue_qk(true);   // the rest of QK(t)
                if (dead) break;
                // while the softmax of tile t runs, QK of tile t+1 on column blocks already landed
                // (it writes the other S^T buffer, whose softmax finished before PV(t-1))
                {
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_test_wait(&tl->p_full, (uint32_t)(t & 1))) {
                        if (qk_t == t + 1 && qk_t < n_tiles && issue_qk(false)) continue;
                        if (*abort || global_timer_ns() - t0 > STI_WAIT_TIMEOUT_NS) {
                            if (!*abort) atomicOr(p.status, 2u /* STI_FLAG_TIMEOUT */);
                            *abort = 1;
                            dead = true;
                            break;
                        }
                    }
                }
                if (dead) break;
                tc_fence_after();
#ifdef STI_ATTN_TIMING
                if (t < 5 && blockIdx.x < 2048) g_hs_p[blockIdx.x][t * 8 + 0] = clock64();
#endif
                for (int m = 0; m < nmb; ++m) {
                    const int slot = (t * ncb + 2 * m) % S;   // column blocks 2m, 2m+1: adjacent slots
                    const uint64_t a = vd0 + (uint64_t)((uint32_t)slot * (kSlotBytes >> 4));
#pragma unroll
                    for (int kk = 0; kk < kHsRows / 16; ++kk)
                        umma_bf16(tmem + (uint32_t)(2 * HC + m * HC), a + (uint64_t)(kk * (2048 >> 4)),
                                  pd0 + (uint64_t)(((kk >> 2) * HC * 128 + (kk & 3) * 32) >> 4), idesc_pv,
                                  (t > 0 || kk > 0) ? 1u : 0u);
#ifdef STI_ATTN_TIMING
                    if (t < 5 && blockIdx.x < 2048) g_hs_p[blockIdx.x][t * 8 + 1 + 2 * m] = clock64();
#endif
                    if (CH == 1) {
                        umma_commit(&tl->empty[slot]);
                        umma_commit(&tl->empty[slot + 1]);
                    } else {
                        umma_commit_mc(&tl->empty[slot], cta_mask);
                        umma_commit_mc(&tl->empty[slot + 1], cta_mask);
                    }
#ifdef STI_ATTN_TIMING
                    if (t < 5 && blockIdx.x < 2048) g_hs_p[blockIdx.x][t * 8 + 2 + 2 * m] = clock64();
#endif
                }
                umma_commit(&tl->o_done);
                if (t < 5) STI_HSTAMP(25 + t);
            }
        }
        __syncwarp();
    } else if ((warp >= 2 && warp <= 5) || (kSets == 2 && warp >= 9)) {
        // ------------------------------------------------------------ softmax
        // kSets groups of four warps; set s owns heads [s*NH, s*NH + NH) of every row
        const int set = warp >= 9 ? 1 : 0;
        const int qd = warp & 3;                       // TMEM lane quarter of this warp
        const int row = 32 * qd + lane;                // KV row of the tile
        const int st = tid - (set == 0 ? 64 : 288);    // 0..127 within the set
        const int hoff = set * NH;
        const uint32_t bar_id = 1u + (uint32_t)set;
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        constexpr int kSpread = 32 / NH;               // lanes holding one head after a reduce-scatter
        if (!ring_tile) griddep_wait();
        bool dead = false;
        for (int t = 0; t < n_tiles; ++t) {
            if (ring_tile && t == 1) griddep_wait();
            bool valid = true;   // the full ring: every row valid
            if (!(ring_tile && t == 0)) {
                const int slot_i = r0 + t * kHsRows + row;
                const int idx = slot_i < r1 ? __ldg(idx_row + slot_i) : -1;
                valid = idx >= 0 && idx < n_rows;
            }
            if (!dead) dead = !attn_wait(&tl->s_full[t & 1], (uint32_t)((t >> 1) & 1), p.status, abort);
            if (set == 0 && st == 0 && t < 5) STI_HSTAMP(15 + t);
            tc_fence_after();
            float x[NH];
            {
                uint32_t r[NH];
                tmem_ld_n<NH>(tmem + lane_base + (uint32_t)((t & 1) * HC + hoff), r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < NH; ++i) x[i] = valid ? __uint_as_float(r[i]) * p.scale_log2 : -INFINITY;
            }
            {
                float v[NH];
#pragma unroll
                for (int i = 0; i < NH; ++i) v[i] = x[i];
                warp_reduce_scatter_n<NH, true>(v);
                if ((lane & (kSpread - 1)) == 0) tl->red_max[qd][hoff + lane / kSpread] = v[0];
            }
            named_bar_sync(bar_id, 128);
            if (st < NH) {
                const int hh = hoff + st;
                const float mt = fmaxf(fmaxf(tl->red_max[0][hh], tl->red_max[1][hh]),
                                       fmaxf(tl->red_max[2][hh], tl->red_max[3][hh]));
                const float m_old = tl->m_run[hh];
                // the running max moves only when a tile's max passes it by more than 8 (log2
                // units): every P stays <= 2^8 and O, l are rescaled only when a max moves
                const float m_new = (m_old == -INFINITY || mt > m_old + 8.f) ? fmaxf(m_old, mt) : m_old;
                tl->alpha[hh] = (m_new == -INFINITY) ? 1.f : exp2f(m_old - m_new);
                tl->m_run[hh] = m_new;
            }
            named_bar_sync(bar_id, 128);
            // the previous tile's PV product has read P^T and O^T before they change
            if (t > 0 && !dead) dead = !attn_wait(&tl->o_done, (uint32_t)((t - 1) & 1), p.status, abort);
            tc_fence_after();
            float v2[NH];
#pragma unroll
            for (int i = 0; i < NH; ++i) {
                const float m = tl->m_run[hoff + i];
                x[i] = (m == -INFINITY) ? 0.f : exp2f(x[i] - m);
                v2[i] = x[i];
            }
            {   // P^T[i][row]: column block row/64, head row i, 16-byte chunk ((row%64)/8) ^ (i%8)
                uint8_t* pb = p_s + (row >> 6) * HC * 128;
                const int kr = row & 63;
#pragma unroll
                for (int i = 0; i < NH; ++i) {
                    const int hi = hoff + i;
                    *reinterpret_cast<__nv_bfloat16*>(pb + hi * 128 + ((((kr >> 3) ^ (hi & 7))) << 4) + (kr & 7) * 2) =
                        __float2bfloat16_rn(x[i]);
                }
            }
            warp_reduce_scatter_n<NH, false>(v2);
            if ((lane & (kSpread - 1)) == 0) tl->red_sum[qd][hoff + lane / kSpread] = v2[0];
            bool rescale = false;
#pragma unroll
            for (int i = 0; i < NH; ++i) rescale = rescale || tl->alpha[hoff + i] != 1.f;
            if (t > 0 && rescale) {   // O^T rows (lane = d within a block) times the heads' factors
                for (int m = 0; m < nmb; ++m) {
                    const uint32_t ta = tmem + lane_base + (uint32_t)(2 * HC + m * HC + hoff);
                    uint32_t r[NH];
                    tmem_ld_n<NH>(ta, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < NH; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * tl->alpha[hoff + i]);
                    tmem_st_n<NH>(ta, r);
                }
                tmem_st_wait();
            }
            fence_proxy_async_smem();   // P^T: generic writes read by the MMA
            tc_fence_before();
            named_bar_sync(bar_id, 128);
            if (st < NH) {
                const int hh = hoff + st;
                tl->l_run[hh] = tl->l_run[hh] * tl->alpha[hh] + (tl->red_sum[0][hh] + tl->red_sum[1][hh]) +
                                (tl->red_sum[2][hh] + tl->red_sum[3][hh]);
            }
            if (st == 0) mbar_arrive(&tl->p_full);   // one arrival per set
            if (set == 0 && st == 0 && t < 5) STI_HSTAMP(20 + t);
        }
        if (!dead && n_tiles > 0) dead = !attn_wait(&tl->o_done, (uint32_t)((n_tiles - 1) & 1), p.status, abort);
        if (set == 0 && st == 0) STI_HSTAMP(12);
    }

    // ---- epilogue: o = O / (l + 2^(sink*log2e - m)); heads with no valid slot give 0
    tc_fence_before();
    __syncthreads();   // every MMA of this CTA has completed; m_run, l_run final
    tc_fence_after();
    if (rope_smem) attn_wait(&tl->rope_bar, 0, p.status, abort);
    const bool sm_warp = warp >= 2 && warp <= 5;
    const int st = tid - 64;                                  // softmax threads: 0..127
    const int row = 32 * (warp & 3) + lane;                   // their TMEM lane (d within a block)
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    // the epilogue runs on every softmax warp: set s takes heads [s*NH, s*NH + NH) of its O^T row
    const bool ep_warp = sm_warp || (kSets == 2 && warp >= 9);
    const int ehoff = warp >= 9 ? NH : 0;
    auto o_part = [&](int m, uint32_t (&r)[NH]) {
        if (n_tiles > 0) {
            tmem_ld_n<NH>(tmem + lane_base + (uint32_t)(2 * HC + m * HC + ehoff), r);
            tmem_ld_wait();
        } else {
#pragma unroll
            for (int i = 0; i < NH; ++i) r[i] = 0u;
        }
    };
    if (CR == 1) {
        if (sm_warp && st < HC) {
            const int hh = hg * HC + st;
            const float m = tl->m_run[st];
            float inv = 0.f, lse = -INFINITY;
            if (m != -INFINITY) {
                const float den = tl->l_run[st] + exp2f(__ldg(p.sink + hh) * kLog2e - m);
                inv = 1.f / den;
                lse = (m + log2f(den)) * kLn2;
            }
            tl->alpha[st] = inv;
            if (p.lse) p.lse[(size_t)query * p.h + hh] = lse;
        }
        __syncthreads();
        // [HC][d] bf16 staged in the Q buffer (every QK product has completed) -> one bulk store
        uint16_t* stage = reinterpret_cast<uint16_t*>(q_s);
        if (ep_warp)
            for (int m = 0; m < nmb; ++m) {
                uint32_t r[NH];
                o_part(m, r);
                const int dd = 128 * m + row;
                float v[NH];
#pragma unroll
                for (int i = 0; i < NH; ++i) v[i] = __uint_as_float(r[i]) * tl->alpha[ehoff + i];
                if (p.rope_dims > 0 && 128 * m + 128 > p.d - p.rope_dims)   // the output's inverse rotation
                    rope_inverse_pairs<NH>(v, dd, p.d, p.rope_dims, rope_tab);
#pragma unroll
                for (int i = 0; i < NH; ++i)
                    stage[(size_t)(ehoff + i) * p.d + dd] = __bfloat16_as_ushort(__float2bfloat16_rn(v[i]));
            }
        fence_proxy_async_smem();
        __syncthreads();
        if (sm_warp && st == 0) {
            bulk_store(p.out + ((size_t)query * p.h + (size_t)hg * HC) * p.d, stage, (uint32_t)(HC * p.d * 2));
            bulk_commit();
            bulk_wait_read_all();   // the stage may be released; the writes complete with the grid
            STI_HSTAMP(13);
        }
    } else {
        // two row groups: this CTA and its partner (same heads, the other half of the slots).
        // Each sends the partner the partner's half of d of its unscaled O^T and its (m, l)
        // (asynchronous stores counted on the partner's barrier) once the partner reports its
        // ring free, then finishes its own half: o = (O_own 2^(m_own-M) + O_peer 2^(m_peer-M)) / L.
        const int partner = (1 - rg) * CH + hg;
        const int half = p.d / 2;
        const int mb_own = rg * (nmb / 2), mb_peer = (1 - rg) * (nmb / 2);
        constexpr int kChunks = HC / 4;                       // 16-byte chunks of a row of HC floats
        float* recv = reinterpret_cast<float*>(ring);         // [half][HC], chunk c of row r at c ^ (r % kChunks)
        if (tid == 0) mbar_arrive_remote(dsmem_addr(&tl->ready_bar, (uint32_t)partner));
        if (tid == 64) STI_ESTAMP(0);
        const bool ready = attn_wait(&tl->ready_bar, 0, p.status, abort);
        if (tid == 64) STI_ESTAMP(1);
        if (ep_warp && ready) {
            const uint32_t rbar = dsmem_addr(&tl->recv_bar, (uint32_t)partner);
            const uint32_t rbase = dsmem_addr(recv, (uint32_t)partner);
            for (int m = mb_peer; m < mb_peer + nmb / 2; ++m) {
                uint32_t r[NH];
                o_part(m, r);
                const int dl = (m - mb_peer) * 128 + row;
#pragma unroll
                for (int c = 0; c < NH / 4; ++c) {
                    const int cc = ehoff / 4 + c;
                    st_async_v4(rbase + (uint32_t)(dl * HC + ((cc ^ (dl % kChunks)) * 4)) * 4u, __uint_as_float(r[4 * c]),
                                __uint_as_float(r[4 * c + 1]), __uint_as_float(r[4 * c + 2]),
                                __uint_as_float(r[4 * c + 3]), rbar);
                }
            }
            if (sm_warp && st < HC)
                st_async_v2(dsmem_addr(&tl->peer_ml[st][0], (uint32_t)partner), tl->m_run[st], tl->l_run[st], rbar);
        }
        if (tid == 64) STI_ESTAMP(2);
        const bool got = attn_wait(&tl->recv_bar, 0, p.status, abort);
        if (tid == 64) STI_ESTAMP(3);
        if (sm_warp && st < HC) {   // scale factors of the two partials; lse (first row group)
            const int hh = hg * HC + st;
            const float mo = tl->m_run[st], lo = tl->l_run[st];
            const float mp = got ? tl->peer_ml[st][0] : -INFINITY, lp = got ? tl->peer_ml[st][1] : 0.f;
            const float M = fmaxf(mo, mp);
            float ao = 0.f, ap = 0.f, lse = -INFINITY;
            if (M != -INFINITY) {
                const float eo = mo == -INFINITY ? 0.f : exp2f(mo - M), ep = mp == -INFINITY ? 0.f : exp2f(mp - M);
                const float L = lo * eo + lp * ep + exp2f(__ldg(p.sink + hh) * kLog2e - M);
                ao = eo / L;
                ap = ep / L;
                lse = (M + log2f(L)) * kLn2;
            }
            tl->alpha[st] = ao;
            tl->red_max[0][st] = ap;   // the peer's factor (the softmax scratch is free now)
            if (rg == 0 && p.lse) p.lse[(size_t)query * p.h + hh] = lse;
        }
        __syncthreads();
        if (ep_warp && got)   // own half of d: combine and write bf16 rows straight to global
            for (int m = mb_own; m < mb_own + nmb / 2; ++m) {
                uint32_t r[NH];
                o_part(m, r);
                const int dl = (m - mb_own) * 128 + row;
                const float4* rv = reinterpret_cast<const float4*>(recv + (size_t)dl * HC);
                uint16_t* orow = p.out + ((size_t)query * p.h + (size_t)hg * HC) * p.d + (size_t)rg * half + dl;
                float v[NH];
#pragma unroll
                for (int c = 0; c < NH / 4; ++c) {
                    const int cc = ehoff / 4 + c;
                    const float4 q4 = rv[cc ^ (dl % kChunks)];
                    const float pv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = 4 * cc + e;
                        v[4 * c + e] = __uint_as_float(r[4 * c + e]) * tl->alpha[i] + pv[e] * tl->red_max[0][i];
                    }
                }
                const int dd = rg * half + dl;
                if (p.rope_dims > 0 && rg * half + (m - mb_own) * 128 + 128 > p.d - p.rope_dims)
                    rope_inverse_pairs<NH>(v, dd, p.d, p.rope_dims, rope_tab);
#pragma unroll
                for (int j = 0; j < NH; ++j)
                    orow[(size_t)(ehoff + j) * p.d] = __bfloat16_as_ushort(__float2bfloat16_rn(v[j]));
            }
        if (tid == 64) STI_ESTAMP(4);
        if (sm_warp && st == 0) STI_HSTAMP(13);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, hs_tmem_cols(HC));
    }
    cluster_sync();   // no CTA leaves while a partner may still signal or fill its shared memory
    if (tid == 0) STI_HSTAMP(14);
#ifdef STI_ATTN_TIMING
    if (tid == 0 && blockIdx.x < 2048) g_hs_t[blockIdx.x][31] = global_timer_ns();
#endif
}

constexpr int kSmemLimit = 232448;   // opt-in dynamic shared memory per CTA

// Ring slots: even (a d-block's two column blocks sit in adjacent slots) and at least one tile's
// column blocks (a tile's last block must not wait for a slot its own PV product frees).
int hs_slots(int hc, int d) {
    for (int s = kHsMaxSlots; s >= d / 64 && s >= 2; s -= 2)
        if (hs_smem_bytes(hc, d, s) <= (size_t)kSmemLimit) return s;
    return 0;
}

template <int HC>
cudaError_t launch_hs(const CUtensorMap& tm_q, const CUtensorMap& tm_kv1, const CUtensorMap& tm_kv2,
                      const CUtensorMap& tm_win, const AttnParams& p, cudaStream_t stream) {
    const int slots = hs_slots(HC, p.d);
    const size_t smem = hs_smem_bytes(HC, p.d, slots);
    cudaError_t err =
        cudaFuncSetAttribute(sparse_attn_hs_kernel<HC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.B * p.s * p.cluster));
    cfg.blockDim = dim3(kHsThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.pdl ? 2 : 1;
    err = cudaLaunchKernelEx(&cfg, sparse_attn_hs_kernel<HC>, tm_q, tm_kv1, tm_kv2, tm_win, p, slots);
    return err != cudaSuccess ? err : cudaGetLastError();
}

template <int HC>
bool hs_resident(int n_queries, int c, int d) {
    const int slots = hs_slots(HC, d);
    if (slots < 2) return false;
    const size_t smem = hs_smem_bytes(HC, d, slots);
    if (cudaFuncSetAttribute(sparse_attn_hs_kernel<HC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_queries * c));
    cfg.blockDim = dim3(kHsThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, sparse_attn_hs_kernel<HC>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return active >= n_queries;
}

// Candidates in order of preference: (heads per CTA, CTAs, row groups).  Two head groups x two
// row groups halve both the MMAs and the slot gathers of a CTA against four head groups (a
// tcgen05 MMA costs about the same for N = 16 or 32); they need d to split in two d-block halves.
int attn_hs_pick_uncached(int n_queries, int h, int d, int* rows) {
    struct Cand {
        int hc, c, r;
    };
    const Cand c64[] = {{32, 4, 2}, {16, 4, 1}, {32, 2, 1}};
    const Cand c32[] = {{32, 2, 2}, {16, 2, 1}};
    const Cand* cands = h == 64 ? c64 : c32;
    const int n = h == 64 ? 3 : 2;
    for (int i = 0; i < n; ++i) {
        const Cand& c = cands[i];
        if (c.hc * c.c / c.r != h) continue;
        if (c.r == 2 && d % 256 != 0) continue;
        const bool ok = c.hc == 16 ? hs_resident<16>(n_queries, c.c, d) : hs_resident<32>(n_queries, c.c, d);
        if (ok) {
            *rows = c.r;
            return c.c;
        }
    }
    return 0;
}

}  // namespace

int attn_hs_pick(int n_queries, int h, int d, int* rows) {
    *rows = 1;
    if ((h != 64 && h != 32) || d % 128 != 0 || d > 512 || n_queries < 1) return 0;
    struct Entry {
        int dev, n_queries, h, d, c, r;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> g(mu);
        for (const Entry& e : cache)
            if (e.dev == dev && e.n_queries == n_queries && e.h == h && e.d == d) {
                *rows = e.r;
                return e.c;
            }
    }
    int r = 1;
    const int c = attn_hs_pick_uncached(n_queries, h, d, &r);
    *rows = r;
    std::lock_guard<std::mutex> g(mu);
    if (cache.size() < 4096) cache.push_back({dev, n_queries, h, d, c, r});
    return c;
}

cudaError_t launch_sparse_attn_hs(const CUtensorMap& tm_q, const CUtensorMap& tm_kv1, const CUtensorMap& tm_kv2,
                                  const CUtensorMap& tm_win, const AttnParams& p, cudaStream_t stream) {
    if (p.B * p.s == 0) return cudaSuccess;
    const int hc = p.h * p.hs_rows / p.cluster;
    if (hc == 16) return launch_hs<16>(tm_q, tm_kv1, tm_kv2, tm_win, p, stream);
    if (hc == 32) return launch_hs<32>(tm_q, tm_kv1, tm_kv2, tm_win, p, stream);
    if (hc == 64) return launch_hs<64>(tm_q, tm_kv1, tm_kv2, tm_win, p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace sti

#ifdef STI_ATTN_TIMING
// profiling builds only: per-CTA clock64 stamps of the head-split attention
extern "C" int sti_dbg_hs_times(unsigned long long* host, int n_blocks) {
    return (int)cudaMemcpyFromSymbol(host, sti::g_hs_t, sizeof(unsigned long long) * 32 * (size_t)n_blocks);
}
extern "C" int sti_dbg_hs_merge(unsigned long long* host, int n_blocks) {
    return (int)cudaMemcpyFromSymbol(host, sti::g_hs_e, sizeof(unsigned long long) * 8 * (size_t)n_blocks);
}
extern "C" int sti_dbg_hs_prod(unsigned long long* host, int n_blocks) {
    return (int)cudaMemcpyFromSymbol(host, sti::g_hs_p, sizeof(unsigned long long) * 40 * (size_t)n_blocks);
}
#endif
