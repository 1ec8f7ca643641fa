// decode_attn.cu -- the decode step's top-k selection and its sparse sink attention, fused into
// one kernel: a thread-block cluster of four CTAs per query.
//
// DeepSeek V4.1, attention "attend/selected" page:
//   Indexer.forward (its last lines)  topk of the visible scores, re-sorted by position, + offset
//   get_window_topk_idxs (decode)     the W-slot ring, oldest first, -1 for slots past start_pos
//   sparse_attn_kernel / sparse_attn  o = sum_i e^{s_i} kv_i / (sum_i e^{s_i} + e^{sink_h}) over the
//                                     non -1 slots of [ring ; top-k compressed rows],
//                                     s_i = softmax_scale * q . kv_i, one latent row as K and V
// "read-weights" page, Attention.forward: _compress_topk_idxs feeds sparse_attn.
//
// Shape: 64 heads x 512, window 128, index_topk 512: 640 rows per query, the ring's 128 and 512
// compressed.  CTA r of a query's cluster owns
//   * ring slots [32r, 32r+32): rows 96..127 of its tile, run through QK, softmax and PV before the
//     indices exist (while the scores kernel drains);
//   * the compressed rows of output slots [128r, 128r+128) of the index row: one 128-row tile;
//   * d-block r (dims [128r, 128r+128)) of the output in the merge.
// Top-k (exact; ties go to the lower position), computed whole by every CTA of the cluster -- its
// inputs are a few tens of KB from L2, and no CTA waits on another: the scores kernel's first
// radix pass (top 11 key bits) gives the threshold bin d1; one pass over the row marks the keys
// above the bin in a position bitmap and lists the bin's members; two radix passes over the
// members (shared-memory histograms of the next 11 and 10 bits) give the exact k-th key tau and
// how many keys equal to it are taken; a second bitmap marks the keys equal to tau; one block scan
// over both bitmaps gives every selected position its output slot, in ascending position order.
// A bin with more than 1024 members (heavy ties) takes the two passes over the whole row instead.
// Each CTA keeps the slots it owns: its tile's index list and its quarter of the published row.
// Attention, per tile: S^T = KV.Q^T (tcgen05, M = 128 rows, N = 64 heads, K = 512) into TMEM; an
// online softmax with thread = row in two warp groups of 32 heads; O^T += V^T.P^T (M = 128 d-rows
// per d-block, N = 64, K = rows) reading the same tile as an MN-major operand.  The compressed
// rows arrive by 16-byte cp.async from the eight math warps (one column block each; masked rows
// zero-filled).
// Merge, through L2: each CTA writes the three d-blocks of its unnormalised O^T that the others
// own, and its (max, sum) per head, to the workspace and signals the cluster (one remote barrier
// arrive per CTA); each then reads its d-block from the three others:
//   o = sum_c O_c 2^(m_c - M) / (sum_c l_c 2^(m_c - M) + 2^(sink - M)).
//
// Roles (13 warps): warp 0 and warps 10-12 load Q and the ring slice; warp 1 allocates TMEM and
// issues the MMAs; warps 2-9 (256 "math" threads) run the top-k, gather the compressed tile
// (warp 2 + j: column block j), the softmax (warps 2-5: heads 0-31, warps 6-9: heads 32-63) and
// the merge.
#include <cuda_bf16.h>
#include <cstddef>
#include <math.h>

#include <mutex>
#include <type_traits>
#include <vector>

#include "sti_internal.h"
#include "sti_ptx.cuh"
#include "sti_attn_util.cuh"

namespace sti {
namespace {

#ifdef STI_DA_TIMING
// global-timer stamps per CTA (profiling builds): [0, 16) math-thread phases, [16, 24) MMA issuer
__device__ unsigned long long g_da_t[1024][32];
#define STI_DSTAMP(i)                                                                                  \
    do {                                                                                               \
        if (blockIdx.x < 1024) g_da_t[blockIdx.x][i] = global_timer_ns();                              \
    } while (0)
#define STI_DCLOCK(i)                                                                                  \
    do {                                                                                               \
        if (blockIdx.x < 1024) g_da_t[blockIdx.x][i] = clock64();                                      \
    } while (0)
#else
#define STI_DCLOCK(i) \
    do {              \
    } while (0)
#define STI_DSTAMP(i) \
    do {              \
    } while (0)
#endif

constexpr int kCtas = 4;                  // CTAs per query
constexpr int kThreads = 416;
constexpr int kH = 64;                    // heads
constexpr int kD = 512;                   // head dim
constexpr int kW = 128;                   // window ring slots
constexpr int kK = 512;                   // index_topk
constexpr int kRows = 128;                // tile rows
constexpr int kRingRows = kW / kCtas;     // ring slots per CTA
constexpr int kRingRow0 = kRows - kRingRows;   // tile row of the first ring slot
constexpr int kBins = 2048;
constexpr int kMemCap = 1024;             // threshold-bin members resolved from a list (more: row passes)
constexpr uint32_t kBlkBytes = kRows * 128;    // one column block of the tile (128 rows x 128 B)
constexpr uint32_t kQBlkBytes = kH * 128;      // one column block of Q (64 heads x 128 B)
constexpr uint32_t kTileBytes = 8 * kBlkBytes;
constexpr uint32_t kQBytes = 8 * kQBlkBytes;
constexpr uint32_t kPBytes = 2 * kQBlkBytes;   // P^T: 2 row blocks x 64 heads x 128 B
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr uint32_t kBarMath = 1, kBarSet0 = 2;   // named barriers: the 256 math threads; each set of 128

struct __align__(16) DaTail {
    uint64_t full[8];          // compressed tile, column block j landed (its math warp's copies)
    uint64_t q_bar;            // Q landed
    uint64_t ring_bar;         // the ring slice landed (4 loader arrivals + bytes)
    uint64_t s_full[2];        // S^T of the ring slice / of the compressed tile in TMEM
    uint64_t p_full;           // P^T written (one arrival per softmax set), phase 0 ring, 1 tile
    uint64_t o_done;           // PV complete, phase 0 ring, 1 tile
    uint64_t ring_free;        // the ring slice's PV complete: rows 96..127 may be overwritten
    uint64_t pub_bar;          // merge: every CTA's partial outputs written (4 CTAs)
    uint32_t tmem_base;
    int abort;
    int n_mem;                 // threshold-bin members listed
    int warp_tot[8], warp_tot2[8];
    int misc[4];
    float m_run[kH], l_run[kH], alpha[kH];
    float red_max[4][kH], red_sum[4][kH];
    float wgt[kCtas][kH];
    int tile_idx[kRows];
};

constexpr size_t kSmemBytes = 1024 + kTileBytes + kQBytes + kPBytes + sizeof(DaTail);
static_assert(kSmemBytes <= 232448, "shared memory of the fused decode kernel");

__device__ __forceinline__ void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

// Publish this CTA's writes made before the call (by all 256 math threads; shared or global
// memory) to the cluster: one release arrive on `bar` in each of the four CTAs.
__device__ __forceinline__ void publish_to_cluster(uint64_t* bar, int mt) {
    fence_acq_rel_cluster();
    named_bar_sync(kBarMath, 256);
    if (mt == 0)
        for (int c = 0; c < kCtas; ++c) mbar_arrive_remote(dsmem_addr(bar, (uint32_t)c));
}

// Exclusive scan of two counts over the 256 math threads; returns the two totals too.
__device__ __forceinline__ void scan2_m(int a, int b, DaTail* tl, int mt, int& a_before, int& b_before, int& a_tot,
                                        int& b_tot) {
    const int lane = mt & 31, w = mt >> 5;
    int ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int xa = __shfl_up_sync(kFull, ia, o), xb = __shfl_up_sync(kFull, ib, o);
        if (lane >= o) {
            ia += xa;
            ib += xb;
        }
    }
    if (lane == 31) {
        tl->warp_tot[w] = ia;
        tl->warp_tot2[w] = ib;
    }
    named_bar_sync(kBarMath, 256);
    int pa = 0, pb = 0, ta = 0, tb = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int xa = tl->warp_tot[i], xb = tl->warp_tot2[i];
        pa += i < w ? xa : 0;
        pb += i < w ? xb : 0;
        ta += xa;
        tb += xb;
    }
    named_bar_sync(kBarMath, 256);   // warp_tot may be rewritten after this
    a_before = pa + ia - a;
    b_before = pb + ib - b;
    a_tot = ta;
    b_tot = tb;
}

// The bin d* (of 2048, eight per math thread in h8) where the count from the top first reaches
// `remaining`; *above = matching keys in higher bins, *cnt = keys in d*.  256 math threads.
__device__ int select_bin_m(const uint32_t (&h8)[8], int remaining, DaTail* tl, int mt, int* above_out,
                            int* cnt_out) {
    const int lane = mt & 31, w = mt >> 5;
    int local = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) local += (int)h8[i];
    int inc = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += x;
    }
    if (lane == 31) tl->warp_tot[w] = inc;
    if (mt == 0) tl->misc[0] = -1;
    named_bar_sync(kBarMath, 256);
    int wpre = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int x = tl->warp_tot[i];
        wpre += i < w ? x : 0;
        tot += x;
    }
    int above = tot - (wpre + inc);   // keys in the bins of higher threads
#pragma unroll
    for (int i = 7; i >= 0; --i) {
        const int c = (int)h8[i];
        if (above < remaining && above + c >= remaining) {
            tl->misc[0] = 8 * mt + i;
            tl->misc[1] = above;
            tl->misc[2] = c;
        }
        above += c;
    }
    named_bar_sync(kBarMath, 256);
    const int d = tl->misc[0];
    *above_out = tl->misc[1];
    *cnt_out = tl->misc[2];
    named_bar_sync(kBarMath, 256);   // misc and warp_tot are rewritten by the next call
    return d;
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_topk_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_ring,
                            const __grid_constant__ CUtensorMap tm_ring_rows, const DecodeAttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* tile = smem;                          // 8 column blocks x [128 rows x 128 B], SW128
    uint8_t* q_s = tile + kTileBytes;              // 8 column blocks x [64 heads x 128 B], SW128
    uint8_t* p_s = q_s + kQBytes;                  // P^T: 2 row blocks x [64 heads x 128 B], SW128
    DaTail* tl = reinterpret_cast<DaTail*>(p_s + kPBytes);
    volatile int* abort = &tl->abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int query = blockIdx.x / kCtas, rank = blockIdx.x - (blockIdx.x / kCtas) * kCtas;
    const int b = query;
    const int sp = __ldg(p.start_pos + b);
    const int n2 = p.n_cols;
    int32_t* idx_row = p.idx_out + (size_t)b * (kW + kK);
    if (tid == 0) {
        STI_DSTAMP(0);
        STI_DCLOCK(30);
    }
    griddep_launch_dependents();

    if (warp == 1) {
        tmem_alloc(&tl->tmem_base, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int j = 0; j < 8; ++j) mbar_init(&tl->full[j], 1);
        mbar_init(&tl->q_bar, 1);
        mbar_init(&tl->ring_bar, 4);
        mbar_init(&tl->s_full[0], 1);
        mbar_init(&tl->s_full[1], 1);
        mbar_init(&tl->p_full, 2);
        mbar_init(&tl->o_done, 1);
        mbar_init(&tl->ring_free, 1);
        mbar_init(&tl->pub_bar, kCtas);
        tl->abort = 0;
        tl->n_mem = 0;
        fence_mbar_init();
    }
    if (tid < kH) {
        tl->m_run[tid] = -INFINITY;
        tl->l_run[tid] = 0.f;
    }
    if (tid < kRows) tl->tile_idx[tid] = -1;
    {   // tile rows no load writes stay finite (zero); the ring slice's QK reads rows 0..95 as zeros
        uint4* t4 = reinterpret_cast<uint4*>(tile);
        for (int i = tid; i < (int)(kTileBytes / 16); i += kThreads) t4[i] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    cluster_sync();   // barriers initialised (and visible to the cluster) before any remote arrive
    tc_fence_after();
    const uint32_t tmem = tl->tmem_base;
    // TMEM columns: S^T of the ring slice [0, 64), of the compressed tile [64, 128), O^T [128, 384)
    constexpr uint32_t kTmemO = 128;

    // ring slot 32*rank + i (tile row 96 + i) holds a position <= start_pos: every slot of a full
    // ring, slot s itself (position s) while the ring is filling
    auto ring_valid = [&](int i) { return sp >= kW - 1 || kRingRows * rank + i <= sp; };

    if (warp == 0 || warp >= 10) {
        // ---------------------------------------------------------------- loaders
        const int pi = warp == 0 ? 0 : warp - 9;   // 0..3
        if (warp == 0) {
            if (lane == 0) {
                tma_prefetch_desc(&tm_ring);
                tma_prefetch_desc(&tm_ring_rows);
                mbar_arrive_expect_tx(&tl->q_bar, kQBytes);
                for (int cb = 0; cb < 8; ++cb)
                    tma_load_2d(q_s + (size_t)cb * kQBlkBytes, &tm_q, &tl->q_bar, cb * 64, b * kH);
            }
            // window indices of the published row: entries [32 rank, 32 rank + 32), oldest first
            {
                const int i = kRingRows * rank + lane;
                const int oldest = sp % kW + 1;
                const int slot = i < kW - oldest ? oldest + i : i - (kW - oldest);
                idx_row[i] = slot > sp ? -1 : slot;
            }
        }
        // the ring slice: one 2-D box per column block when the ring is full, else the valid rows
        // by four-row gathers (rows of a group past start_pos repeat its first valid row; groups
        // with none are not fetched and stay zero)
        if (sp >= kW - 1) {
            if (lane == 0) {
                if (pi == 0) {
                    mbar_arrive_expect_tx(&tl->ring_bar, 8 * kRingRows * 128);
                    for (int cb = 0; cb < 8; ++cb)
                        tma_load_2d(tile + (size_t)cb * kBlkBytes + kRingRow0 * 128, &tm_ring, &tl->ring_bar, cb * 64,
                                    b * (int)p.rows1 + kRingRows * rank);
                } else {
                    mbar_arrive(&tl->ring_bar);
                }
            }
        } else {
            const int cb = 2 * pi + (lane >> 3), g = lane & 7;   // lanes 0..15: 2 column blocks x 8 groups
            int ys[4], first = -1;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 4 * g + i;
                const bool v = ring_valid(r);
                ys[i] = b * (int)p.rows1 + kRingRows * rank + r;
                if (v && first < 0) first = ys[i];
                if (!v) ys[i] = -1;
            }
            const bool issue = lane < 16 && first >= 0;
            const uint32_t bytes = (uint32_t)__popc(__ballot_sync(kFull, issue)) * 512u;
            if (lane == 0) mbar_arrive_expect_tx(&tl->ring_bar, bytes);
            __syncwarp();
            if (issue)   // four-row gathers take the one-row-box map of the ring
                tma_gather4(tile + (size_t)cb * kBlkBytes + (kRingRow0 + 4 * g) * 128, &tm_ring_rows, &tl->ring_bar,
                            cb * 64, ys[0] >= 0 ? ys[0] : first, ys[1] >= 0 ? ys[1] : first, ys[2] >= 0 ? ys[2] : first,
                            ys[3] >= 0 ? ys[3] : first);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t idesc_qk = idesc_bf16_f32(kRows, kH, false, false);
            const uint32_t idesc_pv = idesc_bf16_f32(128, kH, true, false);
            const uint64_t kd0 = sdesc(smem_u32(tile), 16, 1024, kLayoutSW128);          // K-major tile
            const uint64_t vd0 = sdesc(smem_u32(tile), kBlkBytes, 1024, kLayoutSW128);   // MN-major tile
            const uint64_t qd0 = sdesc(smem_u32(q_s), 16, 1024, kLayoutSW128);
            const uint64_t pd0 = sdesc(smem_u32(p_s), 16, 1024, kLayoutSW128);
            // descriptors advance in 16-byte units: +2 per 32-byte K step of a K-major operand
            auto qk_block = [&](uint32_t s_col, int j) {
                const uint64_t a = kd0 + (uint64_t)((uint32_t)j * (kBlkBytes >> 4));
                const uint64_t bq = qd0 + (uint64_t)((uint32_t)j * (kQBlkBytes >> 4));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(tmem + s_col, a + 2 * kk, bq + 2 * kk, idesc_qk, (j > 0 || kk > 0) ? 1u : 0u);
            };
            auto pv = [&](int kk0, bool first) {   // K steps kk0..7 of 16 rows, every d-block
                for (int m = 0; m < 4; ++m) {
                    const uint64_t a = vd0 + (uint64_t)((uint32_t)(2 * m) * (kBlkBytes >> 4));
                    for (int kk = kk0; kk < 8; ++kk)
                        umma_bf16(tmem + kTmemO + (uint32_t)(m * kH), a + (uint64_t)(kk * (2048 >> 4)),
                                  pd0 + (uint64_t)(((kk >> 2) * kQBlkBytes + (kk & 3) * 32) >> 4), idesc_pv,
                                  (!first || kk > kk0) ? 1u : 0u);
                }
            };
            bool ok = attn_wait(&tl->q_bar, 0, p.status, abort);
            ok = ok && attn_wait(&tl->ring_bar, 0, p.status, abort);
            STI_DSTAMP(16);
            if (ok) {   // QK of the ring slice (rows 0..95 are zero)
                tc_fence_after();
                for (int j = 0; j < 8; ++j) qk_block(0, j);
            }
            umma_commit(&tl->s_full[0]);
            ok = ok && attn_wait(&tl->p_full, 0, p.status, abort);
            STI_DSTAMP(17);
            if (ok) {   // PV of the ring slice: rows 96..127 (K steps 6, 7) initialise O^T
                tc_fence_after();
                pv(kRingRow0 / 16, true);
            }
            umma_commit(&tl->o_done);
            umma_commit(&tl->ring_free);
            for (int j = 0; j < 8; ++j) {   // QK of the compressed tile, column block by column block
                ok = ok && attn_wait(&tl->full[j], 0, p.status, abort);
                if (j == 0) STI_DSTAMP(18);
                if (j == 7) STI_DSTAMP(19);
                if (ok) {
                    tc_fence_after();
                    qk_block(64, j);
                }
            }
            umma_commit(&tl->s_full[1]);
            ok = ok && attn_wait(&tl->p_full, 1, p.status, abort);
            STI_DSTAMP(20);
            if (ok) {
                tc_fence_after();
                pv(0, false);
            }
            umma_commit(&tl->o_done);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- math threads (warps 2..9)
        const int mt = tid - 64;                       // 0..255
        const int mw = warp - 2;                       // 0..7
        const int set = mw >> 2;                       // softmax set: heads [32 set, 32 set + 32)
        const int qd = warp & 3;                       // TMEM lane quarter of this warp
        const int row = 32 * qd + lane;                // tile row = TMEM lane
        const int st = mt & 127;                       // 0..127 within the set
        const int hoff = 32 * set;
        const uint32_t bar_set = kBarSet0 + (uint32_t)set;
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        bool dead = false;
        // bounded waits of the math warps; `dead` stays warp-uniform (it guards warp collectives)
        auto mwait = [&](uint64_t* bar, uint32_t parity) {
            if (!dead) dead = !attn_wait(bar, parity, p.status, abort);
            dead = __any_sync(kFull, dead);
        };

        // online softmax over one tile's S^T (t = 0: the ring slice, 1: the compressed tile)
        auto softmax_tile = [&](int t, bool valid) {
            mwait(&tl->s_full[t], 0);
            if (t == 1 && mt == 0) STI_DSTAMP(11);
            tc_fence_after();
            float x[32];
            {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + (uint32_t)(t * kH + hoff), r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = (valid && !dead) ? __uint_as_float(r[i]) * p.scale_log2 : -INFINITY;
            }
            {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = x[i];
                warp_reduce_scatter_n<32, true>(v);
                tl->red_max[qd][hoff + lane] = v[0];
            }
            if (t == 1 && mt == 0) STI_DSTAMP(21);
            named_bar_sync(bar_set, 128);
            if (t == 1 && mt == 0) STI_DSTAMP(22);
            if (st < 32) {
                const int hh = hoff + st;
                const float mx = fmaxf(fmaxf(tl->red_max[0][hh], tl->red_max[1][hh]),
                                       fmaxf(tl->red_max[2][hh], tl->red_max[3][hh]));
                const float m_old = tl->m_run[hh];
                // the running max moves only when a tile's max passes it by more than 8 (log2 units)
                const float m_new = (m_old == -INFINITY || mx > m_old + 8.f) ? fmaxf(m_old, mx) : m_old;
                tl->alpha[hh] = (m_new == -INFINITY) ? 1.f : exp2f(m_old - m_new);
                tl->m_run[hh] = m_new;
            }
            named_bar_sync(bar_set, 128);
            // the ring slice's PV has read P^T and written O^T before the tile's P^T and rescale
            if (t == 1) mwait(&tl->o_done, 0);
            tc_fence_after();
            float v2[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float m = tl->m_run[hoff + i];
                x[i] = (m == -INFINITY) ? 0.f : exp2f(x[i] - m);
                v2[i] = x[i];
            }
            {   // P^T[h][row]: row block row/64, head h, 16-byte chunk ((row%64)/8) ^ (h%8)
                uint8_t* pb = p_s + (row >> 6) * kQBlkBytes;
                const int kr = row & 63;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int hi = hoff + i;
                    *reinterpret_cast<__nv_bfloat16*>(pb + hi * 128 + (((kr >> 3) ^ (hi & 7)) << 4) + (kr & 7) * 2) =
                        __float2bfloat16_rn(x[i]);
                }
            }
            if (t == 1 && mt == 0) STI_DSTAMP(23);
            warp_reduce_scatter_n<32, false>(v2);
            tl->red_sum[qd][hoff + lane] = v2[0];
            if (t == 1 && mt == 0) STI_DSTAMP(24);
            if (t == 1) {
                bool rescale = false;
#pragma unroll
                for (int i = 0; i < 32; ++i) rescale = rescale || tl->alpha[hoff + i] != 1.f;
                if (rescale && !dead) {   // O^T rows (lane = d within a block) times the heads' factors
                    for (int m = 0; m < 4; ++m) {
                        const uint32_t ta = tmem + lane_base + kTmemO + (uint32_t)(m * kH + hoff);
                        uint32_t r[32];
                        tmem_ld32(ta, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r[i] = __float_as_uint(__uint_as_float(r[i]) * tl->alpha[hoff + i]);
                        tmem_st32(ta, r);
                    }
                    tmem_st_wait();
                }
            }
            fence_proxy_async_smem();   // P^T: generic writes read by the MMA
            tc_fence_before();
            named_bar_sync(bar_set, 128);
            if (st < 32) {
                const int hh = hoff + st;
                tl->l_run[hh] = tl->l_run[hh] * tl->alpha[hh] + (tl->red_sum[0][hh] + tl->red_sum[1][hh]) +
                                (tl->red_sum[2][hh] + tl->red_sum[3][hh]);
            }
            if (st == 0) mbar_arrive(&tl->p_full);
        };

        // ---- the ring slice (needs nothing of the step)
        softmax_tile(0, row >= kRingRow0 && ring_valid(row - kRingRow0));
        if (mt == 0) STI_DSTAMP(1);

        // ---- top-k of the compressed positions (the scores and histogram are complete from here)
        griddep_wait();
        if (mt == 0) STI_DSTAMP(2);
        const int vis = max(0, min((sp + 1) / p.ratio, n2));
        const int my0 = kRows * rank;   // this CTA's output slots [my0, my0 + 128)
        if (vis <= kK) {
            // every visible position is selected: output slot o holds position o
            if (mt < kRows) {
                const int o = my0 + mt;
                tl->tile_idx[mt] = o < vis ? o : -1;
                idx_row[kW + o] = o < vis ? o + kW : -1;
            }
        } else {
            const uint32_t* ghist = p.hist + (size_t)b * kBins;
            const float* src = p.scores + (size_t)b * n2;
            // scratch in tile rows 0..95 (the first 12 KB of column blocks 0..3), free until the gather
            uint32_t* bm_gt = reinterpret_cast<uint32_t*>(tile);                   // [2048] key > tau
            uint32_t* bm_eq = reinterpret_cast<uint32_t*>(tile + kBlkBytes);       // [2048] key == tau
            uint32_t* mem_key = reinterpret_cast<uint32_t*>(tile + 2 * kBlkBytes); // [1024] bin-d1 members
            int* mem_pos = reinterpret_cast<int*>(tile + 2 * kBlkBytes + 4096);     // [1024]
            uint32_t* h2 = reinterpret_cast<uint32_t*>(tile + 3 * kBlkBytes);      // [2048]
            uint32_t* h3 = h2 + 2048;                                               // [1024]
            // thread mt owns positions [mt*P, mt*P + P) (P a multiple of 32: whole bitmap words)
            const int P = ((vis + 255) / 256 + 31) & ~31;
            const int p0 = min(vis, mt * P), p1 = min(vis, p0 + P);
            const int w0 = mt * (P / 32), nw = P / 32;
            uint32_t h8[8];
            {
                const uint4 a0 = __ldg(reinterpret_cast<const uint4*>(ghist) + 2 * mt);
                const uint4 a1 = __ldg(reinterpret_cast<const uint4*>(ghist) + 2 * mt + 1);
                h8[0] = a0.x; h8[1] = a0.y; h8[2] = a0.z; h8[3] = a0.w;
                h8[4] = a1.x; h8[5] = a1.y; h8[6] = a1.z; h8[7] = a1.w;
            }
            // every key of this thread's segment in 64-key batches: f(valid, position, key); a fixed
            // trip count over the warp (the per-batch ballots need every lane).  Rows start 16-byte
            // aligned only when n_cols is a multiple of 4: otherwise scalar loads
            const bool vec4 = (reinterpret_cast<uintptr_t>(src) & 15u) == 0u;
            auto for_keys = [&](auto&& f) {
                for (int c0 = 0; c0 < P; c0 += 64) {
                    float v[64];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int pos = mt * P + c0 + 4 * i;
                        float4 f4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                        if (vec4 && pos + 3 < p1) {
                            f4 = __ldg(reinterpret_cast<const float4*>(src + pos));
                        } else {
                            if (pos + 3 < p1) f4.w = __ldg(src + pos + 3);
                            if (pos < p1) f4.x = __ldg(src + pos);
                            if (pos + 1 < p1) f4.y = __ldg(src + pos + 1);
                            if (pos + 2 < p1) f4.z = __ldg(src + pos + 2);
                        }
                        v[4 * i] = f4.x; v[4 * i + 1] = f4.y; v[4 * i + 2] = f4.z; v[4 * i + 3] = f4.w;
                    }
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const int pos = mt * P + c0 + i;
                        f(pos < p1, pos, float_key(v[i]));
                    }
                }
            };
            // pass 1 from the scores kernel's histogram: the threshold bin d1
            int above1, c1;
            const int d1 = select_bin_m(h8, kK, tl, mt, &above1, &c1);
            const int remaining1 = kK - above1;   // keys of bin d1 to take (>= 1)
            if (mt == 0) STI_DSTAMP(3);
            // one pass: bitmap of keys above the bin; list of the bin's members
            for (int w = 0; w < nw; ++w) bm_eq[w0 + w] = 0u;
            {
                uint32_t word = 0u;
                for_keys([&](bool v, int pos, uint32_t key) {
                    const uint32_t dig = key >> 21;
                    if (v && dig > (uint32_t)d1) word |= 1u << (pos & 31);
                    const bool m = v && dig == (uint32_t)d1;
                    const unsigned bal = __ballot_sync(kFull, m);
                    if (bal) {
                        int base = 0;
                        if (lane == 0) base = atomicAdd(&tl->n_mem, __popc(bal));
                        base = __shfl_sync(kFull, base, 0);
                        const int at = base + __popc(bal & ((1u << lane) - 1u));
                        if (m && at < kMemCap) {
                            mem_key[at] = key;
                            mem_pos[at] = pos;
                        }
                    }
                    if ((pos & 31) == 31) {
                        if ((pos >> 5) < w0 + nw) bm_gt[pos >> 5] = word;
                        word = 0u;
                    }
                });
            }
            named_bar_sync(kBarMath, 256);
            if (mt == 0) STI_DSTAMP(4);
            const int n_mem = tl->n_mem;
            const bool listed = n_mem <= kMemCap && n_mem == c1;
            // passes 2 and 3: the next 11 and 10 bits, over the listed members (or the whole row)
            uint32_t prefix = (uint32_t)d1;
            int remaining = remaining1;
            for (int pass = 0; pass < 2; ++pass) {
                uint32_t* hh = pass == 0 ? h2 : h3;
                const int nb = pass == 0 ? 2048 : 1024;
                const int hi_shift = pass == 0 ? 21 : 10, shift = pass == 0 ? 10 : 0;
                const uint32_t mask = pass == 0 ? 0x7FFu : 0x3FFu;
                for (int i = mt; i < nb; i += 256) hh[i] = 0u;
                named_bar_sync(kBarMath, 256);
                if (listed) {
                    for (int i = mt; i < n_mem; i += 256) {
                        const uint32_t key = mem_key[i];
                        if ((key >> hi_shift) == prefix) atomicAdd(&hh[(key >> shift) & mask], 1u);
                    }
                } else {
                    for_keys([&](bool v, int, uint32_t key) {
                        const bool m = v && (key >> hi_shift) == prefix;
                        const uint32_t dig = m ? (key >> shift) & mask : 0xFFFFFFFFu;
                        const unsigned peers = __match_any_sync(kFull, dig);
                        if (m && lane == __ffs(peers) - 1) atomicAdd(&hh[dig], (uint32_t)__popc(peers));
                    });
                }
                named_bar_sync(kBarMath, 256);
                uint32_t hs[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) hs[i] = 8 * mt + i < nb ? hh[8 * mt + i] : 0u;
                int above_p, cnt_p;
                const int dp = select_bin_m(hs, remaining, tl, mt, &above_p, &cnt_p);
                remaining -= above_p;
                prefix = (prefix << (pass == 0 ? 11 : 10)) | (uint32_t)max(dp, 0);
            }
            if (mt == 0) STI_DSTAMP(5);
            const uint32_t tau = prefix;    // the exact k-th key
            const int need_eq = remaining;  // keys == tau taken, lowest positions first (>= 1)
            // the bin's keys above tau join the bitmap; keys equal to tau get their own
            if (listed) {
                for (int i = mt; i < n_mem; i += 256) {
                    const uint32_t key = mem_key[i];
                    const int pos = mem_pos[i];
                    if (key > tau) atomicOr(&bm_gt[pos >> 5], 1u << (pos & 31));
                    else if (key == tau) atomicOr(&bm_eq[pos >> 5], 1u << (pos & 31));
                }
            } else {
                for_keys([&](bool v, int pos, uint32_t key) {
                    if (v && (key >> 21) == (uint32_t)d1) {
                        if (key > tau) bm_gt[pos >> 5] |= 1u << (pos & 31);
                        else if (key == tau) bm_eq[pos >> 5] |= 1u << (pos & 31);
                    }
                });
            }
            named_bar_sync(kBarMath, 256);
            // output slots in ascending position order: keys above tau, and the first need_eq keys
            // equal to tau
            int gt = 0, eq = 0;
            for (int w = 0; w < nw; ++w) {
                gt += __popc(bm_gt[w0 + w]);
                eq += __popc(bm_eq[w0 + w]);
            }
            if (mt == 0) STI_DSTAMP(6);
            int gt_before, eq_before, gt_tot, eq_tot;
            scan2_m(gt, eq, tl, mt, gt_before, eq_before, gt_tot, eq_tot);
            if (mt == 0) STI_DSTAMP(7);
            int o = gt_before + min(eq_before, need_eq);
            int eq_left = max(0, need_eq - eq_before);
            for (int w = 0; w < nw && o < my0 + kRows; ++w) {
                uint32_t e = bm_eq[w0 + w];
                uint32_t take_e = 0u;
                while (e && eq_left > 0) {   // the lowest positions first
                    const uint32_t lo_bit = e & (0u - e);
                    take_e |= lo_bit;
                    e ^= lo_bit;
                    --eq_left;
                }
                uint32_t sel = bm_gt[w0 + w] | take_e;
                while (sel) {
                    const int bit = __ffs(sel) - 1;
                    sel &= sel - 1u;
                    if (o >= my0 && o < my0 + kRows) {
                        const int pos = 32 * (w0 + w) + bit;
                        tl->tile_idx[o - my0] = pos;
                        idx_row[kW + o] = pos + kW;
                    }
                    ++o;
                }
            }
            if (mt == 0) STI_DSTAMP(8);
        }
        // every index is in tile_idx; the scratch rows are free for the gather
        named_bar_sync(kBarMath, 256);
        if (mt == 0) STI_DSTAMP(9);
        // ---- gather the compressed tile: math warp mw copies column block mw (16-byte cp.async
        // into the 128-byte-swizzled layout; masked rows zero-filled); rows 96..127 once the ring
        // slice's PV has read them
        {
            const uint16_t* comp = p.comp_kv + (size_t)b * p.comp_bstride + (size_t)mw * 64;
            const uint32_t blk = smem_u32(tile) + (uint32_t)mw * kBlkBytes;
            const int ch = lane & 7;
            auto copy_rows = [&](int i0, int i1) {
                for (int i = i0; i < i1; ++i) {
                    const int r = 4 * i + (lane >> 3);
                    const int raw = tl->tile_idx[r];
                    const bool ok = raw >= 0 && raw < n2 && !dead;
                    if (raw < -1 || raw >= n2) atomicOr(p.status, 1u /* STI_FLAG_INDEX_RANGE */);   // masked
                    const uint16_t* s = ok ? comp + (size_t)raw * kD + ch * 8 : comp;
                    cp_async_16(blk + (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4)), s, ok ? 16u : 0u);
                }
            };
            copy_rows(0, 24);
            mwait(&tl->ring_free, 0);
            copy_rows(24, 32);
            cp_async_commit();
            cp_async_wait<0>();
            fence_proxy_async_smem();   // generic-proxy copies, read by the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(&tl->full[mw]);
            if (mt == 0) STI_DSTAMP(10);
        }
        // ---- the compressed tile
        softmax_tile(1, !dead && tl->tile_idx[row] >= 0 && tl->tile_idx[row] < n2);
        if (mt == 0) STI_DSTAMP(12);
        mwait(&tl->o_done, 1);
        tc_fence_after();

        // ---- merge through L2: the three d-blocks others own, [128 d][64 heads] fp32 each, and
        // (m, l); then this CTA's d-block from the three others
        const int d_loc = row;   // TMEM lane = d within a block
        auto xblk = [&](int owner, int src) -> float* {   // block `owner` written by CTA `src` != owner
            const int slot = src < owner ? src : src - 1;
            return p.xchg + ((size_t)(b * kCtas + owner) * 3 + slot) * (kRows * kH);
        };
        if (!dead) {
            for (int m = 0; m < kCtas; ++m) {
                if (m == rank) continue;
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + kTmemO + (uint32_t)(m * kH + hoff), r);
                tmem_ld_wait();
                float4* dst = reinterpret_cast<float4*>(xblk(m, rank) + (size_t)d_loc * kH + hoff);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    dst[c] = make_float4(__uint_as_float(r[4 * c]), __uint_as_float(r[4 * c + 1]),
                                         __uint_as_float(r[4 * c + 2]), __uint_as_float(r[4 * c + 3]));
            }
        }
        if (mt == 0) STI_DSTAMP(25);
        float* xml = p.xml + (size_t)(b * kCtas + rank) * 2 * kH;   // this CTA's (m, l) per head
        if (mt < kH) {
            xml[mt] = tl->m_run[mt];
            xml[kH + mt] = tl->l_run[mt];
        }
        if (mt == 0) STI_DSTAMP(13);
        publish_to_cluster(&tl->pub_bar, mt);
        if (!dead) dead = !attn_wait_cluster(&tl->pub_bar, 0, p.status, abort);
        dead = __any_sync(kFull, dead);
        if (mt == 0) STI_DSTAMP(14);
        if (rank == 0) {   // every CTA has read the histogram: ready for the next call
            uint4* gh = reinterpret_cast<uint4*>(p.hist + (size_t)b * kBins);
            gh[2 * mt] = make_uint4(0, 0, 0, 0);
            gh[2 * mt + 1] = make_uint4(0, 0, 0, 0);
        }
        if (mt < kH) {   // the four partials' weights for head mt
            float mc[kCtas], lc[kCtas];
            float M = -INFINITY;
#pragma unroll
            for (int c = 0; c < kCtas; ++c) {
                const float* xc = p.xml + (size_t)(b * kCtas + c) * 2 * kH;
                mc[c] = dead ? -INFINITY : (c == rank ? tl->m_run[mt] : __ldcg(xc + mt));
                lc[c] = dead ? 0.f : (c == rank ? tl->l_run[mt] : __ldcg(xc + kH + mt));
                M = fmaxf(M, mc[c]);
            }
            float L = 0.f;
            float e[kCtas];
#pragma unroll
            for (int c = 0; c < kCtas; ++c) {
                e[c] = (M == -INFINITY || mc[c] == -INFINITY) ? 0.f : exp2f(mc[c] - M);
                L += lc[c] * e[c];
            }
            if (M != -INFINITY) L += exp2f(__ldg(p.sink + mt) * kLog2e - M);
#pragma unroll
            for (int c = 0; c < kCtas; ++c) tl->wgt[c][mt] = M == -INFINITY ? 0.f : e[c] / L;
        }
        named_bar_sync(kBarMath, 256);
        if (mt == 0) STI_DSTAMP(26);
        {
            float v[32];
            {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + kTmemO + (uint32_t)(rank * kH + hoff), r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * tl->wgt[rank][hoff + i];
            }
            // the three others' partials of this CTA's d-block (peer k is CTA k + (k >= rank)):
            // two peers' loads in flight, then the third (128 registers a thread at 416 threads)
            auto add_peers = [&](auto k0_c, auto n_c) {
                constexpr int k0 = decltype(k0_c)::value, n = decltype(n_c)::value;
                float4 q4[n][8];
#pragma unroll
                for (int k = 0; k < n; ++k) {
                    const int c = (k0 + k) + (k0 + k >= rank ? 1 : 0);
                    const float4* src4 = reinterpret_cast<const float4*>(xblk(rank, c) + (size_t)d_loc * kH + hoff);
#pragma unroll
                    for (int j = 0; j < 8; ++j) q4[k][j] = dead ? make_float4(0.f, 0.f, 0.f, 0.f) : __ldcg(src4 + j);
                }
#pragma unroll
                for (int k = 0; k < n; ++k) {
                    const int c = (k0 + k) + (k0 + k >= rank ? 1 : 0);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        v[4 * j] += q4[k][j].x * tl->wgt[c][hoff + 4 * j];
                        v[4 * j + 1] += q4[k][j].y * tl->wgt[c][hoff + 4 * j + 1];
                        v[4 * j + 2] += q4[k][j].z * tl->wgt[c][hoff + 4 * j + 2];
                        v[4 * j + 3] += q4[k][j].w * tl->wgt[c][hoff + 4 * j + 3];
                    }
                }
            };
            add_peers(std::integral_constant<int, 0>(), std::integral_constant<int, 2>());
            add_peers(std::integral_constant<int, 2>(), std::integral_constant<int, 1>());
            const int dd = kRows * rank + d_loc;
            if (p.rope_dims > 0 && kRows * rank + kRows > kD - p.rope_dims)   // the output's inverse rotation
                rope_inverse_pairs<32>(v, dd, kD, p.rope_dims, p.rope_cs + (size_t)b * p.rope_dims);
            uint16_t* orow = p.out + ((size_t)b * kH + hoff) * kD + dd;
#pragma unroll
            for (int i = 0; i < 32; ++i) orow[(size_t)i * kD] = __bfloat16_as_ushort(__float2bfloat16_rn(v[i]));
        }
        if (mt == 0) {
            STI_DSTAMP(15);
            STI_DCLOCK(31);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    cluster_sync();   // no CTA leaves while another may still signal it
}

}  // namespace

size_t decode_topk_attn_smem_bytes() { return kSmemBytes; }

// Whether the fused kernel can run b queries on this device: 4-CTA clusters of its shared memory
// footprint must be launchable (cached per device).
bool decode_topk_attn_available() {
    static std::mutex mu;
    static int state[64] = {0};   // 0 unknown, 1 yes, 2 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> g(mu);
    if (state[dev] == 0) {
        bool ok = cudaFuncSetAttribute(decode_topk_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes) == cudaSuccess;
        if (ok) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(kCtas);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = kSmemBytes;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = kCtas;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int active = 0;
            ok = cudaOccupancyMaxActiveClusters(&active, decode_topk_attn_kernel, &cfg) == cudaSuccess && active >= 1;
        }
        if (!ok) cudaGetLastError();
        state[dev] = ok ? 1 : 2;
    }
    return state[dev] == 1;
}

cudaError_t launch_decode_topk_attn(const CUtensorMap& tm_q, const CUtensorMap& tm_ring, const CUtensorMap& tm_ring_rows,
                                    const DecodeAttnParams& p, bool pdl, cudaStream_t stream) {
    if (p.B == 0) return cudaSuccess;
    cudaError_t err =
        cudaFuncSetAttribute(decode_topk_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.B * kCtas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    err = cudaLaunchKernelEx(&cfg, decode_topk_attn_kernel, tm_q, tm_ring, tm_ring_rows, p);
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace sti

#ifdef STI_DA_TIMING
// profiling builds only: global-timer stamps of the fused decode kernel's CTAs
extern "C" int sti_dbg_da_times(unsigned long long* host, int n_blocks) {
    return (int)cudaMemcpyFromSymbol(host, sti::g_da_t, sizeof(unsigned long long) * 32 * (size_t)n_blocks);
}
#endif
