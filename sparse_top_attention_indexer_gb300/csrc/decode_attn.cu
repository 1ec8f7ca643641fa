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
//   * ring slots [32r, 32r+32): rows 96..127 of its tile, run through QK and softmax before the
//     scores are complete (the kernel is a programmatic dependent of the scores kernel);
//   * the compressed rows of output slots [128r, 128r+128) of the index row: one 128-row tile;
//   * d-block r (dims [128r, 128r+128)) of the output in the merge.
// Top-k (exact; ties go to the lower position): the scores kernel's first radix pass (top 11 key
// bits) gives the threshold bin d1, found by every warp from a shared-memory copy of the
// histogram.  Each CTA scans a quarter of the row: a bitmap of the keys above the bin and, per
// warp, a segment of the bin's members, which it bulk-copies into the other three CTAs (shared to
// shared, counted on their barrier).  Every CTA then holds the whole row's bitmap and members:
// two radix passes over the members (shared-memory histograms of the next 11 and 10 bits, a bin
// taken whole ending them) give the k-th key tau and how many keys equal to it are taken; the
// members above tau join the bitmap, those equal to tau mark a second one; one block scan over
// both gives every selected position its output slot, in ascending position order.  A warp with
// more than 64 members (heavy ties) sends the passes over the whole row instead.  Each CTA keeps
// the slots it owns: its tile's index list and its quarter of the published row.
// Attention, per tile: S^T = KV.Q^T (tcgen05, M = 128 rows, N = 64 heads, K = 512) into TMEM; an
// online softmax with thread = row in two warp groups of 32 heads; O^T += V^T.P^T (M = 128 d-rows
// per d-block, N = 64, K = rows) reading the same tile as an MN-major operand.  The compressed
// rows arrive by four-row TMA gathers issued by the eight math warps (masked rows repeat a valid
// row of their group, whose probability is zero; groups with none are zeroed).
// Merge, in shared memory: each CTA sends its (max, sum) per head to the other three, computes
// every CTA's weight
//   w_c = 2^(m_c - M) / (sum_c' l_c' 2^(m_c' - M) + 2^(sink - M)),
// and bulk-copies the three d-blocks of its O^T that the others own, times its own weight, as bf16
// into their Q buffers; each owner adds the three to its own weighted block:  o = sum_c w_c O_c.
//
// Roles (13 warps): warp 0 and warps 10-12 load Q and the ring slice, warp 11 then runs the ring
// slice's softmax; warp 1 allocates TMEM and issues the MMAs; warps 2-9 (256 "math" threads) run
// the top-k, gather the compressed tile, the softmax (warps 2-5: heads 0-31, warps 6-9: heads
// 32-63) and the merge.
#include <cuda_bf16.h>
#include <cstddef>
#include <math.h>

#include <mutex>
#include <type_traits>
#include <vector>

#include "sti_internal.h"
#include "sti_kvfp4.h"
#include "sti_ptx.cuh"
#include "sti_attn_util.cuh"

namespace sti {
namespace {

#ifdef STI_DA_TIMING
// global-timer stamps per CTA (profiling builds): [0, 16) math-thread phases, [16, 24) MMA issuer
__device__ unsigned long long g_da_t[1024][64];
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
constexpr int kSegCap = 64;               // threshold-bin members one warp lists (more: row passes)
constexpr uint32_t kBlkBytes = kRows * 128;    // one column block of the tile (128 rows x 128 B)
constexpr uint32_t kQBlkBytes = kH * 128;      // one column block of Q (64 heads x 128 B)
constexpr uint32_t kTileBytes = 8 * kBlkBytes;
constexpr uint32_t kQBytes = 8 * kQBlkBytes;
constexpr uint32_t kPBytes = 2 * kQBlkBytes;   // P^T: 128 rows x 64 heads bf16 (128 B per row)
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr uint32_t kBarMath = 1, kBarSet0 = 2;   // named barriers: the 256 math threads; each set of 128

struct __align__(16) DaTail {
    uint64_t full[8];          // compressed tile, column block j landed (8 math-warp arrivals + bytes)
    uint64_t q_bar;            // Q landed
    uint64_t ring_bar;         // the ring slice landed (4 loader arrivals + bytes)
    uint64_t s_full[2];        // S^T of the ring slice / of the compressed tile in TMEM
    uint64_t p_full;           // P^T written (one arrival per softmax set), phase 0 ring, 1 tile
    uint64_t o_done;           // the ring slice's PV complete (O^T initialised)
    uint64_t ring_free;        // the ring slice's PV complete: rows 96..127 may be overwritten
    uint64_t pv_bar[4];        // the compressed tile's PV complete for d-block m
    uint64_t qfree_bar;        // merge: every CTA's compressed QK complete, its Q buffer free to receive (4 CTAs)
    uint64_t ml_bar;           // merge: the other CTAs' (max, sum) per head landed (bytes)
    uint64_t tk_bar;           // top-k: the other CTAs' words, members and counts landed (24 arrivals + bytes)
    uint64_t recv_bar;         // merge: the three other CTAs' partials of this CTA's d-block landed (bytes)
    uint64_t f4_bar;           // fp4 compressed rows: the tile's packed rows staged (bytes)
    uint32_t tmem_base;
    int abort;
    int seg_cnt[8 * kCtas];    // top-k: members each warp of the cluster found in the threshold bin
    int warp_tot[8], warp_tot2[8];
    float m_run[kH], l_run[kH], alpha[kH];
    float red_max[4][kH], red_sum[4][kH];
    float wgt[kCtas][kH];      // merge weights per head: [0, 3) the senders in slot order, 3 this CTA
    float2 xml[kCtas - 1][kH]; // the other CTAs' (running max, sum) per head, in slot order
    int tile_idx[kRows];
};

constexpr size_t kSmemBytes = 1024 + kTileBytes + kQBytes + kPBytes + sizeof(DaTail);
static_assert(kSmemBytes <= 232448, "shared memory of the fused decode kernel");

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

// The bin d (of 32 * per bins, per = 32 or 64, in shared memory) where the count from the top
// first reaches `remaining`: (d, keys in higher bins, keys in d); (-1, total, 0) when the histogram
// holds fewer keys.  One warp, no block barrier: every warp that needs the bin computes it.  Lane l
// sums bins [per l, per l + per) (its 16-byte reads rotated by l, so the eight lanes of a phase hit
// distinct banks), a suffix scan over the lanes finds the lane of d, then that lane's bins are
// split over the warp and scanned the same way.
__device__ __forceinline__ int3 select_bin_w(const uint32_t* h, int per, int remaining, int lane) {
    const int nv = per / 4;
    const uint4* h4 = reinterpret_cast<const uint4*>(h + per * lane);
    int local = 0;
#pragma unroll 4
    for (int i = 0; i < nv; ++i) {
        const uint4 v = h4[(i + lane) & (nv - 1)];
        local += (int)(v.x + v.y + v.z + v.w);
    }
    int suf = local;   // keys in the bins of lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_down_sync(kFull, suf, o);
        if (lane + o < 32) suf += x;
    }
    const unsigned hit = __ballot_sync(kFull, suf - local < remaining && suf >= remaining);
    if (hit == 0u) return make_int3(-1, __shfl_sync(kFull, suf, 0), 0);
    const int L = __ffs(hit) - 1;
    const int above_l = __shfl_sync(kFull, suf - local, L);
    const int sub = per / 32;   // bins of lane L per lane: 1 or 2
    const int b0 = per * L + sub * lane;
    const int c_hi = (int)h[b0 + sub - 1];
    const int c_lo = sub == 2 ? (int)h[b0] : 0;
    const int loc2 = c_hi + c_lo;
    int suf2 = loc2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_down_sync(kFull, suf2, o);
        if (lane + o < 32) suf2 += x;
    }
    const int above_j = above_l + suf2 - loc2;   // keys above this lane's bins
    const unsigned hit2 = __ballot_sync(kFull, above_j < remaining && above_j + loc2 >= remaining);
    const int J = hit2 ? __ffs(hit2) - 1 : 0;
    const bool top = above_j + c_hi >= remaining;   // d is this lane's higher bin
    const int d = __shfl_sync(kFull, top ? b0 + sub - 1 : b0, J);
    const int ab = __shfl_sync(kFull, top ? above_j : above_j + c_hi, J);
    const int c = __shfl_sync(kFull, top ? c_hi : c_lo, J);
    return make_int3(d, ab, c);
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_topk_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_ring,
                            const __grid_constant__ CUtensorMap tm_ring_rows,
                            const __grid_constant__ CUtensorMap tm_comp_rows, const DecodeAttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* tile = smem;                          // 8 column blocks x [128 rows x 128 B], SW128
    uint8_t* q_s = tile + kTileBytes;              // 8 column blocks x [64 heads x 128 B], SW128
    uint8_t* p_s = q_s + kQBytes;                  // P^T: [128 rows][64 heads] bf16, SW128 (MN-major B)
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
        for (int j = 0; j < 8; ++j) mbar_init(&tl->full[j], 8);
        mbar_init(&tl->q_bar, 1);
        mbar_init(&tl->ring_bar, 4);
        mbar_init(&tl->s_full[0], 1);
        mbar_init(&tl->s_full[1], 1);
        mbar_init(&tl->p_full, 2);
        mbar_init(&tl->o_done, 1);
        mbar_init(&tl->ring_free, 1);
        for (int m = 0; m < 4; ++m) mbar_init(&tl->pv_bar[m], 1);
        mbar_init(&tl->qfree_bar, kCtas);
        mbar_init(&tl->ml_bar, 1);
        mbar_init(&tl->tk_bar, (kCtas - 1) * 8);
        mbar_init(&tl->recv_bar, 1);
        mbar_init(&tl->f4_bar, 1);
        // the merge's incoming bytes, fixed: three (max, sum) vectors and three partial d-blocks
        mbar_arrive_expect_tx(&tl->ml_bar, (kCtas - 1) * kH * 8);
        mbar_arrive_expect_tx(&tl->recv_bar, (kCtas - 1) * kRows * kH * 2);
        tl->abort = 0;
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
    // [384, 448): the compressed tile's second partial S^T (its QK alternates two accumulators so
    // consecutive MMAs do not wait on each other; the softmax adds the two)
    constexpr uint32_t kTmemS2 = 384;

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
                tma_prefetch_desc(&tm_comp_rows);
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
        if (warp == 11) {
            // ---- the ring slice's softmax, by the one warp whose TMEM lane quarter holds tile rows
            // 96..127 (lane = ring slot 32*rank + lane), while the math warps run the top-k: the
            // first tile, so the running max is its own max and the running sum its own sum
            bool ok = attn_wait(&tl->s_full[0], 0, p.status, abort);
            ok = __all_sync(kFull, ok);
            tc_fence_after();
            const bool valid = ok && ring_valid(lane);
            float x[64];
            {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)kRingRow0 << 16), r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = valid ? __uint_as_float(r[i]) * p.scale_log2 : -INFINITY;
                tmem_ld32(tmem + ((uint32_t)kRingRow0 << 16) + 32u, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) x[32 + i] = valid ? __uint_as_float(r[i]) * p.scale_log2 : -INFINITY;
            }
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {   // per-head maxima over the 32 rows: lane l gets head 32 hb + l
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = x[32 * hb + i];
                warp_reduce_scatter_n<32, true>(v);
                tl->m_run[32 * hb + lane] = v[0];
            }
            __syncwarp();
            const int rr = kRingRow0 + lane;   // this lane's tile row; P^T[rr][h], 16-byte chunk h/8 ^ rr % 8
            uint8_t* prow = p_s + rr * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float m = tl->m_run[8 * c + j];
                    x[8 * c + j] = (m == -INFINITY) ? 0.f : fast_exp2(x[8 * c + j] - m);
                }
                uint4 pk;
                pk.x = pack_bf16x2(x[8 * c + 0], x[8 * c + 1]);
                pk.y = pack_bf16x2(x[8 * c + 2], x[8 * c + 3]);
                pk.z = pack_bf16x2(x[8 * c + 4], x[8 * c + 5]);
                pk.w = pack_bf16x2(x[8 * c + 6], x[8 * c + 7]);
                *reinterpret_cast<uint4*>(prow + ((c ^ (rr & 7)) << 4)) = pk;
            }
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = x[32 * hb + i];
                warp_reduce_scatter_n<32, false>(v);
                tl->l_run[32 * hb + lane] = v[0];
            }
            fence_proxy_async_smem();   // P^T: generic writes read by the MMA
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {   // both arrivals of phase 0 (the math warps' two sets make phase 1's)
                mbar_arrive(&tl->p_full);
                mbar_arrive(&tl->p_full);
            }
            if (lane == 0) STI_DSTAMP(27);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t idesc_qk = idesc_bf16_f32(kRows, kH, false, false);
            const uint32_t idesc_pv = idesc_bf16_f32(128, kH, true, true);
            const uint64_t kd0 = sdesc(smem_u32(tile), 16, 1024, kLayoutSW128);          // K-major tile
            const uint64_t vd0 = sdesc(smem_u32(tile), kBlkBytes, 1024, kLayoutSW128);   // MN-major tile
            const uint64_t qd0 = sdesc(smem_u32(q_s), 16, 1024, kLayoutSW128);
            const uint64_t pd0 = sdesc(smem_u32(p_s), kPBytes, 1024, kLayoutSW128);   // MN-major P^T [row][head]
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
                                  pd0 + (uint64_t)(kk * (2048 >> 4)), idesc_pv,
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
            for (int j = 0; j < 8; ++j) {   // QK of the compressed tile, column block by column block, its
                ok = ok && attn_wait(&tl->full[j], 0, p.status, abort);   // K steps alternating between
                if (j == 0) STI_DSTAMP(18);                                // two accumulators
                if (j == 7) STI_DSTAMP(19);
                if (ok) {
                    tc_fence_after();
                    const uint64_t a = kd0 + (uint64_t)((uint32_t)j * (kBlkBytes >> 4));
                    const uint64_t bq = qd0 + (uint64_t)((uint32_t)j * (kQBlkBytes >> 4));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + ((kk & 1) ? kTmemS2 : (uint32_t)kH), a + 2 * kk, bq + 2 * kk, idesc_qk,
                                  (j > 0 || kk > 1) ? 1u : 0u);
                }
            }
            umma_commit(&tl->s_full[1]);
            STI_DSTAMP(50);
            ok = ok && attn_wait(&tl->p_full, 1, p.status, abort);
            STI_DSTAMP(20);
            if (ok) tc_fence_after();
            // d-block by d-block, the blocks the other CTAs own first (their shares leave as soon as
            // each is done), this CTA's own block last
            for (int j = 1; j <= kCtas; ++j) {
                const int m = (rank + j) & 3;
                if (ok) {
                    const uint64_t a = vd0 + (uint64_t)((uint32_t)(2 * m) * (kBlkBytes >> 4));
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_bf16(tmem + kTmemO + (uint32_t)(m * kH), a + (uint64_t)(kk * (2048 >> 4)),
                                  pd0 + (uint64_t)(kk * (2048 >> 4)), idesc_pv, 1u);
                }
                umma_commit(&tl->pv_bar[m]);
            }
            STI_DSTAMP(45);
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
        auto mwait_c = [&](uint64_t* bar) {   // phase 0 of a barrier the cluster's st.async stores complete
            if (!dead) dead = !attn_wait_cluster(bar, 0, p.status, abort);
            dead = __any_sync(kFull, dead);
        };

        // online softmax over the compressed tile's S^T (t = 1; the sum of its two partial
        // accumulators), continuing the ring slice's running max and sum.  Thread = row, the set's
        // 32 heads in registers (one TMEM pass); lane l of every warp of the set resolves head
        // hoff + l's new max and rescale factor itself (one barrier), P^T rows leave as 16-byte
        // stores.
        auto softmax_tile = [&](int t, bool valid) {
            mwait(&tl->s_full[t], 0);
            if (t == 1 && mt == 0) STI_DSTAMP(11);
            tc_fence_after();
            if (t == 1 && mt == 0 && !dead)   // the QK has read Q: its buffer may receive the merge shares
                for (int c = 0; c < kCtas; ++c) mbar_arrive_remote_relaxed(dsmem_addr(&tl->qfree_bar, (uint32_t)c));
            const uint32_t s_col = tmem + lane_base + (uint32_t)(t * kH + hoff);
            float x[32];   // this row's S of heads hoff .. hoff + 31, log2 units
            {
                uint32_t r[32], r2[32];
                tmem_ld32(s_col, r);
                tmem_ld32(s_col + (kTmemS2 - (uint32_t)kH), r2);   // the second partial
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    x[i] = (valid && !dead) ? (__uint_as_float(r[i]) + __uint_as_float(r2[i])) * p.scale_log2
                                            : -INFINITY;
            }
            {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = x[i];
                warp_reduce_scatter_n<32, true>(v);   // lane l: head hoff + l over this warp's 32 rows
                tl->red_max[qd][hoff + lane] = v[0];
            }
            if (t == 1 && mt == 0) STI_DSTAMP(21);
            named_bar_sync(bar_set, 128);
            if (t == 1 && mt == 0) STI_DSTAMP(22);
            const int hl = hoff + lane;
            const float mx = fmaxf(fmaxf(tl->red_max[0][hl], tl->red_max[1][hl]), fmaxf(tl->red_max[2][hl], tl->red_max[3][hl]));
            const float m_old = tl->m_run[hl];
            // the running max moves only when a tile's max passes it by more than 8 (log2 units)
            const float m_new = (m_old == -INFINITY || mx > m_old + 8.f) ? fmaxf(m_old, mx) : m_old;
            const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2(m_old - m_new);
            // the ring slice's PV has read P^T and written O^T before the tile's P^T and rescale
            if (t == 1) mwait(&tl->o_done, 0);
            tc_fence_after();
            uint8_t* prow = p_s + row * 128;   // P^T[row][h]: 16-byte chunk h/8, swizzled by row % 8
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float mh = __shfl_sync(kFull, m_new, 8 * c + j);
                    x[8 * c + j] = (mh == -INFINITY) ? 0.f : fast_exp2(x[8 * c + j] - mh);
                }
                uint4 pk;
                pk.x = pack_bf16x2(x[8 * c + 0], x[8 * c + 1]);
                pk.y = pack_bf16x2(x[8 * c + 2], x[8 * c + 3]);
                pk.z = pack_bf16x2(x[8 * c + 4], x[8 * c + 5]);
                pk.w = pack_bf16x2(x[8 * c + 6], x[8 * c + 7]);
                *reinterpret_cast<uint4*>(prow + (((4 * set + c) ^ (row & 7)) << 4)) = pk;
            }
            warp_reduce_scatter_n<32, false>(x);   // lane l: the sum of head hoff + l over this warp's rows
            tl->red_sum[qd][hl] = x[0];
            if (t == 1 && mt == 0) STI_DSTAMP(23);
            if (t == 1 && !dead && __any_sync(kFull, alpha != 1.f)) {
                // O^T rows (lane = d within a block) times the heads' factors
#pragma unroll 1
                for (int m = 0; m < 4; ++m) {
                    const uint32_t ta = tmem + lane_base + kTmemO + (uint32_t)(m * kH + hoff);
                    uint32_t r[32];
                    tmem_ld32(ta, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        r[i] = __float_as_uint(__uint_as_float(r[i]) * __shfl_sync(kFull, alpha, i));
                    tmem_st32(ta, r);
                }
                tmem_st_wait();
            }
            if (t == 1 && mt == 0) STI_DSTAMP(24);
            fence_proxy_async_smem();   // P^T: generic writes read by the MMA
            tc_fence_before();
            named_bar_sync(bar_set, 128);
            if (st < 32) {   // warps 2 and 6: lane st holds head hoff + st
                tl->m_run[hl] = m_new;
                tl->alpha[hl] = alpha;
                tl->l_run[hl] = tl->l_run[hl] * alpha + (tl->red_sum[0][hl] + tl->red_sum[1][hl]) +
                                (tl->red_sum[2][hl] + tl->red_sum[3][hl]);
            }
            if (st == 0) mbar_arrive(&tl->p_full);
        };

        // ---- top-k scratch in tile rows 0..95 (free until the gather; the ring slice's QK reads them
        // only into masked rows of S): rows 64..95 of column blocks 0-1 and 2-3 hold the position
        // bitmaps (keys above tau, keys equal to tau), of block 6 the pass-3 histogram; rows 0..63 of
        // blocks 4-5 the threshold bin's members as every warp of the cluster found them (segment
        // 8 * CTA + warp: up to kSegCap (key, position) pairs), and rows 0..63 of every block the
        // staged scores of the row passes (only when the members overflow their segments); P^T rows
        // 0..63 (the ring slice's probabilities use rows 96..127 only) the pass-2 histogram
        auto bm = [&](int blk0, int w) {   // bitmap word w (blk0 = 0: keys > tau, 2: keys == tau)
            return reinterpret_cast<uint32_t*>(tile + (size_t)(blk0 + (w >> 10)) * kBlkBytes + 8192) + (w & 1023);
        };
        auto seg = [&](int sg, int j) {   // member j of segment sg
            const int i = sg * kSegCap + j;
            return reinterpret_cast<uint2*>(tile + (size_t)(4 + (i >> 10)) * kBlkBytes) + (i & 1023);
        };
        uint32_t* h2 = reinterpret_cast<uint32_t*>(p_s);                           // [2048]
        uint32_t* h3 = reinterpret_cast<uint32_t*>(tile + 6 * kBlkBytes + 8192);   // [1024]

        // ---- the Indexer's top-k of one row, exact (ties to the lower position).  Each CTA scans a
        // quarter of the row against the threshold bin of the scores kernel's histogram and sends
        // what it finds to the whole cluster; every CTA then resolves the bin (passes 2 and 3 over
        // its members) and keeps output slots [128 rank, 128 rank + 128): its tile's index list and
        // its quarter of the published row.
        auto topk_row = [&](int vis_) {
            const int my0 = kRows * rank;
            if (vis_ <= kK) {   // every visible position is selected: slot o holds position o
                if (mt < kRows) {
                    const int o = my0 + mt;
                    tl->tile_idx[mt] = o < vis_ ? o : -1;
                    idx_row[kW + o] = o < vis_ ? o + kW : -1;
                }
                if (rank == 0) {   // nobody reads the histogram: ready for the next call
                    uint4* gh = reinterpret_cast<uint4*>(p.hist + (size_t)b * kBins);
                    gh[2 * mt] = make_uint4(0, 0, 0, 0);
                    gh[2 * mt + 1] = make_uint4(0, 0, 0, 0);
                }
                return;
            }
            const uint32_t* ghist = p.hist + (size_t)b * kBins;
            const float* src = p.scores + (size_t)b * n2;
            const int nwords = (vis_ + 31) / 32;
            const bool vec4 = (reinterpret_cast<uintptr_t>(src) & 15u) == 0u;
            constexpr int kStage = 16384;
            auto stage_ptr = [&](int i) {   // staged score i of the current round
                return reinterpret_cast<const uint32_t*>(tile + (size_t)(i >> 11) * kBlkBytes) + (i & 2047);
            };
            // all words of the row in rounds: f(word, valid, position, key), warp mw taking four words
            // per iteration (four independent load-compare-ballot chains), lane = bit
            auto row_pass = [&](auto&& f) {
                for (int r0 = 0; r0 < vis_; r0 += kStage) {
                    const int rn = min(kStage, vis_ - r0);
                    const bool v4 = vec4 && (r0 & 3) == 0;
                    for (int c = mt; c < rn / 4; c += 256) {
                        const int i = 4 * c;
                        const uint32_t dst = smem_u32(stage_ptr(i));
                        if (v4) {
                            cp_async_16(dst, src + r0 + i, 16u);
                        } else {
                            for (int e = 0; e < 4; ++e) cp_async_4(dst + 4u * e, src + r0 + i + e);
                        }
                    }
                    for (int i = (rn & ~3) + mt; i < rn; i += 256) cp_async_4(smem_u32(stage_ptr(i)), src + r0 + i);
                    cp_async_commit();
                    cp_async_wait<0>();
                    named_bar_sync(kBarMath, 256);
                    const int w_lo = r0 / 32, w_hi = (r0 + rn + 31) / 32;
                    for (int w4 = w_lo + 4 * mw; w4 < w_hi; w4 += 32) {
                        uint32_t key[4];
                        bool v[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int pos = 32 * (w4 + q) + lane;
                            v[q] = w4 + q < w_hi && pos < vis_;
                            key[q] = v[q] ? float_key(__uint_as_float(*stage_ptr(pos - r0))) : 0u;
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (w4 + q < w_hi) f(w4 + q, v[q], 32 * (w4 + q) + lane, key[q]);
                    }
                    named_bar_sync(kBarMath, 256);   // before the next round overwrites the staged scores
                }
            };
            // this CTA's quarter of the row; warp mw stages 16 words (32 scores each) at a time in
            // rows 0..63 of column blocks 0-1, lane = bit (each lane reads back only its own copies)
            const int wq = ((nwords + kCtas - 1) / kCtas + 15) & ~15;   // whole 16-word groups
            const int wa = min(nwords, rank * wq), wb = min(nwords, wa + wq);
            float* stg = reinterpret_cast<float*>(tile + (size_t)(mw >> 2) * kBlkBytes + (size_t)(mw & 3) * 2048);
            auto stage16 = [&](int g) {
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const int pos = 32 * (g + q) + lane;
                    if (g + q < wb && pos < vis_) cp_async_4(smem_u32(stg + 32 * q + lane), src + pos);
                }
                cp_async_commit();
            };
            if (wa + 16 * mw < wb) stage16(wa + 16 * mw);   // in flight during the bin selection
            // pass 1 from the scores kernel's histogram, copied to rows 0..63 of block 2: the threshold bin
            uint32_t* h1 = reinterpret_cast<uint32_t*>(tile + 2 * kBlkBytes);
            {
                const uint4* gh = reinterpret_cast<const uint4*>(ghist);
                uint4* h14 = reinterpret_cast<uint4*>(h1);
                const uint4 a0 = __ldcg(gh + 2 * mt), a1 = __ldcg(gh + 2 * mt + 1);
                h14[2 * mt] = a0;
                h14[2 * mt + 1] = a1;
            }
            named_bar_sync(kBarMath, 256);
            const int3 s1 = select_bin_w(h1, 64, kK, lane);
            const int d1 = s1.x, above1 = s1.y, c1 = s1.z;
            const int remaining1 = kK - above1;   // keys of bin d1 to take (>= 1)
            if (mt == 0) STI_DSTAMP(3);
            // this CTA's quarter of the row, 16 words per warp at a time: the words of keys above the
            // bin and the warp's members of the bin (its segment) are written here, then bulk-copied
            // into the other three CTAs (shared to shared, counted on their tk_bar) with the member
            // count and one arrive per CTA that announces the bytes sent to it
            {
                const int sg_own = 8 * rank + mw;
                int cnt = 0, groups = 0;
                for (int g = wa + 16 * mw; g < wb; g += 128, ++groups) {
                    cp_async_wait<0>();
                    if (mt == 0) STI_DSTAMP(52);
                    uint32_t my_above = 0u;
#pragma unroll 4
                    for (int q = 0; q < 16; ++q) {
                        const int pos = 32 * (g + q) + lane;
                        const bool v = g + q < wb && pos < vis_;
                        const uint32_t key = float_key(stg[32 * q + lane]);
                        const uint32_t dig = key >> 21;
                        const unsigned above = __ballot_sync(kFull, v && dig > (uint32_t)d1);
                        const bool m = v && dig == (uint32_t)d1;
                        const unsigned mem = __ballot_sync(kFull, m);
                        if (lane == q) my_above = above;
                        const int at = cnt + __popc(mem & ((1u << lane) - 1u));
                        if (m && at < kSegCap) *seg(sg_own, at) = make_uint2(key, (uint32_t)pos);
                        cnt += __popc(mem);
                    }
                    if (mt == 0) STI_DSTAMP(53);
                    if (g + 128 < wb) stage16(g + 128);
                    if (lane < 16) *bm(0, g + lane) = g + lane < wb ? my_above : 0u;
                    fence_proxy_async_smem();   // generic writes, read by the bulk copies
                    __syncwarp();
                    if (lane < kCtas - 1) {   // the group's 16 words (64 B) to CTA (rank + 1 + lane) % 4
                        const uint32_t peer = (uint32_t)((rank + 1 + lane) & (kCtas - 1));
                        bulk_copy_to_peer(dsmem_addr(bm(0, g), peer), bm(0, g), 64u, dsmem_addr(&tl->tk_bar, peer));
                    }
                    if (mt == 0) STI_DSTAMP(54);
                }
                const uint32_t mem_bytes = (uint32_t)((min(cnt, kSegCap) * 8 + 15) & ~15);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane < kCtas - 1) {   // the members and their count to CTA (rank + 1 + lane) % 4
                    const uint32_t peer = (uint32_t)((rank + 1 + lane) & (kCtas - 1));
                    const uint32_t pbar = dsmem_addr(&tl->tk_bar, peer);
                    if (mem_bytes) bulk_copy_to_peer(dsmem_addr(seg(sg_own, 0), peer), seg(sg_own, 0), mem_bytes, pbar);
                    st_async_b32(dsmem_addr(&tl->seg_cnt[sg_own], peer), (uint32_t)cnt, pbar);
                    mbar_arrive_expect_tx_remote(pbar, 64u * (uint32_t)groups + mem_bytes + 4u);
                }
                if (lane == 0) tl->seg_cnt[sg_own] = cnt;
            }
            named_bar_sync(kBarMath, 256);   // this CTA's words, members and counts
            if (mt == 0) STI_DSTAMP(28);
            if (!dead) dead = !attn_wait_cluster(&tl->tk_bar, 0, p.status, abort);   // the other CTAs'
            dead = __any_sync(kFull, dead);
            if (mt == 0) STI_DSTAMP(4);
            if (rank == 0) {   // every CTA of the cluster has read the histogram: ready for the next call
                uint4* gh = reinterpret_cast<uint4*>(p.hist + (size_t)b * kBins);
                gh[2 * mt] = make_uint4(0, 0, 0, 0);
                gh[2 * mt + 1] = make_uint4(0, 0, 0, 0);
            }
            int n_mem = 0;
            bool fits = true;
#pragma unroll
            for (int i = 0; i < 8 * kCtas; ++i) {
                const int c = tl->seg_cnt[i];
                n_mem += c;
                fits = fits && c <= kSegCap;
            }
            // the members resolve the bin when none overflowed its segment (else: row passes)
            const bool listed = !dead && fits && n_mem == c1;
            const int sgm = mt >> 3, jm = mt & 7;   // thread mt: every eighth member of segment mt / 8
            const int nseg = listed ? tl->seg_cnt[sgm] : 0;
            if (mt == 0) STI_DSTAMP(37);
            // passes 2 and 3: the next 11 and 10 bits (histograms zeroed before the scores were ready)
            // a bin taken whole ends the passes: every key from its prefix up is selected
            uint32_t prefix = (uint32_t)d1;
            int remaining = remaining1;
            bool whole = c1 == remaining1;
            int bits_left = 21;   // key bits below the prefix
            for (int pass = 0; pass < 2 && !whole; ++pass) {
                uint32_t* hh = pass == 0 ? h2 : h3;
                const int nb = pass == 0 ? 2048 : 1024;
                const int hi_shift = pass == 0 ? 21 : 10, shift = pass == 0 ? 10 : 0;
                const uint32_t mask = pass == 0 ? 0x7FFu : 0x3FFu;
                if (listed) {
                    for (int j = jm; j < nseg; j += 8) {
                        const uint32_t key = seg(sgm, j)->x;
                        if ((key >> hi_shift) == prefix) atomicAdd(&hh[(key >> shift) & mask], 1u);
                    }
                    named_bar_sync(kBarMath, 256);
                    if (mt == 0) STI_DSTAMP(40 + 3 * pass);
                } else {
                    row_pass([&](int, bool v, int, uint32_t key) {
                        const bool m = v && (key >> hi_shift) == prefix;
                        const uint32_t dig = m ? (key >> shift) & mask : 0xFFFFFFFFu;
                        const unsigned peers = __match_any_sync(kFull, dig);
                        if (m && lane == __ffs(peers) - 1) atomicAdd(&hh[dig], (uint32_t)__popc(peers));
                    });
                }
                const int3 sp_ = select_bin_w(hh, nb / 32, remaining, lane);
                remaining -= sp_.y;
                prefix = (prefix << (pass == 0 ? 11 : 10)) | (uint32_t)max(sp_.x, 0);
                bits_left = pass == 0 ? 10 : 0;
                whole = sp_.z == remaining;
                if (mt == 0) STI_DSTAMP(41 + 3 * pass);
            }
            // keys > tau are taken, and the first need_eq keys == tau (lowest positions first): tau is
            // the exact k-th key after pass 3, else the smallest key of the bin taken whole (all of
            // whose keys are taken)
            const uint32_t tau = prefix << bits_left;
            const int need_eq = whole ? (1 << 30) : remaining;
            if (mt == 0) STI_DSTAMP(5);
            // the bin's keys above tau join the first bitmap; keys equal to tau get the second
            if (listed) {
                for (int j = jm; j < nseg; j += 8) {
                    const uint2 kp = *seg(sgm, j);
                    if (kp.x > tau) atomicOr(bm(0, (int)(kp.y >> 5)), 1u << (kp.y & 31));
                    else if (kp.x == tau) atomicOr(bm(2, (int)(kp.y >> 5)), 1u << (kp.y & 31));
                }
                named_bar_sync(kBarMath, 256);
            } else {
                row_pass([&](int w, bool v, int, uint32_t key) {
                    const bool in_bin = v && (key >> 21) == (uint32_t)d1;
                    const unsigned g = __ballot_sync(kFull, in_bin && key > tau);
                    const unsigned e = __ballot_sync(kFull, in_bin && key == tau);
                    if (lane == 0) {
                        *bm(0, w) |= g;
                        *bm(2, w) = e;
                    }
                });
            }
            if (mt == 0) STI_DSTAMP(6);
            // output slots in ascending position order: keys above tau, and the first need_eq keys
            // equal to tau; thread mt owns words [mt*nwt, mt*nwt + nwt)
            const int nwt = (nwords + 255) / 256;
            const int ws0 = min(nwords, mt * nwt), ws1 = min(nwords, ws0 + nwt);
            int gt = 0, eq = 0;
            for (int w = ws0; w < ws1; ++w) {
                gt += __popc(*bm(0, w));
                eq += __popc(*bm(2, w));
            }
            int gt_before, eq_before, gt_tot, eq_tot;
            scan2_m(gt, eq, tl, mt, gt_before, eq_before, gt_tot, eq_tot);
            if (mt == 0) STI_DSTAMP(7);
            int o = gt_before + min(eq_before, need_eq);
            int eq_left = max(0, need_eq - eq_before);
            for (int w = ws0; w < ws1 && o < my0 + kRows; ++w) {
                uint32_t e = *bm(2, w), take_e = 0u;
                while (e && eq_left > 0) {   // the lowest positions first
                    const uint32_t lo_bit = e & (0u - e);
                    take_e |= lo_bit;
                    e ^= lo_bit;
                    --eq_left;
                }
                uint32_t sel = *bm(0, w) | take_e;
                if (o + __popc(sel) <= my0) {   // the whole word falls before this CTA's slots
                    o += __popc(sel);
                    continue;
                }
                while (sel) {
                    const int bit = __ffs(sel) - 1;
                    sel &= sel - 1u;
                    if (o >= my0 && o < my0 + kRows) {
                        const int pos = 32 * w + bit;
                        tl->tile_idx[o - my0] = pos;
                        idx_row[kW + o] = pos + kW;
                    }
                    ++o;
                }
            }
            if (mt == 0) STI_DSTAMP(8);
        };

        // ---- gather the compressed tile: math warp mw loads rows 16mw..16mw+15, lane l the four rows
        // of group 4mw + l/8 in column block l%8 by one four-row TMA gather (so the eight pieces of a
        // row leave together; in the tile's 128-byte swizzle; masked rows of a group repeat its first
        // valid row, whose probability is zero; groups with none are zeroed).  Rows 96..127 load once
        // the ring slice's PV has read them.  Column block j is complete when its bytes and one
        // arrive of every math warp reached full[j].
        auto gather_comp = [&]() {
            const int grp = 4 * mw + (lane >> 3), cb = lane & 7;
            int ys[4], first = -1;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int raw = tl->tile_idx[4 * grp + i];
                const bool ok = raw >= 0 && raw < n2 && !dead;
                if (cb == 0 && (raw < -1 || raw >= n2)) atomicOr(p.status, 1u /* STI_FLAG_INDEX_RANGE */);   // masked
                ys[i] = ok ? b * (int)p.rows_c + raw : -1;
                if (ok && first < 0) first = ys[i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) ys[i] = ys[i] >= 0 ? ys[i] : first;
            const bool issue = first >= 0;
            const unsigned im = __ballot_sync(kFull, issue);   // the same for the eight lanes of a group
            if (lane < 8) mbar_expect_tx(&tl->full[lane], (uint32_t)__popc(im) * 64u);
            __syncwarp();
            uint8_t* dst = tile + (size_t)cb * kBlkBytes + (size_t)grp * 512;
            if (mw >= 6) mwait(&tl->ring_free, 0);   // rows 96..127
            if (issue) {
                tma_gather4(dst, &tm_comp_rows, &tl->full[cb], cb * 64, ys[0], ys[1], ys[2], ys[3]);
            } else {
#pragma unroll 4
                for (int i = 0; i < 32; ++i) reinterpret_cast<uint4*>(dst)[i] = make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();   // zeroed rows: generic writes, read by the tensor core
            }
            __syncwarp();
            if (lane < 8) mbar_arrive(&tl->full[lane]);
        };

        // ---- the same tile from fp4 rows (256 code bytes + 32 E4M3 scale bytes per row): the packed
        // rows are staged by bulk copies -- tile rows 0..95 into the ring slice's rows of column
        // blocks 0..6, rows 96..127 into P^T (both free once the ring slice's PV has read them) --
        // then all 256 threads decode 16-byte chunks of 8 elements (4 code bytes and their group's
        // scale) into the tile's swizzled bf16 layout: rows 0..95 first, then, once those stagings
        // are consumed, rows 96..127 over them.  Masked rows are zero.  One arrive per warp
        // completes full[j].
        auto stage_fp4 = [&](int r) -> uint8_t* {   // staged packed row of tile row r (288 bytes)
            return r < 96 ? tile + (size_t)(r / 14) * kBlkBytes + (size_t)kRingRow0 * 128 + (size_t)(r % 14) * 288
                          : p_s + (size_t)(r - 96) * 288;
        };
        auto gather_comp_fp4 = [&]() {
            mwait(&tl->ring_free, 0);
            // one bulk copy of the 256 code bytes and one of the 32 scale bytes per visible row,
            // lane l of warp mw taking row 16 mw + l, all counted on f4_bar
            if (lane < 16) {
                const int r = 16 * mw + lane;
                const int raw = tl->tile_idx[r];
                if (raw < -1 || raw >= n2) atomicOr(p.status, 1u /* STI_FLAG_INDEX_RANGE */);   // masked
                if (raw >= 0 && raw < n2 && !dead) {
                    uint8_t* dst = stage_fp4(r);
                    bulk_load(dst, p.comp_codes + (size_t)b * p.codes_bstride + (size_t)raw * (kD / 2), kD / 2,
                              &tl->f4_bar);
                    bulk_load(dst + kD / 2, p.comp_scales + (size_t)b * p.scales_bstride + (size_t)raw * (kD / 16),
                              kD / 16, &tl->f4_bar);
                }
            }
            if (mw == 0) {   // the bytes of every visible row of the tile
                int nv = 0;
#pragma unroll
                for (int r = lane; r < kRows; r += 32) nv += (tl->tile_idx[r] >= 0 && tl->tile_idx[r] < n2) ? 1 : 0;
                nv = __reduce_add_sync(kFull, nv);
                if (lane == 0) mbar_arrive_expect_tx(&tl->f4_bar, dead ? 0u : (uint32_t)nv * (kD / 2 + kD / 16));
            }
            if (mt == 0) STI_DSTAMP(55);
            mwait(&tl->f4_bar, 0);
            if (mt == 0) STI_DSTAMP(56);
            auto decode = [&](int r0, int r1) {   // four chunks per thread at a time (rows come in
                for (int i0 = mt; i0 < (r1 - r0) * 64; i0 += 1024) {   // multiples of 16): all four
                    uint32_t cw[4], sb[4];                               // loaded before any store, so
                    int rr[4];                                           // the loads need not wait on them
                    bool ok[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = i0 + 256 * u;
                        rr[u] = r0 + (i >> 6);
                        const int raw = tl->tile_idx[rr[u]];
                        ok[u] = raw >= 0 && raw < n2 && !dead;
                        const uint8_t* st8 = stage_fp4(rr[u]);
                        const int c = i & 63;
                        cw[u] = ok[u] ? *reinterpret_cast<const uint32_t*>(st8 + 4 * c) : 0u;
                        sb[u] = ok[u] ? st8[256 + (c >> 1)] : 0u;
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int c = (i0 + 256 * u) & 63, r = rr[u];
                        const uint4 v = ok[u] ? kvfp4_decode8(cw[u], e4m3_to_float(sb[u])) : make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4*>(tile + (size_t)(c >> 3) * kBlkBytes + (size_t)r * 128 +
                                                  ((((uint32_t)(c & 7)) ^ (uint32_t)(r & 7)) << 4)) = v;
                    }
                }
            };
            decode(0, 96);
            if (mt == 0) STI_DSTAMP(57);
            named_bar_sync(kBarMath, 256);   // rows 0..95's stagings are consumed
            decode(96, 128);
            if (mt == 0) STI_DSTAMP(58);
            fence_proxy_async_smem();   // generic writes, read by the tensor core
            __syncwarp();
            if (lane < 8) mbar_arrive(&tl->full[lane]);
        };

        // compressed row of tile row i once the indices are here: -1 when masked or out of range
        auto tile_row = [&](int i) {
            const int v = tl->tile_idx[i];
            return (v >= 0 && v < n2) ? v : -1;
        };
        // the top-k (the step's critical path; warp 11 runs the ring slice's softmax meanwhile),
        // the compressed tile's gather, then its softmax
        // the histograms of passes 2 and 3 and the bitmap of keys equal to tau start at zero
        for (int i = mt; i < 2048; i += 256) {
            h2[i] = 0u;
            *bm(2, i) = 0u;
        }
        for (int i = mt; i < 1024; i += 256) h3[i] = 0u;
        griddep_wait();   // the scores and histogram are complete from here on
        if (mt == 0) STI_DSTAMP(2);
        topk_row(max(0, min((sp + 1) / p.ratio, n2)));
        fence_proxy_async_smem();   // the scratch's generic writes, before the gather's async copies over it
        named_bar_sync(kBarMath, 256);   // every index is in tile_idx; the scratch rows are free
        if (mt == 0) STI_DSTAMP(9);
        if (p.kvfp4) gather_comp_fp4();
        else gather_comp();
        if (mt == 0) STI_DSTAMP(10);
        mwait(&tl->p_full, 0);   // the ring slice's running max and sum (warp 11) are visible
        softmax_tile(1, !dead && tile_row(row) >= 0);
        if (mt == 0) STI_DSTAMP(12);

        // ---- merge in shared memory.  Each CTA sends its (max, sum) per head to the other three as
        // soon as its softmax is done.  Its PV runs d-block by d-block, the three blocks the others own
        // first: as each completes, the block of its O^T is staged as [128 d][64 heads] bf16 (the
        // eight 16-byte chunks of a d row XOR-swizzled by d) and copied into its owner's Q buffer,
        // free since the owner's QK (bulk shared-to-shared copies counted on the owner's recv_bar;
        // slot k, bytes [16K k, 16K k + 16K), comes from CTA k + (k >= owner)).  Meanwhile each CTA
        // computes every CTA's weight per head, 2^(m_c - M) / (sum_c l_c 2^(m_c - M) + 2^(sink - M)),
        // and the owner adds the three shares times their senders' weights to its own block times
        // its own.
        const int d_loc = row;   // TMEM lane = d within a block
        if (st < 32 && !dead) {
            const int hh = hoff + st;
            const float2 ml = make_float2(tl->m_run[hh], tl->l_run[hh]);
#pragma unroll
            for (int c = 1; c < kCtas; ++c) {
                const uint32_t peer = (uint32_t)((rank + c) & (kCtas - 1));
                const int slot = rank < (int)peer ? rank : rank - 1;
                st_async_u2(dsmem_addr(&tl->xml[slot][hh], peer), __float_as_uint(ml.x), __float_as_uint(ml.y),
                            dsmem_addr(&tl->ml_bar, peer));
            }
        }
        constexpr uint32_t kPartBytes = kRows * kH * 2;   // one d-block's share: [128 d][64 heads] bf16
        // the share of d-block m is staged over the first of its own two column blocks of the tile: the
        // PV of block m has read them, and the later PVs read only their own blocks
        auto out_stage = [&](int m) -> uint8_t* { return tile + (size_t)(2 * m) * kBlkBytes; };
        // every Q buffer is free (each CTA's compressed QK has read its Q)
        if (!dead) dead = !attn_wait_cluster(&tl->qfree_bar, 0, p.status, abort);
        dead = __any_sync(kFull, dead);
        if (mt == 0) STI_DSTAMP(14);
        // the others' d-blocks, each as soon as its PV is done: staged as bf16 (unweighted; the owner
        // applies this CTA's weight) in the tile the PV has finished reading, and copied to the owner
        const uint32_t swz = (uint32_t)(d_loc & 7);
#pragma unroll 1
        for (int j = 1; j < kCtas; ++j) {
            const int m = (j + rank) & 3;
            mwait(&tl->pv_bar[m], 0);
            if (mt == 0) STI_DSTAMP(45 + j);
            tc_fence_after();
            if (!dead) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + kTmemO + (uint32_t)(m * kH + hoff), r);
                tmem_ld_wait();
                uint8_t* dst = out_stage(m) + (size_t)d_loc * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 pk;
                    pk.x = pack_bf16x2(__uint_as_float(r[8 * c + 0]), __uint_as_float(r[8 * c + 1]));
                    pk.y = pack_bf16x2(__uint_as_float(r[8 * c + 2]), __uint_as_float(r[8 * c + 3]));
                    pk.z = pack_bf16x2(__uint_as_float(r[8 * c + 4]), __uint_as_float(r[8 * c + 5]));
                    pk.w = pack_bf16x2(__uint_as_float(r[8 * c + 6]), __uint_as_float(r[8 * c + 7]));
                    *reinterpret_cast<uint4*>(dst + ((((uint32_t)(4 * set + c)) ^ swz) << 4)) = pk;
                }
            }
            fence_proxy_async_smem();   // generic writes, read by the bulk copy
            named_bar_sync(kBarMath, 256);
            if (mt == 0 && !dead) {
                const int slot = rank < m ? rank : rank - 1;
                bulk_copy_to_peer(dsmem_addr(q_s, (uint32_t)m) + (uint32_t)slot * kPartBytes, out_stage(m),
                                  kPartBytes, dsmem_addr(&tl->recv_bar, (uint32_t)m));
            }
        }
        if (mt == 0) STI_DSTAMP(25);
        // the weights, while the own block's PV runs
        mwait_c(&tl->ml_bar);
        if (st < 32) {   // the four CTAs' weights for head hoff + st (whose max and sum this thread wrote)
            const int hh = hoff + st;
            float mc[kCtas], lc[kCtas];
            float M = -INFINITY;
#pragma unroll
            for (int k = 0; k < kCtas; ++k) {
                const float2 ml = k < kCtas - 1 ? tl->xml[k][hh] : make_float2(tl->m_run[hh], tl->l_run[hh]);
                mc[k] = dead ? -INFINITY : ml.x;
                lc[k] = dead ? 0.f : ml.y;
                M = fmaxf(M, mc[k]);
            }
            float L = 0.f;
            float e[kCtas];
#pragma unroll
            for (int k = 0; k < kCtas; ++k) {
                e[k] = (M == -INFINITY || mc[k] == -INFINITY) ? 0.f : fast_exp2(mc[k] - M);
                L += lc[k] * e[k];
            }
            if (M != -INFINITY) L += fast_exp2(__ldg(p.sink + hh) * kLog2e - M);
#pragma unroll
            for (int k = 0; k < kCtas; ++k) tl->wgt[k][hh] = M == -INFINITY ? 0.f : e[k] / L;
        }
        named_bar_sync(kBarMath, 256);   // the weights
        if (mt == 0) STI_DSTAMP(26);
        mwait(&tl->pv_bar[rank], 0);   // this CTA's own block
        if (mt == 0) STI_DSTAMP(49);
        tc_fence_after();
        if (mt == 0) STI_DSTAMP(13);
        float v[32];
        {
            const float* w_own = tl->wgt[kCtas - 1] + hoff;
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + kTmemO + (uint32_t)(rank * kH + hoff), r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * w_own[i];
        }
        mwait_c(&tl->recv_bar);
        if (mt == 0) STI_DSTAMP(51);
#pragma unroll 1
        for (int k = 0; k < kCtas - 1; ++k) {   // the three others' shares of this CTA's d-block, weighted
            const uint8_t* part = q_s + (size_t)k * kPartBytes + (size_t)d_loc * 128;
            const float* wk = tl->wgt[k] + hoff;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 x = dead ? make_uint4(0, 0, 0, 0)
                                     : *reinterpret_cast<const uint4*>(part + (((uint32_t)(4 * set + c) ^ swz) << 4));
                const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[i]));
                    v[8 * c + 2 * i] += f.x * wk[8 * c + 2 * i];
                    v[8 * c + 2 * i + 1] += f.y * wk[8 * c + 2 * i + 1];
                }
            }
        }
        const int dd = kRows * rank + d_loc;
        if (p.rope_dims > 0 && kRows * rank + kRows > kD - p.rope_dims)   // the output's inverse rotation
            rope_inverse_pairs<32>(v, dd, kD, p.rope_dims, p.rope_cs + (size_t)b * p.rope_dims);
        {   // the block's [64 heads][128 d] bf16: each warp turns its 32 d x 32 heads around in 2 KB of the
            // free quarter of the Q buffer and stores 16-byte pieces (a head's 32 d: 64 contiguous bytes)
            uint16_t* stg = reinterpret_cast<uint16_t*>(q_s + 3 * kPartBytes) + mw * 32 * 32;
            const bool odd = (lane & 1) != 0;
#pragma unroll
            for (int i = 0; i < 32; i += 2) {   // lane pairs: the even lane head i, the odd lane head i + 1
                const float send = odd ? v[i] : v[i + 1];
                const float recv = __shfl_xor_sync(kFull, send, 1);
                const uint32_t pr = odd ? pack_bf16x2(recv, v[i + 1]) : pack_bf16x2(v[i], recv);
                *reinterpret_cast<uint32_t*>(stg + (i + (odd ? 1 : 0)) * 32 + (lane & ~1)) = pr;
            }
            __syncwarp();
            uint16_t* obase = p.out + (size_t)b * kH * kD + kRows * rank + 32 * qd;
#pragma unroll
            for (int k = 0; k < 4; ++k) {   // piece c: head hoff + c / 4, d 8 (c % 4) .. + 8 of this warp's 32
                const int c = lane + 32 * k;
                const uint4 val = *reinterpret_cast<const uint4*>(stg + c * 8);
                *reinterpret_cast<uint4*>(obase + (size_t)(hoff + (c >> 2)) * kD + 8 * (c & 3)) = val;
            }
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
                                    const CUtensorMap& tm_comp_rows, const DecodeAttnParams& p, bool pdl,
                                    cudaStream_t stream) {
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
    err = cudaLaunchKernelEx(&cfg, decode_topk_attn_kernel, tm_q, tm_ring, tm_ring_rows, tm_comp_rows, p);
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace sti

#ifdef STI_DA_TIMING
// profiling builds only: global-timer stamps of the fused decode kernel's CTAs
extern "C" int sti_dbg_da_times(unsigned long long* host, int n_blocks) {
    return (int)cudaMemcpyFromSymbol(host, sti::g_da_t, sizeof(unsigned long long) * 64 * (size_t)n_blocks);
}
#endif
