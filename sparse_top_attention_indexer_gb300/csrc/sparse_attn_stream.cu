// sparse_attn_stream.cu -- the sparse sink attention for many queries (prefill): persistent CTAs
// that walk a strided list of queries, with each KV tile streamed through shared memory one
// column block at a time.
//
// DeepSeek V4.1, attention "attend/selected" page, sparse_attn_kernel / sparse_attn:
//   for every query and head, over the slots i whose index is not -1:
//     s_i = softmax_scale * q . kv[idx_i];  o = sum_i e^{s_i} kv[idx_i] / (sum_i e^{s_i} + e^{sink_h})
//   one latent row serving as key and value; a query with no valid slot gets 0.
//
// Shape: up to 64 heads x 512 dims, rows from one or two bf16 sources, or (FP4) the second source
// as fp4 rows (E2M1 codes, an E4M3 scale per 16).  One CTA per SM, 320 threads:
//   * warp 0 loads each query's Q (eight TMA boxes of h heads x 64 dims) as soon as the previous
//     query's last QK has read the buffer;
//   * warp 1 issues the MMAs;
//   * warps 2..9 gather the tiles, run the online softmax and write the outputs.
// A query's index slots form tiles of 128 rows; tiles with no valid slot are skipped.  A tile is
// refilled one pair of column blocks (one d-block, 128 dims) at a time, as soon as the previous
// tile's PV of that d-block has released it: bf16 rows 0..63 by four-row TMA gathers (four lanes
// of every math warp), rows 64..127 by 16-byte LSU copies of every math thread, so the TMA unit
// and the LSU work side by side; fp4 rows are loaded into registers as soon as their index is
// known and decoded into the tile once their block is free.  The QK consumes column block j as
// soon as it has landed, so a tile's gather overlaps the previous tile's PV and its own QK.  The
// index slots of the next tile are loaded while the current tile's rows land.
//   * S^T = KV . Q^T: M = 128 rows, N = 64 heads, K = 512, the K steps alternating between two
//     TMEM accumulators so that consecutive MMAs do not wait on each other (the softmax adds
//     the two).
//   * Softmax, thread = row, heads in two groups of 32 (warps 2-5, 6-9): per-head maxima by a
//     warp reduce-scatter and a named barrier, taken only on a query's first tile and when some
//     score passes its head's running max by more than 8 (log2 units), which is also the only time
//     the max moves and O^T is rescaled; otherwise a single barrier (a vote) decides.  Each thread
//     keeps its row's running sums, reduced at the query's end.  P^T is bf16.
//   * O^T += V^T . P^T: M = 128 d-rows per block, N = 64, K = 128 rows, the same tile read as an
//     MN-major operand; one commit per d-block releases its two column blocks to the gather.
//   * A query's epilogue (O^T from TMEM, normalised, optionally rotated back, turned around as
//     bf16 in the free P^T buffer and stored in 16-byte pieces) runs after the next query's first
//     gather has been issued, while its rows are in flight.
#include <cuda_bf16.h>
#include <math.h>
#include <stddef.h>

#include "sti_attn_util.cuh"
#include "sti_internal.h"
#include "sti_kvfp4.h"
#include "sti_ptx.cuh"

namespace sti {
namespace {

constexpr int kSThreads = 320;
constexpr int kSRows = 128;                    // rows per tile (MMA M)
constexpr int kSH = 64;                        // heads, zero-padded (MMA N)
constexpr int kSD = 512;                       // latent dims
constexpr int kSCb = kSD / 64;                 // column blocks of 64 dims (128 bytes)
constexpr uint32_t kQBlkB = kSH * 128;         // one Q column block: 8 KB
constexpr uint32_t kTBlkB = kSRows * 128;      // one tile column block: 16 KB
constexpr uint32_t kTmS0 = 0, kTmS1 = 64;      // TMEM columns of the two S^T partials
constexpr uint32_t kTmO = 128;                 // O^T d-block m at columns [128 + 64 m, 192 + 64 m)
// bf16 rows: a tile column block is filled by 16 four-row TMA gathers (rows 0..63) and by 128
// threads' LSU copies (rows 64..127, 64 bytes each), so the TMA unit and the LSU run side by
// side; fp4 compressed rows: by 128 threads, one row each, decoded from registers
constexpr uint32_t kFullArrivals = 16 + 128;
constexpr uint32_t kFullArrivalsFp4 = 128;
constexpr uint32_t kBarMath = 3;               // named barrier of the 256 math threads (1, 2: head groups)
constexpr float kLog2eS = 1.4426950408889634f;
constexpr float kLn2S = 0.69314718055994531f;

struct __align__(16) StreamTail {
    // float arrays first: the running maxima are read as float4 (16-byte aligned)
    float mcp[2][4][32];      // [head group][warp]: each warp's copy of the group's running maxima
    float red[2][2][4][32];   // [tile parity][head group][warp quarter][head]: per-warp maxima
    float lsum[2][4][32];     // [head group][warp quarter][head]: per-warp sums at a query's end
    float sink_log2[kSH];     // the heads' sinks times log2(e)
    uint64_t full[kSCb];   // column block j of the tile landed (see kFullArrivals; + the TMA bytes)
    uint64_t pv[4];        // the tile's PV of d-block m done (column blocks 2m, 2m+1 free)
    uint64_t s_full;       // the tile's QK done
    uint64_t p_full;       // the tile's P^T written: one arrival per math warp
    uint64_t q_full;       // the query's Q landed
    uint64_t q_free;       // the query's last QK done: the Q buffer may be reloaded
    uint32_t tmem_base;
    int abort;             // a bounded wait gave up: every role winds down
};
static_assert(offsetof(StreamTail, mcp) % 16 == 0, "float4 reads of the running maxima");

size_t stream_smem_bytes() {
    return 1024 + (size_t)kSCb * kQBlkB + (size_t)kSCb * kTBlkB + kSRows * 128 + sizeof(StreamTail);
}

// Bit t set: slots [128 t, 128 t + 128) of the index row hold at least one valid index.  Every
// lane of the warp calls it and gets the same mask; an index outside [-1, n_rows) counts as
// masked and is flagged in *status (when non-null).  Up to 768 slots take one round of loads.
__device__ __forceinline__ uint32_t live_tiles(const int32_t* idx_row, int k, int n_rows, int lane,
                                               uint32_t* status) {
    uint32_t m = 0;
    bool bad = false;
    for (int base = 0; base < k; base += 32 * 24) {
        int v[24];
#pragma unroll
        for (int i = 0; i < 24; ++i) {
            const int s = base + 32 * i + lane;
            v[i] = s < k ? __ldg(idx_row + s) : -1;
        }
#pragma unroll
        for (int i = 0; i < 24; ++i) {
            const int s = base + 32 * i + lane;
            if (v[i] >= 0 && v[i] < n_rows) m |= 1u << (s >> 7);
            bad = bad || v[i] < -1 || v[i] >= n_rows;
        }
    }
    if (bad && status) atomicOr(status, 1u /* STI_FLAG_INDEX_RANGE */);
    return __reduce_or_sync(kWarpFull, m);
}

#ifdef STI_ATTN_TIMING
// profiling builds only: global-timer stamps of the first 16 tiles of every CTA
__device__ unsigned long long g_stream_t[160][16][24];
#define STI_STAMP(n, e)                                                                  \
    do {                                                                                 \
        if (blockIdx.x < 160 && (n) < 16) g_stream_t[blockIdx.x][(n)][(e)] = global_timer_ns(); \
    } while (0)
#else
#define STI_STAMP(n, e) \
    do {                \
    } while (0)
#endif

// FP4: the second source holds fp4 rows (f); every row of a tile is then copied by one thread:
// bf16 rows by LSU copies, fp4 rows loaded into registers before their block is free and decoded.
template <bool FP4>
__global__ void __launch_bounds__(kSThreads, 1)
    sparse_attn_stream_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv1,
                              const __grid_constant__ CUtensorMap tm_kv2, const AttnParams p, const KvFp4 f) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned start (the swizzle atoms), offset from the __shared__ array itself
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* q_s = smem;                            // Q: 8 column blocks of [64 heads][128 B], SW128
    uint8_t* t_s = q_s + kSCb * kQBlkB;             // tile: 8 column blocks of [128 rows][128 B], SW128
    uint8_t* p_s = t_s + kSCb * kTBlkB;             // P^T: [128 rows][64 heads] bf16, SW128
    StreamTail* tl = reinterpret_cast<StreamTail*>(p_s + kSRows * 128);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nq = p.B * p.s;
    const int n_rows = p.n1 + p.n2;
    const int stride = (int)gridDim.x;
    volatile int* abort = &tl->abort;

    if (warp == 0) {
        tmem_alloc(&tl->tmem_base, 512);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int j = 0; j < kSCb; ++j) mbar_init(&tl->full[j], FP4 ? kFullArrivalsFp4 : kFullArrivals);
        for (int m = 0; m < 4; ++m) mbar_init(&tl->pv[m], 1);
        mbar_init(&tl->s_full, 1);
        mbar_init(&tl->p_full, 8);
        mbar_init(&tl->q_full, 1);
        mbar_init(&tl->q_free, 1);
        tl->abort = 0;
        fence_mbar_init();
    }
    if (tid < kSH) tl->sink_log2[tid] = tid < p.h ? __ldg(p.sink + tid) * kLog2eS : 0.f;
    // Q rows of heads >= h are never loaded: zero them once (the MMA reads all 64)
    if (p.h < kSH)
        for (int i = tid; i < kSCb * kSH * 8; i += kSThreads)
            if (((i >> 3) & (kSH - 1)) >= p.h) reinterpret_cast<uint4*>(q_s)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tl->tmem_base;
    griddep_wait();   // the index rows are complete from here on (Q, KV and the sink come from the caller)

    if (warp == 0) {
        // ------------------------------------------------------------------ Q loads
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            if (!FP4) {
                tma_prefetch_desc(&tm_kv1);
                tma_prefetch_desc(&tm_kv2);
            }
        }
        uint32_t qn = 0;
        for (int qi = blockIdx.x; qi < nq; qi += stride) {
            const uint32_t live = live_tiles(p.idx + (size_t)qi * p.idx_stride, p.k, n_rows, lane, nullptr);
            if (!live) continue;
            bool ok = true;
            if (lane == 0) {
                ok = qn == 0 || attn_wait(&tl->q_free, (qn - 1) & 1u, p.status, abort);
                if (ok) {
                    mbar_arrive_expect_tx(&tl->q_full, (uint32_t)(kSCb * p.h * 128));
                    for (int cb = 0; cb < kSCb; ++cb)
                        tma_load_2d(q_s + cb * kQBlkB, &tm_q, &tl->q_full, cb * 64, qi * p.h);
                }
            }
            if (!__shfl_sync(kWarpFull, ok, 0)) break;
            ++qn;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issue
        const uint32_t idesc_qk = idesc_bf16_f32(128, kSH, false, false);
        const uint32_t idesc_pv = idesc_bf16_f32(128, kSH, true, true);
        const uint32_t q0 = smem_u32(q_s), t0 = smem_u32(t_s), p0 = smem_u32(p_s);
        uint32_t n = 0, qn = 0;
        for (int qi = blockIdx.x; qi < nq; qi += stride) {
            const uint32_t live = live_tiles(p.idx + (size_t)qi * p.idx_stride, p.k, n_rows, lane, nullptr);
            if (!live) continue;
            bool ok = true;
            if (lane == 0) {
                ok = attn_wait(&tl->q_full, qn & 1u, p.status, abort);
                const int T = __popc(live);
                for (int t = 0; t < T && ok; ++t, ++n) {
                    // S^T = tile . Q^T, column block by column block as they land
                    for (int j = 0; j < kSCb && ok; ++j) {
                        ok = attn_wait(&tl->full[j], n & 1u, p.status, abort);
                        if (!ok) break;
                        fence_proxy_async_smem();   // rows the LSU wrote, read by the MMA (async proxy)
                        tc_fence_after();
                        if (j == 0) STI_STAMP(n, 4);
#pragma unroll
                        for (int kq = 0; kq < 4; ++kq) {
                            const int kk = 4 * j + kq;
                            umma_bf16(tmem + ((kk & 1) ? kTmS1 : kTmS0),
                                      sdesc(t0 + (uint32_t)j * kTBlkB + (uint32_t)kq * 32u, 16, 1024, kLayoutSW128),
                                      sdesc(q0 + (uint32_t)j * kQBlkB + (uint32_t)kq * 32u, 16, 1024, kLayoutSW128),
                                      idesc_qk, kk >= 2 ? 1u : 0u);
                        }
                    }
                    if (!ok) break;
                    STI_STAMP(n, 5);
                    umma_commit(&tl->s_full);
                    if (t == T - 1) umma_commit(&tl->q_free);
                    // O^T += V^T . P^T, one commit per d-block
                    ok = attn_wait(&tl->p_full, n & 1u, p.status, abort);
                    if (!ok) break;
                    tc_fence_after();
                    STI_STAMP(n, 6);
                    for (int m = 0; m < 4; ++m) {
#pragma unroll
                        for (int kk = 0; kk < kSRows / 16; ++kk)
                            umma_bf16(tmem + kTmO + 64u * (uint32_t)m,
                                      sdesc(t0 + (uint32_t)(2 * m) * kTBlkB + (uint32_t)kk * 2048u, kTBlkB, 1024,
                                            kLayoutSW128),
                                      sdesc(p0 + (uint32_t)kk * 2048u, kSRows * 128u, 1024, kLayoutSW128), idesc_pv,
                                      (t > 0 || kk > 0) ? 1u : 0u);
                        umma_commit(&tl->pv[m]);
                    }
                }
                ++qn;
            }
            if (!__shfl_sync(kWarpFull, ok, 0)) break;
        }
    } else {
        // ------------------------------------------------------------------ math warps
        const int mw = warp - 2;                  // 0..7
        const int set = mw >> 2;                  // head group: heads [32 set, 32 set + 32)
        const int qd = warp & 3;                  // TMEM lane quarter
        const int row = 32 * qd + lane;           // tile row (TMEM lane) of this thread's softmax
        // gather of a tile, one pair of column blocks (one d-block) at a time as the previous tile's
        // PV releases them: rows 0..63 by four-row TMA gathers (lanes 0..3 of every warp: row group
        // tg, block 2m + tb), rows 64..127 by 16-byte LSU copies (every math thread: row lr, block
        // 2m + lb, four of the row's eight 16-byte chunks)
        const int tg = 2 * mw + (lane & 1);
        const int tb = (lane >> 1) & 1;
        const bool tma_lane = lane < 4;
        const int mt = tid - 64;
        const int lr = 64 + ((mt >> 1) & 63);
        const int lb = mt >> 7;
        const int lc0 = 4 * (mt & 1);
        // fp4 compressed rows (FP4): this thread copies row fr of column block 2m + fh of every pair
        const int fr = mt & 127;
        const int fh = mt >> 7;
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        const uint32_t bar_set = 1u + (uint32_t)set;
        uint32_t n = 0;                           // tiles this CTA has processed
        bool dead = false;                        // warp-uniform
        float m_run = -INFINITY;                  // lane l: the running max of head 32 set + l
        float l_thr[32];                          // this row's running sums of the group's 32 heads

        auto mwait = [&](uint64_t* bar, uint32_t parity) {
            if (!dead) dead = !attn_wait(bar, parity, p.status, abort);
            dead = __any_sync(kWarpFull, dead);
        };
        // the index slots a tile needs from this thread: its TMA row group's four (lanes 0..3), its
        // LSU row's and its softmax row's
        struct TileIdx {
            int g[4];
            int l;
            int r;
        };
        auto load_idx = [&](int q, int t, TileIdx& ti) {
            const int32_t* idx_row = p.idx + (size_t)q * p.idx_stride;
            const int s0 = kSRows * t;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int sl = s0 + 4 * tg + i;
                ti.g[i] = (!FP4 && tma_lane && sl < p.k) ? __ldg(idx_row + sl) : -1;
            }
            const int gr = FP4 ? fr : lr;
            ti.l = s0 + gr < p.k ? __ldg(idx_row + s0 + gr) : -1;
            ti.r = s0 + row < p.k ? __ldg(idx_row + s0 + row) : -1;
        };
        // a slot's row: source (-1 masked) and coordinate in the [B * rows, d] view of its source
        auto resolve = [&](int v, int b, int& sid, int& crd) {
            if (v < -1 || v >= n_rows) v = -1;
            sid = v < 0 ? -1 : (v < p.n1 ? 0 : 1);
            crd = sid < 0 ? 0 : sid == 0 ? (int)((int64_t)b * p.rows1 + v) : (int)((int64_t)b * p.rows2 + (v - p.n1));
        };

        auto gather_fp4 = [&](const TileIdx& ti, int b) {
            int sid, crd;
            resolve(ti.l, b, sid, crd);   // fp4 rows: crd is the row within its batch element
            uint4 cw[4][2];
            uint32_t sw[4];
            if (sid == 1) {   // the packed bytes do not wait for the block: load them now
                const uint8_t* cr = f.codes + (size_t)b * f.codes_bstride + (size_t)crd * (kSD / 2);
                const uint8_t* sr = f.scales + (size_t)b * f.scales_bstride + (size_t)crd * (kSD / 16);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int j = 2 * m + fh;
                    cw[m][0] = __ldg(reinterpret_cast<const uint4*>(cr + j * 32));
                    cw[m][1] = __ldg(reinterpret_cast<const uint4*>(cr + j * 32 + 16));
                    sw[m] = __ldg(reinterpret_cast<const uint32_t*>(sr + j * 4));
                }
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                if (n > 0) mwait(&tl->pv[m], (n - 1) & 1u);   // column blocks 2m, 2m+1 are free
                if (mw == 0 && lane == 0 && n > 0) STI_STAMP(n - 1, 7 + m);
                if (dead) continue;
                const int j = 2 * m + fh;
                uint8_t* dst = t_s + (size_t)j * kTBlkB + (size_t)fr * 128;
                if (sid == 0) {   // a bf16 row of the first source
                    const uint16_t* src = p.kv + (size_t)crd * kSD + j * 64;
                    const uint32_t d0 = smem_u32(dst);
#pragma unroll
                    for (int c = 0; c < 8; ++c) cp_async_16(d0 + (uint32_t)((c ^ (fr & 7)) << 4), src + c * 8, 16u);
                    cp_async_mbar_arrive_noinc(&tl->full[j]);
                    continue;
                }
                if (sid == 1) {   // 64 elements: eight words of eight codes, an E4M3 scale per two words
                    const uint32_t w[8] = {cw[m][0].x, cw[m][0].y, cw[m][0].z, cw[m][0].w,
                                           cw[m][1].x, cw[m][1].y, cw[m][1].z, cw[m][1].w};
                    const float2 s01 = e4m3x2_to_float2(sw[m] & 0xFFFFu), s23 = e4m3x2_to_float2(sw[m] >> 16);
                    const __nv_bfloat162 sc[4] = {__float2bfloat162_rn(s01.x), __float2bfloat162_rn(s01.y),
                                                  __float2bfloat162_rn(s23.x), __float2bfloat162_rn(s23.y)};
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(dst + ((c ^ (fr & 7)) << 4)) = kvfp4_decode8_s2(w[c], sc[c >> 1]);
                } else {          // masked: zeros (finite, and P = 0 for them)
#pragma unroll
                    for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(dst + (c << 4)) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                mbar_arrive(&tl->full[j]);
            }
        };

        auto gather = [&](const TileIdx& ti, int b) {
            int sid[4], crd[4];
            int S = -1, fc = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                resolve(ti.g[i], b, sid[i], crd[i]);
                if (sid[i] >= 0 && S < 0) {
                    S = sid[i];
                    fc = crd[i];
                }
            }
            bool mixed = false;
#pragma unroll
            for (int i = 0; i < 4; ++i) mixed = mixed || (sid[i] >= 0 && sid[i] != S);
            if (!mixed)   // masked rows repeat the group's first valid row (their score is -inf)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (sid[i] != S) crd[i] = fc;
            int lsid, lcrd;
            resolve(ti.l, b, lsid, lcrd);
            const uint16_t* lsrc = lsid < 0 ? p.kv2 != nullptr ? p.kv2 : p.kv
                                            : (lsid == 0 ? p.kv : p.kv2) + (size_t)lcrd * kSD;
            const uint32_t lbytes = lsid < 0 ? 0u : 16u;   // masked rows: zeros
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
                if (n > 0) mwait(&tl->pv[m], (n - 1) & 1u);   // column blocks 2m, 2m+1 are free
                if (mw == 0 && lane == 0 && n > 0) STI_STAMP(n - 1, 7 + m);
                if (dead) continue;
                {   // LSU rows
                    const int j = 2 * m + lb;
                    const uint32_t dst = smem_u32(t_s + (size_t)j * kTBlkB + (size_t)lr * 128);
                    const uint16_t* src = lsid < 0 ? lsrc : lsrc + j * 64;
#pragma unroll
                    for (int c = lc0; c < lc0 + 4; ++c)
                        cp_async_16(dst + (uint32_t)((c ^ (lr & 7)) << 4), lsid < 0 ? src : src + c * 8, lbytes);
                    cp_async_mbar_arrive_noinc(&tl->full[j]);
                }
                if (!tma_lane) continue;
                const int j = 2 * m + tb;
                uint8_t* dst = t_s + (size_t)j * kTBlkB + (size_t)tg * 512;
                if (S < 0) {
                    // no valid row in the group: zeros (finite, and P = 0 for them)
                    uint4* z = reinterpret_cast<uint4*>(dst);
#pragma unroll
                    for (int c = 0; c < 32; ++c) z[c] = make_uint4(0, 0, 0, 0);
                    fence_proxy_async_smem();
                    mbar_arrive(&tl->full[j]);
                } else if (!mixed) {
                    mbar_arrive_expect_tx(&tl->full[j], 512u);
                    tma_gather4(dst, S == 0 ? (const void*)&tm_kv1 : (const void*)&tm_kv2, &tl->full[j], j * 64,
                                crd[0], crd[1], crd[2], crd[3]);
                } else {
                    // rows of both sources in one group: 16-byte copies through the LSU, swizzled
                    const uint32_t d0 = smem_u32(dst);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int si = sid[i] < 0 ? S : sid[i];
                        const int ci = sid[i] < 0 ? fc : crd[i];
                        const uint16_t* src = (si == 0 ? p.kv : p.kv2) + (size_t)ci * kSD + j * 64;
                        const int r = 4 * tg + i;
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            cp_async_16(d0 + (uint32_t)(i * 128) + (uint32_t)((c ^ (r & 7)) << 4), src + c * 8, 16u);
                    }
                    cp_async_commit();
                    cp_async_wait<0>();
                    fence_proxy_async_smem();
                    mbar_arrive(&tl->full[j]);
                }
            }
        };

        // online softmax of the CTA's tile n; `vi` is this row's index slot.  The running maxima
        // stay unless some score of the tile passes its head's maximum by more than 8 (log2 units):
        // then (and on a query's first tile) the tile's per-head maxima are reduced over the group
        // and the sums and O^T rescaled; otherwise one barrier decides and P uses the maxima held.
        auto softmax = [&](int vi, bool first) {
            if (mw == 0 && lane == 0) STI_STAMP(n, 11);
            mwait(&tl->s_full, n & 1u);
            tc_fence_after();
            if (mw == 0 && lane == 0) STI_STAMP(n, 2);
            const bool valid = vi >= 0 && vi < n_rows && !dead;
            float x[32];
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem + lane_base + kTmS0 + 32u * (uint32_t)set, r0);
                tmem_ld32(tmem + lane_base + kTmS1 + 32u * (uint32_t)set, r1);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    x[i] = valid ? (__uint_as_float(r0[i]) + __uint_as_float(r1[i])) * p.scale_log2 : -INFINITY;
            }
            const float* mc = &tl->mcp[set][qd][0];   // this warp's copy of the group's running maxima
            bool need = first;
            if (!first) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 m4 = *reinterpret_cast<const float4*>(mc + 4 * c);
                    need = need || x[4 * c] > m4.x + 8.f || x[4 * c + 1] > m4.y + 8.f || x[4 * c + 2] > m4.z + 8.f ||
                           x[4 * c + 3] > m4.w + 8.f;
                }
            }
            need = !named_bar_and(bar_set, 128, !need);   // any row of the group
            if (need) {
                {
                    float v2[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v2[i] = x[i];
                    warp_reduce_scatter_n<32, true>(v2);   // lane l: the max of head 32 set + l over this warp's rows
                    tl->red[n & 1u][set][qd][lane] = v2[0];
                }
                named_bar_sync(bar_set, 128);
                const float* rr = &tl->red[n & 1u][set][0][0];
                const float mt = fmaxf(fmaxf(rr[lane], rr[32 + lane]), fmaxf(rr[64 + lane], rr[96 + lane]));
                const float m_new = (m_run == -INFINITY || mt > m_run + 8.f) ? fmaxf(m_run, mt) : m_run;
                const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
                m_run = m_new;
                tl->mcp[set][qd][lane] = m_new;
                __syncwarp();
                if (!first && !dead && __any_sync(kWarpFull, alpha != 1.f)) {
                    // O^T rows of this lane (d = 32 qd + lane of every block) and this row's sums times
                    // the heads' factors; the previous tile's PV has completed (it precedes this QK)
#pragma unroll 1
                    for (int m = 0; m < 4; ++m) {
                        const uint32_t ta = tmem + lane_base + kTmO + 64u * (uint32_t)m + 32u * (uint32_t)set;
                        uint32_t r[32];
                        tmem_ld32(ta, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r[i] = __float_as_uint(__uint_as_float(r[i]) * __shfl_sync(kWarpFull, alpha, i));
                        tmem_st32(ta, r);
                    }
                    tmem_st_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) l_thr[i] *= __shfl_sync(kWarpFull, alpha, i);
                }
            }
            // probabilities as bf16 P^T (row = this thread's tile row, heads of this group); this row's sums
            uint8_t* prow = p_s + row * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float4 ma = *reinterpret_cast<const float4*>(mc + 8 * c);
                const float4 mb = *reinterpret_cast<const float4*>(mc + 8 * c + 4);
                const float mm[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float e = (mm[j] == -INFINITY) ? 0.f : fast_exp2(x[8 * c + j] - mm[j]);
                    x[8 * c + j] = e;
                    l_thr[8 * c + j] += e;
                }
                uint4 pk;
                pk.x = pack_bf16x2(x[8 * c + 0], x[8 * c + 1]);
                pk.y = pack_bf16x2(x[8 * c + 2], x[8 * c + 3]);
                pk.z = pack_bf16x2(x[8 * c + 4], x[8 * c + 5]);
                pk.w = pack_bf16x2(x[8 * c + 6], x[8 * c + 7]);
                *reinterpret_cast<uint4*>(prow + (((4 * set + c) ^ (row & 7)) << 4)) = pk;
            }
            fence_proxy_async_smem();              // P^T: generic writes the MMA reads
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&tl->p_full);
                if (mw == 0) STI_STAMP(n, 3);
            }
        };

        // o = O / (l + 2^(sink log2e - m)) for query qe, whose last tile was this CTA's tile last_n.
        // A d-block at a time, each warp turns its 32 d x 32 heads around in its own 2 KB of the P^T
        // buffer (free from the last PV until this tile's softmax) and stores 16-byte pieces: a head's
        // 32 d of this warp are 64 contiguous bytes of the output.
        auto epilogue = [&](int qe, uint32_t last_n) {
            mwait(&tl->pv[3], last_n & 1u);   // the query's last PV has completed
            tc_fence_after();
            if (mw == 0 && lane == 0) STI_STAMP(n, 15);
            {
                float v2[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v2[i] = l_thr[i];
                warp_reduce_scatter_n<32, false>(v2);   // lane l: head 32 set + l over this warp's rows
                tl->lsum[set][qd][lane] = v2[0];
            }
            if (mw == 0 && lane == 0) STI_STAMP(n, 16);
            named_bar_sync(bar_set, 128);
            if (mw == 0 && lane == 0) STI_STAMP(n, 17);
            const float* ls = &tl->lsum[set][0][0];
            const float lt = (ls[lane] + ls[32 + lane]) + (ls[64 + lane] + ls[96 + lane]);
            const int hh = 32 * set + lane;
            float inv = 0.f, lse = -INFINITY;
            if (m_run != -INFINITY && hh < p.h) {
                const float den = lt + exp2f(tl->sink_log2[hh] - m_run);
                inv = 1.f / den;
                lse = (m_run + log2f(den)) * kLn2S;
            }
            if (p.lse && qd == 0 && hh < p.h) p.lse[(size_t)qe * p.h + hh] = lse;
            float invh[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) invh[i] = __shfl_sync(kWarpFull, inv, i);
            uint16_t* orow = p.out + (size_t)qe * p.h * kSD;
            uint16_t* stg = reinterpret_cast<uint16_t*>(p_s) + mw * 32 * 32;   // this warp's [32 heads][32 d]
            const bool odd = (lane & 1) != 0;
            if (mw == 0 && lane == 0) STI_STAMP(n, 18);
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
                const int dd = 128 * m + 32 * qd + lane;
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + kTmO + 64u * (uint32_t)m + 32u * (uint32_t)set, r);
                tmem_ld_wait();
                float vv[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) vv[i] = dead ? 0.f : __uint_as_float(r[i]) * invh[i];
                if (p.rope_dims > 0 && 128 * m + 128 > kSD - p.rope_dims)   // the output's inverse rotation
                    rope_inverse_pairs<32>(vv, dd, kSD, p.rope_dims, p.rope_cs + (size_t)qe * p.rope_dims);
                // lane pairs (dd even, dd + 1) write 4 bytes: the even lane head i, the odd lane head i + 1
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float send = odd ? vv[i] : vv[i + 1];
                    const float recv = __shfl_xor_sync(kWarpFull, send, 1);
                    const uint32_t pr = odd ? pack_bf16x2(recv, vv[i + 1]) : pack_bf16x2(vv[i], recv);
                    *reinterpret_cast<uint32_t*>(stg + (i + (odd ? 1 : 0)) * 32 + (lane & ~1)) = pr;
                }
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 4; ++k) {   // piece c: head c / 4, d 8 (c % 4) .. + 8 of this warp's 32
                    const int c = lane + 32 * k;
                    const int hw = 32 * set + (c >> 2);
                    const uint4 v = *reinterpret_cast<const uint4*>(stg + c * 8);
                    if (hw < p.h)
                        *reinterpret_cast<uint4*>(orow + (size_t)hw * kSD + 128 * m + 32 * qd + 8 * (c & 3)) = v;
                }
                __syncwarp();
                if (mw == 0 && lane == 0) STI_STAMP(n, 19 + m);
            }
            // the warps' pieces of the P^T buffer span its rows: no warp writes P^T before every warp
            // has read its last piece back
            named_bar_sync(kBarMath, 256);
        };

        // the next query of this CTA's list (from q + stride on) with a valid slot; queries without
        // one get their zero output (and lse -inf) on the way
        auto next_live = [&](int q, uint32_t& mask) {
            for (q += stride; q < nq; q += stride) {
                mask = live_tiles(p.idx + (size_t)q * p.idx_stride, p.k, n_rows, lane, mw == 0 ? p.status : nullptr);
                if (mask) return q;
                uint16_t* orow = p.out + (size_t)q * p.h * kSD;
                for (int hh = mw; hh < p.h; hh += 8) {
                    uint4* o = reinterpret_cast<uint4*>(orow + (size_t)hh * kSD);
                    o[lane] = make_uint4(0, 0, 0, 0);
                    o[lane + 32] = make_uint4(0, 0, 0, 0);
                }
                if (p.lse && mw == 0)
                    for (int hh = lane; hh < p.h; hh += 32) p.lse[(size_t)q * p.h + hh] = -INFINITY;
            }
            mask = 0u;
            return nq;
        };

        uint32_t live = 0u;
        int qi = next_live((int)blockIdx.x - stride, live);
        TileIdx cur;
        if (qi < nq) load_idx(qi, __ffs(live) - 1, cur);
        int prev = -1;   // the query whose epilogue is pending
        while (qi < nq) {
            const int b = qi / p.s;
            uint32_t rem = live;
            bool first = true;
            int qn = nq;
            uint32_t live_n = 0u;
            while (rem) {
                rem &= rem - 1u;
                if (mw == 0 && lane == 0) STI_STAMP(n, 0);
                if constexpr (FP4) gather_fp4(cur, b);
                else gather(cur, b);
                if (mw == 0 && lane == 0) STI_STAMP(n, 1);
                // the next tile's index slots load while this tile's rows land
                if (!rem) qn = next_live(qi, live_n);
                if (mw == 0 && lane == 0) STI_STAMP(n, 12);
                TileIdx nxt;
                nxt.g[0] = nxt.g[1] = nxt.g[2] = nxt.g[3] = nxt.l = nxt.r = -1;
                if (rem) load_idx(qi, __ffs(rem) - 1, nxt);
                else if (qn < nq) load_idx(qn, __ffs(live_n) - 1, nxt);
                if (mw == 0 && lane == 0) STI_STAMP(n, 13);
                if (first) {
                    if (prev >= 0) epilogue(prev, n - 1);
                    if (mw == 0 && lane == 0) STI_STAMP(n, 14);
                    prev = -1;
                    m_run = -INFINITY;
#pragma unroll
                    for (int i = 0; i < 32; ++i) l_thr[i] = 0.f;
                }
                softmax(cur.r, first);
                cur = nxt;
                first = false;
                ++n;
            }
            prev = qi;
            qi = qn;
            live = live_n;
        }
        if (prev >= 0) epilogue(prev, n - 1);
    }

    tc_fence_before();
    __syncthreads();
    if (*abort) {
        // a wait gave up: let copies and MMAs already issued land before the CTA's memory goes
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 50000ull) {
        }
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool sparse_attn_stream_fits(const AttnParams& p) {
    return p.use_tma && p.cluster == 1 && p.d == kSD && p.d_pad == kSD && p.h >= 1 && p.h <= kSH && p.k >= 1 &&
           p.k <= 32 * kSRows && p.rope_dims <= kSD;
}

bool sparse_attn_stream_fits_fp4(const AttnParams& p) {
    // the first source's rows are addressed as kv + (b * rows1 + idx) * d: whole rows per batch element
    return p.cluster == 1 && p.d == kSD && p.d_pad == kSD && p.h >= 1 && p.h <= kSH && p.k >= 1 &&
           p.k <= 32 * kSRows && p.rope_dims <= kSD && (p.n1 == 0 || p.kv_bstride == p.rows1 * kSD);
}

template <bool FP4>
static cudaError_t launch_stream(const CUtensorMap& tm_q, const CUtensorMap& tm_kv1, const CUtensorMap& tm_kv2,
                                 const AttnParams& p, const KvFp4& f, cudaStream_t stream) {
    const int nq = p.B * p.s;
    if (nq == 0) return cudaSuccess;
    const size_t smem = stream_smem_bytes();
    cudaError_t err =
        cudaFuncSetAttribute(sparse_attn_stream_kernel<FP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const int sms = device_num_sms();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nq < sms ? nq : sms));
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    int na = 0;
    if (p.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (unsigned)na;
    err = cudaLaunchKernelEx(&cfg, sparse_attn_stream_kernel<FP4>, tm_q, tm_kv1, tm_kv2, p, f);
    return err != cudaSuccess ? err : cudaGetLastError();
}

cudaError_t launch_sparse_attn_stream(const CUtensorMap& tm_q, const CUtensorMap& tm_kv1, const CUtensorMap& tm_kv2,
                                      const AttnParams& p, cudaStream_t stream) {
    if (!sparse_attn_stream_fits(p)) return cudaErrorInvalidValue;
    KvFp4 none{};
    return launch_stream<false>(tm_q, tm_kv1, tm_kv2, p, none, stream);
}

cudaError_t launch_sparse_attn_stream_fp4(const CUtensorMap& tm_q, const AttnParams& p, const KvFp4& f,
                                          cudaStream_t stream) {
    if (!sparse_attn_stream_fits_fp4(p) || !f.on) return cudaErrorInvalidValue;
    return launch_stream<true>(tm_q, tm_q, tm_q, p, f, stream);
}

}  // namespace sti

#ifdef STI_ATTN_TIMING
// profiling builds only: per-CTA global-timer stamps of the streamed attention's first tiles
extern "C" int sti_dbg_stream_times(unsigned long long* host, int n_blocks) {
    return (int)cudaMemcpyFromSymbol(host, sti::g_stream_t, sizeof(unsigned long long) * 16 * 24 * (size_t)n_blocks);
}
#endif
