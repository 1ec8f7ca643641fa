// idx_scores.cu -- Indexer scores on the tcgen05 tensor cores.
//
// DeepSeek V4.1, attention "attend/selected" page, Indexer.forward (score block):
//   index_score[b,t,j] = sum_h relu(q[b,t,h,:] . k[b,j,:]) * weights[b,t,h]*c,  -inf where j >= vis(b,t)
//
// Shape of the GEMM: keys go in the MMA M dimension (128 keys per tile) and (queries x index
// heads) in N, K = index_head_dim.  One TMEM lane then holds every head of one key for the
// unit's queries, so the head-weighted ReLU reduction is an in-thread FMA chain in the
// epilogue, with no cross-lane traffic.  Keys stream from HBM by TMA (128-byte swizzle) through
// a multi-stage shared-memory ring; the index queries of a unit (<= 256 rows) stay resident.
//
// Persistent kernel, one CTA per SM, warp-specialised:
//   warp 0      TMA producer (index-key tiles, and the unit's query tile)
//   warp 1      TMEM allocator + single-thread MMA issuer
//   warps 2..5  epilogue: TMEM -> registers -> sum_h w*relu(acc) -> fp32 scores (coalesced)
// Work = the flattened list of (unit, key tile) pairs over all units (unit = one sequence and
// nq consecutive queries), cut into equal contiguous ranges, one per CTA.  Key tiles past the
// last visible position of a unit are not computed; the epilogue writes -inf there.
#include <cuda.h>
#include <cuda_bf16.h>

#include "sti_internal.h"
#include "sti_ptx.cuh"

namespace sti {
namespace {

constexpr int kTileKeys = 128;
constexpr int kThreads = 192;      // bf16 keys: producer, MMA, 4 epilogue warps
constexpr int kThreadsFp4 = 320;   // MXFP4 keys: + 4 warps that dequantise keys and quantise queries
constexpr int kMaxStages = 8;
constexpr uint32_t kFull = 0xFFFFFFFFu;

struct __align__(8) Barriers {
    uint64_t full_a[kMaxStages];
    uint64_t empty_a[kMaxStages];
    uint64_t full_c[kMaxStages];    // MXFP4: packed key tile (codes + scales) landed
    uint64_t empty_c[kMaxStages];   // MXFP4: packed key tile dequantised (stage free)
    uint64_t b_ready;               // MXFP4: the unit's queries quantised in place
    uint64_t full_b, empty_b;
    uint64_t acc_full[2], acc_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t abort;
};

__device__ __forceinline__ int unit_tiles(const IdxScoresParams& p, int u) {
    const int b = u / p.QT, qt = u - b * p.QT;
    const int t_last = min(p.s, (qt + 1) * p.nq) - 1;
    int vis = (__ldg(p.start_pos + b) + t_last + 1) / p.ratio;
    vis = max(0, min(vis, p.n_cols));
    return (vis + kTileKeys - 1) / kTileKeys;
}

// Warp-cooperative: total number of compute tiles over all units.
__device__ int total_tiles(const IdxScoresParams& p) {
    const int lane = threadIdx.x & 31;
    int sum = 0;
    for (int u0 = 0; u0 < p.total_units; u0 += 32) {
        const int u = u0 + lane;
        sum += (u < p.total_units) ? unit_tiles(p, u) : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
    return sum;
}

// Warp-cooperative: (unit, tile) of flattened tile index g (unit == total_units past the end).
__device__ void locate(const IdxScoresParams& p, int g, int& u_out, int& tile_out) {
    const int lane = threadIdx.x & 31;
    int base = 0;
    for (int u0 = 0; u0 < p.total_units; u0 += 32) {
        const int u = u0 + lane;
        const int n = (u < p.total_units) ? unit_tiles(p, u) : 0;
        int inc = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += v;
        }
        const int chunk_total = __shfl_sync(kFull, inc, 31);
        if (g < base + chunk_total) {
            const unsigned m = __ballot_sync(kFull, base + inc > g);
            const int l = __ffs(m) - 1;
            const int excl = __shfl_sync(kFull, inc - n, l);
            u_out = u0 + l;
            tile_out = g - base - excl;
            return;
        }
        base += chunk_total;
    }
    u_out = p.total_units;
    tile_out = 0;
}

__device__ __forceinline__ void advance(const IdxScoresParams& p, int& u, int& tile) {
    ++tile;
    while (u < p.total_units && tile >= unit_tiles(p, u)) {
        ++u;
        tile = 0;
    }
}

// K-major operand descriptor of K-step kk (16 bf16) for a tile of `rows` rows stored as column
// blocks of rows x 128 bytes (128-byte swizzle, Di >= 64) or one block of 64-byte rows (Di == 32).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk, int Di, int rows) {
    if (Di >= 64) {
        const uint32_t addr = base + (uint32_t)(kk >> 2) * (uint32_t)rows * 128u + (uint32_t)(kk & 3) * 32u;
        return sdesc(addr, 16, 1024, kLayoutSW128);
    }
    const uint32_t addr = base + (uint32_t)kk * 32u;
    return sdesc(addr, 16, 512, kLayoutSW64);
}

#ifdef STI_STEP_TIMING
__device__ unsigned long long g_sc_t[2048][2];   // global timer at CTA start and end (profiling builds)
#endif

// E2M1 nibble (bit 3 sign, bits 2-1 exponent with bias 1, bit 0 mantissa; exponent 0 is
// subnormal: m * 0.5) as a float.
__device__ __forceinline__ float e2m1_value(uint32_t nib) {
    const uint32_t e = (nib >> 1) & 3u, m = nib & 1u;
    uint32_t bits = e ? ((126u + e) << 23) | (m << 22) : (m ? 0x3F000000u : 0u);
    return __uint_as_float(bits | ((nib & 8u) << 28));
}

// E8M0 scale byte -> 2^(e - 127) (255 is NaN).
__device__ __forceinline__ float e8m0_value(uint32_t e) {
    return e == 0u ? __uint_as_float(0x00400000u) : (e == 255u ? __uint_as_float(0x7FC00000u) : __uint_as_float(e << 23));
}

// |x| / 2^X onto the E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}: nearest, ties to the even code,
// saturating at 6.
__device__ __forceinline__ float e2m1_round(float a) {
    return a <= 0.25f ? 0.f : a < 0.75f ? 0.5f : a <= 1.25f ? 1.f : a < 1.75f ? 1.5f
         : a <= 2.5f ? 2.f : a < 3.5f ? 3.f : a <= 5.f ? 4.f : 6.f;
}

// One 32-element block of bf16 queries (four 16-byte chunks at c0..c3), quantised to MXFP4 and
// decoded back in place (Indexer.forward's fp4_act_quant on q, read as OCP MXFP4: scale 2^X with
// X = floor(log2 max|x|) - 2).  The decoded values are exact in bf16.
__device__ __forceinline__ void mxfp4_fake_quant_block(uint4* c0, uint4* c1, uint4* c2, uint4* c3) {
    uint4 v[4] = {*c0, *c1, *c2, *c3};
    uint32_t* w = reinterpret_cast<uint32_t*>(v);
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
    }
    const int X = amax > 0.f ? max(-127, min(127, ilogbf(amax) - 2)) : -127;
    const float sc = ldexpf(1.f, X), inv = ldexpf(1.f, -X);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
        const float ql = copysignf(e2m1_round(fabsf(lo) * inv), lo) * sc;
        const float qh = copysignf(e2m1_round(fabsf(hi) * inv), hi) * sc;
        w[i] = (__float_as_uint(ql) >> 16) | (__float_as_uint(qh) & 0xFFFF0000u);
    }
    *c0 = v[0];
    *c1 = v[1];
    *c2 = v[2];
    *c3 = v[3];
}

template <int HI, bool FP4>
__global__ void __launch_bounds__(FP4 ? kThreadsFp4 : kThreads, FP4 ? 2 : 1)
    idx_scores_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_s, const IdxScoresParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned start, offset from the __shared__ array itself so every derived pointer
    // stays a known shared-memory pointer (ld/st.shared, not generic accesses)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
#ifdef STI_STEP_TIMING
    if (threadIdx.x == 0 && blockIdx.x < 2048) g_sc_t[blockIdx.x][0] = global_timer_ns();
#endif
    griddep_launch_dependents();   // the top-k may be scheduled now; it waits for this grid's end
    const int a_bytes = kTileKeys * p.Di * 2;
    const int b_bytes = p.n_pad * p.Di * 2;
    uint8_t* a_ring = smem;
    uint8_t* b_buf = smem + (size_t)p.stages * a_bytes;
    // MXFP4: packed key tiles, [128 keys x Di/2 code bytes | 128 keys x Di/32 scale bytes] per stage
    const int c_code_bytes = kTileKeys * p.Di / 2;
    const int c_bytes = FP4 ? c_code_bytes + kTileKeys * p.Di / 32 : 0;
    uint8_t* c_ring = b_buf + b_bytes;
    Barriers* bars = reinterpret_cast<Barriers*>(c_ring + (size_t)(FP4 ? p.c_stages : 0) * c_bytes);
    float* w_s = reinterpret_cast<float*>(bars + 1);   // [nq * HI], pre-multiplied by c
    int* vis_s = reinterpret_cast<int*>(w_s + 256);     // [nq]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&bars->full_a[i], FP4 ? 4 : 1);   // MXFP4: the four dequantising warps
            mbar_init(&bars->empty_a[i], 1);
        }
        if (FP4) {
            for (int i = 0; i < p.c_stages; ++i) {
                mbar_init(&bars->full_c[i], 1);
                mbar_init(&bars->empty_c[i], 4);
            }
            mbar_init(&bars->b_ready, 1);
        }
        mbar_init(&bars->full_b, 1);
        mbar_init(&bars->empty_b, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->acc_full[i], 1);
            mbar_init(&bars->acc_empty[i], 4);
        }
        mbar_init(&bars->mma_done, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, (uint32_t)p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    // this CTA's contiguous range of the flattened (unit, tile) list
    const int T = total_tiles(p);
    const int g0 = (int)(((int64_t)T * blockIdx.x) / gridDim.x);
    const int g1 = (int)(((int64_t)T * (blockIdx.x + 1)) / gridDim.x);
    int u, tile;
    locate(p, g0, u, tile);
    const int ncb = p.Di >= 64 ? p.Di / 64 : 1;  // column blocks per row
    const int box_inner = p.Di >= 64 ? 64 : p.Di;

    auto aborted = [&]() { return *(volatile uint32_t*)&bars->abort != 0u; };

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        // Every iteration runs even after an abort (with the waits skipped), so all roles stay
        // in step; at the end the producer waits for the last load of each stage so no TMA
        // write is in flight when the CTA exits.
        if (lane == 0) {
            tma_prefetch_desc(&tm_a);
            tma_prefetch_desc(&tm_b);
            if (FP4) tma_prefetch_desc(&tm_s);
        }
        const int n_st = FP4 ? p.c_stages : p.stages;   // the ring this producer fills
        int stage = 0;
        uint32_t phase = 0, b_phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;  // per stage: armed at least once, parity of last arm
        bool b_issued = false;
        int cur_unit = -1;
        for (int g = g0; g < g1; ++g) {
            const int b = u / p.QT, qt = u - (u / p.QT) * p.QT;
            if (lane == 0 && !aborted()) {
                bool ok = true;
                if (u != cur_unit) {
                    ok = mbar_wait(&bars->empty_b, b_phase ^ 1u, p.status);
                    if (ok) {
                        mbar_arrive_expect_tx(&bars->full_b, (uint32_t)b_bytes);
                        for (int cb = 0; cb < ncb; ++cb)
                            tma_load_3d(b_buf + (size_t)cb * p.n_pad * box_inner * 2, &tm_b, &bars->full_b,
                                        cb * box_inner, qt * p.nq * HI, b);
                        b_issued = true;
                    }
                }
                if (FP4) {
                    // packed keys: 128 rows of Di/2 code bytes, then their Di/32 scale bytes per
                    // key viewed as rows of 16 bytes (Di/4 rows per tile)
                    ok = ok && mbar_wait(&bars->empty_c[stage], phase ^ 1u, p.status);
                    if (ok) {
                        uint8_t* dst = c_ring + (size_t)stage * c_bytes;
                        mbar_arrive_expect_tx(&bars->full_c[stage], (uint32_t)c_bytes);
                        tma_load_3d(dst, &tm_a, &bars->full_c[stage], 0, tile * kTileKeys, b);
                        tma_load_3d(dst + c_code_bytes, &tm_s, &bars->full_c[stage], 0, tile * (p.Di / 4), b);
                    }
                } else {
                    ok = ok && mbar_wait(&bars->empty_a[stage], phase ^ 1u, p.status);
                    if (ok) {
                        uint8_t* dst = a_ring + (size_t)stage * a_bytes;
                        mbar_arrive_expect_tx(&bars->full_a[stage], (uint32_t)a_bytes);
                        for (int cb = 0; cb < ncb; ++cb)
                            tma_load_3d(dst + (size_t)cb * kTileKeys * box_inner * 2, &tm_a, &bars->full_a[stage],
                                        cb * box_inner, tile * kTileKeys, b);
                    }
                }
                if (ok) {
                    issued_mask |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                } else {
                    atomicExch(&bars->abort, 1u);
                }
            }
            if (u != cur_unit) b_phase ^= 1u;
            cur_unit = u;
            if (++stage == n_st) {
                stage = 0;
                phase ^= 1u;
            }
            advance(p, u, tile);
        }
        if (lane == 0) {
            for (int st = 0; st < n_st; ++st)
                if (issued_mask & (1u << st))
                    mbar_wait(FP4 ? &bars->full_c[st] : &bars->full_a[st], (issued_parity >> st) & 1u, p.status);
            if (b_issued) mbar_wait(&bars->full_b, b_phase ^ 1u, p.status);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        const uint32_t idesc = idesc_bf16_f32(128, p.n_pad, false, false);
        const int ksteps = p.Di / 16;
        int stage = 0, acc = 0;
        uint32_t phase = 0, acc_phase = 0, b_phase = 0;
        int cur_unit = -1;
        for (int g = g0; g < g1; ++g) {
            if (lane == 0 && !aborted()) {
                bool ok = true;
                if (u != cur_unit) {
                    if (cur_unit >= 0) umma_commit(&bars->empty_b);
                    ok = mbar_wait(FP4 ? &bars->b_ready : &bars->full_b, b_phase, p.status);
                }
                ok = ok && mbar_wait(&bars->acc_empty[acc], acc_phase ^ 1u, p.status);
                ok = ok && mbar_wait(&bars->full_a[stage], phase, p.status);
                if (ok) {
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(a_ring + (size_t)stage * a_bytes);
                    const uint32_t b_base = smem_u32(b_buf);
                    const uint32_t d_tmem = tmem + (uint32_t)(acc * p.n_alloc);
                    for (int kk = 0; kk < ksteps; ++kk)
                        umma_bf16(d_tmem, kmajor_desc(a_base, kk, p.Di, kTileKeys),
                                  kmajor_desc(b_base, kk, p.Di, p.n_pad), idesc, kk > 0 ? 1u : 0u);
                    umma_commit(&bars->empty_a[stage]);
                    umma_commit(&bars->acc_full[acc]);
                } else {
                    atomicExch(&bars->abort, 1u);
                }
            }
            if (u != cur_unit) b_phase ^= 1u;
            cur_unit = u;
            if (++stage == p.stages) {
                stage = 0;
                phase ^= 1u;
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
            advance(p, u, tile);
        }
        if (lane == 0) {  // every MMA this thread issued has finished before TMEM is freed
            umma_commit(&bars->mma_done);
            mbar_wait(&bars->mma_done, 0, p.status);
        }
    } else if (FP4 && warp >= 6) {
        // ---------------------------------------------------------------- MXFP4 keys and queries
        // Thread dq owns key row dq of every tile: its Di/2 code bytes and Di/32 scale bytes become
        // Di bf16 values (exact: an E2M1 value times a power of two) in the 128-byte-swizzled tile
        // the MMA reads.  At each new unit the four warps first quantise the unit's queries in
        // place (32-element blocks of every query row), as the forward pass quantises q.
        const int dq = threadIdx.x - 192;               // 0..127
        const int nblk = p.Di / 32;
        int astage = 0, cstage = 0;
        uint32_t aphase = 0, cphase = 0, b_phase = 0;
        int cur_unit = -1;
        for (int g = g0; g < g1; ++g) {
            bool ok = !aborted();
            if (u != cur_unit) {
                ok = ok && mbar_wait(&bars->full_b, b_phase, p.status);
                if (ok) {
                    for (int i = dq; i < p.n_pad * nblk; i += 128) {
                        const int r = i / nblk, j = i - (i / nblk) * nblk;
                        uint8_t* rowp = b_buf + (size_t)(j >> 1) * p.n_pad * 128 + (size_t)r * 128;
                        const int c0 = (j & 1) * 4;
                        mxfp4_fake_quant_block(reinterpret_cast<uint4*>(rowp + (((c0 + 0) ^ (r & 7)) << 4)),
                                               reinterpret_cast<uint4*>(rowp + (((c0 + 1) ^ (r & 7)) << 4)),
                                               reinterpret_cast<uint4*>(rowp + (((c0 + 2) ^ (r & 7)) << 4)),
                                               reinterpret_cast<uint4*>(rowp + (((c0 + 3) ^ (r & 7)) << 4)));
                    }
                }
                fence_proxy_async_smem();   // generic stores, read by the tensor core
                named_bar_sync(2, 128);
                if (dq == 0 && ok) mbar_arrive(&bars->b_ready);
                b_phase ^= 1u;
                cur_unit = u;
            }
            ok = ok && mbar_wait(&bars->empty_a[astage], aphase ^ 1u, p.status);
            ok = ok && mbar_wait(&bars->full_c[cstage], cphase, p.status);
            if (ok) {
                const uint8_t* cst = c_ring + (size_t)cstage * c_bytes;
                const uint8_t* crow = cst + (size_t)dq * (p.Di / 2);
                const uint8_t* srow = cst + c_code_bytes + (size_t)dq * nblk;
                uint8_t* arow = a_ring + (size_t)astage * a_bytes + (size_t)dq * 128;
                for (int q4 = 0; q4 < p.Di / 32; ++q4) {
                    // 16 code bytes = 32 elements = one scale block; rows start 64 bytes apart, so
                    // lanes take the blocks in rotated order to spread the shared-memory banks
                    const int qb = (q4 + dq) % (p.Di / 32);
                    const uint4 cw4 = *reinterpret_cast<const uint4*>(crow + qb * 16);
                    const float sc = e8m0_value(srow[qb]);
                    const uint32_t cw[4] = {cw4.x, cw4.y, cw4.z, cw4.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {   // 8 elements -> one 16-byte chunk of the tile
                        uint32_t pk[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t byte = (cw[h] >> (8 * j)) & 0xFFu;
                            const float lo = e2m1_value(byte & 0xFu) * sc, hi = e2m1_value(byte >> 4) * sc;
                            pk[j] = (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);
                        }
                        const int ch = qb * 4 + h;                 // chunk of 8 elements along Di
                        *reinterpret_cast<uint4*>(arow + (size_t)(ch >> 3) * kTileKeys * 128 +
                                                  (size_t)(((ch & 7) ^ (dq & 7)) << 4)) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
            } else {
                atomicExch(&bars->abort, 1u);
            }
            fence_proxy_async_smem();   // generic stores, read by the tensor core
            __syncwarp();
            if (lane == 0 && ok) {
                mbar_arrive(&bars->full_a[astage]);
                mbar_arrive(&bars->empty_c[cstage]);
            }
            if (++astage == p.stages) {
                astage = 0;
                aphase ^= 1u;
            }
            if (++cstage == p.c_stages) {
                cstage = 0;
                cphase ^= 1u;
            }
            advance(p, u, tile);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int ep_tid = threadIdx.x - 64;           // 0..127
        const int quarter = warp & 3;                  // TMEM lane quarter this warp may access
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        constexpr int QPC = HI >= 32 ? 1 : 32 / HI;    // queries per 32-column load
        constexpr int CPQ = HI >= 32 ? HI / 32 : 1;    // 32-column loads per query
        int acc = 0;
        uint32_t acc_phase = 0;
        int cur_unit = -1;
        for (int g = g0; g < g1; ++g) {
            const int b = u / p.QT, qt = u - (u / p.QT) * p.QT;
            const int t0 = qt * p.nq;
            const int nq_here = min(p.nq, p.s - t0);
            if (u != cur_unit) {
                named_bar_sync(1, 128);
                for (int i = ep_tid; i < nq_here * HI; i += 128) {
                    const uint16_t wb = p.w[((size_t)b * p.s + t0) * HI + i];
                    w_s[i] = __uint_as_float((uint32_t)wb << 16) * p.c;
                }
                for (int i = ep_tid; i < nq_here; i += 128)
                    vis_s[i] = max(0, min(p.n_cols, (__ldg(p.start_pos + b) + t0 + i + 1) / p.ratio));
                named_bar_sync(1, 128);
                cur_unit = u;
            }
            bool ok = !aborted() && mbar_wait(&bars->acc_full[acc], acc_phase, p.status);
            ok = __all_sync(kFull, ok);   // warp-uniform: the loop below holds warp collectives
            if (!ok) atomicExch(&bars->abort, 1u);
            tc_fence_after();
            const int key = tile * kTileKeys + quarter * 32 + lane;
            const uint32_t col_base = tmem + lane_base + (uint32_t)(acc * p.n_alloc);
            if (ok) {
                for (int q0 = 0; q0 < nq_here; q0 += QPC) {
                    float sacc[QPC];
#pragma unroll
                    for (int i = 0; i < QPC; ++i) sacc[i] = 0.f;
#pragma unroll
                    for (int cq = 0; cq < CPQ; ++cq) {
                        uint32_t r[32];
                        tmem_ld32(col_base + (uint32_t)(q0 * HI + cq * 32), r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int qq = HI >= 32 ? 0 : i / HI;
                            const int hh = HI >= 32 ? cq * 32 + i : i % HI;
                            const float v = fmaxf(__uint_as_float(r[i]), 0.f);
                            sacc[qq] = fmaf(w_s[(q0 + qq) * HI + hh], v, sacc[qq]);
                        }
                    }
#pragma unroll
                    for (int qq = 0; qq < QPC; ++qq) {
                        const int q = q0 + qq;
                        const bool in_row = q < nq_here && key < p.n_cols;
                        const bool visible = in_row && key < vis_s[q];
                        if (in_row) p.scores[((size_t)b * p.s + t0 + q) * p.n_cols + key] = visible ? sacc[qq] : -INFINITY;
                        if (p.hist != nullptr) {
                            // first radix pass of the top-k: top 11 bits of the order-preserving key,
                            // one aggregated shared-L2 atomic per distinct bin in the warp
                            const uint32_t dig = visible ? (float_key(sacc[qq]) >> 21) : 0xFFFFFFFFu;
                            const unsigned peers = __match_any_sync(kFull, dig);
                            if (visible && lane == __ffs(peers) - 1)
                                atomicAdd(p.hist + ((size_t)b * p.s + t0 + q) * 2048 + dig, (uint32_t)__popc(peers));
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->acc_empty[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
            advance(p, u, tile);
        }
        // -inf for key tiles no query of a unit can see (units strided over CTAs)
        for (int uu = blockIdx.x; uu < p.total_units; uu += gridDim.x) {
            const int b = uu / p.QT, qt = uu - (uu / p.QT) * p.QT;
            const int t0 = qt * p.nq;
            const int nq_here = min(p.nq, p.s - t0);
            const int first = unit_tiles(p, uu) * kTileKeys;
            for (int q = 0; q < nq_here; ++q) {
                float* row = p.scores + ((size_t)b * p.s + t0 + q) * p.n_cols;
                for (int j = first + ep_tid; j < p.n_cols; j += 128) row[j] = -INFINITY;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
    }
#ifdef STI_STEP_TIMING
    if (threadIdx.x == 0 && blockIdx.x < 2048) g_sc_t[blockIdx.x][1] = global_timer_ns();
#endif
}

}  // namespace

int idx_scores_pick_nq(int Hi, int s) {
    // N = nq * Hi <= 256 (one MMA), never more queries than the sequence has
    int nq = 256 / Hi;
    if (nq > s) nq = s;
    if (nq < 1) nq = 1;
    return nq;
}

size_t idx_scores_smem_bytes(const IdxScoresParams& p) {
    const size_t a_bytes = (size_t)kTileKeys * p.Di * 2;
    const size_t b_bytes = (size_t)p.n_pad * p.Di * 2;
    const size_t c_bytes = p.fp4 ? (size_t)kTileKeys * p.Di / 2 + (size_t)kTileKeys * p.Di / 32 : 0;
    return 1024 + p.stages * a_bytes + b_bytes + (p.fp4 ? p.c_stages : 0) * c_bytes + sizeof(Barriers) + 256 * 4 +
           256 * 4;
}

cudaError_t launch_idx_scores(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_s,
                              const IdxScoresParams& p, int num_sms, cudaStream_t stream) {
    size_t smem = idx_scores_smem_bytes(p);
    // p.ctas_per_sm CTAs share an SM (together they fit the SM's 512 TMEM columns); pad shared
    // memory so no more than that many become resident
    const size_t floor_smem = (size_t)(228 * 1024 / (p.ctas_per_sm + 1)) + 1024;
    if (smem < floor_smem) smem = floor_smem;
    const int grid = num_sms * p.ctas_per_sm;
    cudaError_t err = cudaSuccess;
#define STI_LAUNCH_HI(HV)                                                                              \
    case HV: {                                                                                         \
        auto kern = p.fp4 ? idx_scores_kernel<HV, true> : idx_scores_kernel<HV, false>;               \
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);      \
        if (err != cudaSuccess) return err;                                                            \
        kern<<<grid, p.fp4 ? kThreadsFp4 : kThreads, smem, stream>>>(tm_a, tm_b, tm_s, p);            \
        return cudaGetLastError();                                                                     \
    }
    switch (p.Hi) {
        STI_LAUNCH_HI(4)
        STI_LAUNCH_HI(8)
        STI_LAUNCH_HI(16)
        STI_LAUNCH_HI(32)
        STI_LAUNCH_HI(64)
        default:
            return cudaErrorInvalidValue;
    }
#undef STI_LAUNCH_HI
}

}  // namespace sti

#ifdef STI_STEP_TIMING
// profiling builds only: global-timer stamps (ns) of the scores kernel's CTAs
extern "C" int sti_dbg_scores_times(unsigned long long* host, int n_blocks) {
    return (int)cudaMemcpyFromSymbol(host, sti::g_sc_t, sizeof(unsigned long long) * 2 * (size_t)n_blocks);
}
#endif
