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
// Persistent kernel, one or two CTAs per SM (two when both accumulators fit the SM's TMEM),
// warp-specialised:
//   warp 0      TMA producer (index-key tiles, and the unit's query tile)
//   warp 1      TMEM allocator + single-thread MMA issuer
//   warps 2..9  epilogue: TMEM -> registers -> sum_h w*relu(acc) -> fp32 scores (coalesced); two
//               warps per TMEM lane quarter, taking alternate query chunks of a unit (one query per
//               unit, as in decode, and MXFP4 decoded in shared memory: warps 2..5, one per quarter;
//               MXFP4 as E2M1 operands: two groups of four take the CTA's tiles in turn)
// With MXFP4 keys (Indexer.forward's fp4 keys and queries) and one query per unit (decode, Di ==
// 128), warp 0 loads each tile's codes by TMA straight into the layout kind::f8f6f4 reads as E2M1
// operands (16 codes in the first 8 bytes of each 16-byte chunk) plus its scale bytes; the epilogue
// warps quantise the unit's queries into the same layout, every 32-code scale block has its own
// accumulator and the epilogue applies both blocks' 2^X.  Otherwise warp 0 stages packed tiles
// (E2M1 codes + E8M0 scales) by bulk copy and warps 6..13 decode them in shared memory -- to E5M2
// for kind::f8f6f4 MMAs where every block's scale allows an exact E5M2 value, else to bf16 --
// after quantising each unit's queries in place.
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
constexpr int kThreads = 320;      // producer, MMA, 8 epilogue warps (two per TMEM lane quarter): bf16 keys with
                                   // several queries per unit, and MXFP4 keys as E2M1 operands
constexpr int kThreadsOneQ = 192;  // bf16 keys, one query per unit (decode): 4 epilogue warps
constexpr int kThreadsFp4 = 448;   // MXFP4 keys: + 8 warps that dequantise keys and quantise queries
constexpr int kDqWarps = 8;
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
    uint32_t fmt[kMaxStages];       // MXFP4: 1 when the stage holds E5M2 keys, 0 for bf16
    uint32_t tmem_base;
    uint32_t abort;
};

// Keys visible to the last (so to any) query of unit u.
__device__ __forceinline__ int unit_vis(const IdxScoresParams& p, int u) {
    const int b = u / p.QT, qt = u - b * p.QT;
    const int t_last = min(p.s, (qt + 1) * p.nq) - 1;
    const int vis = (__ldg(p.start_pos + b) + t_last + 1) / p.ratio;
    return max(0, min(vis, p.n_cols));
}

__device__ __forceinline__ int unit_tiles(const IdxScoresParams& p, int u) {
    return (unit_vis(p, u) + kTileKeys - 1) / kTileKeys;
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

// Warp-cooperative: this CTA's contiguous range [g0, g1) of the flattened tile list and the
// (unit, tile) of g0.  Up to 32 units (a decode batch) take one round of start_pos reads.
__device__ void cta_range(const IdxScoresParams& p, int& g0, int& g1, int& u_out, int& tile_out) {
    if (p.total_units <= 32) {
        const int lane = threadIdx.x & 31;
        const int n = lane < p.total_units ? unit_tiles(p, lane) : 0;
        int inc = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += v;
        }
        const int T = __shfl_sync(kFull, inc, 31);
        g0 = (int)(((int64_t)T * blockIdx.x) / gridDim.x);
        g1 = (int)(((int64_t)T * (blockIdx.x + 1)) / gridDim.x);
        const unsigned m = __ballot_sync(kFull, inc > g0);
        const int l = m ? __ffs(m) - 1 : 31;
        const int excl = __shfl_sync(kFull, inc - n, l);
        u_out = m ? l : p.total_units;
        tile_out = m ? g0 - excl : 0;
        return;
    }
    const int T = total_tiles(p);
    g0 = (int)(((int64_t)T * blockIdx.x) / gridDim.x);
    g1 = (int)(((int64_t)T * (blockIdx.x + 1)) / gridDim.x);
    locate(p, g0, u_out, tile_out);
}

__device__ __forceinline__ int unit_tiles_at(const IdxScoresParams& p, int u) {
    return u < p.total_units ? unit_tiles(p, u) : 0;
}

// Next (unit, tile) of the flattened list.  n caches the current unit's tile count and n_next the
// following unit's, read one unit ahead: a step touches global memory only when it enters a new
// unit, and then never waits for that read (a per-tile read of start_pos sat on the MMA issuer's
// critical path, about 0.4 us a tile).
__device__ __forceinline__ void advance(const IdxScoresParams& p, int& u, int& tile, int& n, int& n_next) {
    if (++tile < n) return;
    tile = 0;
    ++u;
    n = n_next;
    while (u < p.total_units && n == 0) {
        ++u;
        n = unit_tiles_at(p, u);
    }
    n_next = unit_tiles_at(p, u + 1);
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
#ifdef STI_SC_TILE_TIMING
__device__ unsigned long long g_sc_pro[2048][4];  // prologue: after the barrier, after the range, first copy issued
#endif
#ifdef STI_SC_TILE_TIMING
// profiling builds only: global-timer stamps of the first 16 tiles of every CTA (e: 0 packed tile
// landed, 1 tile decoded, 2 MMAs issued, 3 epilogue done, 4 copy issued; with E2M1 operands 0 is the
// MMA issuer seeing the tile landed and 1 the epilogue seeing the accumulators ready)
__device__ unsigned long long g_sc_tile[2048][16][5];
#define STI_SCSTAMP(li, e)                                                                              \
    do {                                                                                                \
        if (blockIdx.x < 2048 && (li) >= 0 && (li) < 16) g_sc_tile[blockIdx.x][(li)][(e)] = global_timer_ns(); \
    } while (0)
#else
#define STI_SCSTAMP(li, e) \
    do {                   \
    } while (0)
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

// 2^e for e in [-149, 127], exactly.
__device__ __forceinline__ float exp2i(int e) {
    return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(1u << (e + 149));
}

// a = |x| / 2^X onto the E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}: the index 0..7 of the
// nearest one, ties to the even code, saturating at 6.
__device__ __forceinline__ uint32_t e2m1_index(float a) {
    return (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) + (uint32_t)(a >= 1.75f) +
           (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) + (uint32_t)(a > 5.f);
}

// E5M2 bytes of the eight E2M1 magnitudes times 2^X as a byte-permute table (t0: 0, .5, 1, 1.5;
// t1: 2, 3, 4, 6).  For X in [-13, 13] every such product is a normal E5M2 number (exponent field
// 1..30), so X only adds 4X to each non-zero byte, without carries between bytes.
__device__ __forceinline__ void e5m2_table(int X, uint32_t& t0, uint32_t& t1) {
    t0 = 0x3E3C3800u + (uint32_t)X * 0x04040400u;
    t1 = 0x46444240u + (uint32_t)X * 0x04040404u;
}

// Eight E2M1 codes (nibble i of cw = element i) -> their E5M2 bytes (element i in byte i of the
// pair) through the table of e5m2_table.  The sign comes from a second permute that takes each
// whole nibble as its selector: a set sign bit replicates the top bit of 0x7F (0x00), a clear one
// copies 0x7F; adding 1 per byte gives 0x01 or 0x80, and its complement's top bit is the sign.
__device__ __forceinline__ uint2 e2m1x8_to_e5m2(uint32_t cw, uint32_t t0, uint32_t t1) {
    const uint32_t hi = cw >> 16;
    const uint32_t m0 = prmt(t0, t1, cw & 0x7777u), m1 = prmt(t0, t1, hi & 0x7777u);
    const uint32_t n0 = prmt(0x7F7F7F7Fu, 0x7F7F7F7Fu, cw) + 0x01010101u;
    const uint32_t n1 = prmt(0x7F7F7F7Fu, 0x7F7F7F7Fu, hi) + 0x01010101u;
    return make_uint2(m0 | (~n0 & 0x80808080u), m1 | (~n1 & 0x80808080u));
}

// The block scale exponent X = floor(log2 max|x|) - 2 of an MXFP4 block, clamped to E8M0's range
// (-127 for an all-zero block).  floor(log2 amax) is the exponent field of a normal amax; zero and
// subnormals are rare.
__device__ __forceinline__ int mxfp4_block_exp(float amax) {
    const int eb = (int)(__float_as_uint(amax) >> 23);
    return eb > 0 ? max(-127, min(127, eb - 129)) : (amax > 0.f ? max(-127, ilogbf(amax) - 2) : -127);
}

// One 16-byte chunk (8 bf16 queries) of a 32-element block whose four chunks sit in lanes 4k..4k+3
// of the warp: the block is quantised to MXFP4 and decoded back in place (Indexer.forward's
// fp4_act_quant on q, read as OCP MXFP4: scale 2^X with X = floor(log2 max|x|) - 2); the decoded
// values are exact in bf16.  e5 (if not null) receives the same eight values as E5M2 bytes.
// Returns whether they are exact in E5M2: X in [-13, 13], or an all-zero block.
__device__ __forceinline__ bool mxfp4_fake_quant_chunk(uint4* chunk, uint2* e5) {
    const uint4 v = *chunk;
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
    }
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
    const int X = mxfp4_block_exp(amax);
    const float sc = exp2i(X), inv = exp2i(-X);
    uint32_t t0, t1;
    e5m2_table(max(-13, min(13, X)), t0, t1);
    uint32_t e[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
        const uint32_t il = e2m1_index(fabsf(lo) * inv), ih = e2m1_index(fabsf(hi) * inv);
        const float ql = copysignf(e2m1_value(il), lo) * sc;
        const float qh = copysignf(e2m1_value(ih), hi) * sc;
        w[i] = (__float_as_uint(ql) >> 16) | (__float_as_uint(qh) & 0xFFFF0000u);
        const uint32_t bl = prmt(t0, t1, il) | ((__float_as_uint(lo) >> 24) & 0x80u);
        const uint32_t bh = prmt(t0, t1, ih) | ((__float_as_uint(hi) >> 24) & 0x80u);
        e[i >> 1] |= (bl | (bh << 8)) << (16 * (i & 1));
    }
    *chunk = make_uint4(w[0], w[1], w[2], w[3]);
    if (e5 != nullptr) *e5 = make_uint2(e[0], e[1]);
    return amax == 0.f || (X >= -13 && X <= 13);
}

// KM: 0 bf16 keys, 1 MXFP4 keys decoded in shared memory, 2 MXFP4 keys as E2M1 MMA operands.
// The same quantisation of a chunk, returned as its eight E2M1 codes (element i in nibble i: sign in
// bit 3, magnitude index in bits 0-2) with the block's X.
__device__ __forceinline__ uint32_t mxfp4_quant_e2m1(const uint4 v, int& X) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
    }
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
    X = mxfp4_block_exp(amax);
    const float inv = exp2i(-X);
    uint32_t nib = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = w[i] << 16, hi = w[i] & 0xFFFF0000u;
        const uint32_t cl = e2m1_index(fabsf(__uint_as_float(lo)) * inv) | ((lo >> 28) & 8u);
        const uint32_t ch = e2m1_index(fabsf(__uint_as_float(hi)) * inv) | ((hi >> 28) & 8u);
        nib |= (cl | (ch << 4)) << (8 * i);
    }
    return nib;
}

template <int HI, int KM>
__global__ void __launch_bounds__(KM == 1 ? kThreadsFp4 : kThreads, KM == 0 ? 1 : 2)
    idx_scores_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_s, const IdxScoresParams p) {
    constexpr bool FP4 = KM == 1;
    constexpr bool E2 = KM == 2;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned start, offset from the __shared__ array itself so every derived pointer
    // stays a known shared-memory pointer (ld/st.shared, not generic accesses)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
#ifdef STI_STEP_TIMING
    if (threadIdx.x == 0 && blockIdx.x < 2048) g_sc_t[blockIdx.x][0] = global_timer_ns();
#endif
    griddep_launch_dependents();   // the top-k may be scheduled now; it waits for this grid's end
    // E2M1 operands (Di == 128): a key tile is 128 rows of 128 bytes, each 16-byte chunk holding 16
    // codes in its first 8 bytes (the layout TMA's 16 x U4 / 16-byte-aligned load writes)
    const int a_bytes = E2 ? kTileKeys * 128 : kTileKeys * p.Di * 2;
    const int b_bytes = p.n_pad * p.Di * 2;
    uint8_t* a_ring = smem;
    uint8_t* b_buf = smem + (size_t)p.stages * a_bytes;
    // MXFP4: packed key tiles, [128 keys x Di/2 code bytes | 128 keys x Di/32 scale bytes] per stage;
    // E2M1 operands: only the scale bytes, one ring slot per key stage
    const int c_code_bytes = kTileKeys * p.Di / 2;
    const int c_bytes = FP4 ? c_code_bytes + kTileKeys * p.Di / 32 : (E2 ? kTileKeys * 4 : 0);
    // MXFP4 with Di == 128: the quantised queries again as E5M2, or (E2M1 operands) as E2M1 codes in
    // the key tile's layout; rows of 128 bytes, 128-byte swizzle
    uint8_t* b8 = b_buf + b_bytes;
    const int b8_bytes = ((FP4 && p.f8) || E2) ? p.n_pad * 128 : 0;
    uint8_t* c_ring = b8 + b8_bytes;
    Barriers* bars = reinterpret_cast<Barriers*>(c_ring + (size_t)(FP4 ? p.c_stages : (E2 ? p.stages : 0)) * c_bytes);
    float* w_s = reinterpret_cast<float*>(bars + 1);   // [nq * HI], pre-multiplied by c
    int* vis_s = reinterpret_cast<int*>(w_s + 256);     // [nq], nq <= 64
    float* sq_s = reinterpret_cast<float*>(vis_s + 64); // E2M1 operands: 2^X of query block j, head h at [32 j + h]
    uint32_t* hs = reinterpret_cast<uint32_t*>(sq_s + 128);   // E2M1 operands: the unit's first-pass histogram

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&bars->full_a[i], FP4 ? kDqWarps / 2 : 1);   // MXFP4: the decoding group's warps
            // E2M1 operands: the MMAs' commit and the four epilogue warps of the tile's group, which
            // read the stage's scales
            mbar_init(&bars->empty_a[i], E2 ? 5 : 1);
        }
        if (E2) mbar_init(&bars->b_ready, 1);
        if (FP4) {
            for (int i = 0; i < p.c_stages; ++i) {
                mbar_init(&bars->full_c[i], 1);
                mbar_init(&bars->empty_c[i], kDqWarps / 2);
            }
            mbar_init(&bars->b_ready, 1);
        }
        mbar_init(&bars->full_b, 1);
        mbar_init(&bars->empty_b, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->acc_full[i], 1);
            // one arrival per epilogue warp (E2M1 operands: per warp of the group that owns the buffer)
            mbar_init(&bars->acc_empty[i], (FP4 || E2) ? 4u : (blockDim.x - 64u) / 32u);
        }
        mbar_init(&bars->mma_done, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, (uint32_t)p.tmem_cols);
        tmem_relinquish();
    }
    if (FP4) {   // rows a partial last tile does not fill keep zeros (never scored, but finite)
        uint4* c4 = reinterpret_cast<uint4*>(c_ring);
        for (int i = threadIdx.x; i < p.c_stages * c_bytes / 16; i += kThreadsFp4) c4[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
#ifdef STI_SC_TILE_TIMING
    if (threadIdx.x == 0 && blockIdx.x < 2048) g_sc_pro[blockIdx.x][0] = global_timer_ns();
#endif

    // this CTA's contiguous range of the flattened (unit, tile) list
    int g0, g1, u, tile;
    cta_range(p, g0, g1, u, tile);
    int un = unit_tiles_at(p, u), un_next = unit_tiles_at(p, u + 1);
#ifdef STI_SC_TILE_TIMING
    if (threadIdx.x == 0 && blockIdx.x < 2048) g_sc_pro[blockIdx.x][1] = global_timer_ns();
#endif
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
                        // a tile's packed keys are contiguous: two bulk copies, the keys past n_cols
                        // left out (their rows keep finite earlier contents and are never scored)
                        uint8_t* dst = c_ring + (size_t)stage * c_bytes;
                        const int nk = min(kTileKeys, p.n_cols - tile * kTileKeys);
                        const uint32_t cb_bytes = (uint32_t)(nk * (p.Di / 2));
                        const uint32_t sb_bytes = (uint32_t)((nk * (p.Di / 32) + 15) & ~15);
                        mbar_arrive_expect_tx(&bars->full_c[stage], cb_bytes + sb_bytes);
                        bulk_load(dst, p.k_codes + (size_t)b * p.k_codes_bstride + (size_t)tile * kTileKeys * (p.Di / 2),
                                  cb_bytes, &bars->full_c[stage]);
                        bulk_load(dst + c_code_bytes,
                                  p.k_scales + (size_t)b * p.k_scales_bstride + (size_t)tile * kTileKeys * (p.Di / 32),
                                  sb_bytes, &bars->full_c[stage]);
                        STI_SCSTAMP(g - g0, 4);
                    }
                } else {
                    ok = ok && mbar_wait(&bars->empty_a[stage], phase ^ 1u, p.status);
                    if (ok && E2) {
                        // codes by one TMA box (128 codes x 128 keys: 8 KB of codes spread over 16 KB,
                        // the box's transfer count; keys past n_cols read as zero codes), scale bytes
                        // by a bulk copy of the tile's keys
                        uint8_t* dst = a_ring + (size_t)stage * a_bytes;
                        const int nk = min(kTileKeys, p.n_cols - tile * kTileKeys);
                        const uint32_t sb_bytes = (uint32_t)((nk * 4 + 15) & ~15);
                        mbar_arrive_expect_tx(&bars->full_a[stage], (uint32_t)a_bytes / 2 + sb_bytes);
                        tma_load_3d(dst, &tm_a, &bars->full_a[stage], 0, tile * kTileKeys, b);
                        bulk_load(c_ring + (size_t)stage * c_bytes,
                                  p.k_scales + (size_t)b * p.k_scales_bstride + (size_t)tile * kTileKeys * 4, sb_bytes,
                                  &bars->full_a[stage]);
                        STI_SCSTAMP(g - g0, 4);
                    } else if (ok) {
                        uint8_t* dst = a_ring + (size_t)stage * a_bytes;
                        mbar_arrive_expect_tx(&bars->full_a[stage], (uint32_t)a_bytes);
                        for (int cb = 0; cb < ncb; ++cb)
                            tma_load_3d(dst + (size_t)cb * kTileKeys * box_inner * 2, &tm_a, &bars->full_a[stage],
                                        cb * box_inner, tile * kTileKeys, b);
#ifdef STI_SC_TILE_TIMING
                        if (g == g0 && blockIdx.x < 2048) g_sc_pro[blockIdx.x][2] = global_timer_ns();
#endif
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
            advance(p, u, tile, un, un_next);
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
        const uint32_t idesc8 = idesc_e5m2_f32(128, p.n_pad);
        const uint32_t idesc4 = idesc_e2m1_f32(128, p.n_pad);
        const int ksteps = p.Di / 16;
        int stage = 0, acc = 0;
        uint32_t phase = 0, acc_phase = 0, b_phase = 0;
        int cur_unit = -1;
        for (int g = g0; g < g1; ++g) {
            if (lane == 0 && !aborted()) {
                bool ok = true;
                if (u != cur_unit) {
                    if (cur_unit >= 0) umma_commit(&bars->empty_b);
                    ok = mbar_wait((FP4 || E2) ? &bars->b_ready : &bars->full_b, b_phase, p.status);
                }
                ok = ok && mbar_wait(&bars->acc_empty[acc], acc_phase ^ 1u, p.status);
                ok = ok && mbar_wait(&bars->full_a[stage], phase, p.status);
                if (ok) {
                    if (E2) STI_SCSTAMP(g - g0, 0);
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(a_ring + (size_t)stage * a_bytes);
                    const uint32_t b_base = smem_u32(b_buf);
                    const uint32_t d_tmem = tmem + (uint32_t)(acc * (E2 ? 4 : 1) * p.n_alloc);
                    if (E2) {
                        // one K = 32 step per scale block, each into its own accumulator (the block's
                        // two E8M0 scales are applied in the epilogue)
                        const uint32_t b8_base = smem_u32(b8);
                        for (int kk = 0; kk < 4; ++kk)
                            umma_f8f6f4(d_tmem + (uint32_t)(kk * p.n_alloc), kmajor_desc(a_base, kk, 64, kTileKeys),
                                        kmajor_desc(b8_base, kk, 64, p.n_pad), idesc4, 0u);
                    } else if (FP4 && *(volatile uint32_t*)&bars->fmt[stage] != 0u) {
                        // E5M2 keys and queries: rows of 128 bytes, K = 32 per instruction, so the
                        // descriptors step like a 64-wide bf16 tile
                        const uint32_t b8_base = smem_u32(b8);
                        for (int kk = 0; kk < 4; ++kk)
                            umma_f8f6f4(d_tmem, kmajor_desc(a_base, kk, 64, kTileKeys),
                                        kmajor_desc(b8_base, kk, 64, p.n_pad), idesc8, kk > 0 ? 1u : 0u);
                    } else {
                        for (int kk = 0; kk < ksteps; ++kk)
                            umma_bf16(d_tmem, kmajor_desc(a_base, kk, p.Di, kTileKeys),
                                      kmajor_desc(b_base, kk, p.Di, p.n_pad), idesc, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(&bars->empty_a[stage]);
                    umma_commit(&bars->acc_full[acc]);
                    STI_SCSTAMP(g - g0, 2);
#ifdef STI_SC_TILE_TIMING
                    if (g == g0 && blockIdx.x < 2048) g_sc_pro[blockIdx.x][3] = global_timer_ns();
#endif
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
            advance(p, u, tile, un, un_next);
        }
        if (lane == 0) {  // every MMA this thread issued has finished before TMEM is freed
            umma_commit(&bars->mma_done);
            mbar_wait(&bars->mma_done, 0, p.status);
        }
    } else if (FP4 && warp >= 6) {
        // ---------------------------------------------------------------- MXFP4 keys and queries
        // At each new unit the eight warps first quantise the unit's queries in place (32-element
        // blocks of every query row, four lanes to a block), as the forward pass quantises q, and
        // with Di == 128 also write them as E5M2.  Then the warps form two groups of four that take
        // the CTA's tiles in turn, thread dq of a group owning key row dq of its tiles.  When the unit's queries and every scale block
        // of the tile's visible keys have X in [-13, 13], each E2M1 code times 2^X is an exact
        // E5M2 number: the row becomes 128 E5M2 bytes (kind::f8f6f4, half the bytes and MMAs of
        // bf16).  Otherwise the Di/2 code bytes and Di/32 scale bytes become Di bf16 values (also
        // exact).  Either way the tile lands 128-byte-swizzled where the MMA reads it, and the
        // stage's fmt word tells the MMA which it is.
        const int dq_t = threadIdx.x - 192;             // 0..255
        const int dq = dq_t & 127;                      // key row of a tile
        const int dg = dq_t >> 7;                       // decode group: the CTA's tiles alternate between the two
        const int nblk = p.Di / 32;
        int astage = 0, cstage = 0;
        uint32_t aphase = 0, cphase = 0, b_phase = 0;
        int cur_unit = -1, vis_unit = 0;
        bool q_f8 = false;
        for (int g = g0; g < g1; ++g) {
            bool ok = !aborted();
            if (u != cur_unit) {
                vis_unit = unit_vis(p, u);
                ok = ok && mbar_wait(&bars->full_b, b_phase, p.status);
                ok = __all_sync(kFull, ok);   // warp-uniform: the quantiser shuffles within the warp
                bool q_in = true;
                if (ok) {
                    // n_pad * nblk * 4 is a multiple of 32: a warp's lanes run the same trips
                    for (int i = dq_t; i < p.n_pad * nblk * 4; i += 32 * kDqWarps) {
                        const int blk = i >> 2, t4 = i & 3;
                        const int r = blk / nblk, j = blk - (blk / nblk) * nblk;
                        uint8_t* rowp = b_buf + (size_t)(j >> 1) * p.n_pad * 128 + (size_t)r * 128;
                        const int c = (j & 1) * 4 + t4;
                        uint2* e5 = p.f8 ? reinterpret_cast<uint2*>(b8 + (size_t)r * 128 +
                                                                    ((((2 * j + (t4 >> 1)) ^ (r & 7))) << 4) +
                                                                    (t4 & 1) * 8)
                                         : nullptr;
                        q_in = mxfp4_fake_quant_chunk(reinterpret_cast<uint4*>(rowp + ((c ^ (r & 7)) << 4)), e5) && q_in;
                    }
                }
                fence_proxy_async_smem();   // generic stores, read by the tensor core
                q_f8 = named_bar_and(2, 32 * kDqWarps, q_in) && p.f8;
                if (dq_t == 0 && ok) mbar_arrive(&bars->b_ready);
                b_phase ^= 1u;
                cur_unit = u;
            }
            // every warp walks every tile (units change in step); a group decodes every other one, so
            // two tiles are in decoding at once
            if (((g - g0) & 1) == dg) {
                ok = ok && mbar_wait(&bars->empty_a[astage], aphase ^ 1u, p.status);
                ok = ok && mbar_wait(&bars->full_c[cstage], cphase, p.status);
                if (dq == 0) STI_SCSTAMP(g - g0, 0);
                const uint8_t* cst = c_ring + (size_t)cstage * c_bytes;
                const uint8_t* crow = cst + (size_t)dq * (p.Di / 2);
                const uint8_t* srow = cst + c_code_bytes + (size_t)dq * nblk;
                uint8_t* arow = a_ring + (size_t)astage * a_bytes + (size_t)dq * 128;
                // Every warp checks all 512 scale bytes of the tile (16 a lane: keys 4*lane .. 4*lane+3),
                // so the group's four reach the same decision without a barrier.  Keys no query of the unit
                // sees may hold anything.  ok is warp-uniform here (the vote below needs every lane).
                ok = __all_sync(kFull, ok);
                bool f8 = false;
                if (ok && q_f8) {
                    const uint4 sc4 = *reinterpret_cast<const uint4*>(cst + c_code_bytes + lane * 16);
                    const uint32_t sw[4] = {sc4.x, sc4.y, sc4.z, sc4.w};
                    bool in = true;
    #pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t r = __vcmpgeu4(sw[k], 0x72727272u) & __vcmpleu4(sw[k], 0x8C8C8C8Cu);  // 114..140
                        in = in && (r == 0xFFFFFFFFu || tile * kTileKeys + lane * 4 + k >= vis_unit);
                    }
                    f8 = __all_sync(kFull, in);
                }
                if (ok && f8) {
                    for (int q4 = 0; q4 < nblk; ++q4) {
                        const int qb = (q4 + dq) & 3;   // rotated, as below; Di == 128 here
                        const uint4 cw4 = *reinterpret_cast<const uint4*>(crow + qb * 16);
                        uint32_t t0, t1;
                        e5m2_table(max(-13, min(13, (int)srow[qb] - 127)), t0, t1);
                        const uint2 o0 = e2m1x8_to_e5m2(cw4.x, t0, t1), o1 = e2m1x8_to_e5m2(cw4.y, t0, t1);
                        const uint2 o2 = e2m1x8_to_e5m2(cw4.z, t0, t1), o3 = e2m1x8_to_e5m2(cw4.w, t0, t1);
                        *reinterpret_cast<uint4*>(arow + (((2 * qb) ^ (dq & 7)) << 4)) = make_uint4(o0.x, o0.y, o1.x, o1.y);
                        *reinterpret_cast<uint4*>(arow + (((2 * qb + 1) ^ (dq & 7)) << 4)) = make_uint4(o2.x, o2.y, o3.x, o3.y);
                    }
                } else if (ok) {
                    for (int q4 = 0; q4 < p.Di / 32; ++q4) {
                        // 16 code bytes = 32 elements = one scale block; rows start 64 bytes apart, so
                        // lanes take the blocks in rotated order to spread the shared-memory banks
                        const int qb = (q4 + dq) % (p.Di / 32);
                        const uint4 cw4 = *reinterpret_cast<const uint4*>(crow + qb * 16);
                        const uint32_t e8 = srow[qb];
                        const bool fast = e8 >= 2u && e8 <= 252u;   // the exponent stays in the normal range
                        const float sc = e8m0_value(e8);
                        const uint32_t k16 = ((e8 - 127u) << 7) & 0xFFFFu;
                        const uint32_t expadd = k16 | (k16 << 16);
                        const uint32_t cw[4] = {cw4.x, cw4.y, cw4.z, cw4.w};
    #pragma unroll
                        for (int h = 0; h < 4; ++h) {   // 8 elements -> one 16-byte chunk of the tile
                            uint32_t pk[4];
                            if (fast) {
                                e2m1x8_to_bf16(cw[h], expadd, pk);
                            } else {
    #pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const uint32_t byte = (cw[h] >> (8 * j)) & 0xFFu;
                                    const float lo = e2m1_value(byte & 0xFu) * sc, hi = e2m1_value(byte >> 4) * sc;
                                    pk[j] = (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);
                                }
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
                if (dq == 0) {
                    bars->fmt[astage] = f8 ? 1u : 0u;
                    STI_SCSTAMP(g - g0, 1);
                }
                fence_proxy_async_smem();   // generic stores, read by the tensor core
                __syncwarp();
                if (lane == 0 && ok) {
                    mbar_arrive(&bars->full_a[astage]);
                    mbar_arrive(&bars->empty_c[cstage]);
                }
            }
            if (++astage == p.stages) {
                astage = 0;
                aphase ^= 1u;
            }
            if (++cstage == p.c_stages) {
                cstage = 0;
                cphase ^= 1u;
            }
            advance(p, u, tile, un, un_next);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        // bf16 keys with several queries per unit: two warps per TMEM lane quarter, each taking every
        // other query chunk of a unit
        const int EPI = FP4 ? 4 : ((int)blockDim.x - 64) / 32;   // epilogue warps (4 or 8)
        const int NG = EPI / 4;                                  // warps per lane quarter
        const int ep_tid = threadIdx.x - 64;           // 0 .. 32 EPI - 1
        const int eg = (warp - 2) >> 2;                // this warp's group: query chunks eg, eg + NG, ...
        const int quarter = warp & 3;                  // TMEM lane quarter this warp may access
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        constexpr int QPC = HI >= 32 ? 1 : 32 / HI;    // queries per 32-column load
        constexpr int CPQ = HI >= 32 ? HI / 32 : 1;    // 32-column loads per query
        int acc = 0;
        uint32_t acc_phase = 0;
        int cur_unit = -1;
        int st_e = 0;                  // E2M1 operands: the key stage of this tile (its scale bytes)
        uint32_t st_phase = 0, qb_phase = 0;
        // E2M1 operands: the first-pass histogram of the top-k gathers in shared memory (one shared
        // atomic per visible key) and goes to the unit's row in global memory when the CTA leaves the
        // unit (one atomic per non-empty bin); called after a barrier of the epilogue warps
        auto flush_hist = [&](int uu) {
            const int fb = uu / p.QT, ft0 = (uu - fb * p.QT) * p.nq;
            uint32_t* row = p.hist + ((size_t)fb * p.s + ft0) * 2048;
            for (int i = ep_tid; i < 2048; i += 32 * EPI) {
                const uint32_t v = hs[i];
                if (v != 0u) {
                    atomicAdd(row + i, v);
                    hs[i] = 0u;
                }
            }
        };
        if (E2 && p.hist != nullptr)
            for (int i = ep_tid; i < 2048; i += 32 * EPI) hs[i] = 0u;   // ordered by the first unit's barrier
        for (int g = g0; g < g1; ++g) {
            const int b = u / p.QT, qt = u - (u / p.QT) * p.QT;
            const int t0 = qt * p.nq;
            const int nq_here = min(p.nq, p.s - t0);
            if (u != cur_unit && E2) {
                // one query per unit.  First the unit's queries, quantised to MXFP4 into the E2M1 operand
                // (codes of a 32-element block in two 16-code chunks) and the block scales 2^X, so the
                // MMAs of the unit can start; then the previous unit's histogram and this unit's weights.
                // Every tile of the previous unit has been scored, so its MMAs are done.
                named_bar_sync(1, 32 * EPI);
                const bool has_w = ep_tid < HI;   // the unit's weights and start position, read early
                const uint16_t wb = has_w ? p.w[((size_t)b * p.s + t0) * HI + ep_tid] : (uint16_t)0;
                const int spv = ep_tid == 0 ? __ldg(p.start_pos + b) : 0;
                bool okb = !aborted() && mbar_wait(&bars->full_b, qb_phase, p.status);
                okb = __all_sync(kFull, okb);   // warp-uniform: the quantiser shuffles within the warp
                if (okb) {
                    // n_pad * 16 is a multiple of 32 * EPI: a warp's lanes run the same trips
                    for (int i = ep_tid; i < p.n_pad * 16; i += 32 * EPI) {
                        const int r = i >> 4, j = (i >> 2) & 3, t4 = i & 3;
                        const uint8_t* rowp = b_buf + (size_t)(j >> 1) * p.n_pad * 128 + (size_t)r * 128;
                        const int c = (j & 1) * 4 + t4;
                        int X;
                        const uint32_t nib = mxfp4_quant_e2m1(*reinterpret_cast<const uint4*>(rowp + ((c ^ (r & 7)) << 4)), X);
                        const int grp = 2 * j + (t4 >> 1);
                        uint8_t* dst = b8 + (size_t)r * 128 + ((grp ^ (r & 7)) << 4) + (t4 & 1) * 4;
                        // the chunk's second half is never read as codes; it gets the same bytes
                        *reinterpret_cast<uint32_t*>(dst) = nib;
                        *reinterpret_cast<uint32_t*>(dst + 8) = nib;
                        if (t4 == 0) sq_s[j * 32 + r] = exp2i(X);
                    }
                } else {
                    atomicExch(&bars->abort, 1u);
                }
                fence_proxy_async_smem();   // generic stores, read by the tensor core
                qb_phase ^= 1u;
                named_bar_sync(1, 32 * EPI);
                if (ep_tid == 0 && !aborted()) mbar_arrive(&bars->b_ready);
                if (p.hist != nullptr && cur_unit >= 0) flush_hist(cur_unit);
                if (has_w) w_s[ep_tid] = __uint_as_float((uint32_t)wb << 16) * p.c;
                if (ep_tid == 0) vis_s[0] = max(0, min(p.n_cols, (spv + t0 + 1) / p.ratio));
                named_bar_sync(1, 32 * EPI);
                cur_unit = u;
            } else if (u != cur_unit) {
                named_bar_sync(1, 32 * EPI);
                for (int i = ep_tid; i < nq_here * HI; i += 32 * EPI) {
                    const uint16_t wb = p.w[((size_t)b * p.s + t0) * HI + i];
                    w_s[i] = __uint_as_float((uint32_t)wb << 16) * p.c;
                }
                for (int i = ep_tid; i < nq_here; i += 32 * EPI)
                    vis_s[i] = max(0, min(p.n_cols, (__ldg(p.start_pos + b) + t0 + i + 1) / p.ratio));
                named_bar_sync(1, 32 * EPI);
                cur_unit = u;
            }
            // E2M1 operands: the two warp groups take the CTA's tiles in turn, group eg the tiles of
            // accumulator buffer eg; every warp walks every tile so unit changes stay in step
            const bool mine = !E2 || ((g - g0) & 1) == eg;
            bool ok = true;
            if (mine) {
                ok = !aborted() && mbar_wait(&bars->acc_full[acc], acc_phase, p.status);
                // E2M1 operands: the stage's scale bytes landed with its codes (already complete)
                if (E2) ok = ok && mbar_wait(&bars->full_a[st_e], st_phase, p.status);
                ok = __all_sync(kFull, ok);   // warp-uniform: the loop below holds warp collectives
                if (!ok) atomicExch(&bars->abort, 1u);
                if (E2 && ep_tid == 0) STI_SCSTAMP(g - g0, 1);
                tc_fence_after();
            }
            const int key = tile * kTileKeys + quarter * 32 + lane;
            const uint32_t col_base = tmem + lane_base + (uint32_t)(acc * (E2 ? 4 : 1) * p.n_alloc);
            if (E2 && mine && ok) {
                // one query: y_h = sum over the four 32-code blocks of acc_hj * 2^(Xq_hj + Xk_j) (products
                // of E2M1 values are exact, so is each block's fp32 sum), score = sum_h w_h relu(y_h);
                // heads in pairs (packed fp32x2 math), 16 columns of two blocks per TMEM wait
                constexpr int HE = HI <= 32 ? HI : 32;
                const uint32_t skw = *reinterpret_cast<const uint32_t*>(
                    c_ring + (size_t)st_e * c_bytes + (size_t)(quarter * 32 + lane) * 4);
                float2 y[HE / 2];
#pragma unroll
                for (int h = 0; h < HE / 2; ++h) y[h] = make_float2(0.f, 0.f);
#pragma unroll
                for (int hg = 0; hg < (HE + 15) / 16; ++hg) {
#pragma unroll
                    for (int k2 = 0; k2 < 4; k2 += 2) {
                        uint32_t r[2][16];
                        tmem_ld16(col_base + (uint32_t)(k2 * p.n_alloc + hg * 16), r[0]);
                        tmem_ld16(col_base + (uint32_t)((k2 + 1) * p.n_alloc + hg * 16), r[1]);
                        tmem_ld_wait();
#pragma unroll
                        for (int i2 = 0; i2 < 2; ++i2) {
                            const int kb = k2 + i2;
                            const float sk = e8m0_value((skw >> (8 * kb)) & 0xFFu);
                            const float2 sk2 = make_float2(sk, sk);
#pragma unroll
                            for (int h = 0; h < (HE < 16 ? HE : 16) / 2; ++h) {
                                const int hh = hg * 8 + h;   // head pair
                                const float2 f = __fmul2_rn(*reinterpret_cast<const float2*>(sq_s + kb * 32 + 2 * hh), sk2);
                                y[hh] = __ffma2_rn(make_float2(__uint_as_float(r[i2][2 * h]), __uint_as_float(r[i2][2 * h + 1])),
                                                   f, y[hh]);
                            }
                        }
                    }
                }
                float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int h = 0; h < HE / 2; ++h)
                    s2 = __ffma2_rn(*reinterpret_cast<const float2*>(w_s + 2 * h),
                                    make_float2(fmaxf(y[h].x, 0.f), fmaxf(y[h].y, 0.f)), s2);
                const float sc = s2.x + s2.y;
                const bool in_row = key < p.n_cols;
                const bool visible = in_row && key < vis_s[0];
                if (in_row) p.scores[((size_t)b * p.s + t0) * p.n_cols + key] = visible ? sc : -INFINITY;
                if (p.hist != nullptr && visible) atomicAdd(&hs[float_key(sc) >> 21], 1u);
            } else if (!E2 && ok) {
                for (int q0 = eg * QPC; q0 < nq_here; q0 += QPC * NG) {
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
            if (mine) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->acc_empty[acc]);
                if (E2 && lane == 0) mbar_arrive(&bars->empty_a[st_e]);
            }
            if (E2) {
                if (++st_e == p.stages) {
                    st_e = 0;
                    st_phase ^= 1u;
                }
            }
            if (ep_tid == 0) STI_SCSTAMP(g - g0, 3);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
            advance(p, u, tile, un, un_next);
        }
        if (E2 && p.hist != nullptr && cur_unit >= 0) {
            named_bar_sync(1, 32 * EPI);
            flush_hist(cur_unit);
        }
        // -inf for key tiles no query of a unit can see (units strided over CTAs)
        for (int uu = blockIdx.x; uu < p.total_units; uu += gridDim.x) {
            const int b = uu / p.QT, qt = uu - (uu / p.QT) * p.QT;
            const int t0 = qt * p.nq;
            const int nq_here = min(p.nq, p.s - t0);
            const int first = unit_tiles(p, uu) * kTileKeys;
            for (int q = 0; q < nq_here; ++q) {
                float* row = p.scores + ((size_t)b * p.s + t0 + q) * p.n_cols;
                for (int j = first + ep_tid; j < p.n_cols; j += 32 * EPI) row[j] = -INFINITY;
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
    const size_t b_bytes = (size_t)p.n_pad * p.Di * 2;
    if (p.fp4 == 2) {   // E2M1 operands: padded code tiles + scale bytes per stage, E2M1 queries, 2^X table,
                        // histogram
        return 1024 + (size_t)p.stages * (kTileKeys * 128 + kTileKeys * 4) + b_bytes + (size_t)p.n_pad * 128 +
               sizeof(Barriers) + 256 * 4 + 64 * 4 + 128 * 4 + 2048 * 4;
    }
    const size_t a_bytes = (size_t)kTileKeys * p.Di * 2;
    const size_t c_bytes = p.fp4 ? (size_t)kTileKeys * p.Di / 2 + (size_t)kTileKeys * p.Di / 32 : 0;
    const size_t b8_bytes = (p.fp4 && p.f8) ? (size_t)p.n_pad * 128 : 0;
    return 1024 + p.stages * a_bytes + b_bytes + b8_bytes + (p.fp4 ? p.c_stages : 0) * c_bytes + sizeof(Barriers) +
           256 * 4 + 64 * 4;
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
        auto kern = p.fp4 == 2 ? idx_scores_kernel<HV, 2>                                              \
                               : (p.fp4 ? idx_scores_kernel<HV, 1> : idx_scores_kernel<HV, 0>);        \
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);      \
        if (err != cudaSuccess) return err;                                                            \
        const int threads = p.fp4 == 2 ? kThreads                                                     \
                                       : (p.fp4 ? kThreadsFp4 : (p.nq > 1 ? kThreads : kThreadsOneQ)); \
        kern<<<grid, threads, smem, stream>>>(tm_a, tm_b, tm_s, p);                                    \
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

#ifdef STI_SC_TILE_TIMING
// profiling builds only: per-tile global-timer stamps of the scores kernel's first 16 tiles per CTA
extern "C" int sti_dbg_scores_tile_times(unsigned long long* host, int n_blocks) {
    return (int)cudaMemcpyFromSymbol(host, sti::g_sc_tile, sizeof(unsigned long long) * 16 * 5 * (size_t)n_blocks);
}
extern "C" int sti_dbg_scores_prologue_times(unsigned long long* host, int n_blocks) {
    return (int)cudaMemcpyFromSymbol(host, sti::g_sc_pro, sizeof(unsigned long long) * 4 * (size_t)n_blocks);
}
#endif
#ifdef STI_STEP_TIMING
// profiling builds only: global-timer stamps (ns) of the scores kernel's CTAs
extern "C" int sti_dbg_scores_times(unsigned long long* host, int n_blocks) {
    return (int)cudaMemcpyFromSymbol(host, sti::g_sc_t, sizeof(unsigned long long) * 2 * (size_t)n_blocks);
}
#endif
