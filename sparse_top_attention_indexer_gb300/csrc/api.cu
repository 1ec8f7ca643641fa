// api.cu -- the C ABI declared in include/sti.h: argument checks, TMA tensor-map encoding,
// workspace carving, launch sequencing and device-status reporting.  No allocation, no
// synchronisation (except sti_read_device_status), no torch types.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "sti.h"
#include "sti_internal.h"
#include "sti_kvfp4.h"
#include "sti_ptx.cuh"

namespace {

thread_local char g_last_cuda_error[256] = "";

sti_status cuda_fail(cudaError_t e, const char* where) {
    snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
    return STI_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 3-D bf16 tensor map: dims {inner, rows, batch}, strides in bytes for rows and batch.
sti_status make_map_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t batch,
                       uint64_t row_stride_bytes, uint64_t batch_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                       CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "cuTensorMapEncodeTiled unavailable");
        return STI_ERR_CUDA;
    }
    cuuint64_t dims[3] = {inner, rows, batch};
    cuuint64_t strides[2] = {row_stride_bytes, batch_stride_bytes};
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "cuTensorMapEncodeTiled failed (%d)", (int)r);
        return STI_ERR_CUDA;
    }
    return STI_OK;
}

// 2-D bf16 tensor map: dims {inner, rows}, row stride in bytes, 128-byte swizzle.
sti_status make_map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride_bytes,
                       uint32_t box_inner, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "cuTensorMapEncodeTiled unavailable");
        return STI_ERR_CUDA;
    }
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "cuTensorMapEncodeTiled failed (%d)", (int)r);
        return STI_ERR_CUDA;
    }
    return STI_OK;
}

// 3-D byte tensor map (no swizzle): dims {inner bytes, rows, batch}, strides in bytes.
sti_status make_map_3d_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t batch,
                          uint64_t row_stride_bytes, uint64_t batch_stride_bytes, uint32_t box_inner,
                          uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "cuTensorMapEncodeTiled unavailable");
        return STI_ERR_CUDA;
    }
    cuuint64_t dims[3] = {inner, rows, batch};
    cuuint64_t strides[2] = {row_stride_bytes, batch_stride_bytes};
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "cuTensorMapEncodeTiled failed (%d)", (int)r);
        return STI_ERR_CUDA;
    }
    return STI_OK;
}

// 3-D tensor map of MXFP4 codes for E2M1 MMA operands: dims {128 codes, rows, batch}, strides in
// bytes (row 64 B); a box of 128 codes x 128 rows lands as 128-byte rows of 16-byte chunks, each
// holding 16 codes in its first 8 bytes, 128-byte swizzled.  False when the driver declines the map
// (the caller then decodes the codes in shared memory instead); no error is recorded.
static bool make_map_3d_e2m1(CUtensorMap* m, const void* base, uint64_t rows, uint64_t batch,
                             uint64_t batch_stride_bytes) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {128, rows, batch};
    cuuint64_t strides[2] = {64, batch_stride_bytes};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uint32_t* status_word(void* ws) { return reinterpret_cast<uint32_t*>(ws); }

bool ws_ok(void* ws, size_t ws_bytes, size_t need) {
    return ws != nullptr && aligned(ws, sti::kWsAlign) && ws_bytes >= need;
}

}  // namespace

namespace sti {
int device_num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    static int cached[64] = {0};
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return n;
}
}  // namespace sti

// ---------------------------------------------------------------------- shared implementations

static sti_status window_impl(const int32_t* start_pos, int b, int seqlen, int window_size, int32_t* idxs,
                              int64_t row_stride, int* width_out, uint32_t* status, cudaStream_t st) {
    if (b < 0 || seqlen < 1 || window_size < 1) return STI_ERR_INVALID_ARG;
    const int width = seqlen > 1 ? (seqlen < window_size ? seqlen : window_size) : window_size;
    if (width_out) *width_out = width;
    if (b == 0) return STI_OK;
    if (!start_pos || !idxs || row_stride < width) return STI_ERR_INVALID_ARG;
    cudaError_t e = sti::launch_window_idxs(start_pos, b, seqlen, window_size, width, idxs, row_stride, status, st);
    return e == cudaSuccess ? STI_OK : cuda_fail(e, "sti_window_idxs");
}

// MXFP4 index keys: E2M1 codes [b, *, Di/2] bytes and E8M0 scales [b, *, Di/32] bytes.
struct Fp4Keys {
    const uint8_t* codes = nullptr;
    int64_t codes_bstride = 0;    // bytes
    const uint8_t* scales = nullptr;
    int64_t scales_bstride = 0;   // bytes
};

// Host checks of MXFP4 keys (done before anything is enqueued).
static sti_status fp4_keys_check(const Fp4Keys& k, int Di, int n_cols) {
    if (!(Di == 64 || Di == 128)) return STI_ERR_UNSUPPORTED;
    if (!k.codes || !k.scales || !aligned(k.codes, 16) || !aligned(k.scales, 16)) return STI_ERR_INVALID_ARG;
    if (k.codes_bstride < (int64_t)n_cols * Di / 2 || k.codes_bstride % 16 != 0) return STI_ERR_INVALID_ARG;
    if (k.scales_bstride < ((int64_t)n_cols * Di / 32 + 15) / 16 * 16 || k.scales_bstride % 16 != 0)
        return STI_ERR_INVALID_ARG;
    return STI_OK;
}

static sti_status idx_scores_impl(const uint16_t* iq, const uint16_t* ik, int64_t ik_bstride, const uint16_t* w,
                                  float c, const int32_t* start_pos, int b, int seqlen, int Hi, int Di, int n_cols,
                                  int ratio, float* scores, uint32_t* status, cudaStream_t st,
                                  uint32_t* hist = nullptr, const Fp4Keys* fp4 = nullptr) {
    if (b < 0 || seqlen < 1 || n_cols < 0 || ratio < 1) return STI_ERR_INVALID_ARG;
    if (!(Di == 32 || Di == 64 || Di == 128)) return STI_ERR_UNSUPPORTED;
    if (!(Hi == 4 || Hi == 8 || Hi == 16 || Hi == 32 || Hi == 64)) return STI_ERR_UNSUPPORTED;
    if (fp4) {
        const sti_status fs = fp4_keys_check(*fp4, Di, n_cols);
        if (fs != STI_OK) return fs;
    }
    if (b == 0 || n_cols == 0) return STI_OK;
    if (!iq || (!fp4 && !ik) || !w || !start_pos || !scores) return STI_ERR_INVALID_ARG;
    if (!fp4 && (ik_bstride < (int64_t)n_cols * Di || (ik_bstride % 8) != 0)) return STI_ERR_INVALID_ARG;
    if (!aligned(iq, 16) || (!fp4 && !aligned(ik, 16))) return STI_ERR_INVALID_ARG;
    if ((int64_t)seqlen * Hi > 0x7FFFFFFF || (int64_t)b * seqlen > 0x7FFFFFFF) return STI_ERR_UNSUPPORTED;

    sti::IdxScoresParams p{};
    p.w = w;
    p.start_pos = start_pos;
    p.scores = scores;
    p.hist = hist;
    p.status = status;
    p.c = c;
    p.B = b;
    p.s = seqlen;
    p.Hi = Hi;
    p.Di = Di;
    p.n_cols = n_cols;
    p.ratio = ratio;
    p.nq = sti::idx_scores_pick_nq(Hi, seqlen);
    p.QT = (seqlen + p.nq - 1) / p.nq;
    p.n_pad = ((p.nq * Hi + 15) / 16) * 16;
    p.n_alloc = ((p.n_pad + 31) / 32) * 32;
    int cols = 32;
    while (cols < 2 * p.n_alloc) cols *= 2;
    p.tmem_cols = cols;
    p.total_units = b * p.QT;
    const size_t a_bytes = (size_t)128 * Di * 2, b_bytes = (size_t)p.n_pad * Di * 2;
    // Two CTAs per SM stream faster than one with the same total stage count (two independent
    // TMA producers); possible when both CTAs' accumulators fit the SM's 512 TMEM columns.
    p.ctas_per_sm = p.tmem_cols <= 256 ? 2 : 1;
    const size_t budget = p.ctas_per_sm == 2 ? 104 * 1024 : 200 * 1024;
    p.fp4 = fp4 ? 1 : 0;
    if (fp4) {
        p.k_codes = fp4->codes;
        p.k_codes_bstride = fp4->codes_bstride;
        p.k_scales = fp4->scales;
        p.k_scales_bstride = fp4->scales_bstride;
    }
    // MXFP4: three or four stages of packed tiles (a quarter of the bytes) feed two decoded tiles
    // (E5M2, or bf16 when a block's scale is out of E5M2's exact range); with Di == 128 the
    // queries are held a second time as E5M2
    p.c_stages = fp4 ? 3 : 0;
    p.f8 = (fp4 && Di == 128) ? 1 : 0;
    const size_t c_total = fp4 ? (size_t)p.c_stages * ((size_t)128 * Di / 2 + (size_t)128 * Di / 32) : 0;
    const size_t b8_bytes = p.f8 ? (size_t)p.n_pad * 128 : 0;
    int stages = (int)((budget - b_bytes - b8_bytes - c_total) / a_bytes);
    if (stages > (fp4 ? 3 : 8)) stages = fp4 ? 3 : 8;
    if (stages < 2) stages = 2;
    p.stages = stages;
    // a fourth packed-tile stage when two CTAs still fit an SM's 228 KB (1 KB reserved per CTA)
    if (fp4) {
        p.c_stages = 4;
        if (p.ctas_per_sm == 2 && sti::idx_scores_smem_bytes(p) > (size_t)(228 * 1024 / 2 - 1024)) p.c_stages = 3;
    }

    const uint32_t box_inner = Di >= 64 ? 64u : (uint32_t)Di;
    const CUtensorMapSwizzle swz = Di >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUtensorMap tm_a, tm_b, tm_s;
    memset(&tm_s, 0, sizeof tm_s);
    sti_status s = STI_OK;
    // One query per unit (decode) with Di == 128: the codes go to the tensor core as E2M1 operands,
    // one accumulator per 32-code scale block (4 x n_alloc TMEM columns per buffer), the scales
    // applied in the epilogue; no decode in shared memory.
    const bool e2 = fp4 && Di == 128 && p.nq == 1 && p.n_pad <= 32 && aligned(fp4->codes, 32) &&
                    fp4->codes_bstride % 32 == 0 &&
                    make_map_3d_e2m1(&tm_a, fp4->codes, (uint64_t)n_cols, (uint64_t)b, (uint64_t)fp4->codes_bstride);
    if (e2) {
        p.fp4 = 2;
        p.f8 = 0;
        p.c_stages = 0;
        p.tmem_cols = 256;   // 2 buffers x 4 blocks x 32 columns
        p.ctas_per_sm = 2;
        for (p.stages = 8; p.stages > 2 && sti::idx_scores_smem_bytes(p) > (size_t)(228 * 1024 / 2 - 1024); --p.stages) {
        }
    } else if (fp4) {
        // codes: rows of Di/2 bytes; scales: each batch's Di/32 bytes per key as rows of 16 bytes
        s = make_map_3d_u8(&tm_a, fp4->codes, (uint64_t)Di / 2, (uint64_t)n_cols, (uint64_t)b, (uint64_t)Di / 2,
                           (uint64_t)fp4->codes_bstride, (uint32_t)Di / 2, 128);
        if (s == STI_OK)
            s = make_map_3d_u8(&tm_s, fp4->scales, 16, ((uint64_t)n_cols * Di / 32 + 15) / 16, (uint64_t)b, 16,
                               (uint64_t)fp4->scales_bstride, 16, (uint32_t)Di / 4);
    } else {
        s = make_map_3d(&tm_a, ik, (uint64_t)Di, (uint64_t)n_cols, (uint64_t)b, (uint64_t)Di * 2,
                        (uint64_t)ik_bstride * 2, box_inner, 128, swz);
    }
    if (s != STI_OK) return s;
    s = make_map_3d(&tm_b, iq, (uint64_t)Di, (uint64_t)seqlen * Hi, (uint64_t)b, (uint64_t)Di * 2,
                    (uint64_t)seqlen * Hi * Di * 2, box_inner, (uint32_t)p.n_pad, swz);
    if (s != STI_OK) return s;
    cudaError_t e = sti::launch_idx_scores(tm_a, tm_b, tm_s, p, sti::device_num_sms(), st);
    return e == cudaSuccess ? STI_OK : cuda_fail(e, "sti_idx_scores");
}

static sti_status topk_impl(const float* scores, const int32_t* start_pos, int b, int seqlen, int n_cols, int ratio,
                            int k, int32_t offset, int32_t* idxs, int64_t row_stride, uint32_t* status,
                            cudaStream_t st, uint32_t* hist = nullptr, int32_t* win_out = nullptr, int win_W = 0,
                            int win_width = 0, bool pdl = false) {
    if (b < 0 || seqlen < 1 || n_cols < 0 || ratio < 1 || k < 1 || row_stride < k) return STI_ERR_INVALID_ARG;
    if (k > 4096) return STI_ERR_UNSUPPORTED;
    if ((int64_t)b * seqlen > 0x7FFFFFFF) return STI_ERR_UNSUPPORTED;
    if (b == 0) return STI_OK;
    if (!start_pos || !idxs || (n_cols > 0 && !scores)) return STI_ERR_INVALID_ARG;
    sti::TopkParams p{};
    p.scores = scores;
    p.start_pos = start_pos;
    p.idxs = idxs;
    p.row_stride = row_stride;
    p.hist = hist;
    p.win_out = win_out;
    p.status = status;
    p.B = b;
    p.s = seqlen;
    p.n_cols = n_cols;
    p.ratio = ratio;
    p.k = k;
    p.offset = offset;
    p.win_W = win_W;
    p.win_width = win_width;
    p.pdl = pdl ? 1 : 0;
    cudaError_t e = sti::launch_topk(p, st);
    return e == cudaSuccess ? STI_OK : cuda_fail(e, "sti_idx_topk");
}

static sti_status attn_impl(const uint16_t* q, const uint16_t* kv, int64_t kv_bstride, const uint16_t* kv2,
                            int64_t kv2_bstride, int n1, int n2, const float* attn_sink, const int32_t* idxs,
                            int64_t idx_row_stride, float softmax_scale, int b, int seqlen, int h, int d, int k,
                            uint16_t* out, float* lse, uint32_t* status, float* acc, size_t acc_bytes,
                            cudaStream_t st, bool pdl = false, int win_ring = 0,
                            const int32_t* start_pos = nullptr, const float* rope_cs = nullptr, int rope_dims = 0,
                            const sti::KvFp4* fp4 = nullptr) {
    if (b < 0 || seqlen < 1 || h < 1 || d < 1 || k < 1 || n1 < 0 || n2 < 0) return STI_ERR_INVALID_ARG;
    if (rope_dims < 0 || rope_dims % 2 != 0 || rope_dims > d || (rope_dims > 0 && (!rope_cs || !aligned(rope_cs, 16))))
        return STI_ERR_INVALID_ARG;
    if (h > 64 || (d % 64) != 0 || d > 512) return STI_ERR_UNSUPPORTED;
    if (b == 0) return STI_OK;
    if (!q || !attn_sink || !idxs || !out || (n1 > 0 && !kv) || (n2 > 0 && !kv2 && !fp4)) return STI_ERR_INVALID_ARG;
    if (idx_row_stride < k) return STI_ERR_INVALID_ARG;
    if ((n1 > 0 && (kv_bstride < (int64_t)n1 * d || kv_bstride % 8)) ||
        (n2 > 0 && !fp4 && (kv2_bstride < (int64_t)n2 * d || kv2_bstride % 8)))
        return STI_ERR_INVALID_ARG;
    if (fp4 && n2 > 0 &&
        (!fp4->codes || !fp4->scales || !aligned(fp4->codes, 16) || !aligned(fp4->scales, 16) ||
         fp4->codes_bstride < (int64_t)n2 * (d / 2) || fp4->codes_bstride % 16 ||
         fp4->scales_bstride < (int64_t)n2 * (d / 16) || fp4->scales_bstride % 16))
        return STI_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || (kv && !aligned(kv, 16)) || (kv2 && !aligned(kv2, 16)))
        return STI_ERR_INVALID_ARG;
    if ((int64_t)b * seqlen * 8 > 0x7FFFFFFF) return STI_ERR_UNSUPPORTED;
    const int nq = b * seqlen;

    sti::AttnParams p{};
    p.q = q;
    p.kv = kv;
    p.kv2 = kv2;
    p.sink = attn_sink;
    p.idx = idxs;
    p.out = out;
    p.lse = lse;
    p.status = status;
    p.kv_bstride = kv_bstride;
    p.kv2_bstride = kv2_bstride;
    p.idx_stride = idx_row_stride;
    p.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634);
    p.n1 = n1;
    p.n2 = n2;
    p.B = b;
    p.s = seqlen;
    p.h = h;
    p.d = d;
    p.k = k;
    p.d_pad = ((d + 127) / 128) * 128;
    // few queries of 32 or 64 heads: heads split over a cluster, tiles gathered once (multicast);
    // otherwise a query's slots may split over a cluster when the workspace holds the accumulator
    p.acc = (acc != nullptr && acc_bytes >= (size_t)nq * h * d * sizeof(float)) ? acc : nullptr;
    int hs_rows = 1;
    const int c_hs = sti::attn_hs_pick(nq, h, d, &hs_rows);
    p.cluster = c_hs > 0 ? c_hs : (p.acc != nullptr ? sti::attn_pick_cluster(nq, k, d) : 1);
    // TMA gathers need each source to be whole d-element rows: batch stride a multiple of d
    p.rows1 = n1 > 0 ? kv_bstride / d : 0;
    p.rows2 = n2 > 0 ? kv2_bstride / d : 0;
    p.default_src = n1 > 0 ? 0 : 1;
    p.pdl = pdl ? 1 : 0;
    p.use_tma = (n1 + n2 > 0) && (n1 == 0 || kv_bstride % d == 0) && (n2 == 0 || kv2_bstride % d == 0) &&
                (int64_t)b * (p.rows1 > p.rows2 ? p.rows1 : p.rows2) < 0x7FFFFFFF;
    // fp4 compressed rows are gathered with plain loads and decoded into the tile by the
    // one-CTA-per-query kernel (no TMA, no head split)
    if (fp4) {
        p.rows2 = 0;
        p.use_tma = 0;
    }
    CUtensorMap tm_q, tm_kv1, tm_kv2, tm_win;
    memset(&tm_win, 0, sizeof tm_win);
    memset(&tm_q, 0, sizeof tm_q);
    memset(&tm_kv1, 0, sizeof tm_kv1);
    memset(&tm_kv2, 0, sizeof tm_kv2);
    const bool head_split = c_hs > 0 && p.use_tma;
    // the ring block load reads rows [b*rows1, b*rows1 + 128) of the first source
    p.win_ring = (head_split && win_ring == 128 && start_pos != nullptr && seqlen == 1 && n1 == 128 &&
                  p.rows1 >= 128) ? 128 : 0;
    p.start_pos = start_pos;
    p.hs_rows = head_split ? hs_rows : 1;
    p.rope_cs = rope_dims > 0 ? rope_cs : nullptr;
    p.rope_dims = rope_dims;
    if (!head_split && c_hs > 0) p.cluster = p.acc != nullptr ? sti::attn_pick_cluster(nq, k, d) : 1;
    // after the cluster is final: a query's slots split evenly over its CTAs
    p.rows_per_cta = (k + p.cluster - 1) / p.cluster;
    if (p.use_tma) {
        const uint32_t q_rows = head_split ? (uint32_t)(h * hs_rows / c_hs) : (uint32_t)h;
        sti_status s = make_map_2d(&tm_q, q, (uint64_t)d, (uint64_t)nq * h, (uint64_t)d * 2, 64, q_rows);
        if (s == STI_OK && n1 > 0) s = make_map_2d(&tm_kv1, kv, (uint64_t)d, (uint64_t)b * p.rows1, (uint64_t)d * 2, 64, 1);
        if (s == STI_OK && n2 > 0) s = make_map_2d(&tm_kv2, kv2, (uint64_t)d, (uint64_t)b * p.rows2, (uint64_t)d * 2, 64, 1);
        if (s == STI_OK && p.win_ring)
            s = make_map_2d(&tm_win, kv, (uint64_t)d, (uint64_t)b * p.rows1, (uint64_t)d * 2, 64, 128);
        if (s != STI_OK) return s;
        if (n1 == 0) tm_kv1 = tm_kv2;
        if (n2 == 0) tm_kv2 = tm_kv1;
    }
    const bool stream = !head_split && !fp4 && sti::sparse_attn_stream_fits(p);
    const bool stream_fp4 = fp4 && sti::sparse_attn_stream_fits_fp4(p);
    if (stream_fp4) {   // Q by TMA; the rows by LSU copies and fp4 decoding
        sti_status s = make_map_2d(&tm_q, q, (uint64_t)d, (uint64_t)nq * h, (uint64_t)d * 2, 64, (uint32_t)h);
        if (s != STI_OK) return s;
    }
    cudaError_t e = head_split   ? sti::launch_sparse_attn_hs(tm_q, tm_kv1, tm_kv2, tm_win, p, st)
                     : stream_fp4 ? sti::launch_sparse_attn_stream_fp4(tm_q, p, *fp4, st)
                     : fp4        ? sti::launch_sparse_attn_kvfp4(tm_q, tm_kv1, tm_kv2, p, *fp4, st)
                     : stream     ? sti::launch_sparse_attn_stream(tm_q, tm_kv1, tm_kv2, p, st)
                                  : sti::launch_sparse_attn(tm_q, tm_kv1, tm_kv2, p, st);
    return e == cudaSuccess ? STI_OK : cuda_fail(e, "sti_sparse_attn_sink");
}

// Split queries add their partial outputs into a zeroed fp32 [queries, h, d] accumulator that
// follows the status word in the workspace.  Only batches of at most 256 queries split (a split
// needs at least two SMs per query), so larger batches need no accumulator.
static constexpr int64_t kAttnSplitMaxQueries = 256;
static size_t attn_acc_bytes(int b, int seqlen, int h, int d) {
    const int64_t nq = (int64_t)b * seqlen;
    if (nq <= 0 || nq > kAttnSplitMaxQueries || h < 1 || h > 64 || d < 1 || d > 512) return 0;
    return sti::align_up((size_t)nq * (size_t)h * (size_t)d * sizeof(float), sti::kWsAlign);
}

// A wait on a barrier that nothing arrives at: it must give up after limit_ns, flag
// STI_FLAG_TIMEOUT and return, leaving the context usable.
static __global__ void selftest_wait_kernel(uint32_t* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        sti::mbar_init(&bar, 1);
        sti::fence_mbar_init();
    }
    __syncthreads();
    sti::mbar_wait_ns(&bar, 0, threadIdx.x == 0 ? status : nullptr, limit_ns);
}

extern "C" {

const char* sti_status_string(sti_status s) {
    switch (s) {
        case STI_OK: return "STI_OK";
        case STI_ERR_INVALID_ARG: return "STI_ERR_INVALID_ARG";
        case STI_ERR_UNSUPPORTED: return "STI_ERR_UNSUPPORTED";
        case STI_ERR_CUDA: return "STI_ERR_CUDA";
        case STI_ERR_INDEX_RANGE: return "STI_ERR_INDEX_RANGE";
        case STI_ERR_DEVICE_TIMEOUT: return "STI_ERR_DEVICE_TIMEOUT";
        case STI_ERR_DEVICE_UNSUPPORTED: return "STI_ERR_DEVICE_UNSUPPORTED";
        case STI_ERR_TOO_LARGE: return "STI_ERR_TOO_LARGE";
    }
    return "STI_UNKNOWN";
}

const char* sti_last_cuda_error(void) { return g_last_cuda_error; }

int sti_version(void) { return 100; }

sti_status sti_read_device_status(void* ws, uint32_t* flags, sti_stream stream) {
    if (!ws) return STI_ERR_INVALID_ARG;
    uint32_t host = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&host, ws, sizeof host, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof host, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "sti_read_device_status");
    if (flags) *flags = host;
    if (host & STI_FLAG_TIMEOUT) return STI_ERR_DEVICE_TIMEOUT;
    if (host & STI_FLAG_INDEX_RANGE) return STI_ERR_INDEX_RANGE;
    if (host & STI_FLAG_CHUNKED) return STI_ERR_DEVICE_UNSUPPORTED;
    return STI_OK;
}

sti_status sti_window_idxs_chunked(const int32_t* start_pos, int b, int seqlen, int window_size, int32_t* idxs,
                                   int64_t row_stride, void* ws, sti_stream stream) {
    if (ws && !aligned(ws, sti::kWsAlign)) return STI_ERR_INVALID_ARG;
    if (b < 0 || seqlen < 1 || window_size < 1) return STI_ERR_INVALID_ARG;
    if (b == 0) return STI_OK;
    if (!start_pos || !idxs || row_stride < window_size) return STI_ERR_INVALID_ARG;
    cudaError_t e = sti::launch_window_idxs(start_pos, b, seqlen, window_size, window_size, idxs, row_stride,
                                            ws ? status_word(ws) : nullptr, static_cast<cudaStream_t>(stream),
                                            /*chunked=*/true);
    return e == cudaSuccess ? STI_OK : cuda_fail(e, "sti_window_idxs_chunked");
}

sti_status sti_window_idxs(const int32_t* start_pos, int b, int seqlen, int window_size, int32_t* idxs,
                           int64_t row_stride, int* width_out, void* ws, sti_stream stream) {
    if (ws && !aligned(ws, sti::kWsAlign)) return STI_ERR_INVALID_ARG;
    return window_impl(start_pos, b, seqlen, window_size, idxs, row_stride, width_out,
                       ws ? status_word(ws) : nullptr, static_cast<cudaStream_t>(stream));
}

size_t sti_idx_scores_workspace_size(void) { return sti::kWsStatusBytes; }

sti_status sti_idx_scores(const uint16_t* iq, const uint16_t* ik, int64_t ik_bstride, const uint16_t* w, float c,
                          const int32_t* start_pos, int b, int seqlen, int Hi, int Di, int n_cols, int ratio,
                          float* scores, void* ws, size_t ws_bytes, sti_stream stream) {
    if (!ws_ok(ws, ws_bytes, sti_idx_scores_workspace_size())) return STI_ERR_INVALID_ARG;
    return idx_scores_impl(iq, ik, ik_bstride, w, c, start_pos, b, seqlen, Hi, Di, n_cols, ratio, scores,
                           status_word(ws), static_cast<cudaStream_t>(stream));
}

sti_status sti_idx_scores_mxfp4(const uint16_t* iq, const uint8_t* ik_codes, int64_t ik_codes_bstride,
                                const uint8_t* ik_scales, int64_t ik_scales_bstride, const uint16_t* w, float c,
                                const int32_t* start_pos, int b, int seqlen, int Hi, int Di, int n_cols, int ratio,
                                float* scores, void* ws, size_t ws_bytes, sti_stream stream) {
    if (!ws_ok(ws, ws_bytes, sti_idx_scores_workspace_size())) return STI_ERR_INVALID_ARG;
    Fp4Keys k;
    k.codes = ik_codes;
    k.codes_bstride = ik_codes_bstride;
    k.scales = ik_scales;
    k.scales_bstride = ik_scales_bstride;
    return idx_scores_impl(iq, nullptr, 0, w, c, start_pos, b, seqlen, Hi, Di, n_cols, ratio, scores,
                           status_word(ws), static_cast<cudaStream_t>(stream), nullptr, &k);
}

size_t sti_idx_topk_workspace_size(void) { return sti::kWsStatusBytes; }

sti_status sti_idx_topk(const float* scores, const int32_t* start_pos, int b, int seqlen, int n_cols, int ratio,
                        int k, int32_t offset, int32_t* idxs, int64_t row_stride, void* ws, size_t ws_bytes,
                        sti_stream stream) {
    if (!ws_ok(ws, ws_bytes, sti_idx_topk_workspace_size())) return STI_ERR_INVALID_ARG;
    return topk_impl(scores, start_pos, b, seqlen, n_cols, ratio, k, offset, idxs, row_stride, status_word(ws),
                     static_cast<cudaStream_t>(stream));
}

size_t sti_sparse_attn_workspace_size(int b, int seqlen, int h, int d, int k) {
    (void)k;
    return sti::kWsStatusBytes + attn_acc_bytes(b, seqlen, h, d);
}

sti_status sti_sparse_attn_sink(const uint16_t* q, const uint16_t* kv, int64_t kv_bstride, const uint16_t* kv2,
                                int64_t kv2_bstride, int n1, int n2, const float* attn_sink, const int32_t* idxs,
                                int64_t idx_row_stride, float softmax_scale, int b, int seqlen, int h, int d, int k,
                                uint16_t* out, float* lse, void* ws, size_t ws_bytes, sti_stream stream) {
    // the status word is required; the accumulator behind it is optional (without it no query splits)
    if (!ws_ok(ws, ws_bytes, sti::kWsStatusBytes)) return STI_ERR_INVALID_ARG;
    float* acc = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + sti::kWsStatusBytes);
    return attn_impl(q, kv, kv_bstride, kv2, kv2_bstride, n1, n2, attn_sink, idxs, idx_row_stride, softmax_scale, b,
                     seqlen, h, d, k, out, lse, status_word(ws), acc, ws_bytes - sti::kWsStatusBytes,
                     static_cast<cudaStream_t>(stream));
}

sti_status sti_sparse_attn_sink_rope(const uint16_t* q, const uint16_t* kv, int64_t kv_bstride, const uint16_t* kv2,
                                     int64_t kv2_bstride, int n1, int n2, const float* attn_sink, const int32_t* idxs,
                                     int64_t idx_row_stride, float softmax_scale, int b, int seqlen, int h, int d,
                                     int k, const float* rope_cs, int rope_dims, uint16_t* out, float* lse, void* ws,
                                     size_t ws_bytes, sti_stream stream) {
    if (!ws_ok(ws, ws_bytes, sti::kWsStatusBytes)) return STI_ERR_INVALID_ARG;
    if (rope_dims < 1) return STI_ERR_INVALID_ARG;
    float* acc = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + sti::kWsStatusBytes);
    return attn_impl(q, kv, kv_bstride, kv2, kv2_bstride, n1, n2, attn_sink, idxs, idx_row_stride, softmax_scale, b,
                     seqlen, h, d, k, out, lse, status_word(ws), acc, ws_bytes - sti::kWsStatusBytes,
                     static_cast<cudaStream_t>(stream), false, 0, nullptr, rope_cs, rope_dims);
}

sti_status sti_sparse_attn_sink_fp4kv(const uint16_t* q, const uint16_t* kv, int64_t kv_bstride,
                                      const uint8_t* kv2_codes, int64_t kv2_codes_bstride, const uint8_t* kv2_scales,
                                      int64_t kv2_scales_bstride, int n1, int n2, const float* attn_sink,
                                      const int32_t* idxs, int64_t idx_row_stride, float softmax_scale, int b,
                                      int seqlen, int h, int d, int k, uint16_t* out, float* lse, void* ws,
                                      size_t ws_bytes, sti_stream stream) {
    if (!ws_ok(ws, ws_bytes, sti::kWsStatusBytes)) return STI_ERR_INVALID_ARG;
    if (d % 16 != 0) return STI_ERR_INVALID_ARG;
    sti::KvFp4 f{};
    f.codes = kv2_codes;
    f.scales = kv2_scales;
    f.codes_bstride = kv2_codes_bstride;
    f.scales_bstride = kv2_scales_bstride;
    f.on = 1;
    float* acc = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + sti::kWsStatusBytes);
    return attn_impl(q, kv, kv_bstride, nullptr, 0, n1, n2, attn_sink, idxs, idx_row_stride, softmax_scale, b, seqlen,
                     h, d, k, out, lse, status_word(ws), acc, ws_bytes - sti::kWsStatusBytes,
                     static_cast<cudaStream_t>(stream), false, 0, nullptr, nullptr, 0, &f);
}

// The decode step's top-k and attention run as one kernel (decode_attn.cu) for the pages' decode
// shape: 64 heads x 512, window 128, index_topk 512, at most 65536 compressed positions, both KV
// sources in whole rows (TMA).  decode_fusable also needs the device to launch its 4-CTA clusters.
static bool decode_shape_fusable(const sti_decode_args* a) {
    constexpr int64_t kD = 512;
    if (a->b <= 0 || a->n_cols <= 0 || a->n_cols > 65536 || a->h != 64 || a->d != kD || a->window_size != 128 ||
        a->index_topk != 512)
        return false;
    if (!a->q || !a->window_kv || !a->attn_sink || !a->out || !a->topk_idxs) return false;
    if (a->window_bstride % kD != 0 || a->window_bstride < 128 * kD) return false;
    if (!aligned(a->q, 16) || !aligned(a->window_kv, 16) || !aligned(a->out, 16)) return false;
    if ((int64_t)a->b * (a->window_bstride / kD) >= 0x7FFFFFFF || (int64_t)a->b * 64 >= 0x7FFFFFFF) return false;
    if (a->comp_codes) {   // fp4 rows: 256 code bytes and 32 scale bytes per row, 16-byte aligned
        if (!a->comp_scales || !aligned(a->comp_codes, 16) || !aligned(a->comp_scales, 16)) return false;
        if (a->comp_codes_bstride % 16 != 0 || a->comp_scales_bstride % 16 != 0 ||
            a->comp_codes_bstride < (int64_t)a->n_cols * (kD / 2) || a->comp_scales_bstride < (int64_t)a->n_cols * (kD / 16))
            return false;
        return true;
    }
    if (!a->comp_kv || a->comp_bstride % kD != 0 || a->comp_bstride < (int64_t)a->n_cols * kD) return false;
    if (!aligned(a->comp_kv, 16)) return false;
    if ((int64_t)a->b * (a->comp_bstride / kD) >= 0x7FFFFFFF) return false;
    return true;
}
static bool decode_fusable(const sti_decode_args* a) {
    return decode_shape_fusable(a) && sti::decode_topk_attn_available();
}

// fused decode workspace: [status | scores fp32 [b, n_cols] | first-pass histograms u32 [b, 2048] |
//   attention accumulator fp32 [b, h, d] (batches of at most 256; unused when the top-k and
//   attention run as one kernel, which merges its partial outputs in shared memory)]
static size_t decode_scores_bytes(const sti_decode_args* a) {
    return sti::align_up((size_t)a->b * (size_t)(a->n_cols > 0 ? a->n_cols : 1) * sizeof(float), sti::kWsAlign);
}
static size_t decode_hist_bytes(const sti_decode_args* a) { return (size_t)a->b * 2048 * sizeof(uint32_t); }

static size_t decode_acc_bytes(const sti_decode_args* a) { return attn_acc_bytes(a->b, 1, a->h, a->d); }

size_t sti_decode_workspace_size(const sti_decode_args* a) {
    if (!a || a->b <= 0) return sti::kWsStatusBytes;
    return sti::kWsStatusBytes + decode_scores_bytes(a) + decode_hist_bytes(a) + decode_acc_bytes(a);
}

// MXFP4 index keys of a decode step (NULL: bf16 keys).
static const Fp4Keys* decode_fp4(const sti_decode_args* a, Fp4Keys* k) {
    if (!a->ik_codes) return nullptr;
    k->codes = a->ik_codes;
    k->codes_bstride = a->ik_codes_bstride;
    k->scales = a->ik_scales;
    k->scales_bstride = a->ik_scales_bstride;
    return k;
}

// The optional output rotation's arguments (checked before any step is enqueued).
static bool decode_rope_ok(const sti_decode_args* a) {
    return a->rope_dims == 0 || (a->rope_dims > 0 && a->rope_dims % 2 == 0 && a->rope_dims <= a->d && a->rope_cs &&
                                 aligned(a->rope_cs, 16));
}

// Steps 2 and 3 of a decode step as the fused kernel (after the scores kernel filled `scores` and
// `hist`); a programmatic dependent of the scores kernel unless it must wait for q_ready.
static sti_status decode_topk_attn_impl(const sti_decode_args* a, const float* scores, uint32_t* hist,
                                        uint32_t* status, cudaStream_t st) {
    constexpr int kD = 512;
    if (a->q_ready) {
        const cudaError_t e = cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(a->q_ready), 0);
        if (e != cudaSuccess) return cuda_fail(e, "sti_decode_fused: cudaStreamWaitEvent");
    }
    sti::DecodeAttnParams p{};
    p.scores = scores;
    p.hist = hist;
    p.start_pos = a->start_pos;
    p.idx_out = a->topk_idxs;
    p.sink = a->attn_sink;
    p.out = a->out;
    p.rope_cs = a->rope_dims > 0 ? a->rope_cs : nullptr;
    p.rope_dims = a->rope_dims;
    p.status = status;
    p.scale_log2 = (float)((double)a->softmax_scale * 1.4426950408889634);
    p.B = a->b;
    p.n_cols = a->n_cols;
    p.ratio = a->ratio;
    p.rows1 = a->window_bstride / kD;
    p.comp_kv = a->comp_kv;
    p.comp_bstride = a->comp_bstride;
    p.rows_c = a->comp_codes ? 0 : a->comp_bstride / kD;
    p.kvfp4 = a->comp_codes ? 1 : 0;
    p.comp_codes = a->comp_codes;
    p.comp_scales = a->comp_scales;
    p.codes_bstride = a->comp_codes_bstride;
    p.scales_bstride = a->comp_scales_bstride;
    CUtensorMap tm_q, tm_ring, tm_ring_rows, tm_comp_rows;
    memset(&tm_comp_rows, 0, sizeof tm_comp_rows);
    sti_status s = make_map_2d(&tm_q, a->q, kD, (uint64_t)a->b * 64, kD * 2, 64, 64);
    if (s == STI_OK) s = make_map_2d(&tm_ring, a->window_kv, kD, (uint64_t)a->b * p.rows1, kD * 2, 64, 32);
    if (s == STI_OK) s = make_map_2d(&tm_ring_rows, a->window_kv, kD, (uint64_t)a->b * p.rows1, kD * 2, 64, 1);
    if (s == STI_OK && !p.kvfp4)   // fp4 rows are gathered by cp.async (no map)
        s = make_map_2d(&tm_comp_rows, a->comp_kv, kD, (uint64_t)a->b * p.rows_c, kD * 2, 64, 1);
    if (s != STI_OK) return s;
    const cudaError_t e =
        sti::launch_decode_topk_attn(tm_q, tm_ring, tm_ring_rows, tm_comp_rows, p, /*pdl=*/!a->q_ready, st);
    return e == cudaSuccess ? STI_OK : cuda_fail(e, "sti_decode_fused: top-k + attention");
}

sti_status sti_decode_fused(const sti_decode_args* a, void* ws, size_t ws_bytes, sti_stream stream,
                            void* const* events) {
    if (!a) return STI_ERR_INVALID_ARG;
    if (a->b < 0 || a->window_size < 1 || a->index_topk < 1 || a->n_cols < 0) return STI_ERR_INVALID_ARG;
    if (!decode_rope_ok(a)) return STI_ERR_INVALID_ARG;
    Fp4Keys fk;
    if (decode_fp4(a, &fk) && a->n_cols > 0) {
        const sti_status fs = fp4_keys_check(fk, a->Di, a->n_cols);
        if (fs != STI_OK) return fs;
    }
    if (a->b == 0) return STI_OK;
    if (!ws_ok(ws, ws_bytes, sti_decode_workspace_size(a))) return STI_ERR_INVALID_ARG;
    if (!a->topk_idxs || !a->start_pos) return STI_ERR_INVALID_ARG;
    if (a->comp_codes && !decode_fusable(a)) return STI_ERR_UNSUPPORTED;   // fp4 rows: the fused kernel only
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    uint32_t* status = status_word(ws);
    const int W = a->window_size, K = a->index_topk, k_total = W + K;
    float* scores = reinterpret_cast<float*>(wsb + sti::kWsStatusBytes);
    uint32_t* hist = reinterpret_cast<uint32_t*>(wsb + sti::kWsStatusBytes + decode_scores_bytes(a));
    float* acc = reinterpret_cast<float*>(wsb + sti::kWsStatusBytes + decode_scores_bytes(a) + decode_hist_bytes(a));
    // timing events; inside a stream capture they become event-record nodes of the graph
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (events && cudaStreamIsCapturing(st, &cap) != cudaSuccess) cap = cudaStreamCaptureStatusNone;
    auto mark = [&](int i) -> cudaError_t {
        if (!events) return cudaSuccess;
        return cap == cudaStreamCaptureStatusActive
                   ? cudaEventRecordWithFlags(static_cast<cudaEvent_t>(events[i]), st, cudaEventRecordExternal)
                   : cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st);
    };
    cudaError_t e = mark(0);
    if (e != cudaSuccess) return cuda_fail(e, "sti_decode_fused");
    sti_status s = STI_OK;
    if (a->n_cols > 0) {
        s = idx_scores_impl(a->iq, a->ik, a->ik_bstride, a->w, a->index_scale, a->start_pos, a->b, 1, a->Hi, a->Di,
                            a->n_cols, a->ratio, scores, status, st, hist, decode_fp4(a, &fk));
        if (s != STI_OK) return s;
    }
    if ((e = mark(1)) != cudaSuccess) return cuda_fail(e, "sti_decode_fused");
    if (decode_fusable(a)) {
        s = decode_topk_attn_impl(a, scores, hist, status, st);
        if (s != STI_OK) return s;
        if ((e = mark(2)) != cudaSuccess || (e = mark(3)) != cudaSuccess) return cuda_fail(e, "sti_decode_fused");
        return STI_OK;
    }
    // top-k of the compressed positions (+W) and the ring's window indices, one kernel.  It and the
    // attention are programmatic dependents: each is scheduled while its predecessor drains, does
    // the work that needs nothing of the step (window indices; Q load, TMEM and barriers), then
    // waits for the predecessor grid before reading its output.  The scores kernel launches
    // normally, so everything the caller enqueued before this call is complete before either.
    s = topk_impl(scores, a->start_pos, a->b, 1, a->n_cols, a->ratio, K, W, a->topk_idxs + W, k_total, status, st,
                  a->n_cols > 0 ? hist : nullptr, a->topk_idxs, W, W, /*pdl=*/a->n_cols > 0);
    if (s != STI_OK) return s;
    if ((e = mark(2)) != cudaSuccess) return cuda_fail(e, "sti_decode_fused");
    // q may still be uploading on another stream: the attention waits for its event (and then
    // launches as an ordinary dependent)
    if (a->q_ready && (e = cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(a->q_ready), 0)) != cudaSuccess)
        return cuda_fail(e, "sti_decode_fused: cudaStreamWaitEvent");
    s = attn_impl(a->q, a->window_kv, a->window_bstride, a->comp_kv, a->comp_bstride, W, a->n_cols, a->attn_sink,
                  a->topk_idxs, k_total, a->softmax_scale, a->b, 1, a->h, a->d, k_total, a->out, nullptr, status, acc,
                  decode_acc_bytes(a), st, /*pdl=*/a->n_cols > 0 && !a->q_ready, /*win_ring=*/W, a->start_pos,
                  a->rope_cs, a->rope_dims);
    if (s != STI_OK) return s;
    if ((e = mark(3)) != cudaSuccess) return cuda_fail(e, "sti_decode_fused");
    return STI_OK;
}

int sti_decode_kernel_count(const sti_decode_args* a) {
    if (!a || a->b < 0 || a->window_size < 1 || a->index_topk < 1 || a->n_cols < 0) return -1;
    if (a->b == 0) return 0;
    if (decode_fusable(a)) return 2;
    if (a->comp_codes) return -1;   // fp4 compressed rows need the fused kernel
    return a->n_cols > 0 ? 3 : 2;
}

// ---------------------------------------------------------------------- fused decode, no allocation
//
// Scratch of sti_decode_fused_noalloc: [status word | scores fp32 (up to STI_NOALLOC_MAX_SCORES) |
// first-pass histograms u32 (up to STI_NOALLOC_MAX_BATCH rows of 2048 bins)].  A file-scope device
// array: in host code its name is only a stand-in, so the device address is looked up once per
// device with cudaGetSymbolAddress and that pointer is what the kernels get.

static constexpr size_t kNoallocScoresOff = sti::kWsStatusBytes;
static constexpr size_t kNoallocHistOff = kNoallocScoresOff + (size_t)STI_NOALLOC_MAX_SCORES * sizeof(float);
static constexpr size_t kNoallocAccOff = kNoallocHistOff + (size_t)STI_NOALLOC_MAX_BATCH * 2048 * sizeof(uint32_t);
// attention accumulator for split queries: up to 128 queries of 64 heads x 512 (larger batches
// run one CTA per query, which needs none)
static constexpr size_t kNoallocAccBytes = (size_t)128 * 64 * 512 * sizeof(float);
static constexpr size_t kNoallocBytes = kNoallocAccOff + kNoallocAccBytes;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

static std::mutex g_noalloc_mu;
static void* g_noalloc_addr[64];

// Device address of the scratch array on the current device (looked up on first use).
static sti_status noalloc_scratch(uint8_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "sti_decode_fused_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= 64) return STI_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> g(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                             "sti_decode_fused_noalloc: cudaGetSymbolAddress");
        g_noalloc_addr[dev] = p;
    }
    *out = static_cast<uint8_t*>(g_noalloc_addr[dev]);
    return STI_OK;
}

sti_status sti_decode_fused_noalloc(const sti_decode_args* a, sti_stream stream) {
    if (!a) return STI_ERR_INVALID_ARG;
    if (a->b < 0 || a->window_size < 1 || a->index_topk < 1 || a->n_cols < 0) return STI_ERR_INVALID_ARG;
    if (!decode_rope_ok(a)) return STI_ERR_INVALID_ARG;
    Fp4Keys fk;
    if (decode_fp4(a, &fk) && a->n_cols > 0) {
        const sti_status fs = fp4_keys_check(fk, a->Di, a->n_cols);
        if (fs != STI_OK) return fs;
    }
    if (a->b == 0) return STI_OK;
    if (!a->topk_idxs || !a->start_pos) return STI_ERR_INVALID_ARG;
    if (a->comp_codes && !decode_fusable(a)) return STI_ERR_UNSUPPORTED;   // fp4 rows: the fused kernel only
    if (a->b > STI_NOALLOC_MAX_BATCH || (int64_t)a->b * (a->n_cols > 0 ? a->n_cols : 1) > STI_NOALLOC_MAX_SCORES)
        return STI_ERR_TOO_LARGE;
    uint8_t* scratch = nullptr;
    sti_status s = noalloc_scratch(&scratch);
    if (s != STI_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t* status = reinterpret_cast<uint32_t*>(scratch);
    float* scores = reinterpret_cast<float*>(scratch + kNoallocScoresOff);
    uint32_t* hist = reinterpret_cast<uint32_t*>(scratch + kNoallocHistOff);
    float* acc = reinterpret_cast<float*>(scratch + kNoallocAccOff);
    // the fused top-k + attention kernel needs no accumulator; otherwise the split attention's,
    // when it fits
    const bool fused = decode_fusable(a);
    const size_t acc_need = attn_acc_bytes(a->b, 1, a->h, a->d);
    const size_t acc_used = fused ? 0 : (acc_need <= kNoallocAccBytes ? acc_need : 0);
    // the array still holds the previous call's data: zero the status word, the histograms and
    // the part of the accumulator this call may use
    cudaError_t e = cudaMemsetAsync(status, 0, sti::kWsStatusBytes, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(hist, 0, (size_t)a->b * 2048 * sizeof(uint32_t), st);
    if (e == cudaSuccess && acc_used > 0) e = cudaMemsetAsync(acc, 0, acc_used, st);
    if (e != cudaSuccess) return cuda_fail(e, "sti_decode_fused_noalloc: cudaMemsetAsync");
    const int W = a->window_size, K = a->index_topk, k_total = W + K;
    if (a->n_cols > 0) {
        s = idx_scores_impl(a->iq, a->ik, a->ik_bstride, a->w, a->index_scale, a->start_pos, a->b, 1, a->Hi, a->Di,
                            a->n_cols, a->ratio, scores, status, st, hist, decode_fp4(a, &fk));
        if (s != STI_OK) return s;
    }
    if (fused) return decode_topk_attn_impl(a, scores, hist, status, st);
    s = topk_impl(scores, a->start_pos, a->b, 1, a->n_cols, a->ratio, K, W, a->topk_idxs + W, k_total, status, st,
                  a->n_cols > 0 ? hist : nullptr, a->topk_idxs, W, W, /*pdl=*/a->n_cols > 0);
    if (s != STI_OK) return s;
    if (a->q_ready && (e = cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(a->q_ready), 0)) != cudaSuccess)
        return cuda_fail(e, "sti_decode_fused_noalloc: cudaStreamWaitEvent");
    return attn_impl(a->q, a->window_kv, a->window_bstride, a->comp_kv, a->comp_bstride, W, a->n_cols, a->attn_sink,
                     a->topk_idxs, k_total, a->softmax_scale, a->b, 1, a->h, a->d, k_total, a->out, nullptr, status,
                     acc, acc_used, st, /*pdl=*/a->n_cols > 0 && !a->q_ready, /*win_ring=*/W, a->start_pos,
                     a->rope_cs, a->rope_dims);
}

sti_status sti_selftest_wait_timeout(void* ws, size_t ws_bytes, uint32_t limit_us, sti_stream stream) {
    if (!ws_ok(ws, ws_bytes, sti::kWsStatusBytes) || limit_us == 0 || limit_us > 100000) return STI_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    selftest_wait_kernel<<<1, 32, 0, st>>>(status_word(ws), (uint64_t)limit_us * 1000u);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? STI_OK : cuda_fail(e, "sti_selftest_wait_timeout");
}

sti_status sti_decode_noalloc_status(uint32_t* flags, sti_stream stream) {
    uint8_t* scratch = nullptr;
    sti_status s = noalloc_scratch(&scratch);
    if (s != STI_OK) return s;
    uint32_t host = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&host, scratch, sizeof host, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "sti_decode_noalloc_status");
    if (flags) *flags = host;
    if (host & STI_FLAG_TIMEOUT) return STI_ERR_DEVICE_TIMEOUT;
    if (host & STI_FLAG_INDEX_RANGE) return STI_ERR_INDEX_RANGE;
    if (host & STI_FLAG_CHUNKED) return STI_ERR_DEVICE_UNSUPPORTED;
    return STI_OK;
}

}  // extern "C"
