// sti_internal.h -- host-side declarations shared by the C-ABI layer (api.cu) and the
// kernel translation units.  Not installed; the public interface is include/sti.h.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sti {

// Byte offsets inside every workspace: [0, 256) status block, then per-op scratch.
constexpr size_t kWsStatusBytes = 256;
constexpr size_t kWsAlign = 256;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------------ index scores
struct IdxScoresParams {
    const uint16_t* w;      // bf16 [B, s, Hi]
    const int32_t* start_pos;
    float* scores;          // fp32 [B, s, n_cols]
    uint32_t* status;
    float c;
    int B, s, Hi, Di, n_cols, ratio;
    int nq;                 // queries per unit (one B tile)
    int QT;                 // query tiles per sequence = ceil(s / nq)
    int n_pad;              // MMA N = round_up(nq * Hi, 16)
    int n_alloc;            // TMEM columns per accumulator buffer (multiple of 32)
    int tmem_cols;          // power of two >= 2 * n_alloc
    int stages;             // A pipeline depth
    int total_units;        // B * QT
};
// tm_a: index keys, tm_b: index queries.
cudaError_t launch_idx_scores(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const IdxScoresParams& p,
                              int num_sms, cudaStream_t stream);
int idx_scores_pick_nq(int Hi, int s);
size_t idx_scores_smem_bytes(const IdxScoresParams& p);

// ------------------------------------------------------------------ window indices, top-k
cudaError_t launch_window_idxs(const int32_t* start_pos, int B, int s, int W, int width, int32_t* idxs,
                               int64_t row_stride, uint32_t* status, cudaStream_t stream);
cudaError_t launch_topk(const float* scores, const int32_t* start_pos, int B, int s, int n_cols, int ratio, int k,
                        int32_t offset, int32_t* idxs, int64_t row_stride, uint32_t* status, cudaStream_t stream);

// ------------------------------------------------------------------ sparse attention
struct AttnParams {
    const uint16_t* q;       // bf16 [B, s, h, d]
    const uint16_t* kv;      // bf16, batch stride kv_bstride
    const uint16_t* kv2;     // bf16 or null
    const float* sink;       // [h]
    const int32_t* idx;      // [B, s, k] row stride idx_stride
    uint16_t* out;           // bf16 [B, s, h, d]
    float* lse;              // [B, s, h] or null
    float* part_o;           // split partials [B*s, splits, h, d] fp32 (splits > 1)
    float* part_ml;          // [B*s, splits, 2, 64] fp32
    uint32_t* status;
    int64_t kv_bstride, kv2_bstride, idx_stride;
    float scale_log2;        // softmax_scale * log2(e)
    int n1, n2;
    int B, s, h, d, k;
    int d_pad;               // round_up(d, 128)
    int n_tiles;             // ceil(k / 128)
    int splits, tiles_per_split;
};
int attn_pick_splits(int n_queries, int n_tiles, int num_sms);
size_t attn_partials_bytes(int n_queries, int splits, int d);
cudaError_t launch_sparse_attn(const AttnParams& p, cudaStream_t stream);

// ------------------------------------------------------------------ device properties
int device_num_sms();

}  // namespace sti
