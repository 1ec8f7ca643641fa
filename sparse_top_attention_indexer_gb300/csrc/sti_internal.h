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
    uint32_t* hist;         // optional [B*s, 2048] counts of the visible scores' top 11 key bits
    uint32_t* status;
    float c;
    int B, s, Hi, Di, n_cols, ratio;
    int nq;                 // queries per unit (one B tile)
    int QT;                 // query tiles per sequence = ceil(s / nq)
    int n_pad;              // MMA N = round_up(nq * Hi, 16)
    int n_alloc;            // TMEM columns per accumulator buffer (multiple of 32)
    int tmem_cols;          // power of two >= 2 * n_alloc
    int stages;             // A pipeline depth
    int ctas_per_sm;        // 2 when two CTAs' TMEM fits one SM (decode), else 1
    int total_units;        // B * QT
    int fp4;                // keys stored as MXFP4 (codes + E8M0 scales) and queries quantised to MXFP4
    int c_stages;           // fp4: staging depth of the packed key tiles
    int f8;                 // fp4 with Di == 128: tiles whose scales allow it run as E5M2 (kind::f8f6f4)
    const uint8_t* k_codes;   // fp4: E2M1 codes [B, *, Di/2], batch stride in bytes
    int64_t k_codes_bstride;
    const uint8_t* k_scales;  // fp4: E8M0 scales [B, *, Di/32], batch stride in bytes
    int64_t k_scales_bstride;
};
// tm_a: index keys (bf16; fp4: their E2M1 codes, uint8 [Di/2] per key), tm_b: index queries,
// tm_s: fp4 only, the E8M0 scales viewed as rows of 16 bytes.
cudaError_t launch_idx_scores(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_s,
                              const IdxScoresParams& p, int num_sms, cudaStream_t stream);
int idx_scores_pick_nq(int Hi, int s);
size_t idx_scores_smem_bytes(const IdxScoresParams& p);

// ------------------------------------------------------------------ window indices, top-k
cudaError_t launch_window_idxs(const int32_t* start_pos, int B, int s, int W, int width, int32_t* idxs,
                               int64_t row_stride, uint32_t* status, cudaStream_t stream,
                               bool chunked = false);
struct TopkParams {
    const float* scores;      // fp32 [B, s, n_cols]
    const int32_t* start_pos;
    int32_t* idxs;            // row (b,t) at idxs + (b*s+t)*row_stride, k entries
    int64_t row_stride;
    uint32_t* hist;           // optional [B*s, 2048] first-pass histogram (from the scores kernel); re-zeroed
    int32_t* win_out;         // optional: window indices of the row written here too (win_width entries)
    uint32_t* status;
    int B, s, n_cols, ratio, k;
    int32_t offset;
    int win_W, win_width;
    int pdl;                  // launch as a programmatic dependent of the previous kernel in the stream
};
cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream);

// ------------------------------------------------------------------ sparse attention
struct AttnParams {
    const uint16_t* q;       // bf16 [B, s, h, d]
    const uint16_t* kv;      // bf16, batch stride kv_bstride
    const uint16_t* kv2;     // bf16 or null
    const float* sink;       // [h]
    const int32_t* idx;      // [B, s, k] row stride idx_stride
    uint16_t* out;           // bf16 [B, s, h, d]
    float* lse;              // [B, s, h] or null
    uint32_t* status;
    int64_t kv_bstride, kv2_bstride, idx_stride;
    float scale_log2;        // softmax_scale * log2(e)
    int n1, n2;
    int B, s, h, d, k;
    int d_pad;               // round_up(d, 128)
    int cluster;             // CTAs per query (a thread-block cluster when > 1)
    int rows_per_cta;        // index slots each CTA of a cluster handles
    int use_tma;             // gather rows with TMA (tensor maps valid); else 16-byte cp.async
    int64_t rows1, rows2;    // rows per batch element of kv / kv2 (batch stride / d)
    int default_src;         // source whose row 0 stands in for masked slots (0: kv, 1: kv2)
    int pdl;                 // launch as a programmatic dependent of the previous kernel in the stream
    float* acc;              // split queries: zeroed fp32 [B*s, h, d] the cluster adds its partials into
                             // (left zeroed again); nullptr: no split
    int win_ring;            // decode: slots [0, 128) list the 128-row window ring of kv (any order), so a
                             // full ring (start_pos >= 127) is loaded as one block; 0: indices only
    const int32_t* start_pos;  // [B], with win_ring
    int hs_rows;             // head-split kernel: row groups of a query's slots (1 or 2); the cluster
                             // is (cluster / hs_rows) head groups x hs_rows row groups
    // optional inverse rotary rotation of the output's last rope_dims dims: rope_cs[query] holds
    // (cos, sin) of each of the rope_dims/2 interleaved pairs; rope_dims == 0: none
    const float* rope_cs;
    int rope_dims;
};
// CTAs per query for n_queries queries of k slots and head dim d (1 = no cluster); cached per device.
int attn_pick_cluster(int n_queries, int k, int d);
// tm_q: q as [B*s*h, d] (box 64 x h); tm_kv1 / tm_kv2: the sources as [B*rows, d] (box 64 x 1,
// for 4-row gathers).  Ignored unless p.use_tma.
cudaError_t launch_sparse_attn(const CUtensorMap& tm_q, const CUtensorMap& tm_kv1, const CUtensorMap& tm_kv2,
                               const AttnParams& p, cudaStream_t stream);
// Many queries (prefill): persistent CTAs with the tile streamed by column block (64 heads at
// most, d = 512, TMA gathers, no cluster); same maps as launch_sparse_attn.
bool sparse_attn_stream_fits(const AttnParams& p);
cudaError_t launch_sparse_attn_stream(const CUtensorMap& tm_q, const CUtensorMap& tm_kv1, const CUtensorMap& tm_kv2,
                                      const AttnParams& p, cudaStream_t stream);
// Few queries with 32 or 64 heads: CTAs per query of the head-split kernel (0 = not applicable
// or not resident) and, in *rows, how many row groups they form; its launch (tm_q's box is
// {64, heads per CTA}).
int attn_hs_pick(int n_queries, int h, int d, int* rows);
cudaError_t launch_sparse_attn_hs(const CUtensorMap& tm_q, const CUtensorMap& tm_kv1, const CUtensorMap& tm_kv2,
                                  const CUtensorMap& tm_win, const AttnParams& p, cudaStream_t stream);

// ------------------------------------------------------------------ fused decode top-k + attention
// One kernel for the decode step's top-k (with the ring's window indices) and its attention, for
// 64 heads x 512, window 128, index_topk 512: a 4-CTA cluster per query (decode_attn.cu).
struct DecodeAttnParams {
    const float* scores;       // fp32 [B, n_cols] (one query per sequence)
    uint32_t* hist;            // [B, 2048] the scores kernel's first-pass histograms (re-zeroed)
    const int32_t* start_pos;  // [B]
    int32_t* idx_out;          // [B, 128 + 512]: window slots, then compressed positions + 128
    const uint16_t* comp_kv;   // bf16 compressed KV, batch b at + b*comp_bstride, rows of 512
    int64_t comp_bstride;      // elements
    const float* sink;         // [64]
    uint16_t* out;             // bf16 [B, 64, 512]
    const float* rope_cs;      // optional [B, rope_dims/2, 2]: the output's inverse rotation
    int rope_dims;
    uint32_t* status;
    float scale_log2;          // softmax_scale * log2(e)
    int B, n_cols, ratio;
    int64_t rows1;             // rows per batch element of the ring (batch stride / 512)
    int64_t rows_c;            // rows per batch element of the compressed KV (comp_bstride / 512)
    // optional fp4 compressed KV (comp_kv unused): codes [B][*][256] and E4M3 scales [B][*][32]
    const uint8_t* comp_codes;
    const uint8_t* comp_scales;
    int64_t codes_bstride, scales_bstride;   // bytes
    int kvfp4;
};
bool decode_topk_attn_available();
size_t decode_topk_attn_smem_bytes();
// tm_q: q as [B*64, 512] (box 64 x 64); tm_ring: the ring as [B*rows1, 512] (box 64 x 32, a full
// ring's slice per CTA); tm_ring_rows: the same with box 64 x 1, for four-row gathers (whose box is
// one row high); tm_comp_rows: the compressed KV as [B*rows_c, 512], box 64 x 1.
cudaError_t launch_decode_topk_attn(const CUtensorMap& tm_q, const CUtensorMap& tm_ring, const CUtensorMap& tm_ring_rows,
                                    const CUtensorMap& tm_comp_rows, const DecodeAttnParams& p, bool pdl,
                                    cudaStream_t stream);

// ------------------------------------------------------------------ device properties
int device_num_sms();

}  // namespace sti
