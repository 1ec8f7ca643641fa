/*
 * sti.h -- C ABI of the GB300 (sm_103a) library for the DeepSeek V4.1 attention hot path:
 * the Indexer's scores, their top-k, the sliding-window indices, and sparse attention with
 * an attention sink over the selected rows of one shared latent KV.
 *
 * Sources: the "DeepSeek V4.1" model pages -- attention "attend/selected" (prefill) and
 * "attend/allowed" (decode): get_window_topk_idxs, Indexer.forward, sparse_attn_kernel,
 * sparse_attn, Attention.forward; "reindex-layer/read-weights" (decode):
 * Attention._compress_kv and Attention._compress_topk_idxs.
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library never
 *    allocates or frees device memory, never synchronises (except sti_read_device_status),
 *    and enqueues its kernels on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *  - bf16 tensors are passed as uint16_t bit patterns (IEEE bfloat16); float is fp32.
 *  - Layouts are row-major and contiguous unless a stride argument says otherwise; strides
 *    are in ELEMENTS.
 *  - Arguments the host can check (null pointers, shapes, supported sizes, alignment,
 *    workspace size) are checked before anything is enqueued; a failed check returns
 *    STI_ERR_INVALID_ARG or STI_ERR_UNSUPPORTED and enqueues nothing.
 *  - Conditions only the device sees (an index out of range, a bounded wait that timed out,
 *    start_pos != 0 with seqlen > 1) set bits in the workspace's status word; the call still
 *    completes (bad indices are treated as masked).  sti_read_device_status reports them.
 *  - `ws` is a caller-owned device workspace of at least the size the matching
 *    sti_*_workspace_size() returns, aligned to 256 bytes.  It must be zero-filled once
 *    after allocation; the library leaves the parts that must start at zero at zero
 *    (sti_read_device_status clears the status word).  Calls that share one workspace must
 *    not overlap on the device.
 *  - Returns STI_ERR_CUDA if a launch fails (the CUDA error is in sti_last_cuda_error()).
 */
#ifndef STI_H_
#define STI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sti_status {
    STI_OK = 0,
    STI_ERR_INVALID_ARG = 1,       /* null pointer, bad shape or stride, workspace too small */
    STI_ERR_UNSUPPORTED = 2,       /* a size this build does not handle (see each call) */
    STI_ERR_CUDA = 3,              /* a CUDA runtime/driver call failed */
    STI_ERR_INDEX_RANGE = 4,       /* device: an index was < -1 or >= the number of KV rows */
    STI_ERR_DEVICE_TIMEOUT = 5,    /* device: a bounded wait inside a kernel gave up */
    STI_ERR_DEVICE_UNSUPPORTED = 6, /* device: start_pos != 0 with seqlen > 1 (chunked prefill) */
    STI_ERR_TOO_LARGE = 7           /* the sizes exceed the fixed scratch of sti_decode_fused_noalloc */
} sti_status;

/* Bits of the device status word (first 4 bytes of every workspace). */
#define STI_FLAG_INDEX_RANGE 1u
#define STI_FLAG_TIMEOUT 2u
#define STI_FLAG_CHUNKED 4u

typedef void *sti_stream; /* cudaStream_t */

/* Human-readable name of a status code (static storage). */
const char *sti_status_string(sti_status s);

/* Text of this thread's last CUDA failure seen by the library (thread-local storage). */
const char *sti_last_cuda_error(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int sti_version(void);

/*
 * Synchronises `stream`, reads the device status word of `ws` (STI_FLAG_* bits) into
 * *flags (may be NULL), clears it, and returns STI_OK when no bit was set, else the
 * status of the most severe bit (TIMEOUT > INDEX_RANGE > DEVICE_UNSUPPORTED).
 */
sti_status sti_read_device_status(void *ws, uint32_t *flags, sti_stream stream);

/* ------------------------------------------------------------------ window indices */
/*
 * get_window_topk_idxs (attend/selected page): which window-KV rows each query sees.
 *   seqlen > 1 (prefill, start_pos[b] must be 0): row t holds max(0,t-W+1)+i for
 *       i < width = min(seqlen, W); entries > t are -1.  The window KV source is then the
 *       seqlen raw KV rows of the chunk.  (start_pos != 0 raises STI_FLAG_CHUNKED when ws
 *       is given and writes -1 rows: such chunks take sti_window_idxs_chunked.)
 *   seqlen == 1 (decode): width = W; the ring slots oldest first,
 *       (start_pos%W)+1 .. W-1, 0 .. start_pos%W; a slot > start_pos is -1.  Position p
 *       lives in ring slot p % W.  (For start_pos == 0 this lists the same single slot as
 *       the page's prefill branch, at another place in the row; slot order does not matter.)
 * start_pos: int32 [b] device.  idxs: int32, row (b,t) at idxs + (b*seqlen+t)*row_stride,
 * `width` entries written (row_stride >= width).  The width goes to *width_out (host
 * pointer, may be NULL).  ws: optional workspace (NULL: no status reporting).
 */
sti_status sti_window_idxs(const int32_t *start_pos, int b, int seqlen, int window_size, int32_t *idxs,
                           int64_t row_stride, int *width_out, void *ws, sti_stream stream);

/*
 * Window rows of a prefill chunk that continues its sequence (start_pos[b] > 0, any seqlen):
 * not on the pages, which cover prefill from position 0 (the band above) and decode (the ring).
 * The chunk's window KV source is read as [the W-slot ring as it stood before the chunk
 * (slot i: the newest position p < start_pos with p % W == i) ; the chunk's seqlen raw rows
 * (row W + i: position start_pos + i)], W + seqlen rows; compressed indices then take offset
 * W + seqlen.  Query t at P = start_pos + t sees the band of the prefill formula with t -> P:
 * positions max(0, P-W+1) + i for i < W (-1 past P), position p at row W + (p - start_pos)
 * when p >= start_pos, else ring slot p % W.  Row width W (row_stride >= W).  Also valid for
 * start_pos == 0 (an empty ring: the prefill band shifted by W).  ws: optional, as above.
 */
sti_status sti_window_idxs_chunked(const int32_t *start_pos, int b, int seqlen, int window_size, int32_t *idxs,
                                   int64_t row_stride, void *ws, sti_stream stream);

/* ------------------------------------------------------------------ index scores */
/*
 * Indexer.forward (attend/selected page), the score block:
 *   scores[b,t,j] = c * sum_h w[b,t,h] * relu( sum_e iq[b,t,h,e] * ik[b,j,e] )   j < vis(b,t)
 *                 = -inf                                                         otherwise
 *   vis(b,t) = min(n_cols, (start_pos[b] + t + 1) // ratio)   (group j is visible once the
 *   query passed its last token; prefill compress_lens[t] = (t+1)//ratio, decode
 *   end_pos//ratio).  c = index_head_dim^-0.5 * index_n_heads^-0.5 (passed in).
 * Tensor-core (tcgen05) GEMM over bf16 inputs with fp32 accumulation; scores are fp32.
 *   iq: bf16 [b, seqlen, Hi, Di];  w: bf16 [b, seqlen, Hi]
 *   ik: bf16 [b, *, Di], batch b at ik + b*ik_bstride (ik_bstride >= n_cols*Di, a multiple
 *       of 8; rows >= n_cols are never read)
 *   scores: fp32 [b, seqlen, n_cols]
 * Supported: Di in {32, 64, 128}; Hi in {4, 8, 16, 32, 64}; ratio >= 1; iq and ik 16-byte
 * aligned.  ws: sti_idx_scores_workspace_size() bytes.
 */
size_t sti_idx_scores_workspace_size(void);
sti_status sti_idx_scores(const uint16_t *iq, const uint16_t *ik, int64_t ik_bstride, const uint16_t *w, float c,
                          const int32_t *start_pos, int b, int seqlen, int Hi, int Di, int n_cols, int ratio,
                          float *scores, void *ws, size_t ws_bytes, sti_stream stream);

/*
 * The same scores with the Indexer's fp4 keys and queries (Indexer.forward passes both through
 * fp4_act_quant before the einsum; the quantiser is not on the pages).  Reading: OCP MXFP4 --
 * blocks of 32 consecutive elements along Di share an E8M0 scale byte e (2^(e-127)); each
 * element is an E2M1 nibble (bit 3 sign, bits 2-1 exponent with bias 1, bit 0 mantissa;
 * exponent 0: m * 0.5), i.e. one of +-{0, .5, 1, 1.5, 2, 3, 4, 6} times the scale.
 *   ik_codes: uint8 [b, *, Di/2], batch b at + b*ik_codes_bstride bytes; byte j of a key holds
 *       element 2j (low nibble) and 2j+1 (high nibble)
 *   ik_scales: uint8 [b, *, Di/32], batch b at + b*ik_scales_bstride bytes
 *   iq (bf16, as above) is quantised in the kernel: per 32-element block X = floor(log2 max|x|)
 *       - 2 (clamped to [-127, 127]), x / 2^X to the nearest E2M1 value (ties to the even code,
 *       saturating at 6), times 2^X.
 * The score is the einsum/relu/weighted sum above over the decoded values (exact in bf16), with
 * fp32 accumulation.  Keys move as 68 bytes per position at Di = 128 instead of 256.
 * With seqlen == 1, Di == 128, Hi <= 32, ik_codes 32-byte aligned and ik_codes_bstride a multiple
 * of 32, the codes go to the tensor core as they are (E2M1 operands, the scales applied per
 * 32-element block in fp32); other calls decode them in shared memory first.  Both give the
 * scores above up to fp32 rounding order, for scales whose values fit fp32 (a block whose
 * products exceed fp32's range gives a non-finite score).
 * Supported: Di in {64, 128}; ik_codes, ik_scales 16-byte aligned; bstrides multiples of 16
 * covering n_cols keys.  Everything else as sti_idx_scores.
 */
sti_status sti_idx_scores_mxfp4(const uint16_t *iq, const uint8_t *ik_codes, int64_t ik_codes_bstride,
                                const uint8_t *ik_scales, int64_t ik_scales_bstride, const uint16_t *w, float c,
                                const int32_t *start_pos, int b, int seqlen, int Hi, int Di, int n_cols, int ratio,
                                float *scores, void *ws, size_t ws_bytes, sti_stream stream);

/* ------------------------------------------------------------------ top-k */
/*
 * Indexer.forward (attend/selected page), the selection block:
 *   topk = min(k, vis(b,t)); the topk largest scores[b,t,j] over j < vis(b,t) (equal scores:
 *   the lower position first), listed in ascending position order, each plus `offset`;
 *   the row is padded to width k with -1.  (The page's row width is min(index_topk,
 *   end_pos//ratio); the extra -1 slots select nothing.)
 * Radix select on order-preserving keys of the fp32 scores (no sort of the row).
 *   scores: fp32 [b, seqlen, n_cols];  idxs: int32, row (b,t) at idxs + (b*seqlen+t)*row_stride,
 *   k entries written (row_stride >= k; pass idxs+width to write after the window indices).
 * Supported: 1 <= k <= 4096, n_cols >= 0.  ws: sti_idx_topk_workspace_size() bytes.
 */
size_t sti_idx_topk_workspace_size(void);
sti_status sti_idx_topk(const float *scores, const int32_t *start_pos, int b, int seqlen, int n_cols, int ratio,
                        int k, int32_t offset, int32_t *idxs, int64_t row_stride, void *ws, size_t ws_bytes,
                        sti_stream stream);

/* ------------------------------------------------------------------ sparse attention */
/*
 * sparse_attn / sparse_attn_kernel (attend/selected page) with the two KV sources of
 * Attention.forward addressed in place (no concatenation copy): KV row r is
 *   kv[b, r]        for 0 <= r < n1     (window source: the chunk's raw rows, or the ring)
 *   kv2[b, r - n1]  for n1 <= r < n1+n2 (shared compressed KV; kv2 may be NULL when n2 == 0)
 * For every query (b,t) and head h, over the slots i with idx[b,t,i] != -1:
 *   s_i = softmax_scale * q[b,t,h,:] . row_i
 *   out[b,t,h,:] = sum_i e^{s_i} row_i / (sum_i e^{s_i} + e^{attn_sink[h]})
 * the same row serving as key and value; a query with no valid slot gets 0.
 * bf16 inputs, tcgen05 tensor-core MMAs with fp32 accumulation, P rounded to bf16 for the
 * PV product, fp32 online softmax, bf16 output.
 *   q: bf16 [b, seqlen, h, d];  out: bf16 [b, seqlen, h, d]
 *   kv: bf16 batch b at kv + b*kv_bstride, row stride d;  kv2 likewise with kv2_bstride
 *   attn_sink: fp32 [h];  idxs: int32 [b, seqlen, k] with row stride idx_row_stride (>= k)
 *   lse: optional fp32 [b, seqlen, h] = ln(sum_i e^{s_i} + e^{sink}); -inf for a query with
 *        no valid slot; may be NULL.
 * Indices < -1 or >= n1+n2 are treated as masked and raise STI_FLAG_INDEX_RANGE.
 * With few queries (decode) a query's slots are split over a thread-block cluster of 2, 4 or 8
 * CTAs.  They exchange their softmax maxima and sums in distributed shared memory, add their
 * rescaled partial outputs into an fp32 [b*seqlen, h, d] accumulator in the workspace (bulk
 * reductions performed at L2), and each converts a slice of the head dimension to bf16 and
 * zeroes it again.  sti_sparse_attn_workspace_size() includes that accumulator for batches of
 * at most 256 queries (none beyond); a workspace of only 256 bytes is accepted too and then no
 * query splits.
 * Supported: 1 <= h <= 64, d a multiple of 64 up to 512, k >= 1, kv_bstride/kv2_bstride
 * multiples of 8, q/kv/kv2/out 16-byte aligned.  ws: at least 256 bytes, up to
 * sti_sparse_attn_workspace_size(b, seqlen, h, d, k).
 */
size_t sti_sparse_attn_workspace_size(int b, int seqlen, int h, int d, int k);
sti_status sti_sparse_attn_sink(const uint16_t *q, const uint16_t *kv, int64_t kv_bstride, const uint16_t *kv2,
                                int64_t kv2_bstride, int n1, int n2, const float *attn_sink, const int32_t *idxs,
                                int64_t idx_row_stride, float softmax_scale, int b, int seqlen, int h, int d, int k,
                                uint16_t *out, float *lse, void *ws, size_t ws_bytes, sti_stream stream);

/* sti_sparse_attn_sink followed by the output's inverse rotary rotation, in the same kernel
 * (Attention.forward, "attend/selected" page: apply_rotary_emb(o[..., -rd:], freqs_cis, True)
 * right after sparse_attn).  rope_cs: fp32 [b, seqlen, rope_dims/2, 2], (cos, sin) of each
 * interleaved pair's angle at the query's position -- the caller evaluates the frequencies, which
 * the pages do not print.  Pair i = dims (d - rope_dims + 2i, +1) as x + iy is multiplied by
 * cos - i sin: x' = x cos + y sin, y' = y cos - x sin, in fp32 before the bf16 rounding.
 * rope_dims: even, 1 <= rope_dims <= d; rope_cs 16-byte aligned (STI_ERR_INVALID_ARG otherwise, or
 * when rope_cs is NULL).
 * lse is that of the attention (the rotation leaves it unchanged).  Everything else as
 * sti_sparse_attn_sink. */
sti_status sti_sparse_attn_sink_rope(const uint16_t *q, const uint16_t *kv, int64_t kv_bstride, const uint16_t *kv2,
                                     int64_t kv2_bstride, int n1, int n2, const float *attn_sink, const int32_t *idxs,
                                     int64_t idx_row_stride, float softmax_scale, int b, int seqlen, int h, int d,
                                     int k, const float *rope_cs, int rope_dims, uint16_t *out, float *lse, void *ws,
                                     size_t ws_bytes, sti_stream stream);

/* sti_sparse_attn_sink with the second (compressed) KV source stored as fp4 rows, the form
 * Attention._compress_kv ("read-weights" page) gives the compressed latent before writing its
 * cache: fp4_act_quant(latent, 16, True, scale_dtype=float8_e4m3fn) -- groups of 16 elements
 * along the row share one E4M3 scale (float8_e4m3fn: sign, exponent bias 7, 3 mantissa bits),
 * each element an E2M1 code (as in sti_idx_scores_mxfp4).  The quantiser is not on the pages;
 * any codes and scales are accepted and decoded as value = code * scale.
 *   kv2_codes:  uint8 [b, *, d/2], batch b at + b*kv2_codes_bstride bytes; row r of batch b holds
 *               compressed row r (index n1 + r); byte j = elements 2j (low nibble), 2j+1
 *   kv2_scales: uint8 [b, *, d/16], batch b at + b*kv2_scales_bstride bytes; byte g = the E4M3
 *               scale of elements 16g .. 16g+15
 * The window rows (indices < n1) stay bf16 in kv.  A packed 512-wide row is 288 bytes instead of
 * 1 KB.  The decoded values are exact in bf16, so the result is sti_sparse_attn_sink's over
 * those rows.  The rows are gathered with plain loads and decoded in shared memory by the
 * one-CTA-per-query kernel (never the head-split one).
 * Supported: as sti_sparse_attn_sink; kv2_codes and kv2_scales 16-byte aligned, their batch
 * strides multiples of 16 covering n2 rows (STI_ERR_INVALID_ARG otherwise). */
sti_status sti_sparse_attn_sink_fp4kv(const uint16_t *q, const uint16_t *kv, int64_t kv_bstride,
                                      const uint8_t *kv2_codes, int64_t kv2_codes_bstride, const uint8_t *kv2_scales,
                                      int64_t kv2_scales_bstride, int n1, int n2, const float *attn_sink,
                                      const int32_t *idxs, int64_t idx_row_stride, float softmax_scale, int b,
                                      int seqlen, int h, int d, int k, uint16_t *out, float *lse, void *ws,
                                      size_t ws_bytes, sti_stream stream);

/* ------------------------------------------------------------------ fused decode layer */
/*
 * One decode step (seqlen == 1) of an index-source attention layer, as
 * Attention.forward -> _window_kv / _compress_kv -> _compress_topk_idxs -> Indexer ->
 * sparse_attn composes it, three kernels enqueued back to back on one stream:
 *   1. index scores over the n_cols compressed positions (as sti_idx_scores) -> workspace; the
 *      kernel also counts the scores' top 11 key bits, the first radix pass of the top-k
 *   2. top-k of the visible positions, + offset W (as sti_idx_topk) -> topk_idxs[:, W:W+k],
 *      and the W-slot ring's window indices (as sti_window_idxs) -> topk_idxs[:, :W]
 *   3. sparse sink attention over [ring ; compressed KV] (as sti_sparse_attn_sink)
 * Ragged batches: start_pos is per sequence, compress_len = (start_pos+1)//ratio.
 * topk_idxs ([b, W+k] int32) is an output the caller owns, so reuse layers can consume it
 * through sti_sparse_attn_sink without running the Indexer (_compress_topk_idxs).
 */
typedef struct sti_decode_args {
    /* attention */
    const uint16_t *q;          /* bf16 [b, h, d] */
    const uint16_t *window_kv;  /* bf16 ring, batch b at + b*window_bstride, [W, d] */
    int64_t window_bstride;
    const uint16_t *comp_kv;    /* bf16 compressed KV, batch b at + b*comp_bstride, [n_cols, d] */
    int64_t comp_bstride;
    const float *attn_sink;     /* fp32 [h] */
    float softmax_scale;
    int h, d, window_size;
    /* indexer */
    const uint16_t *iq;         /* bf16 [b, Hi, Di] */
    const uint16_t *ik;         /* bf16 index keys, batch b at + b*ik_bstride, [n_cols, Di] */
    int64_t ik_bstride;
    const uint16_t *w;          /* bf16 [b, Hi] */
    float index_scale;          /* c = Di^-0.5 * Hi^-0.5 */
    int Hi, Di, index_topk, ratio, n_cols;
    /* batch */
    const int32_t *start_pos;   /* int32 [b] */
    int b;
    /* outputs */
    uint16_t *out;              /* bf16 [b, h, d] */
    int32_t *topk_idxs;         /* int32 [b, W + index_topk] */
    /* optional: a cudaEvent_t the attention step (step 3) waits for before it reads q, so that
     * q's upload (on another stream) overlaps steps 1 and 2; NULL: q is ready when the call is
     * enqueued */
    void *q_ready;
    /* optional: the inverse rotary rotation Attention.forward applies to the output after
     * sparse_attn ("attend/selected" page: apply_rotary_emb on o[..., -rd:] with the inverse
     * flag), fused into the attention's epilogue.  rope_cs: fp32 [b, rope_dims/2, 2], the
     * (cos, sin) of each interleaved pair's angle at the query's position (the caller evaluates
     * its frequencies); pair i = dims (d - rope_dims + 2i, d - rope_dims + 2i + 1) as x + iy is
     * multiplied by cos - i sin.  rope_dims: 0 (none) or even, <= d; rope_cs 16-byte aligned. */
    const float *rope_cs;
    int rope_dims;
    /* optional: MXFP4 index keys (as sti_idx_scores_mxfp4) instead of ik; the queries are then
     * quantised to MXFP4 in the scores kernel.  NULL ik_codes: bf16 keys from ik. */
    const uint8_t *ik_codes;
    int64_t ik_codes_bstride;   /* bytes */
    const uint8_t *ik_scales;
    int64_t ik_scales_bstride;  /* bytes */
    /* optional: the compressed KV as fp4 rows (as sti_sparse_attn_sink_fp4kv: Attention._compress_kv
     * on the "read-weights" page quantises the compressed latent with fp4_act_quant(latent, 16, ...)
     * before the cache write) instead of comp_kv, which is then unused (it may be NULL):
     *   comp_codes:  uint8 [b, *, d/2], batch b at + b*comp_codes_bstride bytes; byte j of a row holds
     *                element 2j (low nibble) and 2j+1 (high nibble) as E2M1 codes;
     *   comp_scales: uint8 [b, *, d/16], batch b at + b*comp_scales_bstride bytes; byte g is the E4M3
     *                scale of elements 16g .. 16g+15; an element's value is code * scale.
     * Supported only where steps 2 and 3 run as one kernel (sti_decode_kernel_count() == 2 with
     * these arguments): both arrays 16-byte aligned, bstrides multiples of 16 holding n_cols rows;
     * other shapes return STI_ERR_UNSUPPORTED.  NULL comp_codes: bf16 rows from comp_kv. */
    const uint8_t *comp_codes;
    int64_t comp_codes_bstride;  /* bytes */
    const uint8_t *comp_scales;
    int64_t comp_scales_bstride; /* bytes */
} sti_decode_args;

/* Steps 2 and 3 launch as programmatic dependents of the step before them: each is scheduled
 * while its predecessor drains and waits on the device before reading the predecessor's output
 * (step 1 launches normally, so all work enqueued before the call is complete before any step).
 * ws: sti_decode_workspace_size() bytes = status word, scores [b, n_cols] fp32, histograms
 * [b, 2048] u32 and, for b <= 256, the attention accumulator [b, h, d] fp32; zero-filled once,
 * left zeroed by every call that completes.
 * events: NULL, or 4 cudaEvent_t handles recorded on `stream` before step 1 and after steps
 * 1, 2 and 3 (per-kernel timing). */
size_t sti_decode_workspace_size(const sti_decode_args *a);
sti_status sti_decode_fused(const sti_decode_args *a, void *ws, size_t ws_bytes, sti_stream stream,
                            void *const *events);
/* How many kernels sti_decode_fused enqueues for these arguments (the device must be current):
 * 3 (scores; top-k + window indices; attention); 2 when steps 2 and 3 run as one kernel -- the
 * pages' decode shape (h = 64, d = 512, window 128, index_topk 512, n_cols <= 65536, both KV
 * sources in whole rows): a 4-CTA cluster per query selects the top-k and attends over its own
 * quarter of the index row, then merges; events 2 and 3 are then both recorded after it -- or
 * when n_cols == 0 (no scores kernel); 0 for b == 0; -1 if the arguments would be rejected.
 * Enqueues nothing. */
int sti_decode_kernel_count(const sti_decode_args *a);

/* ------------------------------------------------------------------ fused decode, no allocation */
/*
 * Not an operation of the paper (it has no counterpart there): the same decode step as
 * sti_decode_fused, for callers that cannot hand the library a device workspace -- for example
 * a plugin inside a host runtime that owns every device allocation and offers no workspace
 * hook, or a serving loop that must never enter the CUDA allocator once it is running.  The
 * step's scratch (status word, scores, first-pass histograms, attention accumulator) lives in
 * one fixed array inside this library instead: about 26 MiB of device memory that every GPU on
 * which the library is used holds until the process exits.  The call allocates and frees
 * nothing.  Batches of more than 128 queries (of 64 heads x 512) run the attention without
 * splitting a query.
 *  - Limits: b <= STI_NOALLOC_MAX_BATCH and b * n_cols <= STI_NOALLOC_MAX_SCORES; larger calls
 *    return STI_ERR_TOO_LARGE before anything is enqueued.  Other checks as sti_decode_fused.
 *  - The first call on a device looks up the array's device address (once per device, with
 *    that device current); make that first call before any stream capture.
 *  - Every call uses the same array and it keeps the previous call's contents: the call clears
 *    the parts that must start at zero, and calls that overlap on the GPU (other streams, other
 *    threads) race on it -- serialise them.  Device-side status bits are cleared by the next
 *    call; read them with sti_decode_noalloc_status.
 */
#define STI_NOALLOC_MAX_BATCH 256
#define STI_NOALLOC_MAX_SCORES (1 << 21)
sti_status sti_decode_fused_noalloc(const sti_decode_args *a, sti_stream stream);
/* Synchronises `stream` and returns the STI_FLAG_* bits the last no-allocation call left. */
sti_status sti_decode_noalloc_status(uint32_t *flags, sti_stream stream);

/* ------------------------------------------------------------------ diagnostics */
/*
 * Not an operation of the paper: a check of the library's failure handling.  Every wait in the
 * kernels above (on a TMA transfer, an MMA completion or a partner CTA) gives up after 1 s,
 * sets STI_FLAG_TIMEOUT and lets the kernel return, so a stalled step reports an error instead
 * of hanging the GPU.  This launches one small kernel whose wait nothing ever satisfies, with
 * a limit of limit_us microseconds (1..100000): afterwards the workspace's status word holds
 * STI_FLAG_TIMEOUT and the context is still usable.
 */
sti_status sti_selftest_wait_timeout(void *ws, size_t ws_bytes, uint32_t limit_us, sti_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* STI_H_ */
