// sti_kvfp4.h -- the sparse attention's second (compressed) KV source stored as fp4 rows.
//
// Attention._compress_kv ("read-weights" page) passes the compressed latent through
// fp4_act_quant(latent, 16, True, scale_dtype=float8_e4m3fn) before writing it to the cache:
// groups of 16 elements along the row share one E4M3 scale, each element an E2M1 code.  Kept
// packed, a 512-wide row is 256 code bytes + 32 scale bytes instead of 1 KB of bf16; the
// attention decodes the rows it gathers (every decoded value is exact in bf16).
#pragma once

#include "sti_internal.h"

namespace sti {

struct KvFp4 {
    const uint8_t* codes;     // [B, *, d/2]: element 2j of a row in the low nibble of byte j, 2j+1 high
    const uint8_t* scales;    // [B, *, d/16]: E4M3 scale of elements 16g .. 16g + 15 of a row
    int64_t codes_bstride;    // bytes between batch elements
    int64_t scales_bstride;
    int on;                   // 0: the second source is bf16 (AttnParams::kv2)
};

// launch_sparse_attn with the second source given as fp4 rows (f.on != 0; p.kv2 unused); the rows
// are gathered with plain loads and decoded into the tile, so p.use_tma must be 0.
cudaError_t launch_sparse_attn_kvfp4(const CUtensorMap& tm_q, const CUtensorMap& tm_kv1, const CUtensorMap& tm_kv2,
                                     const AttnParams& p, const KvFp4& f, cudaStream_t stream);

}  // namespace sti
