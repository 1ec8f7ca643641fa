// sti_kvfp4.h -- the sparse attention's second (compressed) KV source stored as fp4 rows.
//
// Attention._compress_kv ("read-weights" page) passes the compressed latent through
// fp4_act_quant(latent, 16, True, scale_dtype=float8_e4m3fn) before writing it to the cache:
// groups of 16 elements along the row share one E4M3 scale, each element an E2M1 code.  Kept
// packed, a 512-wide row is 256 code bytes + 32 scale bytes instead of 1 KB of bf16; the
// attention decodes the rows it gathers (every decoded value is exact in bf16).
#pragma once

#include "sti_internal.h"
#ifdef __CUDACC__
#include <cuda_bf16.h>
#include "sti_ptx.cuh"
#endif

namespace sti {

struct KvFp4 {
    const uint8_t* codes;     // [B, *, d/2]: element 2j of a row in the low nibble of byte j, 2j+1 high
    const uint8_t* scales;    // [B, *, d/16]: E4M3 scale of elements 16g .. 16g + 15 of a row
    int64_t codes_bstride;    // bytes between batch elements
    int64_t scales_bstride;
    int on;                   // 0: the second source is bf16 (AttnParams::kv2)
};

#ifdef __CUDACC__
// Two E4M3 bytes (bits 0-7 and 8-15 of `two`; sign, 4-bit exponent with bias 7, 3-bit mantissa;
// exponent 0 subnormal: m * 2^-9; S.1111.111 NaN) -> two floats, by the hardware's E4M3 -> f16
// conversion and f16 -> f32: every E4M3 value, subnormals and NaN included, is an f16 value, so
// both steps are exact.  No branches.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
    float lo, hi;
    asm("{\n\t.reg .b16 t, a, b;\n\t.reg .b32 h;\n\t"
        "cvt.u16.u32 t, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 h, t;\n\t"
        "mov.b32 {a, b}, h;\n\t"
        "cvt.f32.f16 %0, a;\n\t"
        "cvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(two));
    return make_float2(lo, hi);
}
// One E4M3 byte (bits 0-7 of v) -> float.
__device__ __forceinline__ float e4m3_to_float(uint32_t v) { return e4m3x2_to_float2(v & 0xFFu).x; }

// Eight fp4 elements (nibble i of cw = element i) times their E4M3 scale s as eight bf16 (one
// 16-byte chunk of the tile): the E2M1 values by byte-permute lookup (e2m1x8_to_bf16), then four
// bf16x2 products with the scale.  Every factor is exact in bf16 and a product of an E2M1 value
// and an E4M3 value has at most six significant bits, so each product is exact.
__device__ __forceinline__ uint4 kvfp4_decode8_s2(uint32_t cw, __nv_bfloat162 s2) {   // s2 = (s, s)
    uint32_t o[4];
    e2m1x8_to_bf16(cw, 0u, o);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 v = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&o[j]), s2);
        o[j] = *reinterpret_cast<const uint32_t*>(&v);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}
__device__ __forceinline__ uint4 kvfp4_decode8(uint32_t cw, float s) {
    return kvfp4_decode8_s2(cw, __float2bfloat162_rn(s));
}

#endif

// launch_sparse_attn with the second source given as fp4 rows (f.on != 0; p.kv2 unused); the rows
// are gathered with plain loads and decoded into the tile, so p.use_tma must be 0.
cudaError_t launch_sparse_attn_kvfp4(const CUtensorMap& tm_q, const CUtensorMap& tm_kv1, const CUtensorMap& tm_kv2,
                                     const AttnParams& p, const KvFp4& f, cudaStream_t stream);
// The streamed many-query kernel with fp4 rows in the second source (64 heads at most, d = 512, no
// cluster): the first source's rows come by LSU copies, the fp4 rows are loaded into registers
// and decoded into the tile.  tm_q: q as [B*s*h, d] (box 64 x h).
bool sparse_attn_stream_fits_fp4(const AttnParams& p);
cudaError_t launch_sparse_attn_stream_fp4(const CUtensorMap& tm_q, const AttnParams& p, const KvFp4& f,
                                          cudaStream_t stream);

}  // namespace sti
