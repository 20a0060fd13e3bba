// e4m3.cuh -- the tile scale and the E4M3 conversion shared by the quantizers and by the GEMM
// epilogue that re-quantizes its output (one definition, so both produce the same codes).
//
// Online tile scaling (codingmall.com "Định lượng trực tuyến"): for a tile with amax > 0,
// s = amax / 448 and codes E4M3(x * r) with r = 448 / amax (two IEEE FP32 divisions, one
// multiply per element). For amax < 2^-64, r is formed from amax * 2^64 and the values are
// scaled by 2^64 first (both exact). A tile with amax == 0 gets s = 1 and codes 0x00.
#pragma once

#include <cstdint>

namespace fp8bs {

struct TileScale {
    float s;     // dequantization scale
    float r;     // quantization multiplier
    bool tiny;   // amax < 2^-64: r formed from amax * 2^64 (exact), values scaled by 2^64
    bool zero;   // amax == 0: scale 1, codes 0x00
};

__device__ __forceinline__ TileScale tile_scale(float amax)
{
    TileScale t;
    t.zero = (amax == 0.0f);
    t.tiny = !t.zero && (amax < 0x1p-64f);
    const float den = t.tiny ? __fmul_rn(amax, 0x1p64f) : amax;
    t.s = t.zero ? 1.0f : __fdiv_rn(amax, 448.0f);
    t.r = t.zero ? 0.0f : __fdiv_rn(448.0f, den);
    return t;
}

// Power-of-two (UE8M0) tile scale, a variant that is not on the pages (Blackwell's block-scaled
// MMAs take such scales): s = 2^e with e the smallest integer for which 448 * 2^e >= amax (no value
// saturates), clamped below at 2^-127; r = 2^-e, so x * r is exact. With amax = f * 2^E (frexpf,
// f in [0.5, 1)) and 448 = 0.875 * 2^9: e = E - 9 + (f > 0.875).
__device__ __forceinline__ TileScale tile_scale_ue8m0(float amax)
{
    TileScale t;
    t.zero = (amax == 0.0f);
    t.tiny = false;
    int E;
    const float f = frexpf(amax, &E);
    int e = E - 9 + (f > 0.875f ? 1 : 0);
    e = e < -127 ? -127 : e;
    t.s = t.zero ? 1.0f : ldexpf(1.0f, e);
    t.r = t.zero ? 0.0f : ldexpf(1.0f, -e);
    return t;
}

template <bool UE8M0>
__device__ __forceinline__ TileScale tile_scale_of(float amax)
{
    return UE8M0 ? tile_scale_ue8m0(amax) : tile_scale(amax);
}

// Two FP32 values to two E4M3 codes, saturating round-to-nearest-even; `lo` lands in the low
// byte of the result.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// The value a tile's code is formed from: x * r, or (x * 2^64) * r for a tiny tile.
__device__ __forceinline__ float tile_scaled(float x, const TileScale& t)
{
    return t.tiny ? __fmul_rn(__fmul_rn(x, 0x1p64f), t.r) : __fmul_rn(x, t.r);
}

}  // namespace fp8bs
