// Encoding of one row of the quantised K/V cache by one warp ("Qwen3.8-27B on one RTX 4090", section
// "A cheaper cache and state"): keys are rotated by the +-1 Hadamard butterfly and coded E4M3 with one
// fp32 scale per row (the largest magnitude maps to 448), values are coded INT8 with one scale per row
// (the largest magnitude maps to 127).  Lane l codes elements 4 l .. 4 l + 3.  Shared by the separate
// append kernel and the quantised verify step, which appends its live rows inside the attention launch:
// both write the same bytes.
#pragma once

#include <cstdint>

namespace va {
namespace codec {

// Two floats to E4M3 codes (round to nearest even, saturating); a zero result is coded +0.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    uint32_t b = d;
    if ((b & 0x007Fu) == 0) b &= 0xFF00u;
    if ((b & 0x7F00u) == 0) b &= 0x00FFu;
    return b;
}

__device__ __forceinline__ float warp_max(float m) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    return m;
}

// The four bf16 elements of a lane as floats.
__device__ __forceinline__ void bf16x4_to_float(uint2 raw, float (&x)[4]) {
    x[0] = __uint_as_float(raw.x << 16);
    x[1] = __uint_as_float(raw.x & 0xFFFF0000u);
    x[2] = __uint_as_float(raw.y << 16);
    x[3] = __uint_as_float(raw.y & 0xFFFF0000u);
}

// Key row: k' = H k (butterfly stages of width 1 and 2 inside the lane, then 4 .. 64 across lanes), then
// E4M3 codes of k' / s with s = max|k'| / 448.  Writes the lane's four codes and (lane 0) the scale.
__device__ __forceinline__ void code_key_row(uint2 raw, int lane, uint8_t* codes_row, float* scale) {
    float x[4];
    bf16x4_to_float(raw, x);
    const float t0 = __fadd_rn(x[0], x[1]), t1 = __fsub_rn(x[0], x[1]);
    const float t2 = __fadd_rn(x[2], x[3]), t3 = __fsub_rn(x[2], x[3]);
    x[0] = __fadd_rn(t0, t2);
    x[1] = __fadd_rn(t1, t3);
    x[2] = __fsub_rn(t0, t2);
    x[3] = __fsub_rn(t1, t3);
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, x[i], m);
            x[i] = upper ? __fsub_rn(o, x[i]) : __fadd_rn(x[i], o);
        }
    }
    const float mx = warp_max(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
    const float s = __fdiv_rn(mx, 448.0f);
    float q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = s > 0.0f ? __fdiv_rn(x[i], s) : 0.0f;
    const uint32_t codes = e4m3x2(q[0], q[1]) | (e4m3x2(q[2], q[3]) << 16);
    *reinterpret_cast<uint32_t*>(codes_row + 4 * lane) = codes;
    if (lane == 0) *scale = s;
}

// Value row: INT8 codes round(v / s), s = max|v| / 127.  Writes the lane's four codes and (lane 0) the scale.
__device__ __forceinline__ void code_value_row(uint2 raw, int lane, int8_t* codes_row, float* scale) {
    float x[4];
    bf16x4_to_float(raw, x);
    const float mx = warp_max(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
    const float s = __fdiv_rn(mx, 127.0f);
    uint32_t codes = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c = s > 0.0f ? max(-127, min(127, __float2int_rn(__fdiv_rn(x[i], s)))) : 0;
        codes |= ((uint32_t)c & 0xFFu) << (8 * i);
    }
    *reinterpret_cast<uint32_t*>(codes_row + 4 * lane) = codes;
    if (lane == 0) *scale = s;
}

}  // namespace codec
}  // namespace va
