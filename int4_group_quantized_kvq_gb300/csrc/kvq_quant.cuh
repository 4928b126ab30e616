// kvq_quant.cuh -- the quantization of one row of fp16 values into INT4 codes and an fp16
// group scale, shared by the quantize-append kernel and the decode step's fused append, so
// both write the same bytes.
//
// "4-bit KV cache compression" (lpnh.cn/news/2042373), section 2.1: per group of G
// elements along head_dim, scale = amax / 7 (an all-zero group gets 1), code =
// round(x / scale) clamped to [-7, 7].  Here scale = fp16_rne(fp32(amax) / 7.0f), the
// zero test is on that fp16 value, and code = round_half_even(fp32(x) / fp32(scale)).
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

namespace kvq {

// round_half_even(fp32(x) / s) without a division per element.  x and s are fp16
// values (s > 0), so the quotient q = x / s is either exactly a half-integer or more
// than 2^-13 away from every half-integer: with x = X 2^a and s = S 2^b (integers
// X, S < 2048), q - (k + 1/2) = (2 X 2^(a-b) - (2k + 1) S) / (2 S), whose numerator is
// a nonzero multiple of min(1, 2^(a-b)), and 2^(a-b) > S / 4096 whenever |q| >= 1/2.
// The fp32 quotient the definition rounds is therefore on the same side of every
// half-integer as q.  y = x * rs, with rs within 2 ulp of 1/s, is within
// |q| (2^-22 + 2^-24) < 2^-17.6 of q for |q| < 16 (one reciprocal within 2 ulp, one
// rounded product; the quotient never reaches 16 for finite input: the fp16 scale is at least
// two thirds of amax / 7), so rounding y gives the same code unless y is within 2^-10
// of a half-integer h; there the sign of x - h s decides, with ties to even.  One fma
// rounds the exact x - h s once, which keeps its sign and its exact zeros.
__device__ __forceinline__ int exact_code(float x, float s, float y) {
    const float h = floorf(y) + 0.5f;    // the half-integer next to y (when y is near one)
    const float r = fmaf(-h, s, x);      // sign of x - h s, exact
    const int lo = __float2int_rd(h);
    return r > 0.f ? lo + 1 : (r < 0.f ? lo : lo + (lo & 1));
}

// The 8 codes of one lane as nibbles (code + 8, low nibble first) of a 32-bit word.
__device__ __forceinline__ uint32_t quant8(const float (&x)[8], float s, bool plain) {
    int c[8];
    if (plain) {
        // an infinite scale or a NaN input: the plain conversion of the IEEE quotient
        // (a NaN quotient converts to 0)
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = __float2int_rn(__fdiv_rn(x[i], s));
    } else {
        float rs;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rs) : "f"(s));
        constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: adding it rounds to an integer, ties to even
        bool near = false;
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            y[i] = x[i] * rs;
            const float m = y[i] + kMagic;
            c[i] = __float_as_int(m) - 0x4B400000;
            near |= fabsf(y[i] - (m - kMagic)) > 0.4990234375f;
        }
        if (near) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (fabsf(y[i] - rintf(y[i])) > 0.4990234375f) c[i] = exact_code(x[i], s, y[i]);
        }
    }
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) word |= static_cast<uint32_t>(max(-7, min(7, c[i])) + 8) << (4 * i);
    return word;
}

// A row of D values held as 8 values per lane by LPR = D / 8 consecutive lanes (lane tl
// holds values 8 tl .. 8 tl + 7); groups are 8 << lg values, i.e. 1 << lg lanes.  Returns
// the lane's 8 codes as a word of nibbles and the fp16 scale of its group.  Every lane of
// the warp calls this together: the group maximum is a shuffle reduction, and lanes of
// teams with other group widths run the same shuffles, folding in only partners inside
// their own group.
template <int LPR>
__device__ __forceinline__ uint32_t quant_lane8(uint4 raw, int lg, __half& scale_out) {
    float x[8];
    {
        const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(h2[i]);
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int off = 1; off < LPR; off <<= 1) {
        const float other = __shfl_xor_sync(0xffffffffu, amax, off);
        if (off < (1 << lg)) amax = fmaxf(amax, other);
    }
    __half s16 = __float2half_rn(__fdiv_rn(amax, 7.0f));
    if ((__half_as_ushort(s16) & 0x7fffu) == 0) s16 = __ushort_as_half(0x3c00u);
    const float s = __half2float(s16);
    bool nan = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) nan |= x[i] != x[i];
    scale_out = s16;
    return quant8(x, s, nan || isinf(s));
}

}  // namespace kvq
