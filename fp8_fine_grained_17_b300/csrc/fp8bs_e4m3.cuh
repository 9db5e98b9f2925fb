// E4M3 group codec shared by every kernel that writes 1x128 or 128x128
// quantized groups: the group scale s = amax / 448 (s = 1 for an all-zero
// group), its reciprocal, and the code of each bf16 value, E4M3(round(x / s))
// with round-to-nearest-even and saturation to +-448.
//
// Exactness. The stored scale is s = amax / 448 (IEEE division) and each code
// is E4M3(round_f32(x / s)). A full-precision division per element would cost
// more than the memory traffic, so the quotient is formed from the correctly
// rounded reciprocal r = 1/s and one residual correction (Markstein's method:
// y0 = x*r, e = x - y0*s (fused), y = e*r + y0 (fused)), which yields the
// correctly rounded quotient whenever no intermediate underflows. Where the
// quotient is tiny enough for the residual to underflow, its E4M3 code is 0
// either way; only the sign of zero can come out wrong (x = -0 gives +0), so
// every code's sign bit is OR-ed with the sign bit of x, which is the sign
// the exact quotient has. Groups with 0 < amax < 2^-100 (s near the binary32
// subnormal range) take a true IEEE division per element instead. The tests
// check this against the definition over every (bf16 amax, bf16 x) pair.
//
// The per-element arithmetic runs on packed pairs (sm_100+ binary32x2 mul /
// fma, bf16x2 magnitude max), and the per-group scalar work (amax/448 and its
// reciprocal) is done once per group, spread over the lanes that share it.
#pragma once

#include <cstdint>

#include "fp8bs_device.cuh"

namespace fp8bs {

constexpr float kE4M3Max = 448.0f;
constexpr float kFastDivMinAmax = 0x1p-100f;

// Scale of a group and the reciprocal used by the fast quotient; r == 0
// selects the exact-division path.
struct Divider {
    float s;
    float r;
};

__device__ __forceinline__ Divider make_divider(float amax)
{
    Divider d;
    d.s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, kE4M3Max);
    d.r = (amax == 0.0f || amax >= kFastDivMinAmax) ? __frcp_rn(d.s) : 0.0f;
    return d;
}

// Power-of-two scale mode (the scales Blackwell's UE8M0 formats hold): s = 2^e
// for the smallest e in [-127, 127] with amax / 2^e <= 448, taken exactly from
// the bf16 pattern of amax (448 = 1.75 * 2^8, so e = E - 135 for a mantissa
// <= 1.75 and E - 134 above it, E the biased exponent); s = 1 for amax = 0.
// r = 2^-e exactly, so the fast quotient x * r is the exact (or, in the
// binary32 subnormal range, correctly rounded) x / s.
__device__ __forceinline__ Divider make_divider_pow2(uint32_t amax_bits)
{
    Divider d;
    if (amax_bits == 0) {
        d.s = 1.0f;
        d.r = 1.0f;
        return d;
    }
    const int eb = static_cast<int>((amax_bits >> 7) & 0xFFu);
    const int mant = static_cast<int>(amax_bits & 0x7Fu);
    int e = eb == 0 ? -127 : eb - 135 + (mant > 96 ? 1 : 0);
    e = max(e, -127);
    d.s = e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23)
                    : __uint_as_float(0x00400000u);   // 2^-127 (subnormal)
    d.r = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    return d;
}

// Scale and reciprocal of a group from the bf16 pattern of its amax.
__device__ __forceinline__ Divider group_divider(uint32_t amax_bits, int pow2)
{
    return pow2 ? make_divider_pow2(amax_bits) : make_divider(__uint_as_float(amax_bits << 16));
}

// Largest |x| of a bf16 group fragment held as packed words, as the 16-bit
// pattern of a non-negative bf16 (integer order = numeric order).
__device__ __forceinline__ uint32_t absmax_words(const uint4* v, int n)
{
    uint32_t m = 0;
    for (int j = 0; j < n; ++j)
        m = absmax_bf16x2(m, absmax_bf16x2(absmax_bf16x2(v[j].x, v[j].y),
                                           absmax_bf16x2(v[j].z, v[j].w)));
    m &= 0x7FFF7FFFu;
    return max(m & 0xFFFFu, m >> 16);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// Sign bits of the 4 bf16 values in (w0, w1), placed on the sign bits of 4
// E4M3 bytes.
__device__ __forceinline__ uint32_t sign_bytes(uint32_t w0, uint32_t w1)
{
    return __byte_perm(w0, w1, 0x7531) & 0x80808080u;
}

// 2 bf16 (one word) -> 2 E4M3 codes in the low 16 bits, fast quotient.
__device__ __forceinline__ uint32_t quantize2_fast(uint32_t w, uint64_t ns2, uint64_t r2)
{
    const uint64_t x = pack_b32x2(w << 16, w & 0xFFFF0000u);
    const uint64_t y0 = mul_f32x2(x, r2);
    const uint64_t e = fma_f32x2(y0, ns2, x);     // x - y0 * s
    const float2 y = unpack_f32x2(fma_f32x2(e, r2, y0));
    return cvt_e4m3x2(y.x, y.y);
}

// Same with a true IEEE division per element.
__device__ __forceinline__ uint32_t quantize2_exact(uint32_t w, float s)
{
    return cvt_e4m3x2(__fdiv_rn(__uint_as_float(w << 16), s),
                      __fdiv_rn(__uint_as_float(w & 0xFFFF0000u), s));
}

// quantize2_fast with the bf16 pair widened on the FP32 pipe (same result).
__device__ __forceinline__ uint32_t quantize2_fast_fp(uint32_t w, uint64_t ns2, uint64_t r2)
{
    const uint64_t x = bf16x2_add_f32(w, -0.0f);
    const uint64_t y0 = mul_f32x2(x, r2);
    const uint64_t e = fma_f32x2(y0, ns2, x);     // x - y0 * s
    const float2 y = unpack_f32x2(fma_f32x2(e, r2, y0));
    return cvt_e4m3x2(y.x, y.y);
}

// 8 bf16 (one uint4) -> 8 E4M3 codes (one uint2), fast quotient only (the
// caller has checked d.r != 0), widening on the FP32 pipe.
__device__ __forceinline__ uint2 quantize8_fast_fp(const uint4& v, const Divider& d)
{
    const uint64_t ns2 = pack_f32x2(-d.s, -d.s);
    const uint64_t r2 = pack_f32x2(d.r, d.r);
    const uint32_t c0 = quantize2_fast_fp(v.x, ns2, r2);
    const uint32_t c1 = quantize2_fast_fp(v.y, ns2, r2);
    const uint32_t c2 = quantize2_fast_fp(v.z, ns2, r2);
    const uint32_t c3 = quantize2_fast_fp(v.w, ns2, r2);
    return make_uint2(__byte_perm(c0, c1, 0x5410) | sign_bytes(v.x, v.y),
                      __byte_perm(c2, c3, 0x5410) | sign_bytes(v.z, v.w));
}

// 8 bf16 (one uint4) -> 8 E4M3 codes (one uint2), fast quotient only (the
// caller has checked d.r != 0).
__device__ __forceinline__ uint2 quantize8_fast(const uint4& v, const Divider& d)
{
    const uint64_t ns2 = pack_f32x2(-d.s, -d.s);
    const uint64_t r2 = pack_f32x2(d.r, d.r);
    const uint32_t c0 = quantize2_fast(v.x, ns2, r2);
    const uint32_t c1 = quantize2_fast(v.y, ns2, r2);
    const uint32_t c2 = quantize2_fast(v.z, ns2, r2);
    const uint32_t c3 = quantize2_fast(v.w, ns2, r2);
    return make_uint2(__byte_perm(c0, c1, 0x5410) | sign_bytes(v.x, v.y),
                      __byte_perm(c2, c3, 0x5410) | sign_bytes(v.z, v.w));
}

// 8 bf16 (one uint4) -> 8 E4M3 codes (one uint2).
__device__ __forceinline__ uint2 quantize8(const uint4& v, const Divider& d)
{
    if (d.r != 0.0f)
        return quantize8_fast(v, d);
    const uint32_t c0 = quantize2_exact(v.x, d.s);
    const uint32_t c1 = quantize2_exact(v.y, d.s);
    const uint32_t c2 = quantize2_exact(v.z, d.s);
    const uint32_t c3 = quantize2_exact(v.w, d.s);
    return make_uint2(__byte_perm(c0, c1, 0x5410) | sign_bytes(v.x, v.y),
                      __byte_perm(c2, c3, 0x5410) | sign_bytes(v.z, v.w));
}

}  // namespace fp8bs
