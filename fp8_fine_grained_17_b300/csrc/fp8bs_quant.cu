// Activation (1x128 tile) and weight (128x128 block) quantizers: bf16 ->
// E4M3 codes + binary32 dequantization scales.
//
// Grouping follows "personal notes concerning the deepseek core readings"
// (why-be.why-be.co.kr), fine-grained quantization paragraph, Figure 7(a);
// amax-to-FP8-maximum scaling and online quantization follow the Q&A post on
// xn--9g3bo1gtkw0l8ubf92bgle.kr, mixed-precision paragraph.
//
// Exactness. The stored scale is s = amax / 448 (IEEE division) and each code
// is E4M3(round_f32(x / s)). A full-precision division per element would cost
// more than the memory traffic, so the quotient is formed from the correctly
// rounded reciprocal r = 1/s and one residual correction (Markstein's method:
// y0 = x*r, e = fma(-y0, s, x), y = fma(e, r, y0)), which yields the
// correctly rounded quotient whenever no intermediate underflows. Where the
// quotient is tiny enough for the residual to underflow the E4M3 code is 0
// either way, except for the sign of zero, which is restored from x. Groups
// with amax below 2^-100 (s near the binary32 subnormal range) take a true
// IEEE division per element instead. This is checked against the
// definition over every (bf16 amax, bf16 x) pair by the tests.
#include <cstdint>

#include "fp8bs_device.cuh"
#include "fp8bs_host.h"

namespace fp8bs {
namespace {

constexpr float kE4M3Max = 448.0f;
constexpr float kFastDivMinAmax = 0x1p-100f;

struct GroupDivider {
    float s;
    float r;
    bool fast;
};

__device__ __forceinline__ GroupDivider make_divider(float amax)
{
    GroupDivider d;
    d.s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, kE4M3Max);
    d.r = __frcp_rn(d.s);
    d.fast = amax >= kFastDivMinAmax;
    return d;
}

// round_f32(x / s), see the file comment.
__device__ __forceinline__ float divide(float x, const GroupDivider& d)
{
    if (d.fast) {
        const float y0 = __fmul_rn(x, d.r);
        const float e = __fmaf_rn(-y0, d.s, x);
        return copysignf(__fmaf_rn(e, d.r, y0), x);
    }
    return __fdiv_rn(x, d.s);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float absmax_pair(float m, uint32_t w)
{
    return fmaxf(m, fmaxf(fabsf(bf16_lo(w)), fabsf(bf16_hi(w))));
}

// 8 bf16 (one uint4) -> 8 E4M3 codes (one uint2).
__device__ __forceinline__ uint2 quantize8(const uint4& v, const GroupDivider& d)
{
    const uint32_t c0 = cvt_e4m3x2(divide(bf16_lo(v.x), d), divide(bf16_hi(v.x), d));
    const uint32_t c1 = cvt_e4m3x2(divide(bf16_lo(v.y), d), divide(bf16_hi(v.y), d));
    const uint32_t c2 = cvt_e4m3x2(divide(bf16_lo(v.z), d), divide(bf16_hi(v.z), d));
    const uint32_t c3 = cvt_e4m3x2(divide(bf16_lo(v.w), d), divide(bf16_hi(v.w), d));
    return make_uint2(c0 | (c1 << 16), c2 | (c3 << 16));
}

__device__ __forceinline__ float absmax8(float m, const uint4& v)
{
    m = absmax_pair(m, v.x);
    m = absmax_pair(m, v.y);
    m = absmax_pair(m, v.z);
    return absmax_pair(m, v.w);
}

// ---------------------------------------------------------------------------
// Activation quantizer.
//
// Four consecutive lanes own one 1x128 group (256 bytes of bf16): lane
// quarter t loads the 16-byte chunks t, t+4, t+8, t+12 of the group, so one
// warp-wide load instruction touches 8 groups x 64 contiguous bytes, i.e.
// whole 32-byte sectors. The group amax is combined with two xor-shuffles.
// A warp handles kUnroll x 8 groups per iteration of a grid-stride loop;
// all loads of an iteration are issued before any arithmetic.
// ---------------------------------------------------------------------------
constexpr int kActThreads = 256;
constexpr int kActUnroll = 2;

__global__ void __launch_bounds__(kActThreads)
quantize_act_kernel(const uint16_t* __restrict__ x, int64_t ldx, uint8_t* __restrict__ q,
                    int64_t ldq, float* __restrict__ scale, int64_t groups_per_row,
                    int64_t total_groups)
{
    const int lane = threadIdx.x & 31;
    const int quarter = lane & 3;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kActThreads + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * kActThreads) >> 5;
    const int64_t per_iter = 8 * kActUnroll;

    for (int64_t base = warp * per_iter; base < total_groups; base += n_warps * per_iter) {
        uint4 v[kActUnroll][4];
        int64_t row[kActUnroll], col[kActUnroll];
        bool valid[kActUnroll];
#pragma unroll
        for (int u = 0; u < kActUnroll; ++u) {
            const int64_t grp = base + u * 8 + (lane >> 2);
            valid[u] = grp < total_groups;
            row[u] = valid[u] ? grp / groups_per_row : 0;
            col[u] = valid[u] ? (grp - row[u] * groups_per_row) * 128 : 0;
            const uint4* src = reinterpret_cast<const uint4*>(x + row[u] * ldx + col[u]) + quarter;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                v[u][j] = valid[u] ? __ldcs(src + 4 * j) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kActUnroll; ++u) {
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                amax = absmax8(amax, v[u][j]);
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
            const GroupDivider d = make_divider(amax);
            if (valid[u]) {
                uint8_t* dst = q + row[u] * ldq + col[u] + quarter * 8;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<uint2*>(dst + 32 * j) = quantize8(v[u][j], d);
                if (quarter == 0)
                    scale[row[u] * groups_per_row + col[u] / 128] = d.s;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Weight quantizer: one 256-thread CTA per 128x128 block. Thread t holds the
// 16-byte chunk (t & 15) of rows 16i + t/16, i = 0..7, so each warp load
// instruction covers two whole 256-byte block rows. The block amax is reduced
// with shuffles and through shared memory; the codes are written from the
// registers that still hold the inputs.
// ---------------------------------------------------------------------------
constexpr int kWThreads = 256;

__global__ void __launch_bounds__(kWThreads)
quantize_weight_kernel(const uint16_t* __restrict__ w, int64_t N, int64_t ldw,
                       uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ scale,
                       int64_t groups_per_row)
{
    __shared__ float warp_max[kWThreads / 32];
    const int t = threadIdx.x;
    const int64_t kb = blockIdx.x;
    const int64_t nb = blockIdx.y;
    const int chunk = t & 15;
    const int64_t col = kb * 128 + chunk * 8;

    uint4 v[8];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t n = nb * 128 + i * 16 + (t >> 4);
        v[i] = n < N ? __ldcs(reinterpret_cast<const uint4*>(w + n * ldw + col))
                     : make_uint4(0, 0, 0, 0);
        amax = absmax8(amax, v[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((t & 31) == 0)
        warp_max[t >> 5] = amax;
    __syncthreads();
    amax = warp_max[0];
#pragma unroll
    for (int i = 1; i < kWThreads / 32; ++i)
        amax = fmaxf(amax, warp_max[i]);

    const GroupDivider d = make_divider(amax);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t n = nb * 128 + i * 16 + (t >> 4);
        if (n < N)
            *reinterpret_cast<uint2*>(q + n * ldq + col) = quantize8(v[i], d);
    }
    if (t == 0)
        scale[nb * groups_per_row + kb] = d.s;
}

int act_grid(const DeviceInfo& info, int64_t total_groups)
{
    static int blocks_per_sm = 0;
    if (blocks_per_sm == 0) {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, quantize_act_kernel, kActThreads, 0) !=
                cudaSuccess ||
            b <= 0) {
            cudaGetLastError();
            b = 4;
        }
        blocks_per_sm = b;
    }
    const int64_t groups_per_block = (kActThreads / 32) * 8 * kActUnroll;
    const int64_t needed = (total_groups + groups_per_block - 1) / groups_per_block;
    const int64_t full = static_cast<int64_t>(info.sm_count) * blocks_per_sm;
    return static_cast<int>(needed < full ? needed : full);
}

}  // namespace
}  // namespace fp8bs

using namespace fp8bs;

extern "C" fp8bs_status fp8bs_quantize_act_1x128(const void* x, int64_t M, int64_t K, int64_t ldx,
                                                 uint8_t* q, int64_t ldq, float* scale,
                                                 fp8bs_stream_t stream)
{
    if (M < 0 || K < 0)
        return FP8BS_ERR_INVALID_ARG;
    if (K % 128 != 0)
        return FP8BS_ERR_UNSUPPORTED;
    if (M == 0 || K == 0)
        return FP8BS_OK;
    if (x == nullptr || q == nullptr || scale == nullptr)
        return FP8BS_ERR_INVALID_ARG;
    if (ldx < K || ldq < K || (ldx * 2) % 16 != 0 || ldq % 16 != 0)
        return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q) || (reinterpret_cast<uintptr_t>(scale) & 3u) != 0)
        return FP8BS_ERR_INVALID_ARG;
    DeviceInfo info;
    const fp8bs_status st = require_sm103(&info);
    if (st != FP8BS_OK)
        return st;

    const int64_t G = K / 128;
    const int64_t total = M * G;
    const int grid = act_grid(info, total);
    quantize_act_kernel<<<grid, kActThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(x), ldx, q, ldq, scale, G, total);
    return launch_status();
}

extern "C" fp8bs_status fp8bs_quantize_weight_128x128(const void* w, int64_t N, int64_t K,
                                                      int64_t ldw, uint8_t* q, int64_t ldq,
                                                      float* scale, fp8bs_stream_t stream)
{
    if (N < 0 || K < 0)
        return FP8BS_ERR_INVALID_ARG;
    if (K % 128 != 0)
        return FP8BS_ERR_UNSUPPORTED;
    if (N == 0 || K == 0)
        return FP8BS_OK;
    if (w == nullptr || q == nullptr || scale == nullptr)
        return FP8BS_ERR_INVALID_ARG;
    if (ldw < K || ldq < K || (ldw * 2) % 16 != 0 || ldq % 16 != 0)
        return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(q) || (reinterpret_cast<uintptr_t>(scale) & 3u) != 0)
        return FP8BS_ERR_INVALID_ARG;
    const int64_t NB = (N + 127) / 128;
    const int64_t G = K / 128;
    if (NB > 65535 || G > 0x7FFFFFFF)
        return FP8BS_ERR_UNSUPPORTED;
    DeviceInfo info;
    const fp8bs_status st = require_sm103(&info);
    if (st != FP8BS_OK)
        return st;

    const dim3 grid(static_cast<unsigned>(G), static_cast<unsigned>(NB));
    quantize_weight_kernel<<<grid, kWThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(w), N, ldw, q, ldq, scale, G);
    return launch_status();
}
