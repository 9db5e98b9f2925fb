// Normalization fused with the 1x128 activation cast: RMSNorm or LayerNorm of
// each bf16 row, the result rounded to bf16, then quantized exactly as
// fp8bs_quantize_act_1x128 quantizes a bf16 tensor (same per-group codec).
//
// "How I Improved My Deepseek In In The Future", paragraph of hardware
// suggestions: a warp-level cast instruction would allow layer normalization
// and the FP8 cast to be fused. Here the fusion is done in software: the
// normalized row never goes to memory; it is computed, rounded to bf16 and
// cast in registers, so the kernel reads the bf16 input once and writes only
// codes, scales and the row statistics.
//
// Arithmetic, per row (binary32, each step one IEEE operation rounded to
// nearest, none contracted into a fused multiply-add):
//   RMSNorm:   v = sum(x^2) / K
//   LayerNorm: mu = sum(x) / K,  v = sum((x - mu)^2) / K
//   rstd = 1/sqrt(v + eps) (correctly rounded)
//   y = bf16_rne(((x - mu) * rstd) * gamma + beta)   (mu = 0 for RMSNorm,
//       the addition only when beta is given)
// The sums are formed in lane-parallel order (each lane accumulates its
// elements, then a butterfly across lanes and, for long rows, across warps),
// so they may differ from a sequential sum by a few units in the last place;
// everything after the statistics is order-free.
//
// Work split: a CTA of 4 warps (K <= 8192) or 8 warps (K <= 65536) holds one
// row in registers at a time, in a grid-stride loop over rows. Thread t of
// the CTA holds the 16-byte chunks c = j * threads + t, so each warp load
// instruction covers 512 contiguous bytes and a 1x128 group (16 chunks) lies
// in one half-warp. Several CTAs per SM keep enough rows in flight to cover
// the memory latency.
#include <cstdint>

#include "fp8bs_device.cuh"
#include "fp8bs_e4m3.cuh"
#include "fp8bs_host.h"

namespace fp8bs {
namespace {

// Sum of v over the row's threads: butterfly across each warp (every lane
// ends with the same value), then the warps' sums in warp order through
// shared memory (every thread reads the same values in the same order).
template <int kWarps>
__device__ __forceinline__ float row_sum(float v, float* red)
{
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, m);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = v;
    __syncthreads();
    v = red[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i)
        v += red[i];
    __syncthreads();
    return v;
}

__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w)
{
    return pack_b32x2(w << 16, w & 0xFFFF0000u);
}

template <int kWarps, int kJ>
__global__ void __launch_bounds__(32 * kWarps)
norm_quant_kernel(const uint16_t* __restrict__ x, int64_t ldx, const uint16_t* __restrict__ gamma,
                  const uint16_t* __restrict__ beta, int layer, float eps, int64_t M, int K,
                  uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ scale,
                  float* __restrict__ mean_out, float* __restrict__ rstd_out)
{
    constexpr int kThreads = 32 * kWarps;
    static_assert(kJ <= 32, "a lane computes the dividers of at most two groups");
    constexpr int kOwn = (kJ + 15) / 16;   // groups whose divider a lane computes
    __shared__ float red[kWarps];
    const int lane = threadIdx.x & 31;
    const int n_chunks = K >> 3;
    const int64_t G = K >> 7;
    const float k_f = static_cast<float>(K);

    for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
        const uint4* src = reinterpret_cast<const uint4*>(x + row * ldx);
        uint4 v[kJ];
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
            const int c = j * kThreads + threadIdx.x;
            v[j] = c < n_chunks ? __ldcs(src + c) : make_uint4(0, 0, 0, 0);
        }

        // Row statistics (two packed accumulators per sum to shorten the
        // dependency chains).
        float mu = 0.0f;
        uint64_t nmu2 = 0;
        if (layer) {
            const uint64_t one2 = pack_f32x2(1.0f, 1.0f);
            uint64_t acc[2] = {0, 0};
#pragma unroll
            for (int j = 0; j < kJ; ++j) {
                acc[j & 1] = fma_f32x2(bf16x2_to_f32x2(v[j].x), one2, acc[j & 1]);
                acc[j & 1] = fma_f32x2(bf16x2_to_f32x2(v[j].y), one2, acc[j & 1]);
                acc[j & 1] = fma_f32x2(bf16x2_to_f32x2(v[j].z), one2, acc[j & 1]);
                acc[j & 1] = fma_f32x2(bf16x2_to_f32x2(v[j].w), one2, acc[j & 1]);
            }
            const float2 a0 = unpack_f32x2(acc[0]), a1 = unpack_f32x2(acc[1]);
            mu = __fdiv_rn(row_sum<kWarps>((a0.x + a0.y) + (a1.x + a1.y), red), k_f);
            nmu2 = pack_f32x2(-mu, -mu);
        }
        uint64_t acc[2] = {0, 0};
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
            // Chunks past the row end hold zeros; centred they would add mu^2.
            if (j * kThreads + static_cast<int>(threadIdx.x) < n_chunks) {
                const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint64_t t = bf16x2_to_f32x2(w[i]);
                    if (layer)
                        t = add_f32x2(t, nmu2);
                    acc[i & 1] = fma_f32x2(t, t, acc[i & 1]);
                }
            }
        }
        const float2 a0 = unpack_f32x2(acc[0]), a1 = unpack_f32x2(acc[1]);
        const float var = __fdiv_rn(row_sum<kWarps>((a0.x + a0.y) + (a1.x + a1.y), red), k_f);
        const float rstd = __frsqrt_rn(__fadd_rn(var, eps));
        if (threadIdx.x == 0) {
            if (rstd_out != nullptr)
                rstd_out[row] = rstd;
            if (mean_out != nullptr && layer)
                mean_out[row] = mu;
        }

        // Normalize, round to bf16 (kept in v), and take each group's amax
        // (a max-butterfly over the half-warp that holds the group).
        const uint64_t rstd2 = pack_f32x2(rstd, rstd);
        uint32_t own_amax[kOwn];
#pragma unroll
        for (int i = 0; i < kOwn; ++i)
            own_amax[i] = 0;
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
            // gamma and beta are read per row; after the first row they come
            // from L1 (the same 2K bytes for every row of the SM's CTAs).
            const int c = j * kThreads + threadIdx.x;
            const bool ok = c < n_chunks;
            const uint4 g4 = ok ? __ldg(reinterpret_cast<const uint4*>(gamma) + c) : make_uint4(0, 0, 0, 0);
            const uint4 b4 = (ok && beta != nullptr) ? __ldg(reinterpret_cast<const uint4*>(beta) + c)
                                                     : make_uint4(0, 0, 0, 0);
            uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
            const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w};
            const uint32_t bw[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint64_t t = bf16x2_to_f32x2(w[i]);
                if (layer)
                    t = add_f32x2(t, nmu2);
                t = mul_f32x2(t, rstd2);
                t = mul_f32x2(t, bf16x2_to_f32x2(gw[i]));
                if (beta != nullptr) {
                    // Scalar adds: the compiler may fuse a packed multiply
                    // and a packed add into one rounding (measured on
                    // B300); __fadd_rn is never contracted.
                    const float2 u = unpack_f32x2(t);
                    t = pack_f32x2(__fadd_rn(u.x, __uint_as_float(bw[i] << 16)),
                                   __fadd_rn(u.y, __uint_as_float(bw[i] & 0xFFFF0000u)));
                }
                w[i] = cvt_bf16x2(t);
            }
            v[j] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        uint32_t m[kJ];
#pragma unroll
        for (int j = 0; j < kJ; ++j)
            m[j] = absmax_words(&v[j], 1);
#pragma unroll
        for (int s = 8; s >= 1; s >>= 1) {
#pragma unroll
            for (int j = 0; j < kJ; ++j)
                m[j] = max(m[j], __shfl_xor_sync(0xFFFFFFFFu, m[j], s));
        }
#pragma unroll
        for (int j = 0; j < kJ; ++j)
            if ((j & 15) == (lane & 15))
                own_amax[j >> 4] = m[j];

        // Lane l computes the dividers of the groups j = l mod 16 of its
        // half-warp and writes their scales; the half-warp shares them.
        Divider own[kOwn];
        bool fast = true;
#pragma unroll
        for (int i = 0; i < kOwn; ++i) {
            own[i] = make_divider(bf16_bits_to_f32(own_amax[i]));
            fast = fast && own[i].r != 0.0f;
        }
        fast = __all_sync(0xFFFFFFFFu, fast);
        uint8_t* qrow = q + row * ldq;
        float* srow = scale + row * G;
        auto emit = [&](auto quant) {
#pragma unroll
            for (int j = 0; j < kJ; ++j) {
                const int src_lane = (lane & 16) | (j & 15);
                Divider d;
                d.s = __shfl_sync(0xFFFFFFFFu, own[j >> 4].s, src_lane);
                d.r = __shfl_sync(0xFFFFFFFFu, own[j >> 4].r, src_lane);
                const int c = j * kThreads + threadIdx.x;
                if (c < n_chunks) {
                    if ((lane & 15) == (j & 15))
                        srow[c >> 4] = d.s;
                    __stcs(reinterpret_cast<uint2*>(qrow + 8 * static_cast<int64_t>(c)), quant(v[j], d));
                }
            }
        };
        if (fast)
            emit([](const uint4& a, const Divider& d) { return quantize8_fast(a, d); });
        else
            emit([](const uint4& a, const Divider& d) { return quantize8(a, d); });
    }
}

template <int kWarps, int kJ>
fp8bs_status launch_norm(const DeviceInfo& info, const uint16_t* x, int64_t ldx, const uint16_t* gamma,
                         const uint16_t* beta, int layer, float eps, int64_t M, int K, uint8_t* q,
                         int64_t ldq, float* scale, float* mean, float* rstd, cudaStream_t stream)
{
    constexpr int kThreads = 32 * kWarps;
    static int per_sm[64] = {};
    if (info.device < 0 || info.device >= 64)
        return FP8BS_ERR_CUDA;
    if (per_sm[info.device] == 0) {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, norm_quant_kernel<kWarps, kJ>, kThreads, 0) !=
                cudaSuccess || b <= 0) {
            cudaGetLastError();
            b = 1;
        }
        per_sm[info.device] = b;
    }
    const int64_t full = static_cast<int64_t>(info.sm_count) * per_sm[info.device];
    const int grid = static_cast<int>(M < full ? M : full);
    norm_quant_kernel<kWarps, kJ><<<grid, kThreads, 0, stream>>>(x, ldx, gamma, beta, layer, eps, M, K, q,
                                                                 ldq, scale, mean, rstd);
    return launch_status();
}

}  // namespace
}  // namespace fp8bs

using namespace fp8bs;

extern "C" fp8bs_status fp8bs_norm_quantize_act_1x128(const void* x, int64_t M, int64_t K, int64_t ldx,
                                                      const void* gamma, const void* beta,
                                                      fp8bs_norm_kind kind, float eps, uint8_t* q,
                                                      int64_t ldq, float* scale, float* mean,
                                                      float* rstd, fp8bs_stream_t stream)
{
    if (M < 0 || K < 0)
        return FP8BS_ERR_INVALID_ARG;
    if (kind != FP8BS_NORM_RMS && kind != FP8BS_NORM_LAYER)
        return FP8BS_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || eps == __builtin_inff())
        return FP8BS_ERR_INVALID_ARG;
    if (K % 128 != 0)
        return FP8BS_ERR_UNSUPPORTED;
    if (K > 65536)
        return FP8BS_ERR_UNSUPPORTED;
    if (M == 0)
        return FP8BS_OK;
    if (K == 0)
        return FP8BS_ERR_INVALID_ARG;   // the statistics of an empty row are undefined
    if (x == nullptr || gamma == nullptr || q == nullptr || scale == nullptr)
        return FP8BS_ERR_INVALID_ARG;
    if (ldx < K || ldq < K || (ldx * 2) % 16 != 0 || ldq % 16 != 0)
        return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(gamma) || (beta != nullptr && !aligned16(beta)) || !aligned16(q))
        return FP8BS_ERR_INVALID_ARG;
    const uintptr_t f_bits = reinterpret_cast<uintptr_t>(scale) | reinterpret_cast<uintptr_t>(mean) |
                             reinterpret_cast<uintptr_t>(rstd);
    if ((f_bits & 3u) != 0)
        return FP8BS_ERR_INVALID_ARG;
    DeviceInfo info;
    const fp8bs_status st = require_sm103(&info);
    if (st != FP8BS_OK)
        return st;

    const uint16_t* xb = static_cast<const uint16_t*>(x);
    const uint16_t* gb = static_cast<const uint16_t*>(gamma);
    const uint16_t* bb = static_cast<const uint16_t*>(beta);
    const int layer = kind == FP8BS_NORM_LAYER;
    const int k = static_cast<int>(K);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
#define FP8BS_NORM_LAUNCH(W, J) \
    launch_norm<W, J>(info, xb, ldx, gb, bb, layer, eps, M, k, q, ldq, scale, mean, rstd, s)
    // Chunks per thread: K / 8 / threads, rounded up to an instantiated count.
    if (K <= 1024)
        return FP8BS_NORM_LAUNCH(4, 1);
    if (K <= 2048)
        return FP8BS_NORM_LAUNCH(4, 2);
    if (K <= 4096)
        return FP8BS_NORM_LAUNCH(4, 4);
    if (K <= 7168)
        return FP8BS_NORM_LAUNCH(4, 7);
    if (K <= 8192)
        return FP8BS_NORM_LAUNCH(4, 8);
    if (K <= 16384)
        return FP8BS_NORM_LAUNCH(8, 8);
    if (K <= 32768)
        return FP8BS_NORM_LAUNCH(8, 16);
    return FP8BS_NORM_LAUNCH(8, 32);
#undef FP8BS_NORM_LAUNCH
}
