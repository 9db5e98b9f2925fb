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
// Arithmetic, per row (binary32):
//   RMSNorm:   v = sum(x^2) / K
//   LayerNorm: mu = sum(x) / K,  v = sum((x - mu)^2) / K
//   rstd = 1/sqrt(v + eps) (correctly rounded)
//   y = bf16_rne(((x - mu) * rstd) * gamma + beta)   (mu = 0 for RMSNorm,
//       the addition only when beta is given)
// The statistics are sums accumulated with fused multiply-adds (each square
// or centred square added to its lane's accumulator in one rounding) in
// lane-parallel order (each lane accumulates its elements, then a butterfly
// across lanes and, for long rows, across warps), so they may differ from a
// sequentially, separately rounded sum by a few units in the last place.
// Everything after the statistics is one IEEE operation per step, rounded
// to nearest, none contracted into a fused multiply-add, and order-free.
//
// Work split: a CTA holds one row in registers at a time, in a grid-stride
// loop over rows. Thread t of the CTA holds the 16-byte chunks
// c = j * threads + t, so each warp covers 512 contiguous bytes per j and a
// 1x128 group (16 chunks) lies in one half-warp.
#include <atomic>
#include <cstdint>
#include <mutex>

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

// The work on one row once its chunks are in registers (v): statistics,
// normalization to bf16, group amax, dividers, codes and scales.
template <int kWarps, int kJ>
__device__ __forceinline__ void norm_row(uint4 (&v)[kJ], int64_t row, const uint16_t* __restrict__ gamma,
                                         const uint16_t* __restrict__ beta, int layer, float eps, int K,
                                         uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ scale,
                                         float* __restrict__ mean_out, float* __restrict__ rstd_out,
                                         float* red)
{
    constexpr int kThreads = 32 * kWarps;
    static_assert(kJ <= 32, "a lane computes the dividers of at most two groups");
    constexpr int kOwn = (kJ + 15) / 16;   // groups whose divider a lane computes
    const int lane = threadIdx.x & 31;
    const int n_chunks = K >> 3;
    const int64_t G = K >> 7;
    const float k_f = static_cast<float>(K);

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

// Register path: each row is loaded straight into registers (rows of up to
// 65536 elements).
template <int kWarps, int kJ>
__global__ void __launch_bounds__(32 * kWarps)
norm_quant_kernel(const uint16_t* __restrict__ x, int64_t ldx, const uint16_t* __restrict__ gamma,
                  const uint16_t* __restrict__ beta, int layer, float eps, int64_t M, int K,
                  uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ scale,
                  float* __restrict__ mean_out, float* __restrict__ rstd_out)
{
    constexpr int kThreads = 32 * kWarps;
    __shared__ float red[kWarps];
    const int n_chunks = K >> 3;
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
        const uint4* src = reinterpret_cast<const uint4*>(x + row * ldx);
        uint4 v[kJ];
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
            const int c = j * kThreads + threadIdx.x;
            v[j] = c < n_chunks ? __ldcs(src + c) : make_uint4(0, 0, 0, 0);
        }
        norm_row<kWarps, kJ>(v, row, gamma, beta, layer, eps, K, q, ldq, scale, mean_out, rstd_out, red);
    }
}

// Main path (rows of up to 16384 elements): one warp per row, no CTA-wide
// barrier on the row path. The row is read in passes over batches of kB
// chunks per lane (lane l holds chunks c = 32 i + l): LayerNorm's mean, the
// sum of squares, and the output. The first pass brings the row into L2 (and
// L1), so the later passes re-read it from the caches. gamma (and beta) are
// converted to binary32 once per CTA into shared memory, split into the low
// and high halves of each chunk so that a warp's reads are contiguous.
constexpr int kWarpRowsPerCta = 8;
constexpr int kWarpBatch = 4;

template <int kB, bool kFull>
__device__ __forceinline__ void load_batch(uint4 (&v)[kB], const uint4* src, int i0, int lane, int n_chunks,
                                           bool last_use)
{
#pragma unroll
    for (int b = 0; b < kB; ++b) {
        const int c = (i0 + b) * 32 + lane;
        if (kFull || c < n_chunks)
            v[b] = last_use ? __ldcs(src + c) : __ldg(src + c);
        else
            v[b] = make_uint4(0, 0, 0, 0);
    }
}

// kIters > 0: rows of exactly kIters batches (K = 1024 kIters), known at
// compile time: no partial batch, no per-chunk bounds test, fixed trip counts.
// kLayer / kBeta: -1 = taken from the arguments at run time; 0 or 1 = fixed
// at compile time (LayerNorm or RMSNorm; beta present or not).
template <int kIters, int kLayer, int kBeta>
__device__ __forceinline__ void norm_warp_rows(const uint16_t* __restrict__ x, int64_t ldx,
                                               const uint16_t* __restrict__ gamma,
                                               const uint16_t* __restrict__ beta, int layer_arg, float eps,
                                               int64_t M, int K, uint8_t* __restrict__ q, int64_t ldq,
                                               float* __restrict__ scale, float* __restrict__ mean_out,
                                               float* __restrict__ rstd_out)
{
    constexpr int kB = kWarpBatch;
    constexpr bool kFull = kIters > 0;
    extern __shared__ __align__(16) float4 wsm[];   // [gamma lo | gamma hi | beta lo | beta hi] x n_chunks
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int n_chunks = K >> 3;
    const int n_iter = kFull ? kIters : (n_chunks + 32 * kB - 1) / (32 * kB);   // batches per pass
    const int64_t G = K >> 7;
    const float k_f = static_cast<float>(K);
    const bool has_beta = kBeta < 0 ? beta != nullptr : kBeta != 0;
    const int layer = kLayer < 0 ? layer_arg : kLayer;

    auto to_f4 = [](uint32_t a, uint32_t b) {
        return make_float4(__uint_as_float(a << 16), __uint_as_float(a & 0xFFFF0000u),
                           __uint_as_float(b << 16), __uint_as_float(b & 0xFFFF0000u));
    };
    for (int c = threadIdx.x; c < n_chunks; c += blockDim.x) {
        const uint4 g = __ldg(reinterpret_cast<const uint4*>(gamma) + c);
        wsm[c] = to_f4(g.x, g.y);
        wsm[n_chunks + c] = to_f4(g.z, g.w);
        if (has_beta) {
            const uint4 bt = __ldg(reinterpret_cast<const uint4*>(beta) + c);
            wsm[2 * n_chunks + c] = to_f4(bt.x, bt.y);
            wsm[3 * n_chunks + c] = to_f4(bt.z, bt.w);
        }
    }
    __syncthreads();

    auto warp_sum = [](float v) {
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1)
            v += __shfl_xor_sync(0xFFFFFFFFu, v, m);
        return v;
    };

    for (int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpRowsPerCta + warp; row < M;
         row += static_cast<int64_t>(gridDim.x) * kWarpRowsPerCta) {
        const uint4* src = reinterpret_cast<const uint4*>(x + row * ldx);

        // Statistics. Chunks past the row end load as zeros, which add
        // nothing to sum(x) and are skipped in the centred sum.
        float mu = 0.0f;
        if (layer) {
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int it = 0; it < n_iter; ++it) {
                uint4 v[kB];
                load_batch<kB, kFull>(v, src, it * kB, lane, n_chunks, false);
#pragma unroll
                for (int b = 0; b < kB; ++b) {
                    const uint32_t w[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = unpack_f32x2(bf16x2_add_f32(w[i], -0.0f));
                        acc[(i & 1) * 2] += f.x;
                        acc[(i & 1) * 2 + 1] += f.y;
                    }
                }
            }
            mu = __fdiv_rn(warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3])), k_f);
        }
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int it = 0; it < n_iter; ++it) {
            uint4 v[kB];
            load_batch<kB, kFull>(v, src, it * kB, lane, n_chunks, false);
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                if (kFull || (it * kB + b) * 32 + lane < n_chunks) {
                    const uint32_t w[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (layer) {
                            const float2 d = unpack_f32x2(bf16x2_add_f32(w[i], -mu));
                            acc[(i & 1) * 2] = __fmaf_rn(d.x, d.x, acc[(i & 1) * 2]);
                            acc[(i & 1) * 2 + 1] = __fmaf_rn(d.y, d.y, acc[(i & 1) * 2 + 1]);
                        } else {
                            bf16x2_sq_acc(w[i], acc[(i & 1) * 2], acc[(i & 1) * 2 + 1]);
                        }
                    }
                }
            }
        }
        const float var = __fdiv_rn(warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3])), k_f);
        const float rstd = __frsqrt_rn(__fadd_rn(var, eps));
        if (lane == 0) {
            if (rstd_out != nullptr)
                rstd_out[row] = rstd;
            if (mean_out != nullptr && layer)
                mean_out[row] = mu;
        }

        // Output pass: normalize, round to bf16, group amax (half-warp
        // butterfly), dividers (lane l of a half-warp computes batch entry
        // l < kB and shares it), codes and scales.
        const uint64_t rstd2 = pack_f32x2(rstd, rstd);
        const float nmu = layer ? -mu : -0.0f;
        uint8_t* qrow = q + row * ldq;
        float* srow = scale + row * G;
        for (int it = 0; it < n_iter; ++it) {
            uint4 v[kB];
            load_batch<kB, kFull>(v, src, it * kB, lane, n_chunks, true);
            uint32_t m[kB];
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                const int c = (it * kB + b) * 32 + lane;
                const int cs = (kFull || c < n_chunks) ? c : 0;
                const float4 glo = wsm[cs], ghi = wsm[n_chunks + cs];
                const float gg[8] = {glo.x, glo.y, glo.z, glo.w, ghi.x, ghi.y, ghi.z, ghi.w};
                uint32_t w[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
                float bb[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                if (has_beta) {
                    const float4 blo = wsm[2 * n_chunks + cs], bhi = wsm[3 * n_chunks + cs];
                    bb[0] = blo.x; bb[1] = blo.y; bb[2] = blo.z; bb[3] = blo.w;
                    bb[4] = bhi.x; bb[5] = bhi.y; bb[6] = bhi.z; bb[7] = bhi.w;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint64_t t = bf16x2_add_f32(w[i], nmu);   // x - mu (exact widening for RMSNorm)
                    t = mul_f32x2(mul_f32x2(t, rstd2), pack_f32x2(gg[2 * i], gg[2 * i + 1]));
                    if (has_beta) {
                        // Scalar adds: the compiler may fuse a packed multiply
                        // and a packed add into one rounding (measured on
                        // B300); __fadd_rn is never contracted.
                        const float2 u = unpack_f32x2(t);
                        t = pack_f32x2(__fadd_rn(u.x, bb[2 * i]), __fadd_rn(u.y, bb[2 * i + 1]));
                    }
                    w[i] = cvt_bf16x2(t);
                }
                v[b] = make_uint4(w[0], w[1], w[2], w[3]);
                m[b] = absmax_words(&v[b], 1);
            }
#pragma unroll
            for (int sh = 8; sh >= 1; sh >>= 1)
#pragma unroll
                for (int b = 0; b < kB; ++b)
                    m[b] = max(m[b], __shfl_xor_sync(0xFFFFFFFFu, m[b], sh));
            uint32_t mine = 0;
#pragma unroll
            for (int b = 0; b < kB; ++b)
                if ((lane & 15) == b)
                    mine = m[b];
            const Divider own = make_divider(bf16_bits_to_f32(mine));
            const bool fast = __all_sync(0xFFFFFFFFu, own.r != 0.0f);
            Divider d[kB];
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                d[b].s = __shfl_sync(0xFFFFFFFFu, own.s, (lane & 16) | b);
                d[b].r = __shfl_sync(0xFFFFFFFFu, own.r, (lane & 16) | b);
            }
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                const int c = (it * kB + b) * 32 + lane;
                if (kFull || c < n_chunks) {
                    if ((lane & 15) == 0)
                        srow[c >> 4] = d[b].s;
                    __stcs(reinterpret_cast<uint2*>(qrow + 8 * static_cast<int64_t>(c)),
                           fast ? quantize8_fast_fp(v[b], d[b]) : quantize8(v[b], d[b]));
                }
            }
        }
    }
}

#define FP8BS_NORM_WARP_PARAMS                                                                              \
    const uint16_t *__restrict__ x, int64_t ldx, const uint16_t *__restrict__ gamma,                       \
        const uint16_t *__restrict__ beta, int layer, float eps, int64_t M, int K, uint8_t *__restrict__ q, \
        int64_t ldq, float *__restrict__ scale, float *__restrict__ mean_out, float *__restrict__ rstd_out

// The general form: norm kind and beta read at run time, 4 CTAs per SM.
template <int kIters>
__global__ void __launch_bounds__(32 * kWarpRowsPerCta) norm_quant_warp_kernel(FP8BS_NORM_WARP_PARAMS)
{
    norm_warp_rows<kIters, -1, -1>(x, ldx, gamma, beta, layer, eps, M, K, q, ldq, scale, mean_out, rstd_out);
}

// Rows with beta: norm kind and beta fixed at compile time and a larger
// register budget (3 CTAs per SM). Used at K = 7168 and 8192, where it
// measured faster than the general form with beta (K = 7168: RMSNorm 9 %,
// LayerNorm 14 %; K = 8192: 4 % and even); without beta, and at K = 4096, the
// general form is as fast or faster.
template <int kIters, int kLayer>
__global__ void __launch_bounds__(32 * kWarpRowsPerCta, 3) norm_quant_warp_beta_kernel(FP8BS_NORM_WARP_PARAMS)
{
    norm_warp_rows<kIters, kLayer, 1>(x, ldx, gamma, beta, layer, eps, M, K, q, ldq, scale, mean_out, rstd_out);
}
#undef FP8BS_NORM_WARP_PARAMS

template <int kWarps, int kJ>
fp8bs_status launch_norm(const DeviceInfo& info, const uint16_t* x, int64_t ldx, const uint16_t* gamma,
                         const uint16_t* beta, int layer, float eps, int64_t M, int K, uint8_t* q,
                         int64_t ldq, float* scale, float* mean, float* rstd, cudaStream_t stream)
{
    constexpr int kThreads = 32 * kWarps;
    static std::atomic<int> per_sm[64] = {};   // filled once per device; racing fills store the same value
    if (info.device < 0 || info.device >= 64)
        return FP8BS_ERR_CUDA;
    int b = per_sm[info.device].load(std::memory_order_relaxed);
    if (b == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, norm_quant_kernel<kWarps, kJ>, kThreads, 0) !=
                cudaSuccess || b <= 0) {
            cudaGetLastError();
            b = 1;
        }
        per_sm[info.device].store(b, std::memory_order_relaxed);
    }
    const int64_t full = static_cast<int64_t>(info.sm_count) * b;
    const int grid = static_cast<int>(M < full ? M : full);
    norm_quant_kernel<kWarps, kJ><<<grid, kThreads, 0, stream>>>(x, ldx, gamma, beta, layer, eps, M, K, q,
                                                                 ldq, scale, mean, rstd);
    return launch_status();
}

template <int kIters, int kLayer, int kBeta>
fp8bs_status launch_norm_warp_kernel(const DeviceInfo& info, const uint16_t* x, int64_t ldx, const uint16_t* gamma,
                              const uint16_t* beta, int layer, float eps, int64_t M, int K, uint8_t* q,
                              int64_t ldq, float* scale, float* mean, float* rstd, cudaStream_t stream)
{
    constexpr int kThreads = 32 * kWarpRowsPerCta;
    auto* const kernel = [] {
        if constexpr (kBeta < 0)
            return norm_quant_warp_kernel<kIters>;
        else
            return norm_quant_warp_beta_kernel<kIters, kLayer>;
    }();
    constexpr int kMaxK = 16384;
    constexpr int kMaxSmem = 4 * (kMaxK / 8) * 16;
    const int n_chunks = K / 8;
    const size_t smem = static_cast<size_t>(beta != nullptr ? 4 : 2) * n_chunks * 16;
    static std::mutex mu;
    static bool configured[64] = {};
    if (info.device < 0 || info.device >= 64 || K > kMaxK)
        return FP8BS_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!configured[info.device]) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kMaxSmem) != cudaSuccess) {
                cudaGetLastError();
                return FP8BS_ERR_CUDA;
            }
            configured[info.device] = true;
        }
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem) !=
            cudaSuccess ||
        per_sm <= 0) {
        cudaGetLastError();
        per_sm = 1;
    }
    const int64_t needed = (M + kWarpRowsPerCta - 1) / kWarpRowsPerCta;
    const int64_t full = static_cast<int64_t>(info.sm_count) * per_sm;
    const int grid = static_cast<int>(needed < full ? needed : full);
    kernel<<<grid, kThreads, smem, stream>>>(x, ldx, gamma, beta, layer, eps, M, K, q, ldq, scale, mean, rstd);
    return launch_status();
}

template <int kIters>
fp8bs_status launch_norm_warp(const DeviceInfo& info, const uint16_t* x, int64_t ldx, const uint16_t* gamma,
                              const uint16_t* beta, int layer, float eps, int64_t M, int K, uint8_t* q,
                              int64_t ldq, float* scale, float* mean, float* rstd, cudaStream_t stream)
{
    if constexpr (kIters == 7 || kIters == 8) {
        if (beta != nullptr && layer)
            return launch_norm_warp_kernel<kIters, 1, 1>(info, x, ldx, gamma, beta, layer, eps, M, K, q, ldq, scale,
                                                         mean, rstd, stream);
        if (beta != nullptr)
            return launch_norm_warp_kernel<kIters, 0, 1>(info, x, ldx, gamma, beta, layer, eps, M, K, q, ldq, scale,
                                                         mean, rstd, stream);
    }
    return launch_norm_warp_kernel<kIters, -1, -1>(info, x, ldx, gamma, beta, layer, eps, M, K, q, ldq, scale, mean,
                                                   rstd, stream);
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
    // Common hidden sizes get a kernel with the row length built in.
#define FP8BS_NORM_WARP(I) launch_norm_warp<I>(info, xb, ldx, gb, bb, layer, eps, M, k, q, ldq, scale, mean, rstd, s)
    switch (K) {
    case 1024: return FP8BS_NORM_WARP(1);
    case 2048: return FP8BS_NORM_WARP(2);
    case 4096: return FP8BS_NORM_WARP(4);
    case 7168: return FP8BS_NORM_WARP(7);
    case 8192: return FP8BS_NORM_WARP(8);
    default: break;
    }
    if (K <= 16384)
        return FP8BS_NORM_WARP(0);
#undef FP8BS_NORM_WARP
    if (K <= 32768)
        return FP8BS_NORM_LAUNCH(8, 16);
    return FP8BS_NORM_LAUNCH(8, 32);
#undef FP8BS_NORM_LAUNCH
}
