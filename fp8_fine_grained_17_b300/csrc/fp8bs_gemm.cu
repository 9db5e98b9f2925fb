// Block-scaled FP8 GEMM (dense and grouped/MoE) for sm_103a.
//
// C[m, n] = sum_kb sa[m, kb] * sw[n/128, kb] * P_kb[m, n],
// P_kb[m, n] = sum_{k in chunk kb} qa[m, k] * qw[n, k]   (E4M3 x E4M3 -> FP32)
//
// The method: FP8 GEMM on tensor cores with per-group scaling factors along K
// applied on CUDA cores during dequantization, and partial sums promoted to
// FP32 at a fixed K interval because the tensor-core accumulation keeps a
// limited bit width (Q&A post on xn--9g3bo1gtkw0l8ubf92bgle.kr, paragraphs on
// per-group scaling along K and on the two-WGMMA overlap of promotion and
// MMA; "How Google Is Changing How We Method Deepseek", paragraph on limited
// accumulation bit width). The scale group is 128 along K ("personal notes
// concerning the deepseek core readings", Figure 7(a)), so the promotion
// interval here is one 128-wide K chunk.
//
// B300 design (not the pages' Hopper scheme): one persistent CTA per SM,
// 384 threads, output tile 128 x 256.
//   warp 0      TMA producer: A (128x128 B) and W (256x128 B) chunks into a
//               4-stage shared-memory ring, 128-byte swizzled.
//   warp 1      MMA issuer (one thread): 4 x tcgen05.mma.kind::f8f6f4
//               (K = 32 each) per chunk into one of two 256-column FP32 TMEM
//               buffers, overwriting it (the chunk's partial P_kb).
//   warp 2      TMEM allocator (512 columns).
//   warp 3      scale loader: copies each chunk's 128 activation scales and
//               two weight-block scales into an 8-slot shared-memory ring
//               with cp.async (grouped GEMM: first builds the expert tile
//               table), running up to 8 chunks ahead of the promotion warps.
//   warps 4-11  promotion: each thread owns one row and 128 columns; per
//               chunk it reads P_kb from TMEM (tcgen05.ld, the next 32
//               columns in flight while the current ones are accumulated),
//               frees the buffer, and accumulates acc += (sa * sw) * P_kb in
//               FP32 registers. After the last chunk it converts and stores
//               its row segment.
// The two TMEM buffers let the tensor cores compute chunk kb+1 while the
// promotion warps drain chunk kb.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "fp8bs_device.cuh"
#include "fp8bs_host.h"

namespace fp8bs {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr int kStages = 4;
constexpr int kScaleStages = 8;
constexpr int kABytes = BM * BK;
constexpr int kBBytes = BN * BK;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 384;
constexpr int kTmemCols = 2 * BN;
constexpr int kMaxExperts = 1024;
constexpr int kProducerRegs = 56;
constexpr int kEpilogueRegs = 224;
constexpr uint32_t kIdesc = idesc_e4m3_f32(BM, BN);

struct __align__(1024) Smem {
    uint8_t a[kStages][kABytes];
    uint8_t b[kStages][kBBytes];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint64_t scale_full[kScaleStages];    // 32 cp.async arrivals (one per loader lane)
    uint64_t scale_empty[kScaleStages];   // 8 arrivals (one per promotion warp)
    float scale_a[kScaleStages][BM];      // sa[m0 + r, kb]
    float scale_w[kScaleStages][4];       // sw[e, n0/128 + h, kb], h = 0, 1
    uint32_t tmem_base;
    int abort;
    int num_tiles;
    int tile_start[kMaxExperts + 1];   // grouped: first tile index of each expert
    int row_start[kMaxExperts + 1];    // grouped: copy of expert_offsets
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;   // + alignment slack

struct Params {
    const float* sa;          // [rows, KB]
    const float* sw;          // [E, NB, KB]
    void* c;
    int64_t ldc;
    int64_t rows;             // rows of A (M, or total_M)
    int N;
    int KB;
    int NB;                   // N / 128
    int n_tiles;              // ceil(N / 256)
    int out_bf16;
    const int32_t* offsets;   // grouped only
    int E;
    unsigned int* err;
};

struct Tile {
    int64_t m0;        // first row of the tile in A / C
    int64_t row_end;   // rows >= row_end belong to no output of this tile
    int n0;            // first output column (within N)
    int expert;
    int b_row0;        // first row of the W tile in the [E*N, K] weight matrix
};

// Tile t of the launch: the expert e with tile_start[e] <= t < tile_start[e+1]
// (binary search; a dense launch is one expert covering all rows), then the
// m-tile and n-tile within that expert, m-tiles fastest.
__device__ __forceinline__ Tile decode_tile(const Smem& sm, const Params& p, int t)
{
    int lo = 0, hi = p.E;   // invariant: tile_start[lo] <= t < tile_start[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sm.tile_start[mid] <= t)
            lo = mid;
        else
            hi = mid;
    }
    const int e = lo;
    const int local = t - sm.tile_start[e];
    const int rows_e = sm.row_start[e + 1] - sm.row_start[e];
    const int mt_e = (rows_e + BM - 1) / BM;
    const int mt = local % mt_e;
    const int nt = local / mt_e;
    Tile tile;
    tile.m0 = sm.row_start[e] + static_cast<int64_t>(mt) * BM;
    tile.row_end = sm.row_start[e + 1];
    tile.n0 = nt * BN;
    tile.expert = e;
    tile.b_row0 = e * p.N + tile.n0;
    return tile;
}

// Warp 3: copy and validate expert_offsets (a dense launch uses {0, M}),
// then build tile_start[] (exclusive prefix sum of m-tiles x n-tiles per
// expert).
__device__ void build_expert_table(Smem& sm, const Params& p, int lane)
{
    bool ok = true;
    for (int base = 0; base <= p.E; base += 32) {
        const int i = base + lane;
        if (i <= p.E)
            sm.row_start[i] = p.offsets != nullptr ? p.offsets[i] : (i == 0 ? 0 : static_cast<int>(p.rows));
    }
    __syncwarp();
    int carry = 0;
    for (int base = 0; base < p.E; base += 32) {
        const int e = base + lane;
        int tiles = 0;
        if (e < p.E) {
            const int lo = sm.row_start[e], hi = sm.row_start[e + 1];
            if (hi < lo)
                ok = false;
            else
                tiles = ((hi - lo + BM - 1) / BM) * p.n_tiles;
        }
        int incl = tiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int up = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o)
                incl += up;
        }
        if (e < p.E)
            sm.tile_start[e + 1] = carry + incl;
        carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (lane == 0) {
        sm.tile_start[0] = 0;
        if (sm.row_start[0] != 0 || static_cast<int64_t>(sm.row_start[p.E]) > p.rows)
            ok = false;
        if (!ok) {
            if (blockIdx.x == 0)
                atomicOr(p.err, DEVERR_BAD_OFFSETS);
            sm.num_tiles = 0;
        } else {
            sm.num_tiles = carry;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
fp8_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw + (((raw + 1023u) & ~1023u) - raw));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&sm.full[s]), 1);
            mbar_init(smem_addr(&sm.empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&sm.tmem_full[b]), 1);
            mbar_init(smem_addr(&sm.tmem_empty[b]), 8);   // one arrive per promotion warp
        }
        mbar_init(smem_addr(&sm.drain), 1);
        for (int s = 0; s < kScaleStages; ++s) {
            mbar_init(smem_addr(&sm.scale_full[s]), 32);
            mbar_init(smem_addr(&sm.scale_empty[s]), 8);
        }
        sm.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0 && p.KB > 0) {
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b);
    }
    if (warp == 2) {
        tmem_alloc(smem_addr(&sm.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 3)
        build_expert_table(sm, p, lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = sm.tmem_base;
    const int num_tiles = sm.num_tiles;
    volatile int* abort_flag = &sm.abort;

    if (warp < 4) {
        regs_dec<kProducerRegs>();
        if (warp == 0 && lane == 0) {
            // ---------------------------------------------------- TMA producer
            uint32_t chunk = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const Tile tile = decode_tile(sm, p, t);
                for (int kb = 0; kb < p.KB; ++kb, ++chunk) {
                    const uint32_t s = chunk % kStages;
                    const uint32_t ph = (chunk / kStages) & 1u;
                    if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1u, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = smem_addr(&sm.full[s]);
                    mbar_arrive_expect_tx(full, kStageBytes);
                    tma_load_2d(smem_addr(sm.a[s]), &map_a, full, kb * BK, static_cast<int32_t>(tile.m0));
                    tma_load_2d(smem_addr(sm.b[s]), &map_b, full, kb * BK, tile.b_row0);
                }
            }
            if (!ok) {
                // Let the copies already issued land before the CTA exits.
                const uint32_t first = chunk > kStages ? chunk - kStages : 0;
                for (uint32_t c = first; c < chunk; ++c)
                    mbar_wait_drain(smem_addr(&sm.full[c % kStages]), (c / kStages) & 1u,
                                    kWaitLimitNs, p.err);
            }
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------------ MMA issuer
            uint32_t chunk = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                for (int kb = 0; kb < p.KB; ++kb, ++chunk) {
                    const uint32_t s = chunk % kStages;
                    const uint32_t ph = (chunk / kStages) & 1u;
                    const uint32_t b = chunk & 1u;
                    const uint32_t tph = (chunk >> 1) & 1u;
                    if (!mbar_wait(smem_addr(&sm.tmem_empty[b]), tph ^ 1u, abort_flag, p.err) ||
                        !mbar_wait(smem_addr(&sm.full[s]), ph, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + b * BN;
                    const uint32_t a_addr = smem_addr(sm.a[s]);
                    const uint32_t b_addr = smem_addr(sm.b[s]);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        mma_e4m3(d, smem_desc_k_sw128(a_addr + 32 * k),
                                 smem_desc_k_sw128(b_addr + 32 * k), kIdesc, k > 0 ? 1u : 0u);
                    mma_commit(smem_addr(&sm.empty[s]));
                    mma_commit(smem_addr(&sm.tmem_full[b]));
                }
            }
            // All MMAs issued by this thread complete before TMEM is released.
            mma_commit(smem_addr(&sm.drain));
            mbar_wait_drain(smem_addr(&sm.drain), 0, kWaitLimitNs, p.err);
        } else if (warp == 3) {
            // ---------------------------------------------------- scale loader
            uint32_t chunk = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const Tile tile = decode_tile(sm, p, t);
                // Rows past the tile's end read a valid row; their products
                // are never stored.
                const float* src_a[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int64_t row = tile.m0 + lane + 32 * i;
                    src_a[i] = p.sa + (row < p.rows ? row : p.rows - 1) * p.KB;
                }
                const int nbh = min(tile.n0 / 128 + (lane & 1), p.NB - 1);
                const float* src_w = p.sw + (static_cast<int64_t>(tile.expert) * p.NB + nbh) * p.KB;
                for (int kb = 0; kb < p.KB; ++kb, ++chunk) {
                    const uint32_t s = chunk % kScaleStages;
                    const uint32_t ph = (chunk / kScaleStages) & 1u;
                    const bool ready =
                        mbar_wait(smem_addr(&sm.scale_empty[s]), ph ^ 1u, abort_flag, p.err);
                    if (!__all_sync(0xFFFFFFFFu, ready)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        cp_async_4(smem_addr(&sm.scale_a[s][lane + 32 * i]), src_a[i] + kb);
                    if (lane < 2)
                        cp_async_4(smem_addr(&sm.scale_w[s][lane]), src_w + kb);
                    cp_async_arrive_noinc(smem_addr(&sm.scale_full[s]));
                }
            }
            cp_async_wait_all();
        }
    } else {
        regs_inc<kEpilogueRegs>();
        // ------------------------------------------------------- promotion
        const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
        const int half = (warp - 4) >> 2;      // output columns 128*half .. +127
        const int r = quarter * 32 + lane;
        uint32_t chunk = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            const Tile tile = decode_tile(sm, p, t);
            const int64_t row = tile.m0 + r;
            const int n_col = tile.n0 + half * 128;
            const bool live = row < tile.row_end && n_col < p.N;

            // 128 FP32 accumulators as 64 pairs for the packed FMA pipe.
            float2 acc[64];
#pragma unroll
            for (int i = 0; i < 64; ++i)
                acc[i] = make_float2(0.0f, 0.0f);
#pragma unroll 1
            for (int kb = 0; kb < p.KB; ++kb, ++chunk) {
                const uint32_t ss = chunk % kScaleStages;
                const uint32_t sph = (chunk / kScaleStages) & 1u;
                const uint32_t b = chunk & 1u;
                const uint32_t tph = (chunk >> 1) & 1u;
                // The warp continues only if every lane saw the phases
                // complete: the TMEM loads below are warp-collective.
                bool ready = mbar_wait(smem_addr(&sm.scale_full[ss]), sph, abort_flag, p.err);
                float scale = 0.0f;
                if (ready)
                    scale = sm.scale_a[ss][r] * sm.scale_w[ss][half];
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(&sm.scale_empty[ss]));
                ready = ready && mbar_wait(smem_addr(&sm.tmem_full[b]), tph, abort_flag, p.err);
                if (!__all_sync(0xFFFFFFFFu, ready)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr =
                    tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * BN + half * 128;
                const float2 scale2 = make_float2(scale, scale);
                // Column blocks 0..3 of 32: the load of block j+1 is in flight
                // while block j is accumulated.
                uint32_t va[32], vb[32];
                tmem_ld_32x32b_x32(taddr, va);
                tmem_ld_wait(va);
                tmem_ld_32x32b_x32(taddr + 32, vb);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    acc[0 + i] = __ffma2_rn(
                        make_float2(__uint_as_float(va[2 * i]), __uint_as_float(va[2 * i + 1])),
                        scale2, acc[0 + i]);
                tmem_ld_wait(vb);
                tmem_ld_32x32b_x32(taddr + 64, va);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    acc[16 + i] = __ffma2_rn(
                        make_float2(__uint_as_float(vb[2 * i]), __uint_as_float(vb[2 * i + 1])),
                        scale2, acc[16 + i]);
                tmem_ld_wait(va);
                tmem_ld_32x32b_x32(taddr + 96, vb);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    acc[32 + i] = __ffma2_rn(
                        make_float2(__uint_as_float(va[2 * i]), __uint_as_float(va[2 * i + 1])),
                        scale2, acc[32 + i]);
                tmem_ld_wait(vb);
                // Every TMEM read of this buffer is complete: hand it back.
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(&sm.tmem_empty[b]));
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    acc[48 + i] = __ffma2_rn(
                        make_float2(__uint_as_float(vb[2 * i]), __uint_as_float(vb[2 * i + 1])),
                        scale2, acc[48 + i]);
            }
            if (ok && live) {
                if (p.out_bf16) {
                    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.c) + row * p.ldc + n_col;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        uint4 pk;
                        __nv_bfloat162 h0 = __float22bfloat162_rn(acc[4 * i + 0]);
                        __nv_bfloat162 h1 = __float22bfloat162_rn(acc[4 * i + 1]);
                        __nv_bfloat162 h2 = __float22bfloat162_rn(acc[4 * i + 2]);
                        __nv_bfloat162 h3 = __float22bfloat162_rn(acc[4 * i + 3]);
                        memcpy(&pk.x, &h0, 4);
                        memcpy(&pk.y, &h1, 4);
                        memcpy(&pk.z, &h2, 4);
                        memcpy(&pk.w, &h3, 4);
                        reinterpret_cast<uint4*>(dst)[i] = pk;
                    }
                } else {
                    float* dst = static_cast<float*>(p.c) + row * p.ldc + n_col;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        reinterpret_cast<float4*>(dst)[i] = make_float4(
                            acc[2 * i].x, acc[2 * i].y, acc[2 * i + 1].x, acc[2 * i + 1].y);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 get_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// K-major FP8 operand [rows, K] (row stride K bytes), box 128 (K) x box_rows.
bool encode_operand(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows)
{
    auto enc = get_encoder();
    if (enc == nullptr)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

fp8bs_status configure_once(int device)
{
    static std::mutex mu;
    static bool done[64] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64)
        return FP8BS_ERR_CUDA;
    if (!done[device]) {
        if (cudaFuncSetAttribute(fp8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes)) != cudaSuccess) {
            cudaGetLastError();
            return FP8BS_ERR_CUDA;
        }
        done[device] = true;
    }
    return FP8BS_OK;
}

fp8bs_status launch(const uint8_t* qa, int64_t rows, const uint8_t* qw, int64_t w_rows, Params p,
                    int64_t K, int64_t tile_bound, cudaStream_t stream)
{
    DeviceInfo info;
    fp8bs_status st = require_sm103(&info);
    if (st != FP8BS_OK)
        return st;
    p.err = device_error_word();
    if (p.err == nullptr)
        return FP8BS_ERR_CUDA;
    CUtensorMap map_a, map_b;
    memset(&map_a, 0, sizeof map_a);
    memset(&map_b, 0, sizeof map_b);
    if (K > 0) {
        if (!encode_operand(&map_a, qa, rows, K, BM) || !encode_operand(&map_b, qw, w_rows, K, BN))
            return FP8BS_ERR_CUDA;
    }
    st = configure_once(info.device);
    if (st != FP8BS_OK)
        return st;
    const int grid = static_cast<int>(tile_bound < info.sm_count ? tile_bound : info.sm_count);
    if (grid <= 0)
        return FP8BS_OK;
    fp8_gemm_kernel<<<grid, kThreads, kSmemBytes, stream>>>(map_a, map_b, p);
    return launch_status();
}

fp8bs_status check_common(const void* qa, const float* sa, const void* qw, const float* sw,
                          const void* c, fp8bs_out_dtype out_dtype, int64_t N, int64_t K,
                          int64_t ldc)
{
    // With K == 0 the operands are empty and never read; only C is written.
    if (c == nullptr || (K > 0 && (qa == nullptr || sa == nullptr || qw == nullptr || sw == nullptr)))
        return FP8BS_ERR_INVALID_ARG;
    if (out_dtype != FP8BS_OUT_F32 && out_dtype != FP8BS_OUT_BF16)
        return FP8BS_ERR_INVALID_ARG;
    const int64_t esize = out_dtype == FP8BS_OUT_BF16 ? 2 : 4;
    if (ldc < N || (ldc * esize) % 16 != 0 || !aligned16(c))
        return FP8BS_ERR_INVALID_ARG;
    if (K > 0 && (!aligned16(qa) || !aligned16(qw) || (reinterpret_cast<uintptr_t>(sa) & 3u) != 0 ||
                  (reinterpret_cast<uintptr_t>(sw) & 3u) != 0))
        return FP8BS_ERR_INVALID_ARG;
    if (N > (int64_t(1) << 24) || K > (int64_t(1) << 31) - BK)
        return FP8BS_ERR_UNSUPPORTED;
    return FP8BS_OK;
}

}  // namespace
}  // namespace fp8bs

using namespace fp8bs;

extern "C" fp8bs_status fp8bs_gemm(const uint8_t* qa, const float* sa, const uint8_t* qw,
                                   const float* sw, void* c, fp8bs_out_dtype out_dtype, int64_t M,
                                   int64_t N, int64_t K, int64_t ldc, fp8bs_stream_t stream)
{
    if (M < 0 || N < 0 || K < 0)
        return FP8BS_ERR_INVALID_ARG;
    if (K % BK != 0 || N % 128 != 0)
        return FP8BS_ERR_UNSUPPORTED;
    if (M == 0 || N == 0)
        return FP8BS_OK;
    fp8bs_status st = check_common(qa, sa, qw, sw, c, out_dtype, N, K, ldc);
    if (st != FP8BS_OK)
        return st;
    const int64_t m_tiles = (M + BM - 1) / BM;
    const int64_t n_tiles = (N + BN - 1) / BN;
    if (M > 0x7FFFFFFF || m_tiles * n_tiles > 0x7FFFFFFF)
        return FP8BS_ERR_UNSUPPORTED;

    Params p{};
    p.sa = sa;
    p.sw = sw;
    p.c = c;
    p.ldc = ldc;
    p.rows = M;
    p.N = static_cast<int>(N);
    p.KB = static_cast<int>(K / BK);
    p.NB = static_cast<int>(N / 128);
    p.n_tiles = static_cast<int>(n_tiles);
    p.out_bf16 = out_dtype == FP8BS_OUT_BF16;
    p.offsets = nullptr;
    p.E = 1;
    return launch(qa, M, qw, N, p, K, m_tiles * n_tiles,
                         reinterpret_cast<cudaStream_t>(stream));
}

extern "C" fp8bs_status fp8bs_grouped_gemm(const uint8_t* qa, const float* sa,
                                           const int32_t* expert_offsets, int32_t E,
                                           int64_t total_M, const uint8_t* qw, const float* sw,
                                           void* c, fp8bs_out_dtype out_dtype, int64_t N, int64_t K,
                                           int64_t ldc, fp8bs_stream_t stream)
{
    if (E < 1 || total_M < 0 || N < 0 || K < 0)
        return FP8BS_ERR_INVALID_ARG;
    if (E > kMaxExperts || K % BK != 0 || N % 128 != 0)
        return FP8BS_ERR_UNSUPPORTED;
    if (total_M == 0 || N == 0)
        return FP8BS_OK;
    if (expert_offsets == nullptr || (reinterpret_cast<uintptr_t>(expert_offsets) & 3u) != 0)
        return FP8BS_ERR_INVALID_ARG;
    fp8bs_status st = check_common(qa, sa, qw, sw, c, out_dtype, N, K, ldc);
    if (st != FP8BS_OK)
        return st;
    if (total_M > 0x7FFFFFFF || static_cast<int64_t>(E) * N > 0x7FFFFFFF)
        return FP8BS_ERR_UNSUPPORTED;
    const int64_t n_tiles = (N + BN - 1) / BN;
    const int64_t tile_bound = (total_M / BM + E) * n_tiles;
    if (tile_bound > 0x7FFFFFFF)
        return FP8BS_ERR_UNSUPPORTED;

    Params p{};
    p.sa = sa;
    p.sw = sw;
    p.c = c;
    p.ldc = ldc;
    p.rows = total_M;
    p.N = static_cast<int>(N);
    p.KB = static_cast<int>(K / BK);
    p.NB = static_cast<int>(N / 128);
    p.n_tiles = static_cast<int>(n_tiles);
    p.out_bf16 = out_dtype == FP8BS_OUT_BF16;
    p.offsets = expert_offsets;
    p.E = E;
    return launch(qa, total_M, qw, static_cast<int64_t>(E) * N, p, K, tile_bound,
                        reinterpret_cast<cudaStream_t>(stream));
}
