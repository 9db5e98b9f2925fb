// Activation (1x128 tile) and weight (128x128 block) quantizers: bf16 ->
// E4M3 codes + binary32 dequantization scales.
//
// Grouping follows "personal notes concerning the deepseek core readings"
// (why-be.why-be.co.kr), fine-grained quantization paragraph, Figure 7(a);
// amax-to-FP8-maximum scaling and online quantization follow the Q&A post on
// xn--9g3bo1gtkw0l8ubf92bgle.kr, mixed-precision paragraph. The per-group
// codec (scale, reciprocal, codes) is in fp8bs_e4m3.cuh.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fp8bs_device.cuh"
#include "fp8bs_e4m3.cuh"
#include "fp8bs_host.h"

namespace fp8bs {
namespace {

// ---------------------------------------------------------------------------
// Activation quantizer.
//
// Work unit: a lane quad (four consecutive lanes) and four 1x128 groups.
// Lane t of the quad holds the 16-byte chunks t + 4 ((j + rot) & 3),
// j = 0..3, of each of the four groups (rot lets two quads that share a
// shared-memory bank group start at different chunks). The quad's four
// partial maxima are reduced with a transposing exchange (3 shuffles) that
// leaves group t's amax in lane t; lane t computes that group's scale and
// reciprocal once and writes the scale, and the quad broadcasts them.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void quantize_quad(const uint4 (&v)[4][4], const bool (&valid)[4],
                                              uint8_t* const (&qdst)[4], float* my_scale, int t,
                                              int quad_base, int rot, int pow2)
{
    uint32_t m[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
        m[u] = absmax_words(v[u], 4);
    // Transposing max-exchange: after it lane t holds group t's amax.
    const bool b1 = (t & 2) != 0, b0 = (t & 1) != 0;
    uint32_t k[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, b1 ? m[i] : m[2 + i], 2);
        k[i] = max(b1 ? m[2 + i] : m[i], recv);
    }
    const uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, b0 ? k[0] : k[1], 1);
    const uint32_t mine = max(b0 ? k[1] : k[0], recv);

    const Divider own = group_divider(mine, pow2);
    if (my_scale != nullptr)
        *my_scale = own.s;

#pragma unroll
    for (int u = 0; u < 4; ++u) {
        Divider d;
        d.s = __shfl_sync(0xFFFFFFFFu, own.s, quad_base + u);
        d.r = __shfl_sync(0xFFFFFFFFu, own.r, quad_base + u);
        if (valid[u]) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                __stcs(reinterpret_cast<uint2*>(qdst[u] + 8 * (t + 4 * ((j + rot) & 3))),
                       quantize8(v[u][j], d));
        }
    }
}

// Register path: a grid-stride loop over 32-group blocks per warp; all loads
// of an iteration (256 B per lane) are issued before any arithmetic.
// kContiguous: rows back to back (ld == K), group g starts at element 128 g.
constexpr int kActThreads = 256;

// One batch of the register path: the 32 groups starting at group `base`
// (one per lane; the warp's lane quads take four groups each).
template <bool kContiguous>
__device__ __forceinline__ void act_regs_batch(int64_t base, const uint16_t* __restrict__ x, int64_t ldx,
                                               uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ scale,
                                               int64_t groups_per_row, int64_t total_groups, int pow2)
{
    const int lane = threadIdx.x & 31;
    const int t = lane & 3;
    const int quad_base = lane & ~3;
    uint4 v[4][4];
    uint8_t* qdst[4];
    bool valid[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int64_t g = base + quad_base + u;
        valid[u] = g < total_groups;
        int64_t xo, qo;
        if (kContiguous) {
            xo = valid[u] ? g * 128 : 0;
            qo = xo;
        } else {
            const int64_t row = valid[u] ? g / groups_per_row : 0;
            const int64_t col = valid[u] ? (g - row * groups_per_row) * 128 : 0;
            xo = row * ldx + col;
            qo = row * ldq + col;
        }
        qdst[u] = q + qo;
        const uint4* src = reinterpret_cast<const uint4*>(x + xo) + t;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            v[u][j] = valid[u] ? __ldcs(src + 4 * j) : make_uint4(0, 0, 0, 0);
    }
    const int64_t my_g = base + lane;   // scale is [M, K/128] row-major: index = g
    quantize_quad(v, valid, qdst, my_g < total_groups ? scale + my_g : nullptr, t, quad_base, 0, pow2);
}

template <bool kContiguous>
__global__ void __launch_bounds__(kActThreads)
quantize_act_regs_kernel(const uint16_t* __restrict__ x, int64_t ldx, uint8_t* __restrict__ q,
                         int64_t ldq, float* __restrict__ scale, int64_t groups_per_row,
                         int64_t total_groups, int pow2)
{
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kActThreads + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * kActThreads) >> 5;
    for (int64_t base = warp * 32; base < total_groups; base += n_warps * 32)
        act_regs_batch<kContiguous>(base, x, ldx, q, ldq, scale, groups_per_row, total_groups, pow2);
}

// Ring kernel: a persistent grid of 4-warp CTAs (three per SM) that streams
// a list of 32 KB work items through a 2-stage shared-memory ring, so that
// the load of the next item is in flight while one is quantized. Items:
//   activation chunks   128 consecutive 1x128 groups of a contiguous bf16
//                       tensor (ld == K), brought in by one bulk copy;
//   weight blocks       one 128x128 bf16 block, brought in by one 2-D TMA
//                       tile load (rows past N read as zeros).
// Item i of the grid's list goes to CTA i mod grid. The codec is the one of
// the register paths (same codes and scales). Used for the activation
// quantizer on large contiguous inputs and for the activation + weight pair
// of a GEMM step (one launch, both lists back to back). Smaller inputs take
// the register path, whose fill latency is lower (measured on B300:
// [4096, 7168] 22.9 us register path vs 25.2 us ring).
// Ring depth, measured on B300 (interleaved runs): the kernel is bound by
// instruction latency rather than by loads in flight, so resident warps
// matter most. 2 stages (3 CTAs per SM): [16384, 7168] 60.5 us, the step's
// pair 33.0 us; 3 stages (2 CTAs per SM): 65.4 / 37.4 us; 4 stages (1 CTA
// per SM): 105.9 / 58.9 us.
constexpr int kRingThreads = 128;
constexpr int kRingItemGroups = 128;
constexpr int kRingItemBytes = kRingItemGroups * 256;
constexpr int kRingStages = 2;
constexpr int64_t kRingMinGroups = int64_t(1) << 19;

struct __align__(128) RingSmem {
    uint8_t stage[kRingStages][kRingItemBytes];
    uint64_t full[kRingStages];
    uint32_t wmax[kRingThreads / 32];
    int abort;
};
constexpr size_t kRingSmemBytes = sizeof(RingSmem) + 128;

struct RingWork {
    // activation chunks: items [0, n_act)
    const uint16_t* x;
    uint8_t* qx;
    float* sx;
    int64_t x_groups;
    int64_t n_act;
    // weight blocks: items [n_act, n_act + n_w); block (kb, nb) of item
    // n_act + kb + nb * w_gpr
    uint8_t* qw;
    int64_t ldqw;
    float* sw;
    int64_t N;
    int64_t w_gpr;
    int64_t n_w;
    unsigned int* err;
    int pow2;
};

// Weight block from a stage (128 rows x 256 B, row-major): thread t holds the
// 16-byte column chunk t & 15 of rows (t >> 4) + 8 i; block amax by a warp
// max-reduction and the four warps' maxima, codes written per row.
__device__ __forceinline__ void ring_weight_block(const uint8_t* stage, const RingWork& p, int64_t kb,
                                                  int64_t nb, uint32_t* wmax)
{
    const int t = threadIdx.x;
    const int c16 = t & 15;
    const int r0 = t >> 4;
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(stage + (r0 + 8 * i) * 256 + 16 * c16);
        m = max(m, absmax_words(&v, 1));
    }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((t & 31) == 0)
        wmax[t >> 5] = m;
    __syncthreads();
    const uint32_t a = max(max(wmax[0], wmax[1]), max(wmax[2], wmax[3]));
    const Divider d = group_divider(a, p.pow2);
    if (t == 0)
        p.sw[nb * p.w_gpr + kb] = d.s;
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
        const int64_t n = nb * 128 + r0 + 8 * i;
        if (n < p.N) {
            const uint4 v = *reinterpret_cast<const uint4*>(stage + (r0 + 8 * i) * 256 + 16 * c16);
            __stcs(reinterpret_cast<uint2*>(p.qw + n * p.ldqw + kb * 128 + 8 * c16), quantize8(v, d));
        }
    }
}

__global__ void __launch_bounds__(kRingThreads)
quantize_ring_kernel(const __grid_constant__ CUtensorMap wmap, const RingWork p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    RingSmem& sm = *reinterpret_cast<RingSmem*>(smem_raw + (((raw + 127u) & ~127u) - raw));
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int t = lane & 3;
    const int quad_base = lane & ~3;
    const int rot = (lane >> 2) & 1;
    const int64_t n_items = p.n_act + p.n_w;

    // A GEMM launched after this kernel as its programmatic dependent may be
    // scheduled once every CTA here is running; it waits for the results.
    if (threadIdx.x == 0)
        launch_dependents();
    auto issue = [&](int64_t c, int s) {
        const uint32_t bar = smem_addr(&sm.full[s]);
        if (c < p.n_act) {
            const int64_t g0 = c * kRingItemGroups;
            const int64_t n = min(static_cast<int64_t>(kRingItemGroups), p.x_groups - g0);
            const uint32_t bytes = static_cast<uint32_t>(n * 256);
            mbar_arrive_expect_tx(bar, bytes);
            bulk_load(smem_addr(sm.stage[s]), p.x + g0 * 128, bytes, bar);
        } else {
            const int64_t wi = c - p.n_act;
            mbar_arrive_expect_tx(bar, kRingItemBytes);
            tma_load_2d(smem_addr(sm.stage[s]), &wmap, bar, static_cast<int32_t>((wi % p.w_gpr) * 128),
                        static_cast<int32_t>((wi / p.w_gpr) * 128));
        }
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRingStages; ++s)
            mbar_init(smem_addr(&sm.full[s]), 1);
        sm.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (p.n_w > 0)
            tma_prefetch_desc(&wmap);
        for (int s = 0; s < kRingStages; ++s) {
            const int64_t c = blockIdx.x + static_cast<int64_t>(s) * gridDim.x;
            if (c < n_items)
                issue(c, s);
        }
    }
    int s = 0;
    uint32_t ph = 0;
    for (int64_t c = blockIdx.x; c < n_items; c += gridDim.x) {
        const bool ready = mbar_wait(smem_addr(&sm.full[s]), ph, &sm.abort, p.err);
        if (!__syncthreads_and(ready)) {
            // A wait gave up (reported in err): let the copies still in
            // flight land (bounded waits) before the CTA leaves.
            if (threadIdx.x == 0) {
                int ds = s;
                uint32_t dph = ph;
                for (int i = 0; i < kRingStages; ++i) {
                    if (c + static_cast<int64_t>(i) * gridDim.x < n_items)
                        mbar_wait_drain(smem_addr(&sm.full[ds]), dph, kWaitLimitNs, p.err);
                    if (++ds == kRingStages) {
                        ds = 0;
                        dph ^= 1u;
                    }
                }
            }
            break;
        }
        if (c < p.n_act) {
            const int64_t g0 = c * kRingItemGroups;
            const int lq = warp * 32 + quad_base;   // first of the quad's four groups in the chunk
            uint4 v[4][4];
            uint8_t* qdst[4];
            bool valid[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t g = g0 + lq + u;
                valid[u] = g < p.x_groups;
                qdst[u] = p.qx + g * 128;
                const uint8_t* src = sm.stage[s] + (lq + u) * 256;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    v[u][j] = valid[u] ? *reinterpret_cast<const uint4*>(src + 16 * (t + 4 * ((j + rot) & 3)))
                                       : make_uint4(0, 0, 0, 0);
            }
            const int64_t my_g = g0 + warp * 32 + lane;
            quantize_quad(v, valid, qdst, my_g < p.x_groups ? p.sx + my_g : nullptr, t, quad_base, rot, p.pow2);
        } else {
            const int64_t wi = c - p.n_act;
            ring_weight_block(sm.stage[s], p, wi % p.w_gpr, wi / p.w_gpr, sm.wmax);
        }
        __syncthreads();   // every thread is done with stage s (and with wmax)
        if (threadIdx.x == 0) {
            const int64_t c2 = c + static_cast<int64_t>(kRingStages) * gridDim.x;
            if (c2 < n_items)
                issue(c2, s);
        }
        if (++s == kRingStages) {
            s = 0;
            ph ^= 1u;
        }
    }
}

// ---------------------------------------------------------------------------
// Weight quantizer: one 256-thread CTA per 128x128 block. Thread t holds the
// 16-byte chunk (t & 15) of rows 16i + t/16, i = 0..7, so each warp load
// instruction covers two whole 256-byte block rows. The block amax is reduced
// with a warp max-reduction and shared memory; one thread computes the
// scale and reciprocal, and the codes are written from the registers that
// still hold the inputs.
// ---------------------------------------------------------------------------
constexpr int kWThreads = 256;

__device__ __forceinline__ void weight_block(int64_t kb, int64_t nb, const uint16_t* __restrict__ w, int64_t N,
                                             int64_t ldw, uint8_t* __restrict__ q, int64_t ldq,
                                             float* __restrict__ scale, int64_t groups_per_row,
                                             uint32_t* warp_max, Divider* block_div, int pow2)
{
    const int t = threadIdx.x;
    const int chunk = t & 15;
    const int64_t col = kb * 128 + chunk * 8;

    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t n = nb * 128 + i * 16 + (t >> 4);
        v[i] = n < N ? __ldcs(reinterpret_cast<const uint4*>(w + n * ldw + col))
                     : make_uint4(0, 0, 0, 0);
    }
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, absmax_words(v, 8));
    if ((t & 31) == 0)
        warp_max[t >> 5] = m;
    __syncthreads();
    if (t == 0) {
        uint32_t a = warp_max[0];
#pragma unroll
        for (int i = 1; i < kWThreads / 32; ++i)
            a = max(a, warp_max[i]);
        const Divider d = group_divider(a, pow2);
        *block_div = d;
        scale[nb * groups_per_row + kb] = d.s;
    }
    __syncthreads();
    const Divider d = *block_div;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t n = nb * 128 + i * 16 + (t >> 4);
        if (n < N)
            __stcs(reinterpret_cast<uint2*>(q + n * ldq + col), quantize8(v[i], d));
    }
}

__global__ void __launch_bounds__(kWThreads)
quantize_weight_kernel(const uint16_t* __restrict__ w, int64_t N, int64_t ldw,
                       uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ scale,
                       int64_t groups_per_row, int pow2)
{
    __shared__ uint32_t warp_max[kWThreads / 32];
    __shared__ Divider block_div;
    weight_block(blockIdx.x, blockIdx.y, w, N, ldw, q, ldq, scale, groups_per_row, warp_max, &block_div,
                 pow2);
}

// Both quantizers in one launch (a step's activation and weight
// quantizations are independent): blocks [0, act_blocks) each quantize one
// 256-group batch of the activations through the register path, the others
// one 128x128 weight block each, so the two share one wave of the GPU.
static_assert(kActThreads == kWThreads, "one block size for both roles");

// Three CTAs per SM (85 registers): more loads in flight; measured faster on
// B300 than two CTAs at 102 registers (36.4 vs 38.7 us for two [4096, 7168]
// operands) despite a few spilled registers.
template <bool kContiguous>
__global__ void __launch_bounds__(kWThreads, 3)
quantize_pair_kernel(const uint16_t* __restrict__ x, int64_t ldx, uint8_t* __restrict__ qx, int64_t ldqx,
                     float* __restrict__ sx, int64_t x_groups_per_row, int64_t x_groups, int64_t act_blocks,
                     const uint16_t* __restrict__ w, int64_t N, int64_t ldw, uint8_t* __restrict__ qw,
                     int64_t ldqw, float* __restrict__ sw, int64_t w_groups_per_row)
{
    __shared__ uint32_t warp_max[kWThreads / 32];
    __shared__ Divider block_div;
    // The GEMM that follows in a step may be scheduled as soon as every CTA
    // of this grid is running; it waits for this grid's results itself.
    if (threadIdx.x == 0)
        launch_dependents();
    const int64_t b = blockIdx.x;
    if (b < act_blocks) {
        act_regs_batch<kContiguous>((b * (kActThreads / 32) + (threadIdx.x >> 5)) * 32, x, ldx, qx, ldqx, sx,
                                    x_groups_per_row, x_groups, 0);
    } else {
        const int64_t wb = b - act_blocks;
        weight_block(wb % w_groups_per_row, wb / w_groups_per_row, w, N, ldw, qw, ldqw, sw,
                     w_groups_per_row, warp_max, &block_div, 0);
    }
}

// Resident CTAs of a kernel on the device (cached per kernel; at least 1).
// Callers on several host threads may race to fill the cache; they all store
// the same value.
template <typename Kernel>
int resident_blocks(Kernel kernel, int threads, size_t smem, std::atomic<int>* cache)
{
    int b = cache->load(std::memory_order_relaxed);
    if (b == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, threads, smem) != cudaSuccess ||
            b <= 0) {
            cudaGetLastError();
            b = 1;
        }
        cache->store(b, std::memory_order_relaxed);
    }
    return b;
}

// bf16 weights [N, K] (row stride ld elements) as 128 x 128 boxes, rows of
// 256 B in shared memory (no swizzle).
bool encode_weight_blocks(CUtensorMap* map, const void* w, int64_t N, int64_t K, int64_t ld)
{
    auto enc = get_encoder();
    if (enc == nullptr)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    const cuuint32_t box[2] = {128, 128};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launches the ring kernel over `work` (the grid: every resident CTA, at
// most one per item).
fp8bs_status launch_ring(const DeviceInfo& info, RingWork work, const CUtensorMap& wmap, cudaStream_t s)
{
    static std::mutex mu;
    static bool configured[64] = {};
    static std::atomic<int> per_sm{0};
    int resident = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (info.device < 0 || info.device >= 64)
            return FP8BS_ERR_CUDA;
        if (!configured[info.device]) {
            if (cudaFuncSetAttribute(quantize_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kRingSmemBytes)) != cudaSuccess) {
                cudaGetLastError();
                return FP8BS_ERR_CUDA;
            }
            configured[info.device] = true;
        }
        resident = resident_blocks(quantize_ring_kernel, kRingThreads, kRingSmemBytes, &per_sm);
    }
    work.err = device_error_word();
    if (work.err == nullptr)
        return FP8BS_ERR_CUDA;
    const int64_t items = work.n_act + work.n_w;
    const int64_t full = static_cast<int64_t>(info.sm_count) * resident;
    const int grid = static_cast<int>(items < full ? items : full);
    if (grid <= 0)
        return FP8BS_OK;
    quantize_ring_kernel<<<grid, kRingThreads, kRingSmemBytes, s>>>(wmap, work);
    return launch_status();
}

}  // namespace
}  // namespace fp8bs

using namespace fp8bs;

static fp8bs_status quantize_act_impl(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                                      int64_t ldq, float* scale, fp8bs_stream_t stream, int pow2)
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
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    if (ldx == K && ldq == K && total >= kRingMinGroups) {
        RingWork work{};
        work.x = xb;
        work.qx = q;
        work.sx = scale;
        work.x_groups = total;
        work.n_act = (total + kRingItemGroups - 1) / kRingItemGroups;
        work.w_gpr = 1;
        work.pow2 = pow2;
        CUtensorMap none;
        memset(&none, 0, sizeof none);
        return launch_ring(info, work, none, s);
    } else {
        const bool contiguous = ldx == K && ldq == K;
        static std::atomic<int> per_sm[2] = {0, 0};
        const int64_t per_block = (kActThreads / 32) * 32;
        const int64_t needed = (total + per_block - 1) / per_block;
        if (contiguous) {
            const int64_t full = static_cast<int64_t>(info.sm_count) *
                                 resident_blocks(quantize_act_regs_kernel<true>, kActThreads, 0, &per_sm[1]);
            quantize_act_regs_kernel<true><<<static_cast<int>(needed < full ? needed : full), kActThreads, 0,
                                             s>>>(xb, ldx, q, ldq, scale, G, total, pow2);
        } else {
            const int64_t full = static_cast<int64_t>(info.sm_count) *
                                 resident_blocks(quantize_act_regs_kernel<false>, kActThreads, 0, &per_sm[0]);
            quantize_act_regs_kernel<false><<<static_cast<int>(needed < full ? needed : full), kActThreads, 0,
                                              s>>>(xb, ldx, q, ldq, scale, G, total, pow2);
        }
    }
    return launch_status();
}

extern "C" fp8bs_status fp8bs_quantize_act_1x128(const void* x, int64_t M, int64_t K, int64_t ldx,
                                                 uint8_t* q, int64_t ldq, float* scale,
                                                 fp8bs_stream_t stream)
{
    return quantize_act_impl(x, M, K, ldx, q, ldq, scale, stream, 0);
}

extern "C" fp8bs_status fp8bs_quantize_act_1x128_pow2(const void* x, int64_t M, int64_t K, int64_t ldx,
                                                      uint8_t* q, int64_t ldq, float* scale,
                                                      fp8bs_stream_t stream)
{
    return quantize_act_impl(x, M, K, ldx, q, ldq, scale, stream, 1);
}

static fp8bs_status quantize_weight_impl(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q,
                                         int64_t ldq, float* scale, fp8bs_stream_t stream, int pow2)
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
        static_cast<const uint16_t*>(w), N, ldw, q, ldq, scale, G, pow2);
    return launch_status();
}

extern "C" fp8bs_status fp8bs_quantize_weight_128x128(const void* w, int64_t N, int64_t K,
                                                      int64_t ldw, uint8_t* q, int64_t ldq,
                                                      float* scale, fp8bs_stream_t stream)
{
    return quantize_weight_impl(w, N, K, ldw, q, ldq, scale, stream, 0);
}

extern "C" fp8bs_status fp8bs_quantize_weight_128x128_pow2(const void* w, int64_t N, int64_t K,
                                                           int64_t ldw, uint8_t* q, int64_t ldq,
                                                           float* scale, fp8bs_stream_t stream)
{
    return quantize_weight_impl(w, N, K, ldw, q, ldq, scale, stream, 1);
}

extern "C" fp8bs_status fp8bs_quantize_act_and_weight(const void* x, int64_t M, int64_t K, int64_t ldx,
                                                      uint8_t* qx, int64_t ldqx, float* sx,
                                                      const void* w, int64_t N, int64_t Kw,
                                                      int64_t ldw, uint8_t* qw, int64_t ldqw,
                                                      float* sw, fp8bs_stream_t stream)
{
    if (M < 0 || K < 0 || N < 0 || Kw < 0)
        return FP8BS_ERR_INVALID_ARG;
    if (K % 128 != 0 || Kw % 128 != 0)
        return FP8BS_ERR_UNSUPPORTED;
    const bool do_x = M > 0 && K > 0, do_w = N > 0 && Kw > 0;
    if (do_x && (x == nullptr || qx == nullptr || sx == nullptr || ldx < K || ldqx < K ||
                 (ldx * 2) % 16 != 0 || ldqx % 16 != 0 || !aligned16(x) || !aligned16(qx) ||
                 (reinterpret_cast<uintptr_t>(sx) & 3u) != 0))
        return FP8BS_ERR_INVALID_ARG;
    if (do_w && (w == nullptr || qw == nullptr || sw == nullptr || ldw < Kw || ldqw < Kw ||
                 (ldw * 2) % 16 != 0 || ldqw % 16 != 0 || !aligned16(w) || !aligned16(qw) ||
                 (reinterpret_cast<uintptr_t>(sw) & 3u) != 0))
        return FP8BS_ERR_INVALID_ARG;
    if (!do_x && !do_w)
        return FP8BS_OK;
    const int64_t x_groups = do_x ? M * (K / 128) : 0;
    const int64_t act_blocks = (x_groups + kActThreads - 1) / kActThreads;   // 256 groups per block
    const int64_t w_gpr = do_w ? Kw / 128 : 1;
    const int64_t w_blocks = do_w ? ((N + 127) / 128) * w_gpr : 0;
    if (act_blocks + w_blocks > 0x7FFFFFFF)
        return FP8BS_ERR_UNSUPPORTED;
    DeviceInfo info;
    const fp8bs_status st = require_sm103(&info);
    if (st != FP8BS_OK)
        return st;
    const dim3 grid(static_cast<unsigned>(act_blocks + w_blocks));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const auto* xb = static_cast<const uint16_t*>(x);
    const auto* wb = static_cast<const uint16_t*>(w);
    const int64_t x_gpr = do_x ? K / 128 : 1;
    // Contiguous activations: both lists through the ring kernel (activation
    // chunks by bulk copy, weight blocks by 2-D TMA).
    if ((!do_x || (ldx == K && ldqx == K)) && x_groups + w_blocks * 128 >= kRingMinGroups / 2 &&
        (w_blocks == 0 || ((N + 127) / 128 <= 0x7FFFFFFF / 128 && Kw <= 0x7FFFFFFF))) {
        RingWork work{};
        work.x = xb;
        work.qx = qx;
        work.sx = sx;
        work.x_groups = x_groups;
        work.n_act = (x_groups + kRingItemGroups - 1) / kRingItemGroups;
        work.qw = qw;
        work.ldqw = ldqw;
        work.sw = sw;
        work.N = N;
        work.w_gpr = w_gpr;
        work.n_w = w_blocks;
        CUtensorMap wmap;
        memset(&wmap, 0, sizeof wmap);
        if (do_w && !encode_weight_blocks(&wmap, w, N, Kw, ldw))
            return FP8BS_ERR_CUDA;
        return launch_ring(info, work, wmap, s);
    }
    if (!do_x || (ldx == K && ldqx == K))
        quantize_pair_kernel<true><<<grid, kWThreads, 0, s>>>(xb, ldx, qx, ldqx, sx, x_gpr, x_groups, act_blocks,
                                                              wb, N, ldw, qw, ldqw, sw, w_gpr);
    else
        quantize_pair_kernel<false><<<grid, kWThreads, 0, s>>>(xb, ldx, qx, ldqx, sx, x_gpr, x_groups, act_blocks,
                                                               wb, N, ldw, qw, ldqw, sw, w_gpr);
    return launch_status();
}
