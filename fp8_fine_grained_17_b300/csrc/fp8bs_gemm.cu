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
// B300 design (not the pages' Hopper scheme): persistent kernel, 384 threads
// per CTA, one CTA per SM. Each CTA owns 128 output rows x kBN columns of a
// tile (kBN = 128 or 256), and kCtas CTAs share one MMA:
//   kCtas = 1  tile 128 x kBN; the CTA stages A (128 x 128 B) and W
//              (kBN x 128 B) per chunk and issues its own MMAs.
//   kCtas = 2  tile 256 x kBN computed by a CTA pair (cluster of 2) with
//              tcgen05.mma.cta_group::2: each CTA stages its 128 A rows and
//              half of the kBN W rows, the even CTA issues the MMA for both,
//              and each CTA's TMEM gets the accumulator rows of its own A half.
// The 512 TMEM columns hold 512 / kBN accumulator slots: with kBN = 128 four
// chunks can be in flight between the tensor cores and the promotion warps,
// which hides the MMA -> promotion -> MMA hand-off latency.
// Warp roles (each CTA):
//   warp 0      TMA producer: A and W chunks into a shared-memory ring
//               (4 to 8 stages), 128-byte swizzled.
//   warp 1      MMA issuer (one thread; only the even CTA of a pair): 4 x
//               tcgen05.mma.kind::f8f6f4 (K = 32 each) per chunk into the
//               next free TMEM slot, overwriting it (the chunk's partial
//               P_kb).
//   warp 2      TMEM allocator (512 columns).
//   warp 3      builds the expert tile table (a dense launch is one expert).
//   warps 4-11  promotion: each thread owns one row and kBN/2 columns; its
//               scales come straight from global memory, each read two
//               chunks ahead of use. Per chunk it reads P_kb from TMEM
//               (tcgen05.ld, loads in flight during the FMAs), frees the
//               slot, and accumulates acc += (sa * sw) * P_kb in FP32
//               registers with the packed FMA pipe. After the last chunk it
//               converts its row segment and stores it: CTA pairs stage bf16
//               output in shared memory for TMA stores that drain while the
//               next tile runs; single CTAs (and FP32 output) store through a
//               small padded buffer.
// The TMEM slots let the tensor cores compute the next chunks while the
// promotion warps drain earlier ones.
//
// Tiles are dealt to the work units round by round. When the last round
// leaves units idle, its tiles are cut: into K ranges whose partial tiles the
// range owner adds (kSplit = 1, needs a workspace, K >= 4096), or else into
// column pieces computed whole by different units (kSplit = 2, no workspace,
// bit-identical to an uncut launch).
//
// Fused-activation variant (kFused, 128 x 256 tiles, 512 threads): A arrives
// as bf16. Warp 0 also TMA-loads each chunk's A as two 64-wide halves into a
// 3-slot bf16 ring; warps 12-15 (converters) quantize each row's 1x128 group
// with the activation quantizer's codec, write the E4M3 row into the stage's
// A tile in the MMA's swizzled layout (then a proxy fence and one arrival per
// warp on the stage barrier) and put the row's scale into an 8-deep ring that
// the promotion warps read instead of global memory. The result is
// bit-identical to quantizing A first and running the 128 x 256 kernel.
#include <cstdint>
#include <atomic>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "fp8bs_device.cuh"
#include "fp8bs_e4m3.cuh"
#include "fp8bs_host.h"

namespace fp8bs {
namespace {

constexpr int BM = 128;   // output rows per CTA (TMEM lanes)
constexpr int BK = 128;   // K chunk = one scale group
constexpr int kTmemCols = 512;
constexpr int kMaxExperts = 512;
constexpr int kEpiRowBytes = 80;

// kFused: A arrives as bf16 and is quantized to E4M3 1x128 tiles inside the
// kernel (four converter warps, warps 12-15) instead of being read as
// pre-quantized codes; the rest of the pipeline is unchanged.
template <int kCtas, int kBN, bool kFused = false>
struct Cfg {
    // Promotion warps: two column groups of four (TMEM lanes repeat every
    // four warps). Measured on B300: a chunk's promotion is bound by the
    // TMEM read bandwidth plus the packed-FMA pipe, which do not overlap;
    // sixteen warps (four column groups) read TMEM faster in isolation but
    // made the whole kernel 10 % slower.
    static constexpr int kPromo = 8;
    static constexpr int kGroups = kPromo / 4;
    static constexpr int kBRows = kBN / kCtas;            // W rows staged per CTA
    static constexpr int kABytes = BM * BK;
    static constexpr int kBBytes = kBRows * BK;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kSlots = kTmemCols / kBN;        // TMEM accumulator slots
    static constexpr int kCols = kBN / kGroups;           // columns per promotion thread
    // CTA pairs store bf16 output tiles with TMA from a staged copy: each
    // promotion warp's 32 rows x kCols columns as boxes of 32 rows x 64
    // columns (128-byte rows). Single CTAs store synchronously through a
    // small buffer: on B300 the 64 KB a staged 128 x 256 tile needs cost
    // them a pipeline stage, which lost more than the asynchronous store
    // gained.
    static constexpr bool kTmaStore = !kFused && kCtas == 2;
    static constexpr int kOutBoxes = kCols / 64;
    static constexpr int kOutWarpBytes = kTmaStore ? kOutBoxes * 4096 : 32 * kEpiRowBytes;
    // Pipeline stages: the fused kernel gives 48 KB to its bf16 ring and
    // keeps 3; single CTAs take 192 KB (4 or 6 stages); a pair takes what
    // its staged output tile leaves of 220 KB (4 stages for 256 x 256,
    // measured as fast as 6; 7 for 256 x 128).
    static constexpr int kStages = kFused      ? 3
                                   : kTmaStore ? (220 * 1024 - kPromo * kOutWarpBytes) / kStageBytes
                                               : (192 * 1024) / kStageBytes;
    static constexpr int kTileRows = BM * kCtas;          // output rows per tile
    static constexpr int kTileN = kBN;                    // output columns per tile
    static constexpr uint32_t kIdesc = idesc_e4m3_f32(BM * kCtas, kBN);
    static constexpr int kCtrlThreads = kFused ? 256 : 128;   // warps 0-3 (+ the converters)
    static constexpr int kThreads = kCtrlThreads + 32 * kPromo;
    // Registers per thread after setmaxnreg: warps 0-3 (and the converters)
    // shrink, the promotion warps grow; the sums equal the launch budget
    // (the whole register file over the CTA's threads, in steps of 8).
    static constexpr int kLaunchRegs = (65536 / kThreads) & ~7;
    static constexpr int kCtrlRegs = 56;
    static constexpr int kEpilogueRegs =
        ((kLaunchRegs * kThreads - kCtrlRegs * kCtrlThreads) / (32 * kPromo)) & ~7;
    static_assert(kEpilogueRegs <= 256 && kCtrlRegs * kCtrlThreads + kEpilogueRegs * 32 * kPromo <=
                      kLaunchRegs * kThreads, "register split");
    // bf16 A ring (fused only): half chunks of 128 rows x 64 K (16 KB).
    static constexpr int kHalfStages = kFused ? 3 : 1;
    static constexpr int kHalfBytes = kFused ? BM * 64 * 2 : 16;
    static constexpr int kSaRing = kFused ? 8 : 1;       // per-chunk activation scales in flight
};

template <int kCtas, int kBN, bool kFused = false>
struct __align__(1024) Smem {
    using C = Cfg<kCtas, kBN, kFused>;
    uint8_t a[C::kStages][C::kABytes];
    uint8_t b[C::kStages][C::kBBytes];
    uint8_t abf[C::kHalfStages][C::kHalfBytes];   // fused: bf16 A halves, 128-byte swizzled
    uint64_t full[C::kStages];            // even CTA: both CTAs' TMA bytes; fused: the 4 converter warps
    uint64_t empty[C::kStages];
    uint64_t bload[kFused ? C::kStages : 1];   // fused: the stage's W copy landed
    uint64_t bfull[C::kHalfStages];       // fused: bf16 half landed
    uint64_t bempty[C::kHalfStages];      // fused: 4 converter warps done with it
    uint64_t sa_full[C::kSaRing];         // fused: 4 converter warps wrote the chunk's scales
    uint64_t sa_empty[C::kSaRing];        // fused: 8 promotion warps read them
    float sa_ring[C::kSaRing][kFused ? BM : 1];
    uint64_t tmem_full[C::kSlots];
    uint64_t tmem_empty[C::kSlots];       // even CTA: 8 arrivals per CTA of the pair
    uint64_t drain;
    uint64_t part_bar[8];  // split waves: a promotion warp's partial tile landed in shared memory
    uint32_t tmem_base;
    int abort;
    int num_tiles;
    uint32_t issued;     // chunks whose copies the producer issued (or skipped)
    uint32_t consumed;   // chunks the MMA warp consumed
    int skipped;         // chunk left out by the test stall injection, or -1
    // Epilogue staging, one buffer per promotion warp. bf16 output (not
    // fused): the warp's 32 x kCols tile as 128-byte-swizzled boxes that TMA
    // stores read. Otherwise (and for FP32 output) 32 rows x 64 bytes, rows
    // 80 bytes apart so that 16-byte writes of a quarter warp hit distinct
    // banks.
    alignas(C::kTmaStore ? 1024 : 16) uint8_t out[C::kPromo][C::kOutWarpBytes];
    int tile_start[kMaxExperts + 1];   // first tile index of each expert
    int row_start[kMaxExperts + 1];    // copy of expert_offsets
};
template <int kCtas, int kBN, bool kFused = false>
constexpr size_t smem_bytes()
{
    return sizeof(Smem<kCtas, kBN, kFused>) + 1024;   // + alignment slack
}

// 227 KB: the dynamic shared memory a CTA may opt into on sm_100-class GPUs.
constexpr size_t kMaxSmemPerCta = 232448;
static_assert(smem_bytes<1, 256>() <= kMaxSmemPerCta, "shared memory");
static_assert(smem_bytes<1, 128>() <= kMaxSmemPerCta, "shared memory");
static_assert(smem_bytes<2, 256>() <= kMaxSmemPerCta, "shared memory");
static_assert(smem_bytes<2, 128>() <= kMaxSmemPerCta, "shared memory");
static_assert(smem_bytes<1, 256, true>() <= kMaxSmemPerCta, "shared memory");

struct Params {
    const float* sa;          // [rows, KB]
    const float* sw;          // [E, NB, KB]
    void* c;
    int64_t ldc;
    int64_t rows;             // rows of A (M, or total_M)
    int N;
    int KB;
    int NB;                   // N / 128
    int n_tiles;              // N / kBN
    int out_bf16;
    const int32_t* offsets;   // grouped only (nullptr: one expert, rows 0..M)
    int E;
    unsigned int* err;
    unsigned long long wait_ns;   // limit of every bounded wait
    int stall_chunk;              // test fault injection: CTA 0's producer leaves out this chunk's copies (-1: none)
    // Split of the last, partial wave of tiles (dense launches with a
    // workspace): the last sk_tiles tiles are each computed as sk_split
    // ranges of K chunks by different work units. Piece j > 0 writes its
    // FP32 partial tile to sk_part[slot] and sets its warp's flag to `epoch`;
    // piece 0's unit adds the partials in piece order and stores C.
    int sk_tiles;                 // 0: no split
    int sk_split;
    float* sk_part;               // [slot][kCtas][8 warps][kCols / 4][32 lanes] float4
    unsigned int* sk_flag;        // [slot][kCtas][8 warps]
    unsigned int epoch;
    // Or the last wave cut along N (no workspace): each of the last
    // sn_tiles tiles is computed as sn_split column pieces of kBN / sn_split
    // columns by different work units, each over all K chunks.
    int sn_tiles;
    int sn_split;
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
template <typename S>
__device__ __forceinline__ Tile decode_tile(const S& sm, const Params& p, int t)
{
    constexpr int kTileRows = S::C::kTileRows;
    constexpr int kBN = S::C::kTileN;
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
    const int mt_e = (rows_e + kTileRows - 1) / kTileRows;
    const int mt = local % mt_e;
    const int nt = local / mt_e;
    Tile tile;
    tile.m0 = sm.row_start[e] + static_cast<int64_t>(mt) * kTileRows;
    tile.row_end = sm.row_start[e + 1];
    tile.n0 = nt * kBN;
    tile.expert = e;
    tile.b_row0 = e * p.N + tile.n0;
    return tile;
}

// The work of one unit (CTA, or CTA pair): the whole tiles unit,
// unit + n_units, ... below full_end (K chunks [0, KB)), then, when the last
// wave is split, piece `piece` of tile full_end + piece / split: K chunks
// [j KB / split, (j + 1) KB / split) with j = piece % split.
// With kSplit == 2 the pieces are column ranges instead: piece j of a tile
// covers columns [j kBN / split, (j + 1) kBN / split) over all K chunks.
struct Segments {
    int t, step, full_end, KB;
    int piece, split;
    int cur;     // piece index (within its tile) of the range last handed out; 0 for a whole tile
    int ncut;    // 1: pieces are K ranges; > 1: pieces are this many column ranges
    int bn;      // tile width
    int col0;    // columns of the range last handed out: [col0, col0 + width) of its tile
    int width;
    __device__ __forceinline__ bool next(int& tile, int& k0, int& k1)
    {
        if (t < full_end) {
            tile = t;
            k0 = 0;
            k1 = KB;
            t += step;
            cur = 0;
            col0 = 0;
            width = bn;
            return true;
        }
        if (piece < 0)
            return false;
        cur = piece % split;
        tile = full_end + piece / split;
        if (ncut > 1) {
            k0 = 0;
            k1 = KB;
            width = bn / ncut;
            col0 = cur * width;
        } else {
            k0 = cur * KB / split;
            k1 = (cur + 1) * KB / split;
            col0 = 0;
            width = bn;
        }
        piece = -1;
        return true;
    }
};

// kSplit: 0 no split, 1 the last wave's tiles cut into K ranges (hand-over
// through the workspace), 2 cut into column ranges.
template <int kSplit>
__device__ __forceinline__ Segments work_of(const Params& p, int num_tiles, int unit, int n_units, int bn)
{
    Segments w;
    w.KB = p.KB;
    w.t = unit;
    w.step = n_units;
    w.bn = bn;
    w.col0 = 0;
    w.width = bn;
    const int tiles = kSplit == 1 ? p.sk_tiles : (kSplit == 2 ? p.sn_tiles : 0);
    const int cut = kSplit == 1 ? p.sk_split : (kSplit == 2 ? p.sn_split : 1);
    const bool split = kSplit != 0 && tiles > 0 && cut > 1 && num_tiles >= tiles;
    w.full_end = split ? num_tiles - tiles : num_tiles;
    w.split = split ? cut : 1;
    w.ncut = split && kSplit == 2 ? cut : 1;
    w.piece = split && unit < tiles * cut ? unit : -1;
    w.cur = 0;
    return w;
}

// Warp 3: copy and validate expert_offsets (a dense launch uses {0, M}),
// then build tile_start[] (exclusive prefix sum of m-tiles x n-tiles per
// expert).
template <typename S>
__device__ void build_expert_table(S& sm, const Params& p, int lane)
{
    constexpr int kTileRows = S::C::kTileRows;
    bool ok = true;
    for (int base = 0; base <= p.E; base += 32) {
        const int i = base + lane;
        if (i <= p.E)
            sm.row_start[i] =
                p.offsets != nullptr ? p.offsets[i] : (i == 0 ? 0 : static_cast<int>(p.rows));
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
                tiles = ((hi - lo + kTileRows - 1) / kTileRows) * p.n_tiles;
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

// kSplit: the launch splits its last wave, into K ranges (1) or column
// ranges (2) (the instantiations that carry
// the partial-tile hand-over; launches without a split use the other one, so
// their promotion loop is compiled without that code).
template <int kCtas, int kBN, bool kFused = false, int kSplit = 0>
__global__ void __launch_bounds__(Cfg<kCtas, kBN, kFused>::kThreads, 1)
fp8_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                const __grid_constant__ CUtensorMap map_c, const Params p)
{
    using C = Cfg<kCtas, kBN, kFused>;
    using S = Smem<kCtas, kBN, kFused>;
    static_assert(!kFused || (kCtas == 1 && kBN == 256), "the fused kernel is the 128 x 256 tile");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    S& sm = *reinterpret_cast<S*>(smem_raw + (((raw + 1023u) & ~1023u) - raw));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Position in the CTA pair (always 0 for kCtas = 1); tiles are handed out
    // per pair.
    const uint32_t rank = kCtas == 2 ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int unit = static_cast<int>(blockIdx.x) / kCtas;      // work unit of this CTA
    const int n_units = static_cast<int>(gridDim.x) / kCtas;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_addr(&sm.full[s]), kFused ? 4 : 1);   // fused: the 4 converter warps
            mbar_init(smem_addr(&sm.empty[s]), 1);
            if (kFused)
                mbar_init(smem_addr(&sm.bload[s]), 1);
        }
        if constexpr (kFused) {
            for (int h = 0; h < C::kHalfStages; ++h) {
                mbar_init(smem_addr(&sm.bfull[h]), 1);
                mbar_init(smem_addr(&sm.bempty[h]), 4);
            }
            for (int i = 0; i < C::kSaRing; ++i) {
                mbar_init(smem_addr(&sm.sa_full[i]), 4);
                mbar_init(smem_addr(&sm.sa_empty[i]), C::kPromo);
            }
        }
        for (int b = 0; b < C::kSlots; ++b) {
            mbar_init(smem_addr(&sm.tmem_full[b]), 1);
            mbar_init(smem_addr(&sm.tmem_empty[b]), C::kPromo * kCtas);   // one per promotion warp
        }
        mbar_init(smem_addr(&sm.drain), 1);
        for (int w = 0; w < 8; ++w)
            mbar_init(smem_addr(&sm.part_bar[w]), 1);
        sm.abort = 0;
        sm.issued = 0;
        sm.consumed = 0;
        sm.skipped = -1;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0 && p.KB > 0) {
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b);
    }
    if (C::kTmaStore && warp == 1 && lane == 0 && p.out_bf16)
        tma_prefetch_desc(&map_c);
    if (warp == 2) {
        tmem_alloc<kCtas>(smem_addr(&sm.tmem_base), kTmemCols);
        tmem_relinquish<kCtas>();
    }
    // The set-up above touches no global memory, so it may overlap the end
    // of the previous kernel in the stream (programmatic dependent launch);
    // from here on that kernel's results (codes, scales, offsets) are visible.
    grid_dependency_wait();
    if (warp == 3)
        build_expert_table(sm, p, lane);
    tc_fence_before();
    __syncthreads();
    if (kCtas == 2)
        cluster_sync_all();   // both CTAs' barriers exist before any remote use
    tc_fence_after();

    const uint32_t tmem_base = sm.tmem_base;
    const int num_tiles = sm.num_tiles;
    volatile int* abort_flag = &sm.abort;

    if (kFused && warp >= 4 + C::kPromo) {
        regs_dec<C::kCtrlRegs>();
        // -------------------------------------------------- A converters
        // Warp cw handles rows 32 pass + 8 cw + lane/4 (pass = 0..3) of the
        // chunk; the lane quad t = lane & 3 of a row holds its 16-byte
        // pieces 2t, 2t+1 of both bf16 halves (K 16t..16t+15 and
        // 64+16t..64+16t+15), so the row's amax is a quad max-exchange and
        // its codes are the 16-byte E4M3 pieces t and 4+t of the row.
        // Scale and codes are those of the 1x128 activation quantizer
        // (same codec); codes go to the stage's A tile in the MMA's
        // 128-byte-swizzled layout, scales to the ring the promotion warps
        // read.
        const int cw = warp - 4 - C::kPromo;
        const int qrow = lane >> 2;
        const int t4 = lane & 3;
        uint32_t chunk = 0;
        bool ok = true;
        Segments work = work_of<kSplit>(p, num_tiles, unit, n_units, kBN);
        int t, k0, k1;
        while (ok && work.next(t, k0, k1)) {
            for (int kb = k0; kb < k1; ++kb, ++chunk) {
                const uint32_t hs0 = (2 * chunk) % C::kHalfStages, hs1 = (2 * chunk + 1) % C::kHalfStages;
                const uint32_t hp0 = ((2 * chunk) / C::kHalfStages) & 1u;
                const uint32_t hp1 = ((2 * chunk + 1) / C::kHalfStages) & 1u;
                const uint32_t s = chunk % C::kStages, sp = (chunk / C::kStages) & 1u;
                const uint32_t ring = chunk % C::kSaRing, rp = (chunk / C::kSaRing) & 1u;
                const bool ready = mbar_wait(smem_addr(&sm.bfull[hs0]), hp0, abort_flag, p.err, p.wait_ns) &&
                                   mbar_wait(smem_addr(&sm.bfull[hs1]), hp1, abort_flag, p.err, p.wait_ns) &&
                                   mbar_wait(smem_addr(&sm.empty[s]), sp ^ 1u, abort_flag, p.err, p.wait_ns) &&
                                   mbar_wait(smem_addr(&sm.sa_empty[ring]), rp ^ 1u, abort_flag, p.err, p.wait_ns);
                if (!__all_sync(0xFFFFFFFFu, ready)) {
                    ok = false;
                    break;
                }
                const uint8_t* half0 = sm.abf[hs0];
                const uint8_t* half1 = sm.abf[hs1];
                uint8_t* adst = sm.a[s];
#pragma unroll 1
                for (int pass = 0; pass < 4; ++pass) {
                    const int r = pass * 32 + cw * 8 + qrow;   // row of the tile
                    const int sw = r & 7;                       // 128-byte swizzle phase of the row
                    uint4 v[4];
                    v[0] = *reinterpret_cast<const uint4*>(half0 + r * 128 + (((2 * t4) ^ sw) << 4));
                    v[1] = *reinterpret_cast<const uint4*>(half0 + r * 128 + (((2 * t4 + 1) ^ sw) << 4));
                    v[2] = *reinterpret_cast<const uint4*>(half1 + r * 128 + (((2 * t4) ^ sw) << 4));
                    v[3] = *reinterpret_cast<const uint4*>(half1 + r * 128 + (((2 * t4 + 1) ^ sw) << 4));
                    uint32_t m = absmax_words(v, 4);
                    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
                    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
                    const Divider d = make_divider(bf16_bits_to_f32(m));
                    const bool fast = d.r != 0.0f;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint2 lo = fast ? quantize8_fast_fp(v[2 * h], d) : quantize8(v[2 * h], d);
                        const uint2 hi = fast ? quantize8_fast_fp(v[2 * h + 1], d) : quantize8(v[2 * h + 1], d);
                        const int jf = 4 * h + t4;                  // 16-byte piece of the E4M3 row
                        *reinterpret_cast<uint4*>(adst + r * 128 + ((jf ^ sw) << 4)) =
                            make_uint4(lo.x, lo.y, hi.x, hi.y);
                    }
                    if (t4 == 0)
                        sm.sa_ring[ring][r] = d.s;
                }
                // The codes are read by the tensor cores (async proxy).
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_addr(&sm.full[s]));
                    mbar_arrive(smem_addr(&sm.bempty[hs0]));
                    mbar_arrive(smem_addr(&sm.bempty[hs1]));
                    mbar_arrive(smem_addr(&sm.sa_full[ring]));
                }
            }
        }
    } else if (warp < 4) {
        regs_dec<C::kCtrlRegs>();
        if (warp == 0) {
            // ---------------------------------------------------- TMA producer
            // The whole warp runs the loop; one elected lane issues the copies.
            uint32_t chunk = 0;       // chunks whose copies were issued (or left out)
            uint32_t halves = 0;      // fused: bf16 halves issued (or left out)
            int skipped = -1;
            uint32_t s = 0, ph = 0;   // stage and its phase parity
            bool ok = true;
            const bool stall_here = p.stall_chunk >= 0 && blockIdx.x == 0;
            Segments work = work_of<kSplit>(p, num_tiles, unit, n_units, kBN);
            int t, k0, k1;
            while (ok && work.next(t, k0, k1)) {
                const Tile tile = decode_tile(sm, p, t);
                const int32_t a_row = static_cast<int32_t>(tile.m0) + static_cast<int32_t>(rank) * BM;
                // A column piece (kSplit == 2) loads the W rows of its own
                // columns, width / kCtas per CTA, at the front of the stage
                // (the rest of the box is loaded but not used: a box of the
                // piece's rows measured no faster).
                const int32_t b_row =
                    tile.b_row0 + work.col0 + static_cast<int32_t>(rank) * (work.width / kCtas);
                for (int kb = k0; kb < k1; ++kb) {
                    const bool skip = stall_here && chunk == static_cast<uint32_t>(p.stall_chunk);
                    if constexpr (kFused) {
                        // The chunk's bf16 A as two 64-wide halves (128 B
                        // rows, 128-byte swizzle) for the converter warps.
                        for (uint32_t h = 0; h < 2; ++h) {
                            const uint32_t hs = halves % C::kHalfStages;
                            const uint32_t hph = (halves / C::kHalfStages) & 1u;
                            const bool free_ =
                                mbar_wait(smem_addr(&sm.bempty[hs]), hph ^ 1u, abort_flag, p.err, p.wait_ns);
                            if (!__all_sync(0xFFFFFFFFu, free_)) {
                                ok = false;
                                break;
                            }
                            if (!skip && elect_one()) {
                                const uint32_t bar = smem_addr(&sm.bfull[hs]);
                                mbar_arrive_expect_tx(bar, C::kHalfBytes);
                                tma_load_2d(smem_addr(sm.abf[hs]), &map_a, bar, kb * BK + 64 * h, a_row);
                            }
                            __syncwarp();
                            ++halves;
                        }
                        if (!ok)
                            break;
                    }
                    const bool ready = mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1u, abort_flag, p.err, p.wait_ns);
                    if (!__all_sync(0xFFFFFFFFu, ready)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = smem_addr(&sm.full[s]);
                    if (!skip && elect_one()) {
                        if (kFused) {
                            // A comes from the converter warps (their 4 arrivals
                            // on full[s]); W lands on its own barrier.
                            const uint32_t bl = smem_addr(&sm.bload[s]);
                            mbar_arrive_expect_tx(bl, C::kBBytes);
                            tma_load_2d(smem_addr(sm.b[s]), &map_b, bl, kb * BK, b_row);
                        } else if (kCtas == 1) {
                            mbar_arrive_expect_tx(full, C::kStageBytes);
                            tma_load_2d(smem_addr(sm.a[s]), &map_a, full, kb * BK, a_row);
                            tma_load_2d(smem_addr(sm.b[s]), &map_b, full, kb * BK, b_row);
                        } else {
                            // Both CTAs' copies complete on the even CTA's barrier.
                            if (leader)
                                mbar_arrive_expect_tx(full, 2 * C::kStageBytes);
                            const uint32_t full0 = map_to_cta(full, 0);
                            tma_load_2d_pair(smem_addr(sm.a[s]), &map_a, full0, kb * BK, a_row);
                            tma_load_2d_pair(smem_addr(sm.b[s]), &map_b, full0, kb * BK, b_row);
                        }
                    }
                    __syncwarp();
                    if (skip)
                        skipped = static_cast<int>(chunk);
                    ++chunk;
                    if (++s == C::kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (lane == 0) {
                sm.issued = chunk;
                sm.skipped = skipped;
            }
            if (!ok) {
                // Let the copies already issued land before the CTA exits.
                // A stage (a bf16 half) is refilled only after its previous
                // chunk was consumed, which needs that chunk's copies to
                // have landed, so only the last kStages chunks (kHalfStages
                // halves) can still be in flight. CTA pairs retire their
                // copies at the end of the kernel, where the even CTA knows
                // what both CTAs issued.
                const uint32_t c0 = chunk > C::kStages ? chunk - C::kStages : 0;
                if constexpr (kFused) {
                    const uint32_t h0 = halves > C::kHalfStages ? halves - C::kHalfStages : 0;
                    for (uint32_t hc = h0; hc < halves; ++hc)
                        if (static_cast<int>(hc / 2) != skipped)
                            mbar_wait_drain(smem_addr(&sm.bfull[hc % C::kHalfStages]),
                                            (hc / C::kHalfStages) & 1u, p.wait_ns, p.err);
                    for (uint32_t c = c0; c < chunk; ++c)
                        if (static_cast<int>(c) != skipped)
                            mbar_wait_drain(smem_addr(&sm.bload[c % C::kStages]), (c / C::kStages) & 1u,
                                            p.wait_ns, p.err);
                } else if (kCtas == 1) {
                    for (uint32_t c = c0; c < chunk; ++c)
                        if (static_cast<int>(c) != skipped)
                            mbar_wait_drain(smem_addr(&sm.full[c % C::kStages]), (c / C::kStages) & 1u,
                                            p.wait_ns, p.err);
                }
            }
        } else if (warp == 1 && leader) {
            // ------------------------------------------------------ MMA issuer
            // The whole warp runs the loop with warp-uniform values; one
            // elected lane issues each chunk's MMAs and commits (the same
            // lane every time: the warp is converged and fully active).
            uint32_t s = 0, ph = 0;   // smem stage and its phase parity
            uint32_t b = 0, tph = 0;  // TMEM slot and its phase parity
            uint32_t consumed = 0;
            bool ok = true;
            // Descriptors of stage 0; stage s / K step k add their byte offset
            // >> 4 to the start-address field (shared addresses < 256 KB).
            const uint64_t adesc0 = smem_desc_k_sw128(smem_addr(sm.a[0]));
            const uint64_t bdesc0 = smem_desc_k_sw128(smem_addr(sm.b[0]));
            Segments work = work_of<kSplit>(p, num_tiles, unit, n_units, kBN);
            int t, k0, k1;
            while (ok && work.next(t, k0, k1)) {
                // A column piece: an MMA of N = its width into the front of
                // the slot.
                const uint32_t idesc = work.width == kBN ? C::kIdesc : idesc_e4m3_f32(BM * kCtas, work.width);
                for (int kb = k0; kb < k1; ++kb) {
                    const uint32_t empty_bar = smem_addr(&sm.tmem_empty[b]);
                    const uint32_t full_bar = smem_addr(&sm.full[s]);
                    const uint32_t bload_bar = smem_addr(&sm.bload[kFused ? s : 0]);
                    // The conditions are usually met already: test them
                    // together, wait only if one is not.
                    bool ready = mbar_test_wait(empty_bar, tph ^ 1u) & mbar_test_wait(full_bar, ph);
                    if (kFused)
                        ready = ready & mbar_test_wait(bload_bar, ph);
                    if (!__all_sync(0xFFFFFFFFu, ready)) {
                        ready = mbar_wait(empty_bar, tph ^ 1u, abort_flag, p.err, p.wait_ns) &&
                                mbar_wait(full_bar, ph, abort_flag, p.err, p.wait_ns) &&
                                (!kFused || mbar_wait(bload_bar, ph, abort_flag, p.err, p.wait_ns));
                        if (!__all_sync(0xFFFFFFFFu, ready)) {
                            ok = false;
                            break;
                        }
                    }
                    tc_fence_after();
                    if (elect_one()) {
                        const uint32_t d = tmem_base + b * kBN;
                        const uint64_t ad = adesc0 + ((s * C::kABytes) >> 4);
                        const uint64_t bd = bdesc0 + ((s * C::kBBytes) >> 4);
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k)
                            mma_e4m3<kCtas>(d, ad + 2 * k, bd + 2 * k, idesc, k > 0 ? 1u : 0u);
                        mma_commit<kCtas>(smem_addr(&sm.empty[s]));
                        mma_commit<kCtas>(smem_addr(&sm.tmem_full[b]));
                    }
                    __syncwarp();
                    ++consumed;
                    if (++s == C::kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (++b == C::kSlots) {
                        b = 0;
                        tph ^= 1u;
                    }
                }
            }
            if (lane == 0)
                sm.consumed = consumed;
            // All MMAs issued by this warp complete before TMEM is released.
            if (elect_one()) {
                mma_commit<kCtas>(smem_addr(&sm.drain));
                mbar_wait_drain(smem_addr(&sm.drain), 0, p.wait_ns, p.err);
            }
            __syncwarp();
        }
    } else {
        regs_inc<C::kEpilogueRegs>();
        // ------------------------------------------------------- promotion
        const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
        const int half = (warp - 4) >> 2;      // column group: output columns kCols*half .. +kCols-1
        const int r = quarter * 32 + lane;
        // The slot-free arrivals of both CTAs of a pair go to the even CTA
        // (tmem_empty[b] is at tmem_empty[0] + 8 b bytes).
        const uint32_t tmem_empty0 = kCtas == 1 ? smem_addr(&sm.tmem_empty[0])
                                                : map_to_cta(smem_addr(&sm.tmem_empty[0]), 0);
        uint32_t chunk = 0;
        bool ok = true;
        auto give_slot = [&](uint32_t c) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (kCtas == 1)
                    mbar_arrive(tmem_empty0 + 8 * (c % C::kSlots));
                else
                    mbar_arrive_remote(tmem_empty0 + 8 * (c % C::kSlots));
            }
        };
        // Promotes chunk c with the given scale into acc; false if the wait
        // gave up.
        auto promote = [&](uint32_t c, float scale, float2 (&acc)[C::kCols / 2]) -> bool {
            const uint32_t b = c % C::kSlots;
            const bool ready = mbar_wait(smem_addr(&sm.tmem_full[b]), (c / C::kSlots) & 1u,
                                         abort_flag, p.err, p.wait_ns);
            // The warp continues only if every lane saw the phases complete:
            // the TMEM loads below are warp-collective.
            if (!__all_sync(0xFFFFFFFFu, ready))
                return false;
            tc_fence_after();
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * kBN + half * C::kCols;
            const float2 scale2 = make_float2(scale, scale);
            if constexpr (C::kCols == 64) {
                // Both 32-column loads in flight at once, one wait, the slot
                // goes back, then the arithmetic.
                uint32_t x0[32], x1[32];
                tmem_ld_32x32b_x32(taddr, x0);
                tmem_ld_32x32b_x32(taddr + 32, x1);
                tmem_ld_wait(x0);
                tmem_ld_tie(x1);
                give_slot(c);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    acc[i] = __ffma2_rn(
                        make_float2(__uint_as_float(x0[2 * i]), __uint_as_float(x0[2 * i + 1])),
                        scale2, acc[i]);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    acc[16 + i] = __ffma2_rn(
                        make_float2(__uint_as_float(x1[2 * i]), __uint_as_float(x1[2 * i + 1])),
                        scale2, acc[16 + i]);
            } else if constexpr (C::kCols == 128) {
                // Column blocks of 16, loaded two at a time: blocks j+2 and
                // j+3 are in flight while j and j+1 are accumulated (three
                // buffers; one wait per pair of loads); the slot goes back
                // once the last pair has arrived.
                constexpr int kBlocks = 8;
                uint32_t v[3][16];
                tmem_ld_32x32b_x16(taddr, v[0]);
                tmem_ld_32x32b_x16(taddr + 16, v[1]);
                tmem_ld_wait2(v[0], v[1]);
#pragma unroll
                for (int j = 0; j < kBlocks; j += 2) {
                    const bool more = j + 2 < kBlocks;
                    if (more)
                        tmem_ld_32x32b_x16(taddr + 16 * (j + 2), v[(j + 2) % 3]);
                    else
                        give_slot(c);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        acc[8 * j + i] = __ffma2_rn(make_float2(__uint_as_float(v[j % 3][2 * i]),
                                                                __uint_as_float(v[j % 3][2 * i + 1])),
                                                    scale2, acc[8 * j + i]);
                    if (more)
                        tmem_ld_32x32b_x16(taddr + 16 * (j + 3), v[j % 3]);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        acc[8 * (j + 1) + i] =
                            __ffma2_rn(make_float2(__uint_as_float(v[(j + 1) % 3][2 * i]),
                                                   __uint_as_float(v[(j + 1) % 3][2 * i + 1])),
                                       scale2, acc[8 * (j + 1) + i]);
                    if (more)
                        tmem_ld_wait2(v[(j + 2) % 3], v[j % 3]);
                }
            } else {
                // Column blocks j of 16: the load of block j+1 is in flight
                // while block j is accumulated; the slot goes back once the
                // last load has completed.
                constexpr int kBlocks = C::kCols / 16;
                uint32_t v[2][16];
                tmem_ld_32x32b_x16(taddr, v[0]);
                tmem_ld_wait(v[0]);
#pragma unroll
                for (int j = 0; j < kBlocks; ++j) {
                    if (j + 1 < kBlocks)
                        tmem_ld_32x32b_x16(taddr + 16 * (j + 1), v[(j + 1) & 1]);
                    else
                        give_slot(c);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        acc[8 * j + i] = __ffma2_rn(make_float2(__uint_as_float(v[j & 1][2 * i]),
                                                                __uint_as_float(v[j & 1][2 * i + 1])),
                                                    scale2, acc[8 * j + i]);
                    if (j + 1 < kBlocks)
                        tmem_ld_wait(v[(j + 1) & 1]);
                }
            }
            return true;
        };
        Segments work = work_of<kSplit>(p, num_tiles, unit, n_units, kBN);
        int t, k0, k1;
        while (ok && work.next(t, k0, k1)) {
            const Tile tile = decode_tile(sm, p, t);
            const int n_col = tile.n0 + half * C::kCols;
            if constexpr (kSplit == 2) {
                if (work.width != kBN) {
                    // A column piece of a last-wave tile: this thread's
                    // width / 2 columns of its half (16, 32 or 64), promoted
                    // one 16-column TMEM load at a time with the same
                    // arithmetic as a whole tile, then stored straight from
                    // registers.
                    const int hw = work.width / 2;
                    const int nc = tile.n0 + work.col0 + half * hw;
                    const int nblk = hw / 16;
                    const int64_t srow = min(tile.m0 + rank * BM + r, p.rows - 1);
                    const float* sa_row = p.sa + srow * p.KB;
                    const float* sw_row =
                        p.sw + (static_cast<int64_t>(tile.expert) * p.NB + min(nc / 128, p.NB - 1)) * p.KB;
                    const int last = p.KB - 1;
                    float2 nacc[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        nacc[i] = make_float2(0.0f, 0.0f);
                    float a1 = 0.0f, w1 = 0.0f, a2 = 0.0f, w2 = 0.0f;
                    if (k1 > k0) {
                        a1 = __ldg(sa_row + min(k0, last));
                        w1 = __ldg(sw_row + min(k0, last));
                        a2 = __ldg(sa_row + min(k0 + 1, last));
                        w2 = __ldg(sw_row + min(k0 + 1, last));
                    }
#pragma unroll 1
                    for (int kb = k0; kb < k1; ++kb, ++chunk) {
                        const float2 s2 = make_float2(a1 * w1, a1 * w1);
                        a1 = a2;
                        w1 = w2;
                        a2 = __ldg(sa_row + min(kb + 2, last));
                        w2 = __ldg(sw_row + min(kb + 2, last));
                        const uint32_t b = chunk % C::kSlots;
                        const bool ready = mbar_wait(smem_addr(&sm.tmem_full[b]), (chunk / C::kSlots) & 1u,
                                                     abort_flag, p.err, p.wait_ns);
                        if (!__all_sync(0xFFFFFFFFu, ready)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t taddr =
                            tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * kBN + half * hw;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (j < nblk) {
                                uint32_t v[16];
                                tmem_ld_32x32b_x16(taddr + 16 * j, v);
                                tmem_ld_wait(v);
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    nacc[8 * j + i] = __ffma2_rn(
                                        make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), s2,
                                        nacc[8 * j + i]);
                            }
                        }
                        give_slot(chunk);
                    }
                    if (!ok)
                        break;
                    const int64_t grow = tile.m0 + rank * BM + r;
                    if (nc < p.N && grow < tile.row_end) {
                        if (p.out_bf16) {
                            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.c) + grow * p.ldc + nc;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                if (j < hw / 8) {
                                    uint4 pk;
                                    __nv_bfloat162 h0 = __float22bfloat162_rn(nacc[4 * j + 0]);
                                    __nv_bfloat162 h1 = __float22bfloat162_rn(nacc[4 * j + 1]);
                                    __nv_bfloat162 h2 = __float22bfloat162_rn(nacc[4 * j + 2]);
                                    __nv_bfloat162 h3 = __float22bfloat162_rn(nacc[4 * j + 3]);
                                    memcpy(&pk.x, &h0, 4);
                                    memcpy(&pk.y, &h1, 4);
                                    memcpy(&pk.z, &h2, 4);
                                    memcpy(&pk.w, &h3, 4);
                                    *reinterpret_cast<uint4*>(dst + 8 * j) = pk;
                                }
                            }
                        } else {
                            float* dst = static_cast<float*>(p.c) + grow * p.ldc + nc;
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (j < hw / 4)
                                    *reinterpret_cast<float4*>(dst + 4 * j) =
                                        make_float4(nacc[2 * j].x, nacc[2 * j].y, nacc[2 * j + 1].x, nacc[2 * j + 1].y);
                        }
                    }
                    continue;
                }
            }

            // kCols FP32 accumulators as pairs for the packed FMA pipe.
            float2 acc[C::kCols / 2];
#pragma unroll
            for (int i = 0; i < C::kCols / 2; ++i)
                acc[i] = make_float2(0.0f, 0.0f);
            // Scales straight from global memory: a thread's activation
            // scales sa[row, :] are contiguous, and the warp's weight scales
            // sw[e, n-block, :] are one broadcast address. Each is read two
            // chunks ahead of its use (latency hidden; one chunk in the fused
            // kernel). Rows past the end
            // read the last row; their results are never stored.
            const int64_t srow = min(tile.m0 + rank * BM + r, p.rows - 1);
            const float* sa_row = kFused ? nullptr : p.sa + srow * p.KB;
            const float* sw_row =
                p.sw + (static_cast<int64_t>(tile.expert) * p.NB + min(n_col / 128, p.NB - 1)) * p.KB;
            const int last = p.KB - 1;
            // In the fused kernel the activation scales come from the ring.
            auto ld_sa = [&](int kb) { return kFused ? 1.0f : __ldg(sa_row + min(kb, last)); };
            auto ld_sw = [&](int kb) { return __ldg(sw_row + min(kb, last)); };
            float a1 = 0.0f, w1 = 0.0f, a2 = 0.0f, w2 = 0.0f;   // chunks kb and kb + 1
            if (k1 > k0) {
                a1 = ld_sa(k0);
                w1 = ld_sw(k0);
                if (!kFused) {
                    a2 = ld_sa(k0 + 1);
                    w2 = ld_sw(k0 + 1);
                }
            }
#pragma unroll 1
            for (int kb = k0; kb < k1; ++kb, ++chunk) {
                float scale = a1 * w1;
                if constexpr (kFused) {
                    // One chunk ahead: only the weight scale is loaded here.
                    w1 = ld_sw(kb + 1);
                } else {
                    a1 = a2;
                    w1 = w2;
                    a2 = ld_sa(kb + 2);
                    w2 = ld_sw(kb + 2);
                }
                if constexpr (kFused) {
                    // The converter warps' scale of this row and chunk; the
                    // product is formed in the same order as sa * sw above.
                    const uint32_t ring = chunk % C::kSaRing;
                    const bool got = mbar_wait(smem_addr(&sm.sa_full[ring]), (chunk / C::kSaRing) & 1u,
                                               abort_flag, p.err, p.wait_ns);
                    if (!__all_sync(0xFFFFFFFFu, got)) {
                        ok = false;
                        break;
                    }
                    const float sa_v = sm.sa_ring[ring][r];
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(smem_addr(&sm.sa_empty[ring]));
                    scale = sa_v * scale;
                }
                if (!promote(chunk, scale, acc)) {
                    ok = false;
                    break;
                }
            }
            if (!ok)
                break;

            if (kSplit == 1 && work.split > 1 && t >= work.full_end) {
                // A piece of a split tile. It is the unit's last work, so
                // the pipeline's stage memory is idle (every chunk's MMA has
                // completed); each promotion warp stages its 16 KB of the
                // partial tile there (float4 columns interleaved by lane) and
                // moves it with one bulk copy.
                static_assert(8 * 32 * (C::kCols / 4) * 16 <= C::kStages * C::kStageBytes, "staging");
                const int tl = t - work.full_end;
                constexpr uint32_t kWarpBytes = 32 * (C::kCols / 4) * 16;
                float4* stage = reinterpret_cast<float4*>(&sm.a[0][0] + (warp - 4) * kWarpBytes);
                auto part_of = [&](int j) {
                    const size_t slot = static_cast<size_t>(tl) * (work.split - 1) + (j - 1);
                    return reinterpret_cast<float4*>(p.sk_part) +
                           ((slot * kCtas + rank) * 8 + (warp - 4)) * (C::kCols / 4) * 32;
                };
                auto flag_of = [&](int j) {
                    const size_t slot = static_cast<size_t>(tl) * (work.split - 1) + (j - 1);
                    return p.sk_flag + (slot * kCtas + rank) * 8 + (warp - 4);
                };
                if (work.cur > 0) {
                    // Hand the partial to the tile's owner: shared memory,
                    // one bulk copy to the workspace, then this warp's flag
                    // set to the launch's epoch (release).
#pragma unroll
                    for (int i = 0; i < C::kCols / 4; ++i)
                        stage[i * 32 + lane] =
                            make_float4(acc[2 * i].x, acc[2 * i].y, acc[2 * i + 1].x, acc[2 * i + 1].y);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        bulk_store(part_of(work.cur), smem_addr(stage), kWarpBytes);
                        bulk_commit_and_wait();
                        fence_proxy_async_global();
                        __threadfence();
                        st_release_gpu(flag_of(work.cur), p.epoch);
                    }
                    __syncwarp();
                    continue;
                }
                // The owner (piece 0) adds the other pieces in piece order,
                // each brought into shared memory by one bulk copy.
                const uint32_t bar = smem_addr(&sm.part_bar[warp - 4]);
                for (int j = 1; j < work.split; ++j) {
                    unsigned int* flag = flag_of(j);
                    bool got = wait_flag(flag, p.epoch, abort_flag, p.err, p.wait_ns);
                    if (!__all_sync(0xFFFFFFFFu, got)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(bar, kWarpBytes);
                        bulk_load(smem_addr(stage), part_of(j), kWarpBytes, bar);
                    }
                    got = mbar_wait(bar, (j - 1) & 1u, abort_flag, p.err, p.wait_ns);
                    if (!__all_sync(0xFFFFFFFFu, got)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int i = 0; i < C::kCols / 4; ++i) {
                        const float4 v = stage[i * 32 + lane];
                        acc[2 * i] = make_float2(acc[2 * i].x + v.x, acc[2 * i].y + v.y);
                        acc[2 * i + 1] = make_float2(acc[2 * i + 1].x + v.z, acc[2 * i + 1].y + v.w);
                    }
                    __syncwarp();
                    if (lane == 0)
                        *flag = 0u;   // ready for the next launch that uses the workspace
                }
                if (!ok)
                    break;
            }

            const int64_t row0 = tile.m0 + rank * BM + quarter * 32;   // row of lane 0
            if (n_col >= p.N || row0 >= tile.row_end) {
                // Nothing of this warp's part of the tile lies inside C.
            } else if (C::kTmaStore && p.out_bf16) {
                // bf16 epilogue by TMA stores. Each thread converts its row
                // into the warp's boxes (16-byte piece c of row r at piece
                // c ^ (r & 7): the 128-byte swizzle of the store's tensor
                // map, and distinct banks for every 8 lanes); one lane then
                // issues the stores and the warp goes on to its next tile
                // while they drain. The buffer is rewritten only after the
                // previous tile's stores have read it.
                uint8_t* buf = sm.out[warp - 4];
                if (lane == 0)
                    bulk_wait_read();
                __syncwarp();
#pragma unroll
                for (int b = 0; b < C::kOutBoxes; ++b) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int i = 32 * b + 4 * c;   // columns 64 b + 8 c .. + 7
                        uint4 pk;
                        __nv_bfloat162 h0 = __float22bfloat162_rn(acc[i + 0]);
                        __nv_bfloat162 h1 = __float22bfloat162_rn(acc[i + 1]);
                        __nv_bfloat162 h2 = __float22bfloat162_rn(acc[i + 2]);
                        __nv_bfloat162 h3 = __float22bfloat162_rn(acc[i + 3]);
                        memcpy(&pk.x, &h0, 4);
                        memcpy(&pk.y, &h1, 4);
                        memcpy(&pk.z, &h2, 4);
                        memcpy(&pk.w, &h3, 4);
                        *reinterpret_cast<uint4*>(buf + 4096 * b + 128 * lane + ((c ^ (lane & 7)) << 4)) = pk;
                    }
                }
                // A store writes every row of its box that lies inside C:
                // whole boxes, and boxes at the end of C, go to TMA; a box
                // whose rows run into the next expert's is written row by row
                // (8 lanes per 128-byte row) up to the expert's end.
                if (row0 + 32 <= tile.row_end || tile.row_end == p.rows) {   // rows past p.rows are clipped
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
#pragma unroll
                        for (int b = 0; b < C::kOutBoxes; ++b)
                            tma_store_2d(&map_c, smem_addr(buf + 4096 * b), n_col + 64 * b,
                                         static_cast<int32_t>(row0));
                        bulk_commit();
                    }
                } else {
                    __syncwarp();
                    const int pc = lane & 7;
#pragma unroll
                    for (int b = 0; b < C::kOutBoxes; ++b) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int rr = (lane >> 3) + 4 * i;
                            const uint4 v =
                                *reinterpret_cast<const uint4*>(buf + 4096 * b + 128 * rr + ((pc ^ (rr & 7)) << 4));
                            const int64_t grow = row0 + rr;
                            if (grow < tile.row_end)
                                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.c) + grow * p.ldc +
                                                          n_col + 64 * b + 8 * pc) = v;
                        }
                    }
                }
            } else {
                // Synchronous epilogue (single CTAs; FP32 output): each
                // thread writes 64 bytes of its own row into the warp's
                // buffer, then every store instruction writes 8 rows x 64
                // contiguous bytes of C. Rows past the tile's end (M tail, or
                // the next expert's rows) are not written.
                uint8_t* buf = sm.out[warp - 4];
                const int rl = lane >> 2;    // read phase: rows rl + 8 i, 16-byte chunk lane & 3
                const int ch = lane & 3;
                if (p.out_bf16) {
#pragma unroll
                    for (int j = 0; j < C::kCols / 32; ++j) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uint4 pk;
                            __nv_bfloat162 h0 = __float22bfloat162_rn(acc[16 * j + 4 * k + 0]);
                            __nv_bfloat162 h1 = __float22bfloat162_rn(acc[16 * j + 4 * k + 1]);
                            __nv_bfloat162 h2 = __float22bfloat162_rn(acc[16 * j + 4 * k + 2]);
                            __nv_bfloat162 h3 = __float22bfloat162_rn(acc[16 * j + 4 * k + 3]);
                            memcpy(&pk.x, &h0, 4);
                            memcpy(&pk.y, &h1, 4);
                            memcpy(&pk.z, &h2, 4);
                            memcpy(&pk.w, &h3, 4);
                            *reinterpret_cast<uint4*>(buf + lane * kEpiRowBytes + 16 * k) = pk;
                        }
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int rr = rl + 8 * i;
                            const uint4 v = *reinterpret_cast<const uint4*>(buf + rr * kEpiRowBytes + 16 * ch);
                            const int64_t grow = row0 + rr;
                            if (grow < tile.row_end)
                                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.c) + grow * p.ldc +
                                                          n_col + 32 * j + 8 * ch) = v;
                        }
                        __syncwarp();
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < C::kCols / 16; ++j) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            *reinterpret_cast<float4*>(buf + lane * kEpiRowBytes + 16 * k) =
                                make_float4(acc[8 * j + 2 * k].x, acc[8 * j + 2 * k].y,
                                            acc[8 * j + 2 * k + 1].x, acc[8 * j + 2 * k + 1].y);
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int rr = rl + 8 * i;
                            const float4 v = *reinterpret_cast<const float4*>(buf + rr * kEpiRowBytes + 16 * ch);
                            const int64_t grow = row0 + rr;
                            if (grow < tile.row_end)
                                *reinterpret_cast<float4*>(static_cast<float*>(p.c) + grow * p.ldc + n_col +
                                                           16 * j + 4 * ch) = v;
                        }
                        __syncwarp();
                    }
                }
            }
        }
        // The warp's TMA stores have completed before the CTA (and its
        // shared memory) goes away.
        if (C::kTmaStore && lane == 0)
            bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (kCtas == 2) {
        // (A) Both CTAs' roles are done: no MMA is in flight (the even CTA's
        // MMA warp waited for its last commit) and the counts of issued and
        // consumed chunks are in shared memory.
        cluster_sync_all();
        if (leader && warp == 0) {
            // Copies of both CTAs complete on this CTA's stage barriers. After
            // an abort, chunks past the last one consumed may have been
            // issued by one CTA only: make the barrier expect exactly the
            // bytes that were issued (an arrival for a chunk only the odd CTA
            // issued; the odd CTA's bytes retired for a chunk only this CTA
            // issued), then wait (bounded) until they have landed. In a run
            // without abort the range is empty.
            const uint32_t n0 = sm.issued;
            const uint32_t n1 = ld_cluster_u32(map_to_cta(smem_addr(&sm.issued), 1));
            const int sk0 = sm.skipped;
            const int sk1 = static_cast<int>(ld_cluster_u32(map_to_cta(smem_addr(&sm.skipped), 1)));
            const uint32_t hi = n0 > n1 ? n0 : n1;
            for (uint32_t c = sm.consumed; c < hi; ++c) {
                const bool mine = c < n0 && static_cast<int>(c) != sk0;
                const bool theirs = c < n1 && static_cast<int>(c) != sk1;
                const uint32_t bar = smem_addr(&sm.full[c % C::kStages]);
                if (elect_one()) {
                    if (!mine && theirs)
                        mbar_arrive_expect_tx(bar, C::kStageBytes);
                    else if (mine && !theirs)
                        mbar_complete_tx(bar, C::kStageBytes);
                }
                __syncwarp();
                if (mine || theirs)
                    mbar_wait_drain(bar, (c / C::kStages) & 1u, p.wait_ns, p.err);
            }
        }
        // (B) Every copy into either CTA's shared memory has landed.
        cluster_sync_all();
    }
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc<kCtas>(tmem_base, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side

// Fault injection for the failure-detection tests (fp8bs_test_inject_stall):
// read by every GEMM launch.
std::atomic<long long> g_stall_chunk{-1};
std::atomic<unsigned long long> g_wait_ns{kWaitLimitNs};

// Per-device launch counter: each launch that splits tiles marks its partial
// tiles with a fresh nonzero epoch, so a flag left by an earlier (or
// aborted) launch never matches.
std::atomic<unsigned int> g_epoch[64];

// K chunks per piece of a split tile, at least: handing a partial tile over
// costs about as much as 2-3 chunks (measured on B300), so shorter pieces
// lose more than the balance gains.
constexpr int kMinPieceChunks = 16;

inline size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// How the last wave of a dense launch is split: with T tiles on `units`
// work units, the R = T mod units tiles of the last, partial wave are each
// cut into S = min(units / R, KB / kMinPieceChunks) K ranges (S >= 2), so
// that every unit has work in the last round. Workspace: one FP32 partial
// tile per CTA for each piece after the first, then one flag per promotion
// warp.
struct SplitPlan {
    int tiles = 0;
    int split = 1;
    size_t part_bytes = 0;
    size_t bytes = 0;
};

template <int kCtas, int kBN>
SplitPlan split_plan(int64_t rows, int64_t N, int64_t K, int64_t units)
{
    using C = Cfg<kCtas, kBN>;
    SplitPlan sp;
    const int64_t KB = K / BK;
    const int64_t T = ((rows + C::kTileRows - 1) / C::kTileRows) * ((N + kBN - 1) / kBN);
    if (units <= 0 || T <= 0 || KB < 2 * kMinPieceChunks)
        return sp;
    const int64_t R = T % units;
    if (R == 0)
        return sp;
    int64_t S = units / R;
    if (S > KB / kMinPieceChunks)
        S = KB / kMinPieceChunks;
    if (S < 2)
        return sp;
    sp.tiles = static_cast<int>(R);
    sp.split = static_cast<int>(S);
    const size_t slots = static_cast<size_t>(R) * static_cast<size_t>(S - 1);
    sp.part_bytes = slots * kCtas * BM * kBN * sizeof(float);
    sp.bytes = align256(sp.part_bytes) + slots * kCtas * C::kPromo * sizeof(unsigned int);
    return sp;
}

// How the last wave of a dense launch is cut along N when it is not cut
// along K: with T tiles on U resident units (U >= T: one round), the
// R = T mod U tiles of the last round (all T when they fit in one) are each
// cut into S column pieces, S the largest of 8, 4, 2 with at least 32
// columns a piece and R S <= U. A piece computes its columns over all K
// chunks with the same arithmetic as a whole tile, so the results are those
// of the unsplit launch bit for bit, and no workspace is needed.
struct NSplitPlan {
    int tiles = 0;
    int split = 1;
    int64_t units = 0;   // work units the launch runs on
};

NSplitPlan nsplit_plan(int64_t T, int64_t U, int bn)
{
    NSplitPlan sp;
    if (U <= 0 || T <= 0)
        return sp;
    const int64_t R = T % U;
    if (R == 0)
        return sp;
    for (int S = 8; S >= 2; S /= 2) {
        if (bn / S >= 32 && R * S <= U) {
            sp.tiles = static_cast<int>(R);
            sp.split = S;
            sp.units = (T - R) + R * S < U ? (T - R) + R * S : U;
            break;
        }
    }
    return sp;
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

// bf16 activations [rows, K] with row stride ld elements, as boxes of 64 (K)
// x 128 rows (128-byte rows), 128-byte swizzled: the two halves of a K chunk.
bool encode_bf16_halves(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int64_t ld)
{
    auto enc = get_encoder();
    if (enc == nullptr)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(BM)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// bf16 output C [rows, N] with row stride ldc elements, as boxes of 64
// columns (128-byte rows) x 32 rows, 128-byte swizzled: what one promotion
// warp stores per box.
bool encode_out_bf16(CUtensorMap* map, void* base, int64_t rows, int64_t N, int64_t ldc)
{
    auto enc = get_encoder();
    if (enc == nullptr)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldc) * 2};
    const cuuint32_t box[2] = {64, 32};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Per device and shape: the dynamic shared-memory opt-in and the number of
// work units (CTAs, or CTA pairs, which must share a GPC) resident at once.
template <int kCtas, int kBN, bool kFused = false, int kSplit = 0>
fp8bs_status configure_once(int device, int sm_count, int* max_units)
{
    constexpr int kThreads = Cfg<kCtas, kBN, kFused>::kThreads;
    static std::mutex mu;
    static int units[64] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64)
        return FP8BS_ERR_CUDA;
    if (units[device] == 0) {
        using C = Cfg<kCtas, kBN, kFused>;
        const auto kernel = fp8_gemm_kernel<kCtas, kBN, kFused, kSplit>;
        const size_t smem = smem_bytes<kCtas, kBN, kFused>();
        // setmaxnreg.inc waits until the CTA's register pool can grant the
        // request, so the split must fit in what the kernel is launched with.
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) {
            cudaGetLastError();
            return FP8BS_ERR_CUDA;
        }
        if (fa.numRegs * kThreads < C::kCtrlRegs * C::kCtrlThreads + C::kEpilogueRegs * 32 * C::kPromo)
            return FP8BS_ERR_UNSUPPORTED;
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess) {
            cudaGetLastError();
            return FP8BS_ERR_CUDA;
        }
        int n = sm_count;
        if (kCtas == 2) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(2 * (sm_count / 2));
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = smem;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess ||
                clusters <= 0) {
                cudaGetLastError();
                return FP8BS_ERR_CUDA;
            }
            n = clusters;
        }
        units[device] = n;
    }
    *max_units = units[device];
    return FP8BS_OK;
}

// rows: rows of A; w_rows: rows of the stacked W. The number of tiles is
// computed on the device from the expert table (a dense launch is one
// expert); the grid is the resident maximum, capped by an upper bound of the
// tiles.
// kFused: a points at bf16 activations with row stride lda (elements);
// otherwise at E4M3 codes with row stride K.
// Work units (CTAs, or CTA pairs) a launch of `tile_bound` tiles at most
// runs on.
template <int kCtas, int kBN, bool kFused = false>
fp8bs_status launch_units(const DeviceInfo& info, int64_t tile_bound, int64_t* units)
{
    int max_units = 0;
    const fp8bs_status st = configure_once<kCtas, kBN, kFused>(info.device, info.sm_count, &max_units);
    if (st != FP8BS_OK)
        return st;
    *units = tile_bound < max_units ? tile_bound : max_units;
    return FP8BS_OK;
}

// ws / ws_bytes: workspace for splitting the last wave (dense launches only;
// nullptr: no split).
template <int kCtas, int kBN, bool kFused = false>
fp8bs_status launch(const void* a, int64_t rows, const uint8_t* qw, int64_t w_rows, Params p,
                    int64_t K, cudaStream_t stream, int64_t lda = 0, void* ws = nullptr,
                    size_t ws_bytes = 0)
{
    using C = Cfg<kCtas, kBN, kFused>;
    constexpr int kThreads = C::kThreads;
    DeviceInfo info;
    fp8bs_status st = require_sm103(&info);
    if (st != FP8BS_OK)
        return st;
    p.err = device_error_word();
    if (p.err == nullptr)
        return FP8BS_ERR_CUDA;
    p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    p.stall_chunk = static_cast<int>(g_stall_chunk.load(std::memory_order_relaxed));
    p.n_tiles = (p.N + kBN - 1) / kBN;   // a last partial tile is masked
    const int64_t tile_bound = (rows / C::kTileRows + p.E) * static_cast<int64_t>(p.n_tiles);
    if (tile_bound > 0x7FFFFFFF)
        return FP8BS_ERR_UNSUPPORTED;
    CUtensorMap map_a, map_b, map_c;
    memset(&map_a, 0, sizeof map_a);
    memset(&map_b, 0, sizeof map_b);
    memset(&map_c, 0, sizeof map_c);
    if (K > 0) {
        const bool a_ok = kFused ? encode_bf16_halves(&map_a, a, rows, K, lda)
                                 : encode_operand(&map_a, a, rows, K, BM);
        if (!a_ok || !encode_operand(&map_b, qw, w_rows, K, C::kBRows))
            return FP8BS_ERR_CUDA;
    }
    if (C::kTmaStore && p.out_bf16 && rows > 0 && p.N > 0 && !encode_out_bf16(&map_c, p.c, rows, p.N, p.ldc))
        return FP8BS_ERR_CUDA;
    int64_t units64 = 0;
    st = launch_units<kCtas, kBN, kFused>(info, tile_bound, &units64);
    if (st != FP8BS_OK)
        return st;
    auto kernel = fp8_gemm_kernel<kCtas, kBN, kFused, false>;
    int units = static_cast<int>(units64);
    if (units <= 0)
        return FP8BS_OK;
    bool k_split = false;
    if constexpr (!kFused) {
        if (ws != nullptr && p.offsets == nullptr) {
            const SplitPlan sp = split_plan<kCtas, kBN>(rows, p.N, K, units);
            if (sp.tiles > 0) {
                k_split = true;
                if (ws_bytes < sp.bytes || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
                    return FP8BS_ERR_INVALID_ARG;
                unsigned int e = g_epoch[info.device].fetch_add(1) + 1;
                if (e == 0)
                    e = g_epoch[info.device].fetch_add(1) + 1;
                p.sk_tiles = sp.tiles;
                p.sk_split = sp.split;
                p.sk_part = static_cast<float*>(ws);
                p.sk_flag = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + align256(sp.part_bytes));
                p.epoch = e;
                int split_units = 0;
                st = configure_once<kCtas, kBN, false, 1>(info.device, info.sm_count, &split_units);
                if (st != FP8BS_OK)
                    return st;
                kernel = fp8_gemm_kernel<kCtas, kBN, false, 1>;
            }
        }
        if (!k_split && p.offsets == nullptr) {
            int max_units = 0;
            st = configure_once<kCtas, kBN, false, 2>(info.device, info.sm_count, &max_units);
            if (st != FP8BS_OK)
                return st;
            const int64_t T = ((rows + C::kTileRows - 1) / C::kTileRows) * p.n_tiles;
            const NSplitPlan np = nsplit_plan(T, max_units, kBN);
            if (np.tiles > 0) {
                p.sn_tiles = np.tiles;
                p.sn_split = np.split;
                units = static_cast<int>(np.units);
                kernel = fp8_gemm_kernel<kCtas, kBN, false, 2>;
            }
        }
    }
    // Programmatic dependent launch: the kernel's set-up may overlap the tail
    // of the previous kernel in the stream (it waits for that kernel's
    // results before its first global-memory access).
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kCtas;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.gridDim = dim3(kCtas * units);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes<kCtas, kBN, kFused>();
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = kCtas == 2 ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, kernel, map_a, map_b, map_c, p) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    return FP8BS_OK;
}

// sa == nullptr is accepted when need_sa is false (the fused kernels make
// the activation scales themselves).
fp8bs_status check_common(const void* qa, const float* sa, const void* qw, const float* sw,
                          const void* c, fp8bs_out_dtype out_dtype, int64_t N, int64_t K,
                          int64_t ldc, bool need_sa = true)
{
    // With K == 0 the operands are empty and never read; only C is written.
    if (c == nullptr ||
        (K > 0 && (qa == nullptr || (need_sa && sa == nullptr) || qw == nullptr || sw == nullptr)))
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

Params make_params(const float* sa, const float* sw, void* c, fp8bs_out_dtype out_dtype,
                   int64_t rows, int64_t N, int64_t K, int64_t ldc, const int32_t* offsets, int E)
{
    Params p{};
    p.sa = sa;
    p.sw = sw;
    p.c = c;
    p.ldc = ldc;
    p.rows = rows;
    p.N = static_cast<int>(N);
    p.KB = static_cast<int>(K / BK);
    p.NB = static_cast<int>(N / 128);
    p.out_bf16 = out_dtype == FP8BS_OUT_BF16;
    p.offsets = offsets;
    p.E = E;
    return p;
}

// Tile shape of a launch (fp8bs_tile without AUTO): CTAs per MMA and tile
// width. Measured on B300: for dense GEMMs the CTA pair's 256 x 256 tile is
// as fast as 128 x 256 at K = 7168 and 8 % faster at K = 2048 (each CTA
// stages half of the W tile, so it loads a third less per chunk); for the
// MoE grouped GEMM, whose experts hold few rows, the 128-row tile wastes
// less and is 25 % faster. A dense GEMM of at most 128 rows has one row of
// tiles, so 128-wide tiles run twice as many CTAs (at 128 x 7168 x 2048:
// 9.7 us against 12.8 us with 128 x 256). A 256-wide tile needs
// N % 256 == 0 to be fully used; other N take 128-wide tiles.
fp8bs_tile auto_tile(int64_t N, int64_t M, bool grouped)
{
    if (N % 256 != 0 || (!grouped && M <= 128))
        return FP8BS_TILE_128x128;
    return grouped ? FP8BS_TILE_128x256 : FP8BS_TILE_PAIR_256x256;
}

fp8bs_status launch_tile(fp8bs_tile tile, const uint8_t* qa, int64_t rows, const uint8_t* qw,
                         int64_t w_rows, const Params& p, int64_t K, cudaStream_t s, void* ws = nullptr,
                         size_t ws_bytes = 0)
{
    switch (tile) {
    case FP8BS_TILE_128x256: return launch<1, 256>(qa, rows, qw, w_rows, p, K, s, 0, ws, ws_bytes);
    case FP8BS_TILE_128x128: return launch<1, 128>(qa, rows, qw, w_rows, p, K, s, 0, ws, ws_bytes);
    case FP8BS_TILE_PAIR_256x256: return launch<2, 256>(qa, rows, qw, w_rows, p, K, s, 0, ws, ws_bytes);
    case FP8BS_TILE_PAIR_256x128: return launch<2, 128>(qa, rows, qw, w_rows, p, K, s, 0, ws, ws_bytes);
    default: break;
    }
    return FP8BS_ERR_INVALID_ARG;
}

// Workspace bytes a dense launch of this shape and tile needs to split its
// last wave (0: it does not split).
template <int kCtas, int kBN>
fp8bs_status plan_bytes(int64_t M, int64_t N, int64_t K, size_t* bytes)
{
    using C = Cfg<kCtas, kBN>;
    DeviceInfo info;
    fp8bs_status st = require_sm103(&info);
    if (st != FP8BS_OK)
        return st;
    const int64_t n_tiles = (N + kBN - 1) / kBN;
    int64_t units = 0;
    st = launch_units<kCtas, kBN>(info, (M / C::kTileRows + 1) * n_tiles, &units);
    if (st != FP8BS_OK)
        return st;
    *bytes = split_plan<kCtas, kBN>(M, N, K, units).bytes;
    return FP8BS_OK;
}

fp8bs_status tile_plan_bytes(fp8bs_tile tile, int64_t M, int64_t N, int64_t K, size_t* bytes)
{
    switch (tile) {
    case FP8BS_TILE_128x256: return plan_bytes<1, 256>(M, N, K, bytes);
    case FP8BS_TILE_128x128: return plan_bytes<1, 128>(M, N, K, bytes);
    case FP8BS_TILE_PAIR_256x256: return plan_bytes<2, 256>(M, N, K, bytes);
    case FP8BS_TILE_PAIR_256x128: return plan_bytes<2, 128>(M, N, K, bytes);
    default: break;
    }
    return FP8BS_ERR_INVALID_ARG;
}

bool valid_tile(fp8bs_tile tile, int64_t N)
{
    switch (tile) {
    case FP8BS_TILE_AUTO:
    case FP8BS_TILE_128x256:
    case FP8BS_TILE_128x128:
    case FP8BS_TILE_PAIR_256x128: return true;
    case FP8BS_TILE_PAIR_256x256: return N % 256 == 0;   // the pair splits W tiles in halves
    }
    return false;
}

}  // namespace
}  // namespace fp8bs

using namespace fp8bs;

extern "C" fp8bs_status fp8bs_gemm_tiled(const uint8_t* qa, const float* sa, const uint8_t* qw,
                                         const float* sw, void* c, fp8bs_out_dtype out_dtype,
                                         int64_t M, int64_t N, int64_t K, int64_t ldc,
                                         fp8bs_tile tile, fp8bs_stream_t stream)
{
    if (M < 0 || N < 0 || K < 0)
        return FP8BS_ERR_INVALID_ARG;
    if (K % BK != 0 || N % 128 != 0)
        return FP8BS_ERR_UNSUPPORTED;
    if (!valid_tile(tile, N))
        return FP8BS_ERR_INVALID_ARG;
    if (M == 0 || N == 0)
        return FP8BS_OK;
    fp8bs_status st = check_common(qa, sa, qw, sw, c, out_dtype, N, K, ldc);
    if (st != FP8BS_OK)
        return st;
    if (M > 0x7FFFFFFF)
        return FP8BS_ERR_UNSUPPORTED;
    const Params p = make_params(sa, sw, c, out_dtype, M, N, K, ldc, nullptr, 1);
    return launch_tile(tile == FP8BS_TILE_AUTO ? auto_tile(N, M, false) : tile, qa, M, qw, N, p, K,
                       reinterpret_cast<cudaStream_t>(stream));
}

extern "C" fp8bs_status fp8bs_gemm_workspace_size(int64_t M, int64_t N, int64_t K, fp8bs_tile tile,
                                                  size_t* bytes)
{
    if (bytes == nullptr || M < 0 || N < 0 || K < 0)
        return FP8BS_ERR_INVALID_ARG;
    *bytes = 0;
    if (K % BK != 0 || N % 128 != 0)
        return FP8BS_ERR_UNSUPPORTED;
    if (!valid_tile(tile, N))
        return FP8BS_ERR_INVALID_ARG;
    if (M == 0 || N == 0 || K == 0)
        return FP8BS_OK;
    if (M > 0x7FFFFFFF || N > (int64_t(1) << 24) || K > (int64_t(1) << 31) - BK)
        return FP8BS_ERR_UNSUPPORTED;
    return tile_plan_bytes(tile == FP8BS_TILE_AUTO ? auto_tile(N, M, false) : tile, M, N, K, bytes);
}

extern "C" fp8bs_status fp8bs_gemm_ws(const uint8_t* qa, const float* sa, const uint8_t* qw,
                                      const float* sw, void* c, fp8bs_out_dtype out_dtype, int64_t M,
                                      int64_t N, int64_t K, int64_t ldc, fp8bs_tile tile,
                                      void* workspace, size_t workspace_bytes, fp8bs_stream_t stream)
{
    if (M < 0 || N < 0 || K < 0)
        return FP8BS_ERR_INVALID_ARG;
    if (K % BK != 0 || N % 128 != 0)
        return FP8BS_ERR_UNSUPPORTED;
    if (!valid_tile(tile, N))
        return FP8BS_ERR_INVALID_ARG;
    if (M == 0 || N == 0)
        return FP8BS_OK;
    fp8bs_status st = check_common(qa, sa, qw, sw, c, out_dtype, N, K, ldc);
    if (st != FP8BS_OK)
        return st;
    if (M > 0x7FFFFFFF)
        return FP8BS_ERR_UNSUPPORTED;
    const Params p = make_params(sa, sw, c, out_dtype, M, N, K, ldc, nullptr, 1);
    return launch_tile(tile == FP8BS_TILE_AUTO ? auto_tile(N, M, false) : tile, qa, M, qw, N, p, K,
                       reinterpret_cast<cudaStream_t>(stream), workspace, workspace_bytes);
}

extern "C" fp8bs_status fp8bs_gemm(const uint8_t* qa, const float* sa, const uint8_t* qw,
                                   const float* sw, void* c, fp8bs_out_dtype out_dtype, int64_t M,
                                   int64_t N, int64_t K, int64_t ldc, fp8bs_stream_t stream)
{
    return fp8bs_gemm_tiled(qa, sa, qw, sw, c, out_dtype, M, N, K, ldc, FP8BS_TILE_AUTO, stream);
}

extern "C" fp8bs_status fp8bs_grouped_gemm_tiled(const uint8_t* qa, const float* sa,
                                                 const int32_t* expert_offsets, int32_t E,
                                                 int64_t total_M, const uint8_t* qw,
                                                 const float* sw, void* c,
                                                 fp8bs_out_dtype out_dtype, int64_t N, int64_t K,
                                                 int64_t ldc, fp8bs_tile tile,
                                                 fp8bs_stream_t stream)
{
    if (E < 1 || total_M < 0 || N < 0 || K < 0)
        return FP8BS_ERR_INVALID_ARG;
    if (E > kMaxExperts || K % BK != 0 || N % 128 != 0)
        return FP8BS_ERR_UNSUPPORTED;
    if (!valid_tile(tile, N))
        return FP8BS_ERR_INVALID_ARG;
    if (total_M == 0 || N == 0)
        return FP8BS_OK;
    if (expert_offsets == nullptr || (reinterpret_cast<uintptr_t>(expert_offsets) & 3u) != 0)
        return FP8BS_ERR_INVALID_ARG;
    fp8bs_status st = check_common(qa, sa, qw, sw, c, out_dtype, N, K, ldc);
    if (st != FP8BS_OK)
        return st;
    if (total_M > 0x7FFFFFFF || static_cast<int64_t>(E) * N > 0x7FFFFFFF)
        return FP8BS_ERR_UNSUPPORTED;
    const Params p = make_params(sa, sw, c, out_dtype, total_M, N, K, ldc, expert_offsets, E);
    return launch_tile(tile == FP8BS_TILE_AUTO ? auto_tile(N, total_M, true) : tile, qa, total_M, qw,
                       static_cast<int64_t>(E) * N, p, K, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" fp8bs_status fp8bs_grouped_gemm(const uint8_t* qa, const float* sa,
                                           const int32_t* expert_offsets, int32_t E,
                                           int64_t total_M, const uint8_t* qw, const float* sw,
                                           void* c, fp8bs_out_dtype out_dtype, int64_t N, int64_t K,
                                           int64_t ldc, fp8bs_stream_t stream)
{
    return fp8bs_grouped_gemm_tiled(qa, sa, expert_offsets, E, total_M, qw, sw, c, out_dtype, N, K,
                                    ldc, FP8BS_TILE_AUTO, stream);
}

// Row stride checks of a bf16 activation operand of the fused kernels.
static fp8bs_status check_bf16_act(const void* a, int64_t lda, int64_t K)
{
    if (K > 0 && (a == nullptr || lda < K || (lda * 2) % 16 != 0 || !aligned16(a)))
        return FP8BS_ERR_INVALID_ARG;
    return FP8BS_OK;
}

extern "C" fp8bs_status fp8bs_gemm_bf16_act(const void* a, int64_t lda, const uint8_t* qw,
                                            const float* sw, void* c, fp8bs_out_dtype out_dtype,
                                            int64_t M, int64_t N, int64_t K, int64_t ldc,
                                            fp8bs_stream_t stream)
{
    if (M < 0 || N < 0 || K < 0)
        return FP8BS_ERR_INVALID_ARG;
    if (K % BK != 0 || N % 128 != 0)
        return FP8BS_ERR_UNSUPPORTED;
    if (M == 0 || N == 0)
        return FP8BS_OK;
    fp8bs_status st = check_bf16_act(a, lda, K);
    if (st != FP8BS_OK)
        return st;
    st = check_common(a, nullptr, qw, sw, c, out_dtype, N, K, ldc, false);
    if (st != FP8BS_OK)
        return st;
    if (M > 0x7FFFFFFF)
        return FP8BS_ERR_UNSUPPORTED;
    const Params p = make_params(nullptr, sw, c, out_dtype, M, N, K, ldc, nullptr, 1);
    return launch<1, 256, true>(a, M, qw, N, p, K, reinterpret_cast<cudaStream_t>(stream), lda);
}

extern "C" fp8bs_status fp8bs_grouped_gemm_bf16_act(const void* a, int64_t lda,
                                                    const int32_t* expert_offsets, int32_t E,
                                                    int64_t total_M, const uint8_t* qw,
                                                    const float* sw, void* c,
                                                    fp8bs_out_dtype out_dtype, int64_t N, int64_t K,
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
    fp8bs_status st = check_bf16_act(a, lda, K);
    if (st != FP8BS_OK)
        return st;
    st = check_common(a, nullptr, qw, sw, c, out_dtype, N, K, ldc, false);
    if (st != FP8BS_OK)
        return st;
    if (total_M > 0x7FFFFFFF || static_cast<int64_t>(E) * N > 0x7FFFFFFF)
        return FP8BS_ERR_UNSUPPORTED;
    const Params p = make_params(nullptr, sw, c, out_dtype, total_M, N, K, ldc, expert_offsets, E);
    return launch<1, 256, true>(a, total_M, qw, static_cast<int64_t>(E) * N, p, K,
                                reinterpret_cast<cudaStream_t>(stream), lda);
}

extern "C" fp8bs_status fp8bs_test_inject_stall(int64_t chunk, int64_t wait_limit_ns)
{
    if (chunk < 0) {
        g_stall_chunk.store(-1);
        g_wait_ns.store(kWaitLimitNs);
        return FP8BS_OK;
    }
    if (chunk > 0x7FFFFFFF || wait_limit_ns < 100000 || wait_limit_ns > 10000000000ll)
        return FP8BS_ERR_INVALID_ARG;
    g_wait_ns.store(static_cast<unsigned long long>(wait_limit_ns));
    g_stall_chunk.store(chunk);
    return FP8BS_OK;
}

// ----------------------------------------------------------------------------
// Allocation-free variant of fp8bs_gemm_ws, for callers that cannot allocate
// device memory at the point of the call (an allocator that must not be
// re-entered from inside a callback, a plug-in that may not own memory, code
// that runs where a cudaMalloc would synchronize or fail). Its workspace is
// this file-scope array: every GPU that loads the library holds it until the
// process exits, and every call on a device shares it.
namespace fp8bs {
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(12) << 20;   // 12 MiB
// Zero at load. The kernel needs no part of it cleared per call: a flag
// counts only when it holds the launch's own epoch (a per-device counter
// that never repeats a value in practice), and owners reset the flags they
// consume; the partial tiles are always written before they are read.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64];

// Device address of the array on the current device, looked up once per
// device (with that device current) and cached.
fp8bs_status noalloc_scratch(const DeviceInfo& info, void** out)
{
    if (info.device < 0 || info.device >= 64)
        return FP8BS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[info.device] == nullptr) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return FP8BS_ERR_CUDA;
        }
        g_noalloc_addr[info.device] = ptr;
    }
    *out = g_noalloc_addr[info.device];
    return FP8BS_OK;
}
}  // namespace
}  // namespace fp8bs

extern "C" fp8bs_status fp8bs_gemm_noalloc(const uint8_t* qa, const float* sa, const uint8_t* qw,
                                           const float* sw, void* c, fp8bs_out_dtype out_dtype,
                                           int64_t M, int64_t N, int64_t K, int64_t ldc,
                                           fp8bs_tile tile, fp8bs_stream_t stream)
{
    size_t need = 0;
    fp8bs_status st = fp8bs_gemm_workspace_size(M, N, K, tile, &need);
    if (st != FP8BS_OK)
        return st;
    if (need > kNoAllocScratchBytes)
        return FP8BS_ERR_UNSUPPORTED;   // this shape's split needs more than the fixed scratch
    void* ws = nullptr;
    if (need > 0) {
        DeviceInfo info;
        st = require_sm103(&info);
        if (st != FP8BS_OK)
            return st;
        st = noalloc_scratch(info, &ws);
        if (st != FP8BS_OK)
            return st;
    }
    return fp8bs_gemm_ws(qa, sa, qw, sw, c, out_dtype, M, N, K, ldc, tile, ws,
                         need > 0 ? kNoAllocScratchBytes : 0, stream);
}
