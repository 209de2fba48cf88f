// tc_gemv.cuh -- batched-verify decode GEMV (m = 2..8 activation rows) on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// y[i][r] = sum_c e4m3(W[r][c]) * S[r/128][c/128] * x[i][c] ("Module dsv4_gpu"
// page, struct Fp8Dense; "Struct Dsv4Gpu" page, verify_batch_dev: T = k+1 rows).
// At m = 8 the CUDA-core form needs 8 FP32 FMAs per weight byte and the FP32
// pipe caps it near half the HBM rate, so here the tensor cores do the
// products and the CUDA cores only re-encode the weights:
//   * A (M = 128 weight rows x K): f16 = e4m3(code) * S * 2^-q, one cvt and
//     one f16 multiply per pair of codes.  e4m3 values are f16 values; S is a
//     power of two and q (per 128-row scale block) puts every S * 2^-q of the
//     block in [2^-15, 2^7], where the product is an exact f16.
//   * B (N = 16 x K): for each activation row i, v = x_i * 2^p_i split into two
//     f16 planes, hi = f16(v) in row i and lo = f16(v - hi) in row 8 + i (p_i
//     makes max|v| < 2^15 over the whole row).  hi + lo keeps about 22 bits.
//   * D (128 x 16 f32, tensor memory): y[i][r] = (D[r][i] + D[r][8 + i]) * 2^(q - p_i).
// Products of f16 pairs are exact in f32 and accumulate in f32.
//
// Pipeline per CTA (one per SM):
//   producer warp, lane 0: ring stages of two 128-column K-blocks; per K-block
//                  one 2-D TMA box of 128 rows x 128 e4m3 bytes (32 rows for
//                  tiles that short), SWIZZLE_128B and L2 evict-first, plus one
//                  2-D box of the m activation rows x 256 f32 for the stage.
//                  The copy engine pays a fixed cost per request, so requests
//                  are few and large.  The weight boxes of the first stages are
//                  issued before the grid dependency wait (weights are never
//                  outputs of the preceding kernel), x only after it;
//   converter warps: each thread converts one tile row's K slice (two warps
//                  per 32-lane quarter of tensor memory) to f16 and stores it
//                  into its own TMEM lane (tcgen05.st; row r in lane r, two f16
//                  of consecutive K per 32-bit column), and all of them build
//                  the 16 x 128 B tile in shared memory from the x slice (UMMA
//                  K-major, no swizzle: 8 x 16-byte core matrices, LBO = 128 B,
//                  SBO = 2048 B); the first four warps also run the epilogue;
//   MMA warp, lane 0: 8 x tcgen05.mma (K = 16 each, A from tensor memory, B
//                  from shared memory) per K-block, commits to mbarriers that
//                  free the operand stage / publish the accumulator (two
//                  accumulators of 16 columns alternate).
// Keeping A in tensor memory spares shared memory the f16 tile's write and the
// tensor core's read of it (64 KiB per K-block), which bounded the rate.
// The f16 scale factors S * 2^-q are tabulated in shared memory before the
// roles split.
// Every wait is a bounded mbarrier wait; any timeout raises a shared abort
// flag, every role leaves its loop, the status word records it, and the tensor
// memory is freed after the last commit has landed (bounded).  A CTA whose
// 128-row blocks have a scale spread above 2^22, or a scale that is not a
// positive finite power of two, computes its rows with a plain CUDA-core loop
// instead (same sums, no tensor cores).
#pragma once

#include <cuda.h>

#include "stream_gemv.cuh"

#ifndef TC_CONV_WARPS
#define TC_CONV_WARPS 8
#endif
#ifndef TC_E_STAGES
#define TC_E_STAGES 4
#endif
#ifndef TC_AB_STAGES
#define TC_AB_STAGES 4
#endif
#ifndef TC_SPIN
#define TC_SPIN 0
#endif
#ifndef TC_MMA_WARPS
#define TC_MMA_WARPS 2
#endif
#ifndef TC_B_WARPS
#define TC_B_WARPS 4
#endif
#ifndef TC_MMA_SLEEP
#define TC_MMA_SLEEP 1
#endif

namespace fp8blk {

constexpr int kTcM = 128;          // weight rows per tile (MMA M)
constexpr int kTcN = 16;           // B rows: 8 hi planes + 8 lo planes (MMA N)
constexpr int kTcKb = 128;         // columns per K-block (one scale block, one TMA box)
constexpr int kTcKbPerStage = 2;   // K-blocks per TMA ring stage
constexpr int kTcConvWarps = TC_CONV_WARPS;  // converters; the first 4 also run the epilogue
constexpr int kTcEpiWarps = 4;
constexpr int kTcBWarp0 = kTcConvWarps;                // warps that build the B tile
constexpr int kTcBWarps = TC_B_WARPS;
constexpr int kTcProducerWarp = kTcBWarp0 + kTcBWarps;
constexpr int kTcMmaWarp = kTcProducerWarp + 1;        // first MMA-issuing warp
constexpr int kTcMmaWarps = TC_MMA_WARPS;              // MMA-issuing warps (one lane each)
constexpr int kTcStageArrivals = kTcConvWarps + kTcBWarps;  // warps that fill / release a stage
constexpr int kTcThreads = (kTcProducerWarp + 1 + kTcMmaWarps) * 32;
constexpr int kTcKSplit = kTcConvWarps / 4;        // converter warps per TMEM lane quarter
constexpr int kTcKW = kTcKb / kTcKSplit;            // K columns each converter thread converts
constexpr int kTcChunks = kTcKW / 16;               // ... as 16-code chunks
constexpr int kTcEStages = TC_E_STAGES;   // TMA ring depth
constexpr int kTcStages = TC_AB_STAGES;   // operand ring depth: A in tensor memory, B in shared memory
constexpr bool kTcSleep = TC_SPIN == 0;   // converters' and producer's waits: sleeping (true) or polling
constexpr bool kTcMmaSleep = TC_MMA_SLEEP != 0;  // MMA issuer's waits
constexpr int kTcMaxPanel = 4096;         // columns per panel
constexpr int kTcETileBytes = kTcM * kTcKb;          // 16 KiB of e4m3 codes per K-block
constexpr int kTcXCols = kTcKbPerStage * kTcKb;      // x columns per stage (one 2-D box)
constexpr int kTcXStageBytes = 8 * kTcXCols * 4;     // up to 8 rows x 256 f32
constexpr int kTcEStageBytes = kTcKbPerStage * kTcETileBytes + kTcXStageBytes;
constexpr int kTcBTileBytes = kTcN * kTcKb * 2;      // 4 KiB
constexpr int kTcSbo = kTcKb / 8 * 128;              // bytes between the B tile's 8-row core groups
constexpr int kTcMaxSf = 4096;                       // f16 scale factors held in shared memory
constexpr int kTcACols = kTcKb / 2;                  // TMEM columns of one A stage (two f16 per column)
constexpr int kTcDCol = kTcStages * kTcACols;        // first accumulator column
// A tcgen05.mma costs its issuing thread about 120 cycles whatever the
// shape, so the 8 MMAs of a K-block are spread over kTcMmaWarps warps, each
// into its own accumulator (K-steps interleaved); the epilogue adds them.
constexpr int kTcNAcc = kTcMmaWarps;
constexpr int kTcDBuf = kTcNAcc * kTcN;              // accumulator columns per tile buffer
constexpr int kTcTmemUsed = kTcDCol + 2 * kTcDBuf;
constexpr int kTcTmemCols = kTcTmemUsed <= 64 ? 64 : kTcTmemUsed <= 128 ? 128 : kTcTmemUsed <= 256 ? 256 : 512;
constexpr int kTcSmemBytes =
    kTcEStages * kTcEStageBytes + kTcStages * kTcBTileBytes + kTcMaxSf * 2 + 1024;  // + alignment slack
constexpr int kTcMaxRowBlocks = 64;                  // scale row blocks a CTA may span
constexpr int kTcSmallBoxRows = 32;                  // tiles this short load one 32-row box per K-block
static_assert(kTcEStageBytes % 1024 == 0, "swizzled TMA tiles need 1024-byte alignment");
static_assert(kTcConvWarps == 8 || kTcConvWarps == 16, "8 or 16 converter warps");
static_assert(kTcTmemUsed <= 512, "tensor memory holds 512 columns");
static_assert((kTcKb / 16) % kTcMmaWarps == 0, "K-steps split evenly over the MMA warps");
constexpr int kTcBValsPerThread = 8 * kTcKb / (kTcBWarps * 32);  // x values each B thread encodes
static_assert(kTcBValsPerThread == 16 || kTcBValsPerThread == 8, "B split: 8 or 16 values (whole K-cores)");

struct TcArgs {
    const float *scales;
    const float *x;
    float *y;
    uint32_t *tokens;
    float *part_val;
    uint32_t *part_idx;
    uint32_t *counter;
    unsigned int *status;
    const uint8_t *w;        // for the CUDA-core fallback
    int64_t rows, cols;
    int m;
    int panels;
    int panel_cols;          // multiple of kTcKb except possibly the last panel
    int64_t n_units8;        // ceil(rows / 8): CTAs own whole 8-row units
};

__device__ __forceinline__ uint64_t umma_smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // sm_100-family descriptor version; no swizzle
    return d;
}

// kind::f16 instruction descriptor: f16 A and B, f32 D, both K-major.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int m_rows, int n_cols) {
    return (1u << 4) | (static_cast<uint32_t>(n_cols >> 3) << 17) | (static_cast<uint32_t>(m_rows >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(static_cast<uint32_t>(accumulate))
        : "memory");
}

__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// One warp stores N consecutive 32-bit columns of its own 32 TMEM lanes.
template <int N>
__device__ __forceinline__ void tc_st(uint32_t taddr, const uint32_t (&v)[N]);

template <>
__device__ __forceinline__ void tc_st<16>(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

template <>
__device__ __forceinline__ void tc_st<32>(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// kind::f16 MMA with A read from tensor memory (row r in lane r, two f16 of
// consecutive K per 32-bit column) and B from shared memory.
__device__ __forceinline__ void tc_mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(static_cast<uint32_t>(accumulate))
        : "memory");
}

// 2^e as an f32 for -126 <= e <= 127.
__device__ __forceinline__ float pow2f_normal(int e) { return __int_as_float((e + 127) << 23); }

// Power-of-two exponent of a positive power of two f32 (including subnormals);
// -1000 if s is not a positive finite power of two.
__device__ __forceinline__ int pow2_exponent(float s) {
    if (!(s > 0.f) || !isfinite(s)) return -1000;
    int e = 0;
    const float f = frexpf(s, &e);
    return f == 0.5f ? e - 1 : -1000;
}

// Plain CUDA-core rows for a CTA whose scales the f16 encoding cannot carry:
// warp per row, lanes stride the columns, shuffle reduction.
__device__ inline void tc_fallback_rows(const TcArgs &a, int64_t r0, int64_t r1, int warp, int lane, float *best_v,
                                 uint32_t *best_i, bool argmax) {
    const int64_t gcols = (a.cols + 127) / 128;
    for (int64_t r = r0 + warp; r < r1; r += kTcConvWarps) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int64_t c = lane; c < a.cols; c += 32) {
            const uint32_t code = a.w[r * a.cols + c];
            const float wv = e4m3x2_to_f32(code).x * __ldg(a.scales + (r >> 7) * gcols + (c >> 7));
            for (int i = 0; i < a.m; ++i) acc[i] = fmaf(wv, __ldg(a.x + i * a.cols + c), acc[i]);
        }
        for (int i = 0; i < a.m; ++i) {
            float v = acc[i];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
            if (lane == 0) {
                if (a.y) a.y[static_cast<int64_t>(i) * a.rows + r] = v;
                if (argmax && argmax_better(v, static_cast<uint32_t>(r), best_v[i], best_i[i])) {
                    best_v[i] = v;
                    best_i[i] = static_cast<uint32_t>(r);
                }
            }
        }
    }
}

__device__ __forceinline__ bool tc_aborted(const int *flag) { return *reinterpret_cast<const volatile int *>(flag) != 0; }
__device__ __forceinline__ void tc_raise_abort(int *flag) { *reinterpret_cast<volatile int *>(flag) = 1; }

// Rows of one tile: every role derives the same values from the same arguments.
struct TcTile {
    int64_t row0;   // first row of the tile
    int rows;       // rows of the tile that belong to this CTA (1..128)
};

__device__ __forceinline__ TcTile tc_tile(int64_t r0, int64_t r1, int t) {
    TcTile d;
    d.row0 = r0 + static_cast<int64_t>(t) * kTcM;
    d.rows = static_cast<int>(r1 - d.row0 < kTcM ? r1 - d.row0 : kTcM);
    return d;
}

template <bool ARGMAX>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemv_kernel(const __grid_constant__ CUtensorMap wmap_big, const __grid_constant__ CUtensorMap wmap_small,
                   const __grid_constant__ CUtensorMap xmap, const TcArgs a) {
    extern __shared__ __align__(1024) uint8_t tc_smem[];
    __shared__ __align__(8) uint64_t full_e[kTcEStages], empty_e[kTcEStages];
    __shared__ __align__(8) uint64_t conv_a[kTcStages], free_a[kTcStages], d_full[2], d_free[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int s_abort, s_fallback;
    __shared__ int s_q[kTcMaxRowBlocks];
    __shared__ int s_p[8];
    __shared__ int s_xmax_bits[8];
    __shared__ float s_xpart[kTcThreads];
    __shared__ float am_val[kTcThreads / 32][8];
    __shared__ uint32_t am_idx[kTcThreads / 32][8];
    __shared__ int s_is_last;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int m = a.m;

    // Shared memory: [TMA ring: stages of (two 16 KiB e4m3 K-block tiles |
    // x slice m x 256 f32), 1024-aligned for the 128-byte swizzle | operand
    // ring: (f16 A tile 32 KiB | B tile 4 KiB) | f16 scale factors S * 2^-q
    // per (row block, K-block)].
    uint8_t *sE = tc_smem + ((1024u - (smem_addr(tc_smem) & 1023u)) & 1023u);
    uint8_t *sB = sE + kTcEStages * kTcEStageBytes;
    __half *s_sf = reinterpret_cast<__half *>(sB + kTcStages * kTcBTileBytes);

    // This CTA's rows: whole 8-row units, balanced.
    const int64_t u0 = static_cast<int64_t>(blockIdx.x) * a.n_units8 / gridDim.x;
    const int64_t u1 = static_cast<int64_t>(blockIdx.x + 1) * a.n_units8 / gridDim.x;
    const int64_t r0 = u0 * 8;
    const int64_t r1 = u1 * 8 < a.rows ? u1 * 8 : a.rows;
    const int n_tiles = r1 > r0 ? static_cast<int>((r1 - r0 + kTcM - 1) / kTcM) : 0;
    const int64_t gcols = (a.cols + 127) / 128;
    const int rb0 = static_cast<int>(r0 >> 7);
    const int n_rb = r1 > r0 ? static_cast<int>(((r1 - 1) >> 7) - rb0 + 1) : 0;

    auto panel_cols_of = [&](int p) {
        const int64_t pc64 = a.cols - static_cast<int64_t>(p) * a.panel_cols;
        return pc64 < a.panel_cols ? static_cast<int>(pc64) : a.panel_cols;
    };
    auto nkb_of = [&](int p) { return (panel_cols_of(p) + kTcKb - 1) / kTcKb; };
    auto nst_of = [&](int p) { return (nkb_of(p) + kTcKbPerStage - 1) / kTcKbPerStage; };

    if (tid == 0) {
        for (int s = 0; s < kTcEStages; ++s) {
            mbar_init(smem_addr(&full_e[s]), 1);
            mbar_init(smem_addr(&empty_e[s]), kTcStageArrivals);
        }
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(smem_addr(&conv_a[s]), kTcStageArrivals);
            mbar_init(smem_addr(&free_a[s]), kTcMmaWarps);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_addr(&d_full[s]), kTcMmaWarps);
            mbar_init(smem_addr(&d_free[s]), kTcEpiWarps);
        }
        mbar_init_fence();
        for (int i = 0; i < 8; ++i) s_xmax_bits[i] = 0;
        s_abort = 0;
        // Shapes whose scale table does not fit take the CUDA-core loop.
        s_fallback = (n_rb > kTcMaxRowBlocks || static_cast<int64_t>(n_rb) * gcols > kTcMaxSf) ? 1 : 0;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_slot)),
                     "n"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    // ---- TMA ring stage e = (panel p, tile t, stage st): two K-blocks.
    const uint64_t pol = l2_policy_evict_first();
    auto stage_coords = [&](int64_t e, int &p, int &t, int &st) {
        p = 0;
        while (p + 1 < a.panels && e >= static_cast<int64_t>(n_tiles) * nst_of(p)) {
            e -= static_cast<int64_t>(n_tiles) * nst_of(p);
            ++p;
        }
        const int nst = nst_of(p);
        t = static_cast<int>(e / nst);
        st = static_cast<int>(e % nst);
    };
    // Bytes a stage's boxes deliver (a box always delivers its full extent;
    // out-of-range elements arrive as zeros).
    auto stage_bytes = [&](int p, int t, int st) {
        const TcTile tl = tc_tile(r0, r1, t);
        const int nk = min(kTcKbPerStage, nkb_of(p) - st * kTcKbPerStage);
        const uint32_t box = tl.rows > kTcSmallBoxRows ? static_cast<uint32_t>(kTcETileBytes)
                                                       : static_cast<uint32_t>(kTcSmallBoxRows * kTcKb);
        return static_cast<uint32_t>(nk) * box + static_cast<uint32_t>(m) * kTcXCols * 4u;
    };
    auto issue_weights = [&](int64_t e, int p, int t, int st) {
        const TcTile tl = tc_tile(r0, r1, t);
        const int nk = min(kTcKbPerStage, nkb_of(p) - st * kTcKbPerStage);
        const uint32_t bar = smem_addr(&full_e[e % kTcEStages]);
        uint8_t *stg = sE + (e % kTcEStages) * kTcEStageBytes;
        for (int k2 = 0; k2 < nk; ++k2) {
            const int xc = p * a.panel_cols + (st * kTcKbPerStage + k2) * kTcKb;
            uint8_t *dst = stg + k2 * kTcETileBytes;
            tma_load_2d_hint(smem_addr(dst), tl.rows > kTcSmallBoxRows ? &wmap_big : &wmap_small, xc,
                             static_cast<int>(tl.row0), bar, pol);
        }
    };
    auto issue_x = [&](int64_t e, int p, int st) {
        const uint32_t bar = smem_addr(&full_e[e % kTcEStages]);
        uint8_t *xst = sE + (e % kTcEStages) * kTcEStageBytes + kTcKbPerStage * kTcETileBytes;
        tma_load_2d(smem_addr(xst), &xmap, p * a.panel_cols + st * kTcXCols, 0, bar);
    };
    int64_t n_stages = 0;
    for (int p = 0; p < a.panels; ++p) n_stages += static_cast<int64_t>(n_tiles) * nst_of(p);
    const int64_t pre = n_stages < kTcEStages ? n_stages : kTcEStages;

    // Weights are never written by the preceding kernel: start streaming them
    // before the grid dependency wait.  (The producer keeps its own record of
    // whether it did: other warps may raise s_fallback meanwhile.)
    bool early = false;
    if (warp == kTcProducerWarp && lane == 0 && !*reinterpret_cast<volatile int *>(&s_fallback)) {
        early = true;
        for (int64_t e = 0; e < pre; ++e) {
            int p, t, st;
            stage_coords(e, p, t, st);
            mbar_arrive_expect_tx(smem_addr(&full_e[e]), stage_bytes(p, t, st));
            issue_weights(e, p, t, st);
        }
    }

    grid_dependency_wait();
    grid_launch_dependents();

    // All threads, before the roles split: per row block the offset q = (largest
    // scale exponent) - 7 and the f16 factors S * 2^-q of its K-blocks (each in
    // [2^-15, 2^7] unless the CTA falls back), and per activation row the
    // pre-scale p from max|x_i|.
    if (!s_fallback) {
        for (int j = warp; j < n_rb; j += kTcThreads / 32) {
            const float *srow = a.scales + static_cast<int64_t>(rb0 + j) * gcols;
            int emax = -100000, emin = 100000, bad = 0;
            for (int64_t kb = lane; kb < gcols; kb += 32) {
                const int e = pow2_exponent(__ldg(srow + kb));
                if (e == -1000) bad = 1;
                emax = max(emax, e);
                emin = min(emin, e);
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                emax = max(emax, __shfl_xor_sync(0xFFFFFFFFu, emax, off));
                emin = min(emin, __shfl_xor_sync(0xFFFFFFFFu, emin, off));
                bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, off);
            }
            if (bad || emax - emin > 22) {
                if (lane == 0) atomicOr(&s_fallback, 1);
                continue;
            }
            if (lane == 0) s_q[j] = emax - 7;
            for (int64_t kb = lane; kb < gcols; kb += 32)
                s_sf[j * gcols + kb] = __float2half_rn(ldexpf(__ldg(srow + kb), 7 - emax));
        }
        // max|x_i|: threads [i * T, (i + 1) * T) take row i (T = threads per row),
        // each every T-th float4 from its offset, up to 20 loads in flight; the
        // partial maxima meet in s_xpart and one warp per row reduces them.
        {
            const int per_row = kTcThreads / m;
            const int xi = tid / per_row;
            const int j0 = tid - xi * per_row;
            const int c4n = static_cast<int>(a.cols / 4);
            float mxr = 0.f;
            if (xi < m) {
                const float4 *xrow = reinterpret_cast<const float4 *>(a.x + static_cast<int64_t>(xi) * a.cols);
                for (int jb = j0; jb < c4n; jb += 20 * per_row) {
                    float4 v[20];
#pragma unroll
                    for (int k = 0; k < 20; ++k) {
                        const int j = jb + k * per_row;
                        v[k] = j < c4n ? __ldg(xrow + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int k = 0; k < 20; ++k)
                        mxr = fmaxf(mxr, fmaxf(fmaxf(fabsf(v[k].x), fabsf(v[k].y)), fmaxf(fabsf(v[k].z), fabsf(v[k].w))));
                }
            }
            s_xpart[tid] = mxr;
        }
    }
    __syncthreads();
    if (!s_fallback && warp < m) {
        const int per_row = kTcThreads / m;
        float v = 0.f;
        for (int j = lane; j < per_row; j += 32) v = fmaxf(v, s_xpart[warp * per_row + j]);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
        if (lane == 0) s_xmax_bits[warp] = __float_as_int(v);  // non-negative: bits order like values
    }
    __syncthreads();
    if (tid < 8) {
        const float mxv = __int_as_float(s_xmax_bits[tid]);
        int e = 0;
        const bool finite_pos = mxv > 0.f && isfinite(mxv);
        if (finite_pos) (void)frexpf(mxv, &e);  // mx < 2^e
        s_p[tid] = finite_pos ? 15 - e : 0;
    }
    __syncthreads();

    float best_v[8];
    uint32_t best_i[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        best_v[i] = -INFINITY;
        best_i[i] = 0;
    }
    if (s_fallback) {
        if (warp < kTcConvWarps) tc_fallback_rows(a, r0, r1, warp, lane, best_v, best_i, ARGMAX);
        if (early) {
            // Complete the early stages' transactions with their x bytes, then
            // let them land before the CTA exits.
            for (int64_t e = 0; e < pre; ++e) {
                int p, t, st;
                stage_coords(e, p, t, st);
                issue_x(e, p, st);
            }
            for (int64_t e = 0; e < pre; ++e) (void)mbar_wait_bounded(smem_addr(&full_e[e]), 0u);
        }
    } else if (warp == kTcProducerWarp) {
        // ---------------- TMA producer
        if (lane == 0) {
            int64_t e = 0;
            for (; e < n_stages && !tc_aborted(&s_abort); ++e) {
                int p, t, st;
                stage_coords(e, p, t, st);
                if (e >= pre) {
                    const int s = static_cast<int>(e % kTcEStages);
                    if (!mbar_wait_bounded<kTcSleep>(smem_addr(&empty_e[s]), static_cast<uint32_t>((e / kTcEStages - 1) & 1))) {
                        tc_raise_abort(&s_abort);
                        break;
                    }
                    mbar_arrive_expect_tx(smem_addr(&full_e[s]), stage_bytes(p, t, st));
                    issue_weights(e, p, t, st);
                }
                issue_x(e, p, st);
            }
            // Early stages never reached still owe their x bytes; then every
            // copy in flight must land before the CTA's memory is released.
            for (int64_t v = e; v < pre; ++v) {
                int p, t, st;
                stage_coords(v, p, t, st);
                issue_x(v, p, st);
            }
            const int64_t issued = e > pre ? e : pre;
            const int64_t first_open = issued > kTcEStages ? issued - kTcEStages : 0;
            for (int64_t v = first_open; v < issued; ++v)
                (void)mbar_wait_bounded(smem_addr(&full_e[v % kTcEStages]), static_cast<uint32_t>((v / kTcEStages) & 1));
        }
    } else if (warp >= kTcMmaWarp) {
        // ---------------- MMA issuers: warp kTcMmaWarp + j issues K-steps j, j + kTcMmaWarps, ...
        // of every K-block into accumulator j.
        const int mj = warp - kTcMmaWarp;
        if (lane == 0) {
            int64_t u = 0;
            int tile_seq = 0;
            for (int p = 0; p < a.panels && !tc_aborted(&s_abort); ++p) {
                const int nkb = nkb_of(p);
                for (int t = 0; t < n_tiles && !tc_aborted(&s_abort); ++t, ++tile_seq) {
                    const TcTile tl = tc_tile(r0, r1, t);
                    const uint32_t idesc = umma_idesc_f16(kTcM, kTcN);
                    const int acc = tile_seq & 1;
                    if (tile_seq >= 2 && !mbar_wait_bounded<kTcMmaSleep>(smem_addr(&d_free[acc]),
                                                                   static_cast<uint32_t>((tile_seq / 2 - 1) & 1))) {
                        tc_raise_abort(&s_abort);
                        break;
                    }
                    tc_fence_after();
                    bool broke = false;
                    for (int kb = 0; kb < nkb; ++kb, ++u) {
                        const int s = static_cast<int>(u % kTcStages);
                        if (!mbar_wait_bounded<kTcMmaSleep>(smem_addr(&conv_a[s]), static_cast<uint32_t>((u / kTcStages) & 1))) {
                            tc_raise_abort(&s_abort);
                            broke = true;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_col = tmem + static_cast<uint32_t>(s * kTcACols);
                        const uint32_t b_base = smem_addr(sB + s * kTcBTileBytes);
#pragma unroll
                        for (int k = mj; k < kTcKb / 16; k += kTcMmaWarps) {
                            const uint64_t bd = umma_smem_desc(b_base + k * 256u, 128u, kTcSbo);
                            tc_mma_f16_ta(tmem + static_cast<uint32_t>(kTcDCol + acc * kTcDBuf + mj * kTcN),
                                          a_col + 8u * k, bd, idesc, kb > 0 || k >= kTcMmaWarps);
                        }
                        tc_commit(smem_addr(&free_a[s]));
                        if (kb == nkb - 1) tc_commit(smem_addr(&d_full[acc]));
                    }
                    if (broke) break;
                }
            }
            // The last commit must have landed before the tensor memory is freed.
            if (u > 0) {
                const int64_t last = u - 1;
                (void)mbar_wait_bounded(smem_addr(&free_a[last % kTcStages]),
                                        static_cast<uint32_t>((last / kTcStages) & 1));
            }
        }
    } else if (warp >= kTcBWarp0) {
        // ---------------- B builders: per operand stage, x_bi's columns bc.. of the
        // K-block as hi (row bi) and lo (row 8 + bi) f16 planes of x * 2^p; zeros
        // past the panel or for bi >= m.
        auto warp_aborted = [&]() { return __any_sync(0xFFFFFFFFu, tc_aborted(&s_abort)); };
        constexpr int V = kTcBValsPerThread;
        const int bt = tid - kTcBWarp0 * 32;
        const int bi = bt & 7;
        const int bc = (bt >> 3) * V;  // first column within the K-block (whole K-cores)
        const int pb = s_p[bi];
        const float pfa = pow2f_normal(pb / 2), pfb = pow2f_normal(pb - pb / 2);
        int64_t u = 0, e = 0;
        for (int p = 0; p < a.panels && !warp_aborted(); ++p) {
            const int pc = panel_cols_of(p);
            const int nkb = nkb_of(p);
            bool broke = false;
            for (int t = 0; t < n_tiles && !broke && !warp_aborted(); ++t) {
                for (int kb = 0; kb < nkb; ++kb, ++u) {
                    const int k2 = kb % kTcKbPerStage;
                    const int se = static_cast<int>(e % kTcEStages);
                    const int s = static_cast<int>(u % kTcStages);
                    bool ok = true;
                    if (k2 == 0)
                        ok = mbar_wait_bounded<kTcSleep>(smem_addr(&full_e[se]), static_cast<uint32_t>((e / kTcEStages) & 1));
                    if (ok && u >= kTcStages)
                        ok = mbar_wait_bounded<kTcSleep>(smem_addr(&free_a[s]), static_cast<uint32_t>((u / kTcStages - 1) & 1));
                    if (!__all_sync(0xFFFFFFFFu, ok)) {
                        tc_raise_abort(&s_abort);
                        broke = true;
                        break;
                    }
                    const float *xs = reinterpret_cast<const float *>(sE + se * kTcEStageBytes + kTcKbPerStage * kTcETileBytes) +
                                      k2 * kTcKb;
                    uint8_t *btile = sB + s * kTcBTileBytes;
                    uint32_t hw[V / 2], lw[V / 2];
#pragma unroll
                    for (int q = 0; q < V / 2; ++q) hw[q] = lw[q] = 0u;
                    if (bi < m && kb * kTcKb + bc < pc) {
                        float vv[V];
#pragma unroll
                        for (int q = 0; q < V; q += 4) {
                            const float4 v4 = *reinterpret_cast<const float4 *>(xs + bi * kTcXCols + bc + q);
                            vv[q] = v4.x;
                            vv[q + 1] = v4.y;
                            vv[q + 2] = v4.z;
                            vv[q + 3] = v4.w;
                        }
#pragma unroll
                        for (int q = 0; q < V / 2; ++q) {
                            const float s0 = vv[2 * q] * pfa * pfb, s1 = vv[2 * q + 1] * pfa * pfb;
                            const __half2 hh = __floats2half2_rn(s0, s1);
                            const float2 hb = __half22float2(hh);
                            const __half2 ll = __floats2half2_rn(s0 - hb.x, s1 - hb.y);
                            hw[q] = *reinterpret_cast<const uint32_t *>(&hh);
                            lw[q] = *reinterpret_cast<const uint32_t *>(&ll);
                        }
                    }
                    // K-core bc / 8 + c holds columns 8c..8c+7 of this thread's run
#pragma unroll
                    for (int c = 0; c < V / 8; ++c) {
                        uint8_t *bh = btile + ((bc >> 3) + c) * 128 + bi * 16;
                        *reinterpret_cast<uint4 *>(bh) = make_uint4(hw[4 * c], hw[4 * c + 1], hw[4 * c + 2], hw[4 * c + 3]);
                        *reinterpret_cast<uint4 *>(bh + kTcSbo) =
                            make_uint4(lw[4 * c], lw[4 * c + 1], lw[4 * c + 2], lw[4 * c + 3]);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic stores -> the MMA
                    __syncwarp();
                    const bool stage_done = k2 == kTcKbPerStage - 1 || kb == nkb - 1;
                    if (lane == 0) {
                        mbar_arrive(smem_addr(&conv_a[s]));
                        if (stage_done) mbar_arrive(smem_addr(&empty_e[se]));
                    }
                    if (stage_done) ++e;
                }
            }
            if (broke) break;
        }
    } else {
        // ---------------- converters (+ epilogue on the first four warps)
        // Abort checks are warp-uniform: the loops below hold warp-wide votes.
        auto warp_aborted = [&]() { return __any_sync(0xFFFFFFFFu, tc_aborted(&s_abort)); };
        // A work of this thread: tile row tr_a (TMEM lane), K slice kq.
        const int kq = warp >> 2;
        const int tr_a = (warp & 3) * 32 + lane;
        const uint32_t a_taddr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + static_cast<uint32_t>(kq * (kTcKW / 2));
        int64_t u = 0, e = 0;
        int tile_seq = 0;
        for (int p = 0; p < a.panels && !warp_aborted(); ++p) {
            const int pc = panel_cols_of(p);
            const int nkb = nkb_of(p);
            const int kglob0 = p * (a.panel_cols / kTcKb);  // first global K-block of the panel
            for (int t = 0; t < n_tiles && !warp_aborted(); ++t, ++tile_seq) {
                const TcTile tl = tc_tile(r0, r1, t);
                // Scale-table row of this thread's tile row (rows past r1 use the last
                // row's: their accumulator rows are never read).
                const int64_t arow = tl.row0 + tr_a < r1 ? tl.row0 + tr_a : r1 - 1;
                const int sf_row = static_cast<int>((arow >> 7) - rb0) * static_cast<int>(gcols);
                const bool a_live = (tr_a & ~31) < tl.rows;  // warp-uniform: some row of this quarter is in the tile
                bool broke = false;
                for (int kb = 0; kb < nkb; ++kb, ++u) {
                    const int k2 = kb % kTcKbPerStage;
                    const int se = static_cast<int>(e % kTcEStages);
                    const int s = static_cast<int>(u % kTcStages);
                    bool ok = true;
                    if (k2 == 0)
                        ok = mbar_wait_bounded<kTcSleep>(smem_addr(&full_e[se]), static_cast<uint32_t>((e / kTcEStages) & 1));
                    if (ok && u >= kTcStages)
                        ok = mbar_wait_bounded<kTcSleep>(smem_addr(&free_a[s]), static_cast<uint32_t>((u / kTcStages - 1) & 1));
                    if (!__all_sync(0xFFFFFFFFu, ok)) {
                        tc_raise_abort(&s_abort);
                        broke = true;
                        break;
                    }
                    tc_fence_after();  // the MMA that read this operand stage has completed
                    const uint8_t *stg = sE + se * kTcEStageBytes;
                    const uint8_t *et = stg + k2 * kTcETileBytes;
                    const int kglob = kglob0 + kb;
                    // A: this thread's row, K columns [kq * kTcKW, (kq + 1) * kTcKW), codes ->
                    // f16 * S * 2^-q, stored to its TMEM lane (two f16 per column).
                    if (a_live) {
                        const __half sfh = s_sf[sf_row + kglob];
                        const __half2 sf2 = __halves2half2(sfh, sfh);
                        uint32_t o[kTcChunks * 8];
#pragma unroll
                        for (int c = 0; c < kTcChunks; ++c) {
                            const int kc = kq * kTcChunks + c;  // 16-code chunk within the K-block
                            const uint4 q = *reinterpret_cast<const uint4 *>(et + tr_a * 128 + ((kc ^ (tr_a & 7)) << 4));
                            const uint32_t wds[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                uint32_t h01, h23;
                                asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
                                    "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
                                    : "=r"(h01), "=r"(h23)
                                    : "r"(wds[j]));
                                const __half2 p01 = __hmul2(*reinterpret_cast<const __half2 *>(&h01), sf2);
                                const __half2 p23 = __hmul2(*reinterpret_cast<const __half2 *>(&h23), sf2);
                                o[c * 8 + 2 * j] = *reinterpret_cast<const uint32_t *>(&p01);
                                o[c * 8 + 2 * j + 1] = *reinterpret_cast<const uint32_t *>(&p23);
                            }
                        }
                        tc_st<kTcChunks * 8>(a_taddr + static_cast<uint32_t>(s * kTcACols), o);
                        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    }
                    tc_fence_before();  // A's tensor-memory stores -> the MMA
                    __syncwarp();
                    const bool stage_done = k2 == kTcKbPerStage - 1 || kb == nkb - 1;
                    if (lane == 0) {
                        mbar_arrive(smem_addr(&conv_a[s]));
                        if (stage_done) mbar_arrive(smem_addr(&empty_e[se]));
                    }
                    if (stage_done) ++e;
                }
                if (broke || warp_aborted()) break;
                if (warp >= kTcEpiWarps) continue;
                // ---------------- epilogue for this tile (TMEM lanes 32 * warp ..)
                const int acc = tile_seq & 1;
                const bool ok = __all_sync(
                    0xFFFFFFFFu,
                    mbar_wait_bounded<kTcSleep>(smem_addr(&d_full[acc]), static_cast<uint32_t>((tile_seq / 2) & 1)));
                if (!ok) {
                    tc_raise_abort(&s_abort);
                    break;
                }
                tc_fence_after();
                float v[16];
                tc_ld16(tmem + static_cast<uint32_t>(kTcDCol + acc * kTcDBuf) + (static_cast<uint32_t>(warp * 32) << 16), v);
#pragma unroll
                for (int c = 1; c < kTcNAcc; ++c) {
                    float w[16];
                    tc_ld16(tmem + static_cast<uint32_t>(kTcDCol + acc * kTcDBuf + c * kTcN) +
                                (static_cast<uint32_t>(warp * 32) << 16),
                            w);
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] += w[j];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&d_free[acc]));
                const int tr = warp * 32 + lane;
                if (tr < tl.rows) {
                    const int64_t row = tl.row0 + tr;
                    const int qv = s_q[static_cast<int>((row >> 7) - rb0)];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (i >= m) break;
                        float val = ldexpf(v[i] + v[8 + i], qv - s_p[i]);
                        float *yp = a.y ? a.y + static_cast<int64_t>(i) * a.rows + row : nullptr;
                        if (a.panels > 1) {
                            if (p > 0) val += *yp;
                            *yp = val;
                        } else if (yp) {
                            *yp = val;
                        }
                        if (ARGMAX && p == a.panels - 1 &&
                            argmax_better(val, static_cast<uint32_t>(row), best_v[i], best_i[i])) {
                            best_v[i] = val;
                            best_i[i] = static_cast<uint32_t>(row);
                        }
                    }
                }
            }
        }
    }

    if (tid == 0 && tc_aborted(&s_abort)) atomicOr(a.status, 1u);
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTcTmemCols) : "memory");

    if constexpr (ARGMAX) {
        // Per activation row: merge the converter threads' bests, then CTAs.
        for (int i = 0; i < 8; ++i) {
            float bv = best_v[i];
            uint32_t bi = best_i[i];
            warp_argmax_merge<1>(bv, bi);
            if (lane == 0) {
                am_val[warp][i] = bv;
                am_idx[warp][i] = bi;
            }
        }
        __syncthreads();
        if (tid < m) {
            float bv = -INFINITY;
            uint32_t bi = 0;
            for (int w2 = 0; w2 < kTcConvWarps; ++w2)
                if (argmax_better(am_val[w2][tid], am_idx[w2][tid], bv, bi)) {
                    bv = am_val[w2][tid];
                    bi = am_idx[w2][tid];
                }
            __stcg(a.part_val + static_cast<int64_t>(blockIdx.x) * m + tid, bv);
            __stcg(a.part_idx + static_cast<int64_t>(blockIdx.x) * m + tid, bi);
        }
        GemvArgs ga = {};
        ga.part_val = a.part_val;
        ga.part_idx = a.part_idx;
        ga.counter = a.counter;
        ga.tokens = a.tokens;
        switch (m) {  // the cross-CTA merge is templated on the row count
            case 2: argmax_cross_cta<2, kTcThreads, kTcThreads / 32>(ga, am_val, am_idx, &s_is_last); break;
            case 3: argmax_cross_cta<3, kTcThreads, kTcThreads / 32>(ga, am_val, am_idx, &s_is_last); break;
            case 4: argmax_cross_cta<4, kTcThreads, kTcThreads / 32>(ga, am_val, am_idx, &s_is_last); break;
            case 5: argmax_cross_cta<5, kTcThreads, kTcThreads / 32>(ga, am_val, am_idx, &s_is_last); break;
            case 6: argmax_cross_cta<6, kTcThreads, kTcThreads / 32>(ga, am_val, am_idx, &s_is_last); break;
            case 7: argmax_cross_cta<7, kTcThreads, kTcThreads / 32>(ga, am_val, am_idx, &s_is_last); break;
            default: argmax_cross_cta<8, kTcThreads, kTcThreads / 32>(ga, am_val, am_idx, &s_is_last); break;
        }
    }
}

}  // namespace fp8blk
