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
//   converter warps: e4m3 tile -> f16 A tile in the UMMA K-major layout (no
//                  swizzle: 8 x 16-byte core matrices, LBO = 128 B along K,
//                  SBO = 2048 B per 8 rows) and, all of them together, the x
//                  slice -> B tile; the first four warps also run the epilogue;
//   MMA warp, lane 0: 8 x tcgen05.mma (K = 16 each) per K-block, commits to
//                  mbarriers that free the operand stage / publish the
//                  accumulator (two accumulators of 16 columns alternate).
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
#define TC_E_STAGES 3
#endif
#ifndef TC_AK
#define TC_AK 128
#endif
#ifndef TC_AB_STAGES
#define TC_AB_STAGES (2 * 128 / TC_AK)
#endif
#ifndef TC_SPIN
#define TC_SPIN 0
#endif
#ifndef TC_MMA_SLEEP
#define TC_MMA_SLEEP 0
#endif

namespace fp8blk {

constexpr int kTcM = 128;          // weight rows per tile (MMA M)
constexpr int kTcN = 16;           // B rows: 8 hi planes + 8 lo planes (MMA N)
constexpr int kTcKb = 128;         // columns per K-block (one scale block, one TMA box)
constexpr int kTcKbPerStage = 2;   // K-blocks per TMA ring stage
constexpr int kTcConvWarps = TC_CONV_WARPS;  // converters; the first 4 also run the epilogue
constexpr int kTcEpiWarps = 4;
constexpr int kTcProducerWarp = kTcConvWarps;
constexpr int kTcMmaWarp = kTcConvWarps + 1;
constexpr int kTcThreads = (kTcConvWarps + 2) * 32;
constexpr int kTcGroupsPerWarp = (kTcM / 8) / kTcConvWarps;  // 8-row groups each converter owns
constexpr int kTcEStages = TC_E_STAGES;   // TMA ring depth
constexpr int kTcAK = TC_AK;              // columns per operand stage (a K-block or half of one)
constexpr int kTcSub = 128 / kTcAK;       // operand stages per K-block
constexpr int kTcStages = TC_AB_STAGES;   // f16 A + B ring depth (MMA operands)
constexpr bool kTcSleep = TC_SPIN == 0;   // converters' and producer's waits: sleeping (true) or polling
constexpr bool kTcMmaSleep = TC_MMA_SLEEP != 0;  // MMA issuer's waits
constexpr int kTcMaxPanel = 4096;         // columns per panel
constexpr int kTcETileBytes = kTcM * kTcKb;          // 16 KiB of e4m3 codes per K-block
constexpr int kTcXCols = kTcKbPerStage * kTcKb;      // x columns per stage (one 2-D box)
constexpr int kTcXStageBytes = 8 * kTcXCols * 4;     // up to 8 rows x 256 f32
constexpr int kTcEStageBytes = kTcKbPerStage * kTcETileBytes + kTcXStageBytes;
constexpr int kTcATileBytes = kTcM * kTcAK * 2;      // 16 or 32 KiB
constexpr int kTcBTileBytes = kTcN * kTcAK * 2;      // 2 or 4 KiB
constexpr int kTcSbo = kTcAK / 8 * 128;              // bytes between 8-row core groups (A and B)
constexpr int kTcABStageBytes = kTcATileBytes + kTcBTileBytes;
constexpr int kTcMaxSf = 4096;                       // f16 scale factors held in shared memory
constexpr int kTcTmemCols = 2 * kTcN;
constexpr int kTcSmemBytes =
    kTcEStages * kTcEStageBytes + kTcStages * kTcABStageBytes + kTcMaxSf * 2 + 1024;  // + alignment slack
constexpr int kTcMaxRowBlocks = 64;                  // scale row blocks a CTA may span
constexpr int kTcSmallBoxRows = 32;                  // tiles this short load one 32-row box per K-block
static_assert(kTcEStageBytes % 1024 == 0, "swizzled TMA tiles need 1024-byte alignment");
static_assert((kTcM / 8) % kTcConvWarps == 0, "row groups must split evenly");
static_assert(kTcConvWarps == 4 || kTcConvWarps == 8, "4 or 8 converter warps");
constexpr int kTcBValsPerThread = 8 * kTcAK / (kTcConvWarps * 32);  // x values each converter thread encodes
static_assert(kTcBValsPerThread == 2 || kTcBValsPerThread == 4 || kTcBValsPerThread == 8, "B split");
static_assert(kTcAK == 64 || kTcAK == 128, "operand stage width");

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
    __shared__ float am_val[kAmWarps][8];
    __shared__ uint32_t am_idx[kAmWarps][8];
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
    uint8_t *sAB = sE + kTcEStages * kTcEStageBytes;
    __half *s_sf = reinterpret_cast<__half *>(sAB + kTcStages * kTcABStageBytes);

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
            mbar_init(smem_addr(&empty_e[s]), kTcConvWarps);
        }
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(smem_addr(&conv_a[s]), kTcConvWarps);
            mbar_init(smem_addr(&free_a[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_addr(&d_full[s]), 1);
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
        // max|x_i|: warp w takes row w (w < m), lanes stride its float4s with
        // 8 independent loads in flight.
        if (warp < m) {
            const int c4n = static_cast<int>(a.cols / 4);
            const float4 *xrow = reinterpret_cast<const float4 *>(a.x + static_cast<int64_t>(warp) * a.cols);
            float mxr = 0.f;
            for (int j0 = lane; j0 < c4n; j0 += 8 * 32) {
                float4 v[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int j = j0 + k * 32;
                    v[k] = j < c4n ? __ldg(xrow + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mxr = fmaxf(mxr, fmaxf(fmaxf(fabsf(v[k].x), fabsf(v[k].y)), fmaxf(fabsf(v[k].z), fabsf(v[k].w))));
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) mxr = fmaxf(mxr, __shfl_xor_sync(0xFFFFFFFFu, mxr, off));
            const float v = mxr;
            const int r = warp;
            if (lane == 0 && v > 0.f) atomicMax(&s_xmax_bits[r], __float_as_int(v));
        }
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
    } else if (warp == kTcMmaWarp) {
        // ---------------- MMA issuer
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
                    const int nsub = nkb * kTcSub;
                    for (int sb = 0; sb < nsub; ++sb, ++u) {
                        const int s = static_cast<int>(u % kTcStages);
                        if (!mbar_wait_bounded<kTcMmaSleep>(smem_addr(&conv_a[s]), static_cast<uint32_t>((u / kTcStages) & 1))) {
                            tc_raise_abort(&s_abort);
                            broke = true;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_base = smem_addr(sAB + s * kTcABStageBytes);
                        const uint32_t b_base = a_base + kTcATileBytes;
#pragma unroll
                        for (int k = 0; k < kTcAK / 16; ++k) {
                            const uint64_t ad = umma_smem_desc(a_base + k * 256u, 128u, kTcSbo);
                            const uint64_t bd = umma_smem_desc(b_base + k * 256u, 128u, kTcSbo);
                            tc_mma_f16(tmem + static_cast<uint32_t>(acc * kTcN), ad, bd, idesc, sb > 0 || k > 0);
                        }
                        tc_commit(smem_addr(&free_a[s]));
                        if (sb == nsub - 1) tc_commit(smem_addr(&d_full[acc]));
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
    } else {
        // ---------------- converters (+ epilogue on the first four warps)
        // Abort checks are warp-uniform: the loops below hold warp-wide votes.
        auto warp_aborted = [&]() { return __any_sync(0xFFFFFFFFu, tc_aborted(&s_abort)); };
        // B work of this thread: activation row bi, kTcBValsPerThread consecutive
        // columns from bc; the pre-scale 2^p as two normal f32 factors.
        const int bi = tid & 7;
        const int bc = (tid >> 3) * kTcBValsPerThread;
        const int pb = s_p[bi];
        const float pfa = pow2f_normal(pb / 2), pfb = pow2f_normal(pb - pb / 2);
        int64_t u = 0, e = 0;
        int tile_seq = 0;
        for (int p = 0; p < a.panels && !warp_aborted(); ++p) {
            const int pc = panel_cols_of(p);
            const int nkb = nkb_of(p);
            const int kglob0 = p * (a.panel_cols / kTcKb);  // first global K-block of the panel
            for (int t = 0; t < n_tiles && !warp_aborted(); ++t, ++tile_seq) {
                const TcTile tl = tc_tile(r0, r1, t);
                // Scale-table row of each owned 8-row group.
                int sf_row[kTcGroupsPerWarp];
#pragma unroll
                for (int g = 0; g < kTcGroupsPerWarp; ++g) {
                    const int64_t grow = tl.row0 + (warp * kTcGroupsPerWarp + g) * 8;
                    const int64_t growc = grow < r1 ? grow : r1 - 1;  // groups past r1 are never read back
                    sf_row[g] = static_cast<int>((growc >> 7) - rb0) * static_cast<int>(gcols);
                }
                bool broke = false;
                for (int kb = 0; kb < nkb && !broke; ++kb)
                for (int sub = 0; sub < kTcSub; ++sub, ++u) {
                    const int k2 = kb % kTcKbPerStage;
                    const int se = static_cast<int>(e % kTcEStages);
                    const int s = static_cast<int>(u % kTcStages);
                    bool ok = true;
                    if (k2 == 0 && sub == 0)
                        ok = mbar_wait_bounded<kTcSleep>(smem_addr(&full_e[se]), static_cast<uint32_t>((e / kTcEStages) & 1));
                    if (ok && u >= kTcStages)
                        ok = mbar_wait_bounded<kTcSleep>(smem_addr(&free_a[s]), static_cast<uint32_t>((u / kTcStages - 1) & 1));
                    if (!__all_sync(0xFFFFFFFFu, ok)) {
                        tc_raise_abort(&s_abort);
                        broke = true;
                        break;
                    }
                    const uint8_t *stg = sE + se * kTcEStageBytes;
                    const uint8_t *et = stg + k2 * kTcETileBytes;
                    const float *xs = reinterpret_cast<const float *>(stg + kTcKbPerStage * kTcETileBytes) + k2 * kTcKb;
                    uint8_t *at = sAB + s * kTcABStageBytes;
                    uint8_t *btile = at + kTcATileBytes;
                    const int kglob = kglob0 + kb;
                    // A: this warp's 8-row groups; lane = (chunk in half, row in group).
                    // Groups wholly past the tile's rows are skipped: their A rows feed
                    // accumulator rows that are never read.
#pragma unroll
                    for (int g = 0; g < kTcGroupsPerWarp; ++g) {
                        const int G = warp * kTcGroupsPerWarp + g;
                        if (G * 8 >= tl.rows) break;
                        const int tr = G * 8 + (lane & 7);
                        const __half sfh = s_sf[sf_row[g] + kglob];
                        const __half2 sf2 = __halves2half2(sfh, sfh);
#pragma unroll
                        for (int h = 0; h < kTcAK / 64; ++h) {
                            const int kc = (lane >> 3) + 4 * h;        // 16-column chunk within the operand stage
                            const int kcg = sub * (kTcAK / 16) + kc;  // ... within the K-block
                            const uint4 q = *reinterpret_cast<const uint4 *>(et + tr * 128 + ((kcg ^ (tr & 7)) << 4));
                            const uint32_t wds[4] = {q.x, q.y, q.z, q.w};
                            uint32_t o[8];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                uint32_t h01, h23;
                                asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
                                    "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
                                    : "=r"(h01), "=r"(h23)
                                    : "r"(wds[j]));
                                const __half2 p01 = __hmul2(*reinterpret_cast<const __half2 *>(&h01), sf2);
                                const __half2 p23 = __hmul2(*reinterpret_cast<const __half2 *>(&h23), sf2);
                                o[2 * j] = *reinterpret_cast<const uint32_t *>(&p01);
                                o[2 * j + 1] = *reinterpret_cast<const uint32_t *>(&p23);
                            }
                            uint8_t *dst = at + (tr >> 3) * kTcSbo + (2 * kc) * 128 + (tr & 7) * 16;
                            *reinterpret_cast<uint4 *>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
                            *reinterpret_cast<uint4 *>(dst + 128) = make_uint4(o[4], o[5], o[6], o[7]);
                        }
                    }
                    // B (all converter threads): x_bi's columns bc.. as hi (row bi) and lo
                    // (row 8 + bi); zeros past the panel or for bi >= m.
                    {
                        uint32_t hw[kTcBValsPerThread / 2], lw[kTcBValsPerThread / 2];
#pragma unroll
                        for (int q = 0; q < kTcBValsPerThread / 2; ++q) hw[q] = lw[q] = 0u;
                        const int bcol = sub * kTcAK + bc;  // column within the K-block
                        if (bi < m && kb * kTcKb + bcol < pc) {
                            float vv[kTcBValsPerThread];
#pragma unroll
                            for (int q = 0; q < kTcBValsPerThread; q += 2) {
                                const float2 v2 = *reinterpret_cast<const float2 *>(xs + bi * kTcXCols + bcol + q);
                                vv[q] = v2.x;
                                vv[q + 1] = v2.y;
                            }
#pragma unroll
                            for (int q = 0; q < kTcBValsPerThread / 2; ++q) {
                                const float s0 = vv[2 * q] * pfa * pfb, s1 = vv[2 * q + 1] * pfa * pfb;
                                const __half2 hh = __floats2half2_rn(s0, s1);
                                const float2 hb = __half22float2(hh);
                                const __half2 ll = __floats2half2_rn(s0 - hb.x, s1 - hb.y);
                                hw[q] = *reinterpret_cast<const uint32_t *>(&hh);
                                lw[q] = *reinterpret_cast<const uint32_t *>(&ll);
                            }
                        }
                        // core column bc / 8, byte offset (bc % 8) * 2 within the 16-byte row
                        uint8_t *bh = btile + (bc >> 3) * 128 + bi * 16 + (bc & 7) * 2;
#pragma unroll
                        for (int q = 0; q < kTcBValsPerThread / 2; ++q) {
                            *reinterpret_cast<uint32_t *>(bh + 4 * q) = hw[q];
                            *reinterpret_cast<uint32_t *>(bh + kTcSbo + 4 * q) = lw[q];
                        }
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    const bool stage_done = sub == kTcSub - 1 && (k2 == kTcKbPerStage - 1 || kb == nkb - 1);
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
                tc_ld16(tmem + static_cast<uint32_t>(acc * kTcN) + (static_cast<uint32_t>(warp * 32) << 16), v);
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
            case 2: argmax_cross_cta<2, kTcThreads>(ga, am_val, am_idx, &s_is_last); break;
            case 3: argmax_cross_cta<3, kTcThreads>(ga, am_val, am_idx, &s_is_last); break;
            case 4: argmax_cross_cta<4, kTcThreads>(ga, am_val, am_idx, &s_is_last); break;
            case 5: argmax_cross_cta<5, kTcThreads>(ga, am_val, am_idx, &s_is_last); break;
            case 6: argmax_cross_cta<6, kTcThreads>(ga, am_val, am_idx, &s_is_last); break;
            case 7: argmax_cross_cta<7, kTcThreads>(ga, am_val, am_idx, &s_is_last); break;
            default: argmax_cross_cta<8, kTcThreads>(ga, am_val, am_idx, &s_is_last); break;
        }
    }
}

}  // namespace fp8blk
