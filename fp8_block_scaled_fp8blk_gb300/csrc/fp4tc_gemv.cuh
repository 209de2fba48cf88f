// fp4tc_gemv.cuh -- NVFP4 and OCP MXFP4 routed-expert GEMV on the
// fifth-generation tensor cores, all active experts in one launch, the e2m1
// codes fed to the MMA as stored:
//   y[k][r] = g[e] * sum_b s[e][r][b] * sum_{c in block b} e2m1(q[e][r][c]) x[c],
//   e = ids[k]; NVFP4: blocks of 16 columns, s = e4m3; MXFP4: blocks of 32,
//   s = 2^(e8m0 - 127), g = 1.
// Source: "Module dsv4_gpu" page, module header and enums ExpertArm /
// ExpertKind (routed experts stay NVFP4 as stored, the MTP block's are OCP
// MXFP4; each activated expert's weights take the exact values of their
// dequantisation; one launch per projection, expert ids on the device).  The
// sum is the one the CUDA-core kernel forms, grouped by scale block.  The
// description below is NVFP4's; MXFP4 has one block per K = 32 step (B rows
// 0-4) and a scale-ring slot per stage pair.
//
// A (M = 128 weight rows x K): the packed codes.  A 2-D TMA box of 128 e2m1
//   columns with the 16 x U4 / 16-byte-aligned element type writes each 8
//   bytes of codes into a 16-byte shared-memory chunk (8 bytes of zeros
//   after them), the layout kind::f8f6f4 reads e2m1 operands in, under the
//   128-byte swizzle; the CUDA cores never touch a weight.
// B (N = 16 x K, e4m3): x in blocks of 16 columns, v = x 2^e_b with e_b the
//   block's exponent (2^7 <= max|v| < 2^8), split into five e4m3 planes
//   t_0 = v, q_p = e4m3(t_p), t_{p+1} = 16 (t_p - q_p): every subtraction is
//   exact and each plane adds 4 bits (2^-20 of each element).  One K = 32 MMA
//   step covers two blocks; B rows 0-4 hold block 2j's planes (zeros under
//   block 2j + 1), rows 5-9 block 2j + 1's, so the step's D columns are the
//   ten (block, plane) sums of 16 products, each exact in f32.  B is built
//   once per CTA for all of x.
// D (TMEM): 16 columns per step, eight steps per 256-column stage, a ring of
//   four stages (512 columns).  The epilogue forms per row
//   acc += e4m3(s[r][b]) * ((sum_p D[b][p] 2^-4p) * 2^-e_b)   (f32),
//   in block order within four sums (even / odd blocks of even / odd
//   stages), added in a fixed order at the end.  The inner product by the
//   power of two is exact: it is the block sum in x's units, so the scale is
//   applied to the same value as on the CUDA cores, and a block of zero codes
//   adds zero whatever its scale and x (the other grouping could form
//   scale * 2^-e_b = inf and then 0 * inf).
//
// Work: units (active slot, R-row slab of the expert, R <= 128 chosen on the
// host so the units fill the SMs), contiguous ranges per CTA; an MMA always
// covers 128 rows and the lanes past the slab are never read.  Stages of 256
// columns: two code boxes of R rows (a ring freed by the MMAs) and one R x
// 16-byte box of scales (a deeper ring freed by the epilogue, so the copies
// run ahead of it).
// Roles (one CTA per SM, 416 threads):
//   warps 0-7   epilogue: warp w drains TMEM lanes 32 (w % 4).. (slab rows)
//               of the even (w < 4) or odd stages, so a group has two stage
//               times for each stage's waits, loads and sums; the two sums of
//               a row meet in shared memory at the end of the unit; warp 0
//               allocates and frees tensor memory;
//   warp 8      TMA producer (one lane);
//   warps 9-12  MMA issuers (one lane each): warp 9 + i issues the eight
//               steps of every stage g with g % 4 == i, into D stage i (one
//               thread takes about 0.4 us for a stage's MMAs and two
//               commits; four threads on whole stages were measured faster
//               than any split of a stage's steps).
// An expert id outside [0, n_experts) or an unusable global scale makes the
// slot's outputs NaN and sets FP8BLK_STATUS_BAD_EXPERT; an inf or NaN in x
// makes every output NaN (the exact sums are not finite).  Every wait is
// bounded; a timeout raises a CTA-wide abort flag, every role leaves its
// loop, copies in flight land, the MMAs complete before the tensor memory is
// freed, and the status word records it.
#pragma once

#include "launch.h"
#include "nvfp4_gemv.cuh"
#include "tc8_gemv.cuh"

namespace fp8blk {

constexpr int kF4StageCols = kF4StageColsHost;                 // columns per raw stage (256)
constexpr int kF4BoxCols = 128;                                // e2m1 columns per code box
constexpr int kF4RowSmem = 128;                                // one box row in shared memory (gaps included)
constexpr int kF4ScaleSlots = 8;                               // scale ring (R x 16 bytes each)
constexpr int kF4ScaleSlotSmem = 128 * 16;
constexpr int kF4Steps = kF4StageCols / 32;                    // K = 32 MMA steps per stage
constexpr int kF4Planes = 5;
constexpr int kF4N = 16;
constexpr int kF4BTileBytes = kF4N * 128;                      // B for 128 columns (four steps)
constexpr int kF4DStages = 4;                                  // D ring: 4 x 128 columns
constexpr int kF4MaxRawStages = 8;
constexpr int kF4MinRawStages = 4;
constexpr int kF4EpiWarps = 8;                                 // two groups of four (even / odd stages)
constexpr int kF4ProducerWarp = 8;
constexpr int kF4MmaWarp0 = 9;
constexpr int kF4Issuers = 4;                                  // issuer i: the stages g with g % 4 == i
constexpr int kF4Threads = (kF4MmaWarp0 + kF4Issuers) * 32;
// Issuer i owns D stage i and the code slots i, i + 4: it alone waits on and
// commits to their barriers, in stage order, so no parity wait can be met by
// an older phase.  Hence a ring of 4 or 8 stages.
static_assert(kF4DStages == kF4Issuers && kF4MaxRawStages % kF4Issuers == 0 && kF4MinRawStages == kF4Issuers,
              "issuers own their D stage and code slots");
constexpr int kF4TmemCols = 512;
constexpr uint32_t kF4IDesc = t8_idesc(128, kF4N) | (5u << 7);  // A e2m1 (format 5), B e4m3, D f32

// Dynamic shared memory: 1024 (alignment) + B (16 bytes per column) + the
// code ring (two boxes of R rows x 128 bytes per stage) + the scale ring +
// the block factors 2^-e_b (4 bytes per 16 columns) + the row sums of the
// second epilogue group (2 x 128 f32), at least 116 KiB so that one CTA
// holds an SM (and its 512 TMEM columns).  An MMA reads 128 rows of a box:
// past the last stage's second box it reads into the scale ring (16 KiB,
// enough for 120 rows), garbage in lanes that are never read.
constexpr int64_t kF4FixedSmem = 1024 + kF4ScaleSlots * kF4ScaleSlotSmem + 2 * 128 * 4;
__host__ __device__ constexpr int64_t f4_stage_smem(int slab_rows) { return 2 * kF4RowSmem * slab_rows; }
__host__ __device__ constexpr size_t f4_smem_need(int64_t cols, int raw_stages, int slab_rows) {
    return static_cast<size_t>(kF4FixedSmem + 16 * cols + cols / 4 + raw_stages * f4_stage_smem(slab_rows));
}
__host__ __device__ constexpr size_t f4_smem_bytes(int64_t cols, int raw_stages, int slab_rows) {
    return f4_smem_need(cols, raw_stages, slab_rows) < 116 * 1024 ? 116 * 1024
                                                                  : f4_smem_need(cols, raw_stages, slab_rows);
}
// Code ring depth for a budget: the most stages that fit, at most
// kF4MaxRawStages, rounded down to a multiple of kF4Issuers (0 if under 4).
__host__ __device__ constexpr int f4_raw_stages(int64_t cols, int slab_rows, int64_t budget) {
    return ((budget - kF4FixedSmem - 16 * cols - cols / 4) / f4_stage_smem(slab_rows) > kF4MaxRawStages
                ? kF4MaxRawStages
                : static_cast<int>((budget - kF4FixedSmem - 16 * cols - cols / 4) / f4_stage_smem(slab_rows))) /
           kF4Issuers * kF4Issuers;
}

struct F4Args {
    Nvfp4Args nv;        // ids, global scales, x, y, status, sizes
    int64_t n_slabs;     // slabs per expert
    int64_t units;       // n_active * n_slabs
    int slab_rows;       // R, a multiple of 8 in [8, 128]
    int raw_stages;      // kF4MinRawStages .. kF4MaxRawStages
};

// Waits as t8_wait / t8_warp_wait, after a non-blocking test: a phase that
// has already completed is seen without entering the suspending wait.
__device__ __forceinline__ bool f4_wait(uint32_t bar, uint32_t parity, int *abort_flag) {
    return mbar_test_wait(bar, parity) || t8_wait(bar, parity, abort_flag);
}
__device__ __forceinline__ bool f4_warp_wait(uint32_t bar, uint32_t parity, int *abort_flag, int lane) {
    bool ok = true;
    if (lane == 0) ok = f4_wait(bar, parity, abort_flag);
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();
    return ok;
}

__device__ __forceinline__ void f4_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// TMEM -> registers: 8 consecutive 32-bit columns of the warp's 32 lanes
// (MXFP4 uses 5 of a step's 16 columns).
__device__ __forceinline__ void f4_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

template <int FP4>
__global__ void __launch_bounds__(kF4Threads, 1)
    fp4tc_gemv_kernel(const __grid_constant__ CUtensorMap cmap, const __grid_constant__ CUtensorMap smap,
                      const F4Args a) {
    // Scale blocks of SB columns: NVFP4 e4m3 per 16 (two blocks per K = 32
    // step, block-diagonal B), MXFP4 e8m0 per 32 (one block per step).
    constexpr bool kMx = FP4 == kFp4Mx;
    constexpr int SB = fp4_scale_cols<FP4>();
    extern __shared__ __align__(1024) uint8_t f4_smem[];
    __shared__ __align__(8) uint64_t raw_full[kF4MaxRawStages], raw_free[kF4MaxRawStages];
    __shared__ __align__(8) uint64_t sc_full[kF4ScaleSlots], sc_free[kF4ScaleSlots];
    __shared__ __align__(8) uint64_t d_full[kF4DStages], d_free[kF4DStages], mma_done[kF4Issuers];
    __shared__ __align__(8) uint64_t comb_full[2], comb_free[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int s_abort;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const Nvfp4Args &nv = a.nv;
    const int RS = a.raw_stages;
    const int R = a.slab_rows;

    // [B (cols x 16 bytes) | code ring | scale ring | 2^-e_b per block |
    //  second-half row sums], B and the code ring 1024-aligned.
    uint8_t *sB = f4_smem + ((1024u - (smem_addr(f4_smem) & 1023u)) & 1023u);
    uint8_t *sRaw = sB + 16 * nv.cols;
    const int stage_smem = 2 * kF4RowSmem * R;  // a multiple of 1024
    uint8_t *sSc = sRaw + static_cast<size_t>(RS) * stage_smem;
    float *sC = reinterpret_cast<float *>(sSc + kF4ScaleSlots * kF4ScaleSlotSmem);
    float *sAcc = sC + nv.cols / 16;  // [2][128]

    const int64_t U0 = static_cast<int64_t>(blockIdx.x) * a.units / gridDim.x;
    const int64_t U1 = static_cast<int64_t>(blockIdx.x + 1) * a.units / gridDim.x;
    const int n_units = static_cast<int>(U1 - U0);
    const int nrs = static_cast<int>(nv.cols / kF4StageCols);  // raw stages per unit

    if (tid == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(smem_addr(&raw_full[s]), 1);
            mbar_init(smem_addr(&raw_free[s]), 1);  // the stage's issuer
        }
        for (int s = 0; s < kF4ScaleSlots; ++s) {
            mbar_init(smem_addr(&sc_full[s]), 1);
            mbar_init(smem_addr(&sc_free[s]), kF4EpiWarps / 2);  // one epilogue group per stage
        }
        for (int j = 0; j < kF4DStages; ++j) {
            mbar_init(smem_addr(&d_full[j]), 1);  // issuer j
            mbar_init(smem_addr(&d_free[j]), kF4EpiWarps / 2);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(smem_addr(&comb_full[j]), kF4EpiWarps / 2);
            mbar_init(smem_addr(&comb_free[j]), kF4EpiWarps / 2);
        }
        for (int j = 0; j < kF4Issuers; ++j) mbar_init(smem_addr(&mma_done[j]), 1);
        mbar_init_fence();
        s_abort = 0;
    }
    // B starts as zeros: the half of each step row outside its block, and
    // rows 10-15, stay zero.
    for (int64_t i = tid; i < nv.cols; i += kF4Threads) reinterpret_cast<uint4 *>(sB)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_slot)),
                     "r"(kF4TmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    t8_fence_before();
    __syncthreads();
    t8_fence_after();
    const uint32_t tmem = tmem_slot;

    // The ids, global scales and x may be outputs of the preceding kernel.
    grid_dependency_wait();
    grid_launch_dependents();

    // Producer cursor: the next stage to copy (unit, stage of the unit, code
    // and scale ring slots and passes, slot k and slab of the unit),
    // advanced by counters.
    int p_unit = 0, p_rs = 0, p_slot = 0, p_sslot = 0, p_k = static_cast<int>(U0 / a.n_slabs), p_row0 = 0;
    uint32_t p_pass = 0, p_spass = 0, p_issued = 0;
    int64_t p_slab = U0 % a.n_slabs;
    bool p_ok = false;  // the unit's expert is usable
    NvSlot pcache;
    auto p_unit_start = [&]() {
        const int e = nv_slot<FP4>(nv, p_k, pcache).e;
        p_ok = e >= 0;
        p_row0 = p_ok ? static_cast<int>(static_cast<int64_t>(e) * nv.rows + p_slab * R) : 0;
    };
    auto p_issue_next = [&](uint64_t pol) {
        const uint32_t cbar = smem_addr(&raw_full[p_slot]), sbar = smem_addr(&sc_full[p_sslot]);
        if (!p_ok) {  // nothing to copy: complete the phases so the consumers move on
            mbar_arrive(cbar);
            mbar_arrive(sbar);
        } else {
            uint8_t *st = sRaw + static_cast<size_t>(p_slot) * stage_smem;
            mbar_arrive_expect_tx(cbar, static_cast<uint32_t>(R) * kF4BoxCols);  // two boxes of R x 64 packed bytes
            t8_tma_2d(smem_addr(st), &cmap, p_rs * kF4StageCols, p_row0, cbar, pol);
            t8_tma_2d(smem_addr(st + kF4RowSmem * R), &cmap, p_rs * kF4StageCols + kF4BoxCols, p_row0, cbar, pol);
            mbar_arrive_expect_tx(sbar, static_cast<uint32_t>(R) * 16);
            t8_tma_2d(smem_addr(sSc + p_sslot * kF4ScaleSlotSmem), &smap, kMx ? (p_rs >> 1) * 16 : p_rs * 16, p_row0, sbar,
                      pol);
        }
        ++p_issued;
        if (++p_slot == RS) {
            p_slot = 0;
            ++p_pass;
        }
        if (++p_sslot == kF4ScaleSlots) {
            p_sslot = 0;
            ++p_spass;
        }
        if (++p_rs == nrs) {
            p_rs = 0;
            if (++p_slab == a.n_slabs) {
                p_slab = 0;
                ++p_k;
            }
            if (++p_unit < n_units) p_unit_start();
        }
    };
    // The first ring's worth of copies go out before B is built.
    if (warp == kF4ProducerWarp && lane == 0) {
        const uint64_t pol = l2_policy_evict_first();
        p_unit_start();
        for (int v = 0; v < RS && p_unit < n_units; ++v) p_issue_next(pol);
    }

    // ---- B and the block factors, once per CTA, by every warp but the
    // producer's.  Four lanes share a block; four float4 of x are in flight
    // per thread.
    constexpr int kBThreads = kF4Threads - 32;
    const int btid = tid < kF4ProducerWarp * 32 ? tid : tid - 32;
    for (int64_t c0 = 4 * static_cast<int64_t>(btid); warp != kF4ProducerWarp && c0 < nv.cols;
         c0 += 16 * kBThreads) {
        float4 xv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t c = c0 + static_cast<int64_t>(u) * 4 * kBThreads;
            xv[u] = c < nv.cols ? t8_ld_f32x4(nv.x + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t c = c0 + static_cast<int64_t>(u) * 4 * kBThreads;
            if (c >= nv.cols) break;  // the same for the lanes of a block
            const float4 v = xv[u];
            auto fin = [](float f) {  // |f| as bits, 0 for inf / NaN
                const uint32_t b = __float_as_uint(fabsf(f));
                return b < 0x7F800000u ? b : 0u;
            };
            uint32_t mx = max(max(fin(v.x), fin(v.y)), max(fin(v.z), fin(v.w)));
            uint32_t bad = (fabsf(v.x) < INFINITY && fabsf(v.y) < INFINITY && fabsf(v.z) < INFINITY &&
                            fabsf(v.w) < INFINITY)
                               ? 0u
                               : 1u;
            constexpr int GL = SB / 4;  // lanes per scale block
            const uint32_t grp = ((1u << GL) - 1u) << (lane & ~(GL - 1));
#pragma unroll
            for (int o = 1; o < GL; o <<= 1) {
                mx = max(mx, __shfl_xor_sync(grp, mx, o));
                bad |= __shfl_xor_sync(grp, bad, o);
            }
            const int eb = t8_plane_exponent(__uint_as_float(mx));  // 2^7 <= max |x| 2^eb < 2^8 (finite max)
            float f1, f2;
            t8_pow2_split(eb, f1, f2);
            if ((lane & (GL - 1)) == 0) {
                float g1, g2;
                t8_pow2_split(-eb, g1, g2);
                sC[c / SB] = bad ? __int_as_float(0x7FC00000) : g1 * g2;
            }
            float t0 = bad ? 0.f : v.x * f1 * f2, t1 = bad ? 0.f : v.y * f1 * f2;
            float t2 = bad ? 0.f : v.z * f1 * f2, t3 = bad ? 0.f : v.w * f1 * f2;
            // Column c: 128-column tile G, step j, block parity h, offset o in the block.
            const int64_t G = c >> 7;
            const int j = static_cast<int>((c >> 5) & 3), h = static_cast<int>((c >> 4) & 1),
                      o = static_cast<int>(c & 15);
            uint8_t *bt = sB + G * kF4BTileBytes;
#pragma unroll
            for (int p = 0; p < kF4Planes; ++p) {
                const uint32_t lo = t8_to_e4m3x2(t0, t1), hi = t8_to_e4m3x2(t2, t3);
                const int n = kMx ? p : 5 * h + p;  // MXFP4: the step's one block spans both halves
                *reinterpret_cast<uint32_t *>(bt + (n >> 3) * 1024 + (n & 7) * 128 + (((2 * j + h) ^ (n & 7)) << 4) +
                                              o) = lo | (hi << 16);
                if (p + 1 < kF4Planes) {
                    const float2 qlo = e4m3x2_to_f32(lo), qhi = e4m3x2_to_f32(hi);
                    t0 = (t0 - qlo.x) * 16.f;
                    t1 = (t1 - qlo.y) * 16.f;
                    t2 = (t2 - qhi.x) * 16.f;
                    t3 = (t3 - qhi.y) * 16.f;
                }
            }
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic stores -> the MMA
    __syncthreads();

    if (warp == kF4ProducerWarp) {
        // ---------------- TMA producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            while (p_unit < n_units) {
                if ((p_pass > 0 && !f4_wait(smem_addr(&raw_free[p_slot]), (p_pass - 1u) & 1u, &s_abort)) ||
                    (p_spass > 0 && !f4_wait(smem_addr(&sc_free[p_sslot]), (p_spass - 1u) & 1u, &s_abort)))
                    break;
                p_issue_next(pol);
            }
            // Copies still in flight must land before the shared memory is released.
            for (uint32_t w = p_issued > static_cast<uint32_t>(RS) ? p_issued - RS : 0u; w < p_issued; ++w)
                (void)mbar_wait_bounded(smem_addr(&raw_full[w % RS]), (w / RS) & 1u);
            for (uint32_t w = p_issued > static_cast<uint32_t>(kF4ScaleSlots) ? p_issued - kF4ScaleSlots : 0u;
                 w < p_issued; ++w)
                (void)mbar_wait_bounded(smem_addr(&sc_full[w % kF4ScaleSlots]), (w / kF4ScaleSlots) & 1u);
        }
    } else if (warp >= kF4MmaWarp0) {
        // ---------------- MMA issuer i: all steps of the stages g with
        // g % kF4Issuers == i, one commit per barrier per stage.  Issuing
        // threads run in parallel on different stages: a thread's tcgen05
        // ops, not the tensor pipe, set the rate.
        const int iss = warp - kF4MmaWarp0;
        if (lane == 0) {
            int slot = 0;
            uint32_t pass = 0, g = 0;  // ring pass; stages so far
            bool stop = false;
            for (int i = 0; i < n_units && !stop; ++i) {
                for (int rs = 0; rs < nrs; ++rs, ++g) {
                    if (static_cast<int>(g % kF4Issuers) == iss) {
                        const int ds = iss;  // g % kF4DStages
                        if (!f4_wait(smem_addr(&raw_full[slot]), pass & 1u, &s_abort) ||
                            (g >= kF4DStages &&
                             !f4_wait(smem_addr(&d_free[ds]), ((g / kF4DStages) - 1u) & 1u, &s_abort))) {
                            stop = true;
                            break;
                        }
                        t8_fence_after();
                        const uint32_t st = smem_addr(sRaw + static_cast<size_t>(slot) * stage_smem);
#pragma unroll
                        for (int t = 0; t < kF4Steps; ++t) {  // step: code box t / 4, K offset 32 (t % 4) bytes
                            const int box = t >> 2, kk = t & 3;
                            const uint32_t bt = smem_addr(sB + static_cast<size_t>(2 * rs + box) * kF4BTileBytes);
                            t8_mma(tmem + static_cast<uint32_t>(ds * 128 + 16 * t),
                                   t8_desc_sw128(st + box * kF4RowSmem * R + 32u * kk), t8_desc_sw128(bt + 32u * kk),
                                   kF4IDesc, false);
                        }
                        t8_commit(smem_addr(&raw_free[slot]));
                        t8_commit(smem_addr(&d_full[ds]));
                    }
                    if (++slot == RS) {
                        slot = 0;
                        ++pass;
                    }
                }
            }
            t8_commit(smem_addr(&mma_done[iss]));
            (void)mbar_wait_bounded(smem_addr(&mma_done[iss]), 0u);
        }
    } else {
        // ---------------- epilogue: warp w drains TMEM lanes 32 (w % 4) ..
        // + 31 (slab rows) for the stages of its group's parity, w / 4.
        const int qr = warp & 3, hf = warp >> 2;
        const int r = 32 * qr + lane;  // row of the slab
        NvSlot cache;
        int k = static_cast<int>(U0 / a.n_slabs);
        int64_t slab = U0 % a.n_slabs;
        uint32_t g = 0;
        bool stop = false;
        for (int i = 0; i < n_units && !stop; ++i) {
            if (i > 0 && ++slab == a.n_slabs) {
                slab = 0;
                ++k;
            }
            float acc0 = 0.f, acc1 = 0.f;  // even and odd blocks
            for (int rs = 0; rs < nrs; ++rs, ++g) {
                if ((g & 1u) != static_cast<uint32_t>(hf)) continue;
                // This row's block scales of the stage: NVFP4 16 e4m3 bytes;
                // MXFP4 8 e8m0 bytes, the stage pair's slot half (rs & 1).
                const int ss = static_cast<int>(g % kF4ScaleSlots);
                if (!f4_warp_wait(smem_addr(&sc_full[ss]), (g / kF4ScaleSlots) & 1u, &s_abort, lane)) {
                    stop = true;
                    break;
                }
                uint4 sc = make_uint4(0u, 0u, 0u, 0u);
                if (r < R) sc = *reinterpret_cast<const uint4 *>(sSc + ss * kF4ScaleSlotSmem + 16 * r);
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&sc_free[ss]));
                const int ds = static_cast<int>(g % kF4DStages);
                if (!f4_warp_wait(smem_addr(&d_full[ds]), (g / kF4DStages) & 1u, &s_abort, lane)) {
                    stop = true;
                    break;
                }
                t8_fence_after();
                const uint32_t sw[4] = {sc.x, sc.y, sc.z, sc.w};
                const uint32_t mw0 = (rs & 1) ? sc.z : sc.x, mw1 = (rs & 1) ? sc.w : sc.y;  // MXFP4: this stage's 8 bytes
                const float *cb = sC + static_cast<size_t>(rs) * (kF4StageCols / SB);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    // NVFP4 reads a step's ten plane sums, MXFP4 its five
                    uint32_t d[kF4Steps / 2][kMx ? 8 : 16];
#pragma unroll
                    for (int t = 0; t < kF4Steps / 2; ++t) {
                        const uint32_t ta = tmem + static_cast<uint32_t>(ds * 128 + 16 * (4 * half + t)) +
                                            (static_cast<uint32_t>(qr * 32) << 16);
                        if constexpr (kMx)
                            f4_ld8(ta, d[t]);
                        else
                            f4_ld16(ta, d[t]);
                    }
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                    if (half == 1) {
                        t8_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_addr(&d_free[ds]));
                    }
#pragma unroll
                    for (int t = 0; t < kF4Steps / 2; ++t) {
                        const int T = 4 * half + t;
                        if constexpr (kMx) {
                            // block T of the stage: e8m0 byte 8 (rs & 1) + T of the slot row
                            const uint32_t byte = ((T >> 2 ? mw1 : mw0) >> (8 * (T & 3))) & 0xFFu;
                            float u = __uint_as_float(d[t][kF4Planes - 1]);
#pragma unroll
                            for (int p = kF4Planes - 2; p >= 0; --p) u = fmaf(u, 0.0625f, __uint_as_float(d[t][p]));
                            // u * 2^-e_b is exact (a power of two): the block sum
                            // in x's units, scaled as the CUDA-core kernel does
                            if (T & 1)
                                acc1 = fmaf(e8m0_to_f32(byte), u * cb[T], acc1);
                            else
                                acc0 = fmaf(e8m0_to_f32(byte), u * cb[T], acc0);
                        } else {
                            // blocks 2T, 2T + 1 of the stage: scale bytes 2T, 2T + 1
                            const float2 s2 = e4m3x2_to_f32((sw[T >> 1] >> (16 * (T & 1))) & 0xFFFFu);
                            float u[2];
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                u[hh] = __uint_as_float(d[t][5 * hh + kF4Planes - 1]);
#pragma unroll
                                for (int p = kF4Planes - 2; p >= 0; --p)
                                    u[hh] = fmaf(u[hh], 0.0625f, __uint_as_float(d[t][5 * hh + p]));
                            }
                            acc0 = fmaf(s2.x, u[0] * cb[2 * T], acc0);
                            acc1 = fmaf(s2.y, u[1] * cb[2 * T + 1], acc1);
                        }
                    }
                }
            }
            if (stop) break;
            // Row sum = (even stages) + (odd stages), the odd stages' sum passed
            // through shared memory (double-buffered by unit parity).
            const float part = acc0 + acc1;
            const int cbuf = i & 1;
            if (hf == 1) {
                if (i >= 2 && !f4_warp_wait(smem_addr(&comb_free[cbuf]), ((i >> 1) - 1) & 1, &s_abort, lane)) break;
                sAcc[cbuf * 128 + r] = part;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&comb_full[cbuf]));
            } else {
                if (!f4_warp_wait(smem_addr(&comb_full[cbuf]), (i >> 1) & 1, &s_abort, lane)) break;
                const float total = part + sAcc[cbuf * 128 + r];
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&comb_free[cbuf]));
                const NvSlot &sl = nv_slot<FP4>(nv, k, cache);
                const int64_t row = slab * R + r;
                if (r < R && row < nv.rows)
                    nv.y[static_cast<int64_t>(k) * nv.rows + row] = sl.e >= 0 ? total * sl.g : __int_as_float(0x7FC00000);
                if (sl.e < 0 && slab == 0 && tid == 0) atomicOr(nv.status, kStatusBadExpert);
            }
        }
    }

    if (tid == 0 && *reinterpret_cast<volatile int *>(&s_abort)) atomicOr(nv.status, 1u);
    t8_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kF4TmemCols) : "memory");
}

}  // namespace fp8blk
