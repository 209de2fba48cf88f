// tc8_gemv.cuh -- the e4m3 decode / verify GEMV on the fifth-generation
// tensor cores, with the weight codes fed to the MMA exactly as stored.
//
// y[i][r] = sum_c e4m3(W[r][c]) * S[r/128][c/128] * x[i][c] ("Module dsv4_gpu"
// page, struct Fp8Dense; "Struct Dsv4Gpu" page, verify_batch_dev: T = k+1
// activation rows).
//
// A CTA owns whole 128-row tiles, each one row block of the scale grid, so
// within a tile the block scale is one number S_kb per 128-column K-block.
// A (M = 128 weight rows x K): the e4m3 codes themselves.  A 2-D TMA box of
//   128 rows x 128 bytes with the 128-byte swizzle lands each K-block in
//   shared memory in the layout tcgen05.mma reads, so the CUDA cores never
//   touch a weight (kind::f8f6f4, e4m3 x e4m3 -> f32).
// B (N = 16 / 32 / 48 x K): v = x * S_kb * 2^e, split into kPlanes e4m3
//   planes per activation row: t_0 = v, q_p = e4m3(t_p), t_{p+1} = 16 (t_p -
//   q_p).  e is one exponent per activation row and tile, chosen from
//   max_kb |S_kb| * max|x over K-block kb| so that |v| < 256: no plane
//   saturates, every subtraction is exact, and each plane adds 4 bits, so an
//   element keeps 2^-20 of itself (absolute floor 2^-33 of the tile maximum),
//   inside the 1e-5 * sum|w x| bound.  x * S rounds once in f32.
// D (TMEM, 128 lanes x N f32): per tile one accumulator per MMA warp (even
//   and odd K-blocks), double buffered across tiles;
//   y[i][r] = 2^-e * sum_p (D0 + D1)[r][i P + p] 2^-4p, summed in that order.
//
// Roles (one CTA per SM, 480 threads):
//   warps 0-3   epilogue: TMEM lanes 32w.. = tile rows; drain a tile, write y,
//               greedy argmax; warp 0 allocates and frees tensor memory;
//   warps 4-11  B builders: warp 4 + 2s + k builds K-block k of every ring
//               stage in slot s;
//   warp 12     TMA producer (one lane): weight boxes;
//   warps 13-14 MMA issuers (one lane each): warp 13 + k issues the four
//               K = 32 MMAs of K-block k of every stage into its own
//               accumulator (a single issuing thread is the bottleneck
//               otherwise); one commit per stage and one per tile each.
// Before the roles split, every warp takes the block maxima of |x| (x is read
// after the grid dependency wait); the first ring of weight copies follows.  Every wait is bounded; a timeout raises a
// CTA-wide abort flag, every role leaves its loop, copies in flight land
// (fixed bound), the MMAs complete before the tensor memory is freed, and the
// status word records it.
#pragma once

#include <cuda.h>

#include "stream_gemv.cuh"

namespace fp8blk {

constexpr int kT8Planes = 5;           // e4m3 planes per activation row
constexpr int kT8Kb = 128;             // columns per K-block (one scale block, one TMA box)
constexpr int kT8KbPerStage = 2;       // K-blocks per ring stage
constexpr int kT8Stages = 4;           // ring depth (A boxes and B operands share the slot index)
constexpr int kT8EpiWarps = 4;
constexpr int kT8BWarp0 = 4;
constexpr int kT8BWarps = kT8Stages * kT8KbPerStage;  // one builder warp per (slot, K-block)
constexpr int kT8ProducerWarp = kT8BWarp0 + kT8BWarps;
constexpr int kT8MmaWarp = kT8ProducerWarp + 1;   // issues K-block 0 of every stage; the next warp, K-block 1
constexpr int kT8MmaWarps = kT8KbPerStage;
constexpr int kT8Threads = (kT8MmaWarp + kT8MmaWarps) * 32;
constexpr int kT8PrepassRound = 18;                // block maxima in flight per warp
constexpr int64_t kT8PrefetchChunk = 32768;         // bytes per L2 prefetch instruction
constexpr int kT8TileBytes = 128 * kT8Kb;                 // 16 KiB per K-block
constexpr int kT8StageBytes = kT8KbPerStage * kT8TileBytes;
constexpr int kT8MaxN = 48;
constexpr int kT8BTileBytes = kT8MaxN * kT8Kb;            // 6 KiB per K-block
constexpr int kT8MaxKb = 256;                             // K-blocks per row the block-max table holds
constexpr size_t kT8SmemBytes = 1024 + static_cast<size_t>(kT8Stages) * kT8StageBytes +
                                static_cast<size_t>(kT8Stages) * kT8KbPerStage * kT8BTileBytes +
                                static_cast<size_t>(8) * kT8MaxKb * sizeof(float);

__host__ __device__ constexpr int t8_n_cols(int m) { return (m * kT8Planes + 15) / 16 * 16; }
// Two tiles in flight x one accumulator per MMA warp.
__host__ __device__ constexpr int t8_tmem_cols(int n) {
    return 4 * n <= 32 ? 32 : 4 * n <= 64 ? 64 : 4 * n <= 128 ? 128 : 256;
}

struct T8Args {
    const uint8_t *w;        // e4m3 codes [rows, cols] (what the tensor map describes)
    const float *scales;     // f32 grid [ceil(rows/128), ceil(cols/128)]
    const float *x;          // [m, cols]
    float *y;                // [m, rows] or null (argmax only)
    uint32_t *tokens;        // [m] (ARGMAX)
    float *part_val;         // [grid, m] (ARGMAX)
    uint32_t *part_idx;
    uint32_t *counter;
    unsigned int *status;
    int64_t rows, cols;
    int m;
    int64_t n_tiles;         // ceil(rows / 128)
    int64_t l2_prefetch;     // bytes of the CTA's first rows prefetched into L2 at entry (0: none)
};

// UMMA shared-memory descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (what a SWIZZLE_128B TMA box with 128-byte rows produces).
__device__ __forceinline__ uint64_t t8_desc_sw128(uint32_t saddr) {
    uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(16 >> 4) << 16;    // leading byte offset (unused when swizzled)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;  // stride byte offset: 8 rows x 128 B
    d |= static_cast<uint64_t>(1) << 46;          // sm_100-family descriptor version
    d |= static_cast<uint64_t>(2) << 61;          // 128-byte swizzle
    return d;
}

// kind::f8f6f4 instruction descriptor: e4m3 A and B, f32 D, both K-major.
__host__ __device__ constexpr uint32_t t8_idesc(int m_rows, int n_cols) {
    return (1u << 4) | (static_cast<uint32_t>(n_cols >> 3) << 17) | (static_cast<uint32_t>(m_rows >> 4) << 24);
}

__device__ __forceinline__ void t8_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(static_cast<uint32_t>(acc))
        : "memory");
}

__device__ __forceinline__ void t8_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void t8_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void t8_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void t8_tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// 16 consecutive f32 columns of this warp's 32 TMEM lanes (no wait).
__device__ __forceinline__ void t8_ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// Two f32 -> e4m3x2 (round to nearest even, saturating to the finite range);
// `lo` lands in the low byte.
__device__ __forceinline__ uint32_t t8_to_e4m3x2(float lo, float hi) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// 2^e as two normal f32 factors, -252 <= e <= 254 (a product with them is
// exact while the result stays normal).
__device__ __forceinline__ void t8_pow2_split(int e, float &f1, float &f2) {
    const int h = e / 2;
    f1 = __int_as_float((h + 127) << 23);
    f2 = __int_as_float((e - h + 127) << 23);
}

// Plane exponent for a tile maximum g >= 0: g * 2^ex in [128, 256); g = 0 or
// subnormal gives 134 (all planes zero or below 2^8); a non-finite g gives
// kT8Poison.
constexpr int kT8Poison = 1000;
__device__ __forceinline__ int t8_plane_exponent(float g) {
    const int be = (__float_as_int(g) >> 23) & 0xFF;
    return be == 0xFF ? kT8Poison : 134 - (be > 0 ? be : 0);
}

// Read-only global loads issued exactly where they stand (volatile asm is
// not moved, so a prefetch stays a prefetch instead of sinking to its use).
__device__ __forceinline__ float t8_ld_f32(const float *p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ float4 t8_ld_f32x4(const float *p) {
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

// max |v| over a warp's 128 values (4 per lane), as f32 bits.  With the sign
// cleared, the unsigned order of f32 bits is the numeric order and every NaN
// sorts above +inf, so a NaN anywhere is what comes out.
__device__ __forceinline__ uint32_t t8_absmax_bits(const float4 &v) {
    const uint32_t a = __float_as_uint(fabsf(v.x)), b = __float_as_uint(fabsf(v.y));
    const uint32_t c = __float_as_uint(fabsf(v.z)), d = __float_as_uint(fabsf(v.w));
    return __reduce_max_sync(0xFFFFFFFFu, max(max(a, b), max(c, d)));
}

// Single-thread wait for phase `parity`: the hinted try_wait suspends the
// thread until the phase completes (or the hint elapses), so a waiting role
// takes no issue slots from the warps doing arithmetic.  Gives up when the
// CTA aborts or after kWaitLimitNs (then raises the abort flag).
__device__ __forceinline__ bool t8_wait(uint32_t bar, uint32_t parity, int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int *>(abort_flag)) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *reinterpret_cast<volatile int *>(abort_flag) = 1;
            return false;
        }
    }
}

// A whole warp's wait: lane 0 waits (as t8_wait), the outcome is broadcast,
// and __syncwarp orders the warp's later accesses after lane 0's acquire.
__device__ __forceinline__ bool t8_warp_wait(uint32_t bar, uint32_t parity, int *abort_flag, int lane) {
    bool ok = true;
    if (lane == 0) ok = t8_wait(bar, parity, abort_flag);
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();
    return ok;
}

template <bool ARGMAX>
__global__ void __launch_bounds__(kT8Threads, 1)
    tc8_gemv_kernel(const __grid_constant__ CUtensorMap wmap, const T8Args a) {
    extern __shared__ __align__(1024) uint8_t t8_smem[];
    __shared__ __align__(8) uint64_t a_full[kT8Stages], stage_free[kT8Stages], b_full[kT8Stages];
    __shared__ __align__(8) uint64_t d_full[2], d_free[2], mma_done[kT8MmaWarps];
    __shared__ uint32_t tmem_slot;
    __shared__ int s_abort;
    __shared__ float am_val[kT8Threads / 32][8];
    __shared__ uint32_t am_idx[kT8Threads / 32][8];
    __shared__ int s_is_last;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int m = a.m;
    const int N = t8_n_cols(m);

    // Shared memory: [A ring: kT8Stages x two 16 KiB K-block tiles | B
    // operands: kT8Stages x two (N x 128 B) tiles | block maxima M[i][kb]],
    // the tiles 1024-aligned for the 128-byte swizzle.
    uint8_t *sA = t8_smem + ((1024u - (smem_addr(t8_smem) & 1023u)) & 1023u);
    uint8_t *sB = sA + static_cast<size_t>(kT8Stages) * kT8StageBytes;
    float *sM = reinterpret_cast<float *>(sB + static_cast<size_t>(kT8Stages) * kT8KbPerStage * kT8BTileBytes);

    // This CTA's tiles [T0, T1): 128-row blocks, balanced.
    const int64_t T0 = static_cast<int64_t>(blockIdx.x) * a.n_tiles / gridDim.x;
    const int64_t T1 = static_cast<int64_t>(blockIdx.x + 1) * a.n_tiles / gridDim.x;
    const int n_tiles = static_cast<int>(T1 - T0);
    const int nkb = static_cast<int>((a.cols + kT8Kb - 1) / kT8Kb);
    const int nst = (nkb + kT8KbPerStage - 1) / kT8KbPerStage;   // stages per tile
    const int64_t n_stages = static_cast<int64_t>(n_tiles) * nst;
    const int64_t gcols = nkb;

    // The CTA's first weight rows go to L2 at entry, in address order (codes
    // are never outputs of the preceding kernel): HBM streams through the
    // prologue instead of idling with the ring full.  More than about a
    // prologue's worth of streaming crowds out the other CTAs' first stages.
    if (warp == kT8ProducerWarp && lane == 0 && a.l2_prefetch > 0 && n_tiles > 0) {
        const int64_t r0 = T0 * 128, r1 = T1 * 128 < a.rows ? T1 * 128 : a.rows;
        int64_t bytes = (r1 - r0) * a.cols;
        if (bytes > a.l2_prefetch) bytes = a.l2_prefetch;
        bytes &= ~static_cast<int64_t>(15);
        for (int64_t off = 0; off < bytes; off += kT8PrefetchChunk)
            bulk_prefetch_l2(a.w + r0 * a.cols + off,
                             static_cast<uint32_t>(bytes - off < kT8PrefetchChunk ? bytes - off : kT8PrefetchChunk));
    }

    if (tid == 0) {
        for (int s = 0; s < kT8Stages; ++s) {
            mbar_init(smem_addr(&a_full[s]), 1);
            mbar_init(smem_addr(&stage_free[s]), kT8MmaWarps);
            mbar_init(smem_addr(&b_full[s]), kT8KbPerStage);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(smem_addr(&d_full[j]), kT8MmaWarps);
            mbar_init(smem_addr(&d_free[j]), kT8EpiWarps);
        }
        for (int j = 0; j < kT8MmaWarps; ++j) mbar_init(smem_addr(&mma_done[j]), 1);
        mbar_init_fence();
        s_abort = 0;
    }
    // B rows past m * kPlanes stay zero for the whole launch.
    for (int i = tid; i < kT8Stages * kT8KbPerStage * kT8BTileBytes / 16; i += kT8Threads)
        reinterpret_cast<uint4 *>(sB)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_slot)),
                     "r"(t8_tmem_cols(N))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    t8_fence_before();
    __syncthreads();
    t8_fence_after();
    const uint32_t tmem = tmem_slot;

    // ---- ring stage cursor: tile t of the CTA, stage st of the tile, slot s
    struct Cursor {
        int t = 0, st = 0, s = 0;
        uint32_t ph = 0;   // (stage index / kT8Stages) & 1
    };
    auto advance = [&](Cursor &c) {
        if (++c.st == nst) {
            c.st = 0;
            ++c.t;
        }
        if (++c.s == kT8Stages) {
            c.s = 0;
            c.ph ^= 1u;
        }
    };
    auto stage_kbs = [&](int st) { return min(kT8KbPerStage, nkb - st * kT8KbPerStage); };
    const uint64_t pol = l2_policy_evict_first();
    auto issue_stage = [&](const Cursor &c) {
        const int nk = stage_kbs(c.st);
        const uint32_t bar = smem_addr(&a_full[c.s]);
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nk * kT8TileBytes));
        uint8_t *stg = sA + static_cast<size_t>(c.s) * kT8StageBytes;
        const int row0 = static_cast<int>((T0 + c.t) * 128);
        for (int k2 = 0; k2 < nk; ++k2)
            t8_tma_2d(smem_addr(stg + k2 * kT8TileBytes), &wmap, (c.st * kT8KbPerStage + k2) * kT8Kb, row0, bar, pol);
    };
    grid_dependency_wait();
    grid_launch_dependents();

    // ---- block maxima M[i][kb] = max |x[i][128 kb ..]| (NaN kept), every warp,
    // up to kT8PrepassRound blocks in flight per warp; the first tile's scale
    // row rides in the same round of loads.  The first ring of weight copies
    // is issued only after these loads: issued earlier, it fills the memory
    // queues the activation loads then wait behind.
    float sc_first[kT8MaxKb / 32];
    {
#pragma unroll
        for (int j = 0; j < kT8MaxKb / 32; ++j) {
            const int kb = lane + 32 * j;
            sc_first[j] = kb < nkb ? t8_ld_f32(a.scales + T0 * gcols + kb) : 0.f;
        }
        const int nblk = m * nkb;
        constexpr int nw = kT8Threads / 32;
        int bi = warp / nkb, bkb = warp - (warp / nkb) * nkb;  // (row, K-block) of block `warp`
        for (int b0 = warp; b0 < nblk; b0 += kT8PrepassRound * nw) {
            float4 v[kT8PrepassRound];
            int kbj = bkb, ij = bi;
#pragma unroll
            for (int j = 0; j < kT8PrepassRound; ++j) {
                v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                const int64_t c0 = static_cast<int64_t>(kbj) * kT8Kb + 4 * lane;
                if (ij < m && c0 < a.cols) v[j] = t8_ld_f32x4(a.x + ij * a.cols + c0);
                kbj += nw;
                while (kbj >= nkb) {
                    kbj -= nkb;
                    ++ij;
                }
            }
#pragma unroll
            for (int j = 0; j < kT8PrepassRound; ++j) {
                const uint32_t mx = t8_absmax_bits(v[j]);
                const int blk = b0 + j * nw;
                if (lane == 0 && blk < nblk) sM[blk] = __uint_as_float(mx);  // row-major: blk = i * nkb + kb
            }
            bkb = kbj;
            bi = ij;
        }
        __syncthreads();
    }
    const int64_t pre = n_stages < kT8Stages ? n_stages : kT8Stages;
    Cursor pc;
    if (warp == kT8ProducerWarp && lane == 0)
        for (int64_t e = 0; e < pre; ++e) {
            issue_stage(pc);
            advance(pc);
        }

    // The scale row of tile t, lane l holding kb = l + 32 j.
    auto load_scales = [&](int t, float (&sc)[kT8MaxKb / 32]) {
#pragma unroll
        for (int j = 0; j < kT8MaxKb / 32; ++j) {
            const int kb = lane + 32 * j;
            sc[j] = (t < n_tiles && kb < nkb) ? t8_ld_f32(a.scales + (T0 + t) * gcols + kb) : 0.f;
        }
    };
    // Per activation row and tile, the plane exponent from max_kb |S_kb| M[i][kb],
    // given the tile's scale row (warp-collective; every builder and epilogue
    // warp computes the same bits).
    auto tile_exponents = [&](const float (&sc)[kT8MaxKb / 32], int (&ex)[8]) {
        uint32_t gi[8];  // f32 bits of non-negative values (or NaN): ordered as unsigned
#pragma unroll
        for (int i = 0; i < 8; ++i) gi[i] = 0u;
#pragma unroll
        for (int j = 0; j < kT8MaxKb / 32; ++j) {
            const int kb = lane + 32 * j;
            if (kb < nkb) {
                const float s_abs = fabsf(sc[j]);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i < m) gi[i] = max(gi[i], __float_as_uint(fabsf(s_abs * sM[i * nkb + kb])));
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) ex[i] = t8_plane_exponent(__uint_as_float(__reduce_max_sync(0xFFFFFFFFu, gi[i])));
    };

    float best_v[8];
    uint32_t best_i[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        best_v[i] = -INFINITY;
        best_i[i] = 0;
    }

    if (warp == kT8ProducerWarp) {
        // ---------------- TMA producer
        if (lane == 0) {
            int64_t e = pre;
            for (; e < n_stages; ++e) {
                if (!t8_wait(smem_addr(&stage_free[pc.s]), pc.ph ^ 1u, &s_abort)) break;
                issue_stage(pc);
                advance(pc);
            }
            // Copies of the last ring must have landed before the CTA's shared
            // memory is released (fixed bound, whatever the abort flag says).
            const int64_t first_open = e > kT8Stages ? e - kT8Stages : 0;
            for (int64_t v = first_open; v < e; ++v)
                (void)mbar_wait_bounded(smem_addr(&a_full[v % kT8Stages]),
                                        static_cast<uint32_t>((v / kT8Stages) & 1));
        }
    } else if (warp >= kT8MmaWarp) {
        // ---------------- MMA issuers: warp kT8MmaWarp + k2 issues K-block k2 of
        // every stage into its own accumulator
        const int k2 = warp - kT8MmaWarp;
        if (lane == 0) {
            const uint32_t idesc = t8_idesc(128, N);
            Cursor c;
            for (int64_t e = 0; e < n_stages; ++e) {
                if (!t8_wait(smem_addr(&a_full[c.s]), c.ph, &s_abort)) break;
                if (!t8_wait(smem_addr(&b_full[c.s]), c.ph, &s_abort)) break;
                const int tb = c.t & 1;
                // A tile's accumulators are free once the epilogue drained tile t - 2.
                if (c.st == 0 && c.t >= 2 &&
                    !t8_wait(smem_addr(&d_free[tb]), static_cast<uint32_t>(((c.t >> 1) - 1) & 1), &s_abort))
                    break;
                t8_fence_after();
                if (k2 < stage_kbs(c.st)) {
                    const uint32_t a_base = smem_addr(sA + static_cast<size_t>(c.s) * kT8StageBytes + k2 * kT8TileBytes);
                    const uint32_t b_base =
                        smem_addr(sB + (static_cast<size_t>(c.s) * kT8KbPerStage + k2) * kT8BTileBytes);
                    const uint32_t d = tmem + static_cast<uint32_t>((tb * kT8MmaWarps + k2) * N);
                    const bool first = c.st == 0;  // the tile's first K-block of this warp overwrites D
                    t8_mma(d, t8_desc_sw128(a_base), t8_desc_sw128(b_base), idesc, !first);
                    t8_mma(d, t8_desc_sw128(a_base + 32u), t8_desc_sw128(b_base + 32u), idesc, true);
                    t8_mma(d, t8_desc_sw128(a_base + 64u), t8_desc_sw128(b_base + 64u), idesc, true);
                    t8_mma(d, t8_desc_sw128(a_base + 96u), t8_desc_sw128(b_base + 96u), idesc, true);
                }
                t8_commit(smem_addr(&stage_free[c.s]));  // the stage's A and B slots may be refilled
                if (c.st == nst - 1) t8_commit(smem_addr(&d_full[tb]));
                advance(c);
            }
            // Every MMA issued must complete before the tensor memory is freed.
            t8_commit(smem_addr(&mma_done[k2]));
            (void)mbar_wait_bounded(smem_addr(&mma_done[k2]), 0u);
        }
    } else if (warp >= kT8BWarp0) {
        // ---------------- B builders: warp kT8BWarp0 + 2s + k builds K-block k of
        // the stages in slot s.  Lane l encodes columns 4l .. 4l+3 for every
        // activation row.
        const int bw = warp - kT8BWarp0;
        const int slot = bw / kT8KbPerStage, k2 = bw % kT8KbPerStage;
        uint8_t *bs = sB + (static_cast<size_t>(slot) * kT8KbPerStage + k2) * kT8BTileBytes;
        Cursor c;  // position of this warp's next stage (slot `slot`)
        for (int j = 0; j < slot; ++j) advance(c);
        int ex[8];
        int ex_tile = -1;
        float sc_cur[kT8MaxKb / 32], sc_next[kT8MaxKb / 32];
#pragma unroll
        for (int j = 0; j < kT8MaxKb / 32; ++j) sc_cur[j] = sc_first[j];
        uint32_t pw = 1;  // parity of the stage_free phase that frees the slot
        for (int64_t e = slot; e < n_stages; e += kT8Stages) {
            if (c.t != ex_tile) {
                if (ex_tile >= 0) {
#pragma unroll
                    for (int j = 0; j < kT8MaxKb / 32; ++j) sc_cur[j] = c.t == ex_tile + 1 ? sc_next[j] : 0.f;
                    if (c.t != ex_tile + 1) load_scales(c.t, sc_cur);
                }
                tile_exponents(sc_cur, ex);
                ex_tile = c.t;
                load_scales(c.t + 1, sc_next);  // the next tile's scale row, in flight meanwhile
            }
            const int kb = c.st * kT8KbPerStage + k2;
            const bool live = kb < nkb;
            float4 v[8];
            float sc = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (live) {
                sc = __shfl_sync(0xFFFFFFFFu, sc_cur[0], kb & 31);
#pragma unroll
                for (int j = 1; j < kT8MaxKb / 32; ++j) {
                    const float o = __shfl_sync(0xFFFFFFFFu, sc_cur[j], kb & 31);
                    if ((kb >> 5) == j) sc = o;
                }
                const int64_t c0 = static_cast<int64_t>(kb) * kT8Kb + 4 * lane;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i < m && c0 < a.cols) v[i] = t8_ld_f32x4(a.x + static_cast<int64_t>(i) * a.cols + c0);
            }
            // The MMAs that read this slot's previous stage have completed.
            if (e >= kT8Stages && !t8_warp_wait(smem_addr(&stage_free[slot]), pw, &s_abort, lane)) break;
            if (live) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (i < m) {
                        const bool poison = ex[i] == kT8Poison;
                        float f1, f2;
                        t8_pow2_split(poison ? 0 : ex[i], f1, f2);
                        float t0 = v[i].x * sc * f1 * f2, t1 = v[i].y * sc * f1 * f2;
                        float t2 = v[i].z * sc * f1 * f2, t3 = v[i].w * sc * f1 * f2;
#pragma unroll
                        for (int p = 0; p < kT8Planes; ++p) {
                            const uint32_t lo = t8_to_e4m3x2(t0, t1), hi = t8_to_e4m3x2(t2, t3);
                            const uint32_t word = poison ? 0x7F7F7F7Fu : (lo | (hi << 16));
                            const int n = i * kT8Planes + p;
                            *reinterpret_cast<uint32_t *>(bs + (n >> 3) * 1024 + (n & 7) * 128 +
                                                          ((((lane >> 2) ^ (n & 7)) << 4) | ((lane & 3) << 2))) = word;
                            if (p + 1 < kT8Planes) {
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
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&b_full[slot]));
            if (e >= kT8Stages) pw ^= 1u;
            else pw = 0;
            for (int j = 0; j < kT8Stages; ++j) advance(c);
        }
    } else {
        // ---------------- epilogue: warp w drains TMEM lanes 32w .. 32w+31
        const int tr = warp * 32 + lane;
        float sc_t[kT8MaxKb / 32];
#pragma unroll
        for (int j = 0; j < kT8MaxKb / 32; ++j) sc_t[j] = sc_first[j];
        for (int t = 0; t < n_tiles; ++t) {
            int ex[8];
            if (t > 0) load_scales(t, sc_t);
            tile_exponents(sc_t, ex);
            const int tb = t & 1;
            if (!t8_warp_wait(smem_addr(&d_full[tb]), static_cast<uint32_t>((t >> 1) & 1), &s_abort, lane)) break;
            t8_fence_after();
            // D0 + D1, 16 columns at a time (the odd K-blocks' accumulator holds
            // nothing when a row has a single K-block).
            float d[kT8MaxN];
            const uint32_t taddr =
                tmem + static_cast<uint32_t>(tb * kT8MmaWarps * N) + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll
            for (int c16 = 0; c16 < kT8MaxN; c16 += 16) {
                if (c16 < N) {
                    float d1[16];
                    t8_ld16(taddr + c16, d + c16);
                    t8_ld16(taddr + N + c16, d1);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                    for (int n = 0; n < 16; ++n) d[c16 + n] = nkb > 1 ? d[c16 + n] + d1[n] : d[c16 + n];
                }
            }
            t8_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&d_free[tb]));
            const int64_t row = (T0 + t) * 128 + tr;
            if (row < a.rows) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (i < m) {
                        // 2^-ex (D[0] + 2^-4 (D[1] + ...)); a factor 2^-ex below the
                        // normal range is flushed (the tile's |x S| is below 2^-118).
                        float u = d[i * kT8Planes + kT8Planes - 1];
#pragma unroll
                        for (int p = kT8Planes - 2; p >= 0; --p) u = fmaf(u, 0.0625f, d[i * kT8Planes + p]);
                        const int eb = 127 - ex[i];
                        const float f = ex[i] == kT8Poison ? __int_as_float(0x7FC00000)
                                                           : (eb > 0 ? __int_as_float(eb << 23) : 0.f);
                        const float val = u * f;
                        if (a.y) a.y[static_cast<int64_t>(i) * a.rows + row] = val;
                        if (ARGMAX && argmax_better(val, static_cast<uint32_t>(row), best_v[i], best_i[i])) {
                            best_v[i] = val;
                            best_i[i] = static_cast<uint32_t>(row);
                        }
                    }
                }
            }
        }
    }

    if (tid == 0 && *reinterpret_cast<volatile int *>(&s_abort)) atomicOr(a.status, 1u);
    t8_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(t8_tmem_cols(N)) : "memory");

    if constexpr (ARGMAX) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < m) {
                float bv = best_v[i];
                uint32_t bi = best_i[i];
                warp_argmax_all(bv, bi);
                if (lane == 0) {
                    am_val[warp][i] = bv;
                    am_idx[warp][i] = bi;
                }
            }
        }
        __syncthreads();
        if (tid < m) {
            float bv = -INFINITY;
            uint32_t bi = 0;
            for (int w2 = 0; w2 < kT8EpiWarps; ++w2)
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
            case 1: argmax_cross_cta<1, kT8Threads, kT8Threads / 32>(ga, am_val, am_idx, &s_is_last); break;
            case 2: argmax_cross_cta<2, kT8Threads, kT8Threads / 32>(ga, am_val, am_idx, &s_is_last); break;
            case 3: argmax_cross_cta<3, kT8Threads, kT8Threads / 32>(ga, am_val, am_idx, &s_is_last); break;
            case 4: argmax_cross_cta<4, kT8Threads, kT8Threads / 32>(ga, am_val, am_idx, &s_is_last); break;
            case 5: argmax_cross_cta<5, kT8Threads, kT8Threads / 32>(ga, am_val, am_idx, &s_is_last); break;
            case 6: argmax_cross_cta<6, kT8Threads, kT8Threads / 32>(ga, am_val, am_idx, &s_is_last); break;
            case 7: argmax_cross_cta<7, kT8Threads, kT8Threads / 32>(ga, am_val, am_idx, &s_is_last); break;
            default: argmax_cross_cta<8, kT8Threads, kT8Threads / 32>(ga, am_val, am_idx, &s_is_last); break;
        }
    }
}

}  // namespace fp8blk
