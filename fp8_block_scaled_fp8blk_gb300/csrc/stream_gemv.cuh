// stream_gemv.cuh -- the weight-streaming decode GEMV for sm_103a.
//
// y[i][r] = sum_c w(r, c) * x[i][c]   for m = M activation rows (1..8), where
// w is either an e4m3 code times a 128x128 block scale ("Module dsv4_gpu"
// page, struct Fp8Dense) or a bf16 value (the NVFP4 experts' dequantised
// scratch, same page, enum ExpertArm), optionally fused with a greedy argmax
// per activation row ("Struct Dsv4Gpu" page, decode_step_greedy and
// verify_batch_dev; lowest index wins ties, "dflash.rs source" page,
// dflash2_walk_greedy).
//
// The path is HBM-bound (m <= 8 reads each weight byte once and does at most
// 8 FMAs on it), so the kernel is organised around moving bytes:
//   * a persistent grid, one or two CTAs per SM, each owning a contiguous
//     range of row groups;
//   * a ring of shared-memory stages filled by 1-D bulk copies (TMA,
//     cp.async.bulk) that complete on mbarriers, with L2 evict-first hints;
//     a stage holds R whole rows of one column panel (<= 4096 columns), and
//     the last warp to finish reading a stage refills it at once;
//   * each thread owns 16 columns of the panel, keeps x[0..M)[those columns]
//     in registers pre-multiplied by the block scale, decodes its weights in
//     registers (hardware e4m3->f16 conversion, exact) and accumulates with
//     scalar FMAs (measured faster than packed f32x2 FMAs here);
//   * the 8 per-lane partials (RT rows x MP activation rows) are reduced
//     across the warp by a 3-level reduce-scatter whose lane-dependent slot
//     permutation is folded into the smem row address and the x register
//     layout (no selects), then summed across warps in a fixed order.
// Every output is therefore reduced in one fixed order: results are
// deterministic and identical rows give bit-identical outputs.  m = 1 uses the
// row-per-warp variant in rowwarp_gemv.cuh instead.
#pragma once

#include "device_common.cuh"

namespace fp8blk {

constexpr int kThreads = 256;   // 8 warps per CTA, all of them consumers
constexpr int kWarps = kThreads / 32;
constexpr int kMaxStages = 8;
constexpr int kMaxPanelCols = kThreads * 16;  // 4096 columns per panel
constexpr int kMaxRowBatches = 8;

enum WeightFormat : int { kE4M3 = 0, kBF16 = 1 };

struct GemvArgs {
    const uint8_t *w;       // weight bytes [rows, cols * bpw]
    const float *scales;    // e4m3: f32 grid [ceil(rows/128), ceil(cols/128)]; bf16: unused
    const float *x;         // [m, cols]
    float *y;               // [m, rows] outputs / panel accumulator; may be null (argmax only,
                            // single panel)
    uint32_t *tokens;       // [m] argmax tokens (ARGMAX only)
    float *part_val;        // [grid, m] per-CTA argmax partials (ARGMAX only)
    uint32_t *part_idx;     // [grid, m]
    uint32_t *counter;      // CTA-arrival counter, wraps to 0 at the end of every call
    unsigned int *status;   // device status word
    int64_t rows, cols;
    int64_t n_groups;       // ceil(rows / stage_rows)
    int panels;             // column panels
    int panel_cols;         // columns of every panel but the last (multiple of 16)
    int team_warps_log2;    // warps per team (1, 2, 4, 8) as log2
    int rb;                 // row batches per team per stage
    int stages;             // ring depth
    int stage_bytes;        // bytes per stage
    int stage_rows;         // R = teams * rb * RT
    int l2_prefetch;        // issue L2 prefetches before the grid-dependency wait
    uint64_t wait_limit_ns; // consumer-side weight-tile wait limit (drains keep kWaitLimitNs)
};

__host__ __device__ constexpr int pow2_ceil(int v) {
    return v <= 1 ? 1 : 2 * pow2_ceil((v + 1) / 2);
}
__host__ __device__ constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

// Greedy order: higher value first, then lower index.  NaN is never better.
__device__ __forceinline__ bool argmax_better(float v, uint32_t i, float bv, uint32_t bi) {
    return v > bv || (v == bv && i < bi);
}

// Warp reduce-scatter of 8 per-lane values.  Lane L holds in slot j the value
// for output j ^ perm(L), perm(L) = (L4 L3 L2) as a 3-bit number.  Returns,
// at every lane L, the 32-lane sum for output perm(L).  The combination tree
// is the same for every output (pairs differ in lane bit 4, then 3, 2, 1, 0).
__device__ __forceinline__ float warp_reduce_scatter8(const float p[8]) {
    const unsigned full = 0xFFFFFFFFu;
    float q0 = p[0] + __shfl_xor_sync(full, p[4], 16);
    float q1 = p[1] + __shfl_xor_sync(full, p[5], 16);
    float q2 = p[2] + __shfl_xor_sync(full, p[6], 16);
    float q3 = p[3] + __shfl_xor_sync(full, p[7], 16);
    float r0 = q0 + __shfl_xor_sync(full, q2, 8);
    float r1 = q1 + __shfl_xor_sync(full, q3, 8);
    float t = r0 + __shfl_xor_sync(full, r1, 4);
    t += __shfl_xor_sync(full, t, 2);
    t += __shfl_xor_sync(full, t, 1);
    return t;
}

template <int FMT>
struct Fmt {
    static constexpr int kBytesPerWeight = FMT == kE4M3 ? 1 : 2;
    static constexpr int kChunksPerThread = kBytesPerWeight;  // 16-byte chunks -> 16 columns
    static constexpr int kColsPerChunk = 16 / kBytesPerWeight;
};

// Issue the bulk copies of unit u into a stage.  Unit u = (panel u / n_my,
// row group g0 + u % n_my).  Rows of a group are contiguous in memory, so a
// single-panel unit is one copy; a multi-panel unit is one copy per row.
template <int FMT>
__device__ __forceinline__ void issue_unit(const GemvArgs &a, int64_t u, int64_t n_my, int64_t g0,
                                           uint32_t stage, uint32_t bar, uint64_t policy,
                                           bool prefetch_only) {
    constexpr int BPW = Fmt<FMT>::kBytesPerWeight;
    const int panel = static_cast<int>(u / n_my);
    const int64_t grp = g0 + u % n_my;
    const int64_t row0 = grp * a.stage_rows;
    const int64_t nr64 = a.rows - row0 < a.stage_rows ? a.rows - row0 : a.stage_rows;
    const int nr = static_cast<int>(nr64);
    const int64_t pc64 = a.cols - static_cast<int64_t>(panel) * a.panel_cols;
    const int pc = pc64 < a.panel_cols ? static_cast<int>(pc64) : a.panel_cols;
    const uint32_t pwb = static_cast<uint32_t>(pc * BPW);
    const int64_t row_bytes = a.cols * BPW;
    const uint8_t *src0 = a.w + row0 * row_bytes + static_cast<int64_t>(panel) * a.panel_cols * BPW;
    if (prefetch_only) {
        if (a.panels == 1) {
            bulk_prefetch_l2(src0, pwb * nr);
        } else {
            for (int r = 0; r < nr; ++r) bulk_prefetch_l2(src0 + r * row_bytes, pwb);
        }
        return;
    }
    mbar_arrive_expect_tx(bar, pwb * nr);
    if (a.panels == 1) {
        bulk_g2s(stage, src0, pwb * nr, bar, policy);
    } else {
        for (int r = 0; r < nr; ++r) bulk_g2s(stage + r * pwb, src0 + r * row_bytes, pwb, bar, policy);
    }
}

// Decode this thread's 16 columns of one staged row into 8 f32 pairs.
// Chunks past the panel edge read nothing and decode to zero; FULL: the panel
// is a whole kMaxPanelCols wide, so no chunk is past the edge.
template <int FMT, bool FULL>
__device__ __forceinline__ void load_row_weights(const uint8_t *row, int tt, int team_threads,
                                                 int pwb, float2 wv[8]) {
    if constexpr (FMT == kE4M3) {
        if (FULL || tt * 16 < pwb) {
            const uint4 q = *reinterpret_cast<const uint4 *>(row + tt * 16);
            e4m3x4_to_f32(q.x, wv[0], wv[1]);
            e4m3x4_to_f32(q.y, wv[2], wv[3]);
            e4m3x4_to_f32(q.z, wv[4], wv[5]);
            e4m3x4_to_f32(q.w, wv[6], wv[7]);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) wv[k] = make_float2(0.f, 0.f);
        }
    } else {
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const int chunk = s * team_threads + tt;
            if (FULL || chunk * 16 < pwb) {
                const uint4 q = *reinterpret_cast<const uint4 *>(row + chunk * 16);
                wv[4 * s + 0] = bf16x2_to_f32(q.x);
                wv[4 * s + 1] = bf16x2_to_f32(q.y);
                wv[4 * s + 2] = bf16x2_to_f32(q.z);
                wv[4 * s + 3] = bf16x2_to_f32(q.w);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) wv[4 * s + k] = make_float2(0.f, 0.f);
            }
        }
    }
}

// All row batches of one staged unit: per lane, per batch, 8 partial sums
// (RT rows x MP activation rows), reduced across the warp into red_w[b][*].
// Scalar FMAs, two independent chains per (row, activation row).
template <int M, int FMT, bool FULL>
__device__ __forceinline__ void team_stage_compute(const uint8_t *st, int pwb, int rb, int team,
                                                   int team_rows, int tt, int team_threads, int prt,
                                                   int lane, const float2 (&xr)[pow2_ceil(M)][8],
                                                   float (*red_w)[8]) {
    constexpr int MP = pow2_ceil(M);
    constexpr int RT = 8 / MP;
    // Partial sums of one row batch: 8 slots (RT rows x MP activation rows).
    auto batch_partials = [&](int b, float (&p)[8]) {
#pragma unroll
        for (int rt = 0; rt < RT; ++rt) {
            const int lrow = team * team_rows + b * RT + (rt ^ prt);
            float2 wv[8];
            load_row_weights<FMT, FULL>(st + lrow * pwb, tt, team_threads, pwb, wv);
#pragma unroll
            for (int i = 0; i < MP; ++i) {
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    a0 = fmaf(wv[k].x, xr[i][k].x, a0);
                    a1 = fmaf(wv[k].y, xr[i][k].y, a1);
                }
                p[rt * MP + i] = a0 + a1;
            }
        }
    };
    // Two batches per step, so that one batch's shuffle chain can overlap the
    // other's arithmetic.
    int b = 0;
    for (; b + 1 < rb; b += 2) {
        float p0[8], p1[8];
        batch_partials(b, p0);
        batch_partials(b + 1, p1);
        const float v0 = warp_reduce_scatter8(p0);
        const float v1 = warp_reduce_scatter8(p1);
        if ((lane & 3) == 0) {
            red_w[b][lane >> 2] = v0;
            red_w[b + 1][lane >> 2] = v1;
        }
    }
    if (b < rb) {
        float p0[8];
        batch_partials(b, p0);
        const float v0 = warp_reduce_scatter8(p0);
        if ((lane & 3) == 0) red_w[b][lane >> 2] = v0;
    }
}

// x[i ^ pi][this thread's 16 columns of the panel] * block scale, as pairs.
template <int M, int FMT>
__device__ __forceinline__ void load_x_regs(const GemvArgs &a, int panel, int pwb, int64_t rblk,
                                            int tt, int team_threads, int pi,
                                            float2 (&xr)[pow2_ceil(M)][8]) {
    constexpr int MP = pow2_ceil(M);
    constexpr int CPC = Fmt<FMT>::kColsPerChunk;
    const int64_t gcols = (a.cols + 127) / 128;
#pragma unroll
    for (int s = 0; s < Fmt<FMT>::kChunksPerThread; ++s) {
        const int chunk = s * team_threads + tt;
        const bool col_ok = chunk * 16 < pwb;
        const int64_t c0 = static_cast<int64_t>(panel) * a.panel_cols + static_cast<int64_t>(chunk) * CPC;
        float sc = 1.f;
        if constexpr (FMT == kE4M3) {
            if (col_ok) sc = __ldg(a.scales + rblk * gcols + c0 / 128);
        }
#pragma unroll
        for (int i = 0; i < MP; ++i) {
            const int mi = i ^ pi;
            const bool ok = col_ok && mi < M;
#pragma unroll
            for (int q = 0; q < CPC / 4; ++q) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (ok) v = __ldg(reinterpret_cast<const float4 *>(a.x + mi * a.cols + c0) + q);
                if constexpr (FMT == kE4M3) {
                    v.x *= sc;
                    v.y *= sc;
                    v.z *= sc;
                    v.w *= sc;
                }
                xr[i][s * (CPC / 2) + 2 * q] = make_float2(v.x, v.y);
                xr[i][s * (CPC / 2) + 2 * q + 1] = make_float2(v.z, v.w);
            }
        }
    }
}

// Warp-level greedy merge over lanes that differ in bits >= log2(MP): after
// it, lane l < MP holds the warp's best for activation row l.
template <int MP>
__device__ __forceinline__ void warp_argmax_merge(float &v, uint32_t &i) {
#pragma unroll
    for (int off = 16; off >= MP; off >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, v, off);
        const uint32_t oi = __shfl_xor_sync(0xFFFFFFFFu, i, off);
        if (argmax_better(ov, oi, v, i)) {
            v = ov;
            i = oi;
        }
    }
}

// Warp-wide greedy argmax, every lane ending with the warp's best: one
// redux.sync takes the largest order key, a second the lowest index among the
// lanes holding it.  The key orders floats as argmax_better compares them
// (-0 as +0); NaN, which argmax_better never prefers, is never a lane's best
// (each starts from -inf), so it needs no key.  Same result as the shuffle
// tree of warp_argmax_merge<1>, in two instructions instead of ten.
__device__ __forceinline__ void warp_argmax_all(float &v, uint32_t &i) {
    const uint32_t b = __float_as_uint(v + 0.0f);  // -0 -> +0
    const uint32_t key = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    const uint32_t kmax = __reduce_max_sync(0xFFFFFFFFu, key);
    i = __reduce_min_sync(0xFFFFFFFFu, key == kmax ? i : 0xFFFFFFFFu);
    v = __uint_as_float((kmax & 0x80000000u) ? (kmax & 0x7FFFFFFFu) : ~kmax);
}

constexpr int kAmWarps = 16;  // rows of the argmax merge scratch (one per warp)

// Called by every thread of the CTA after its per-activation-row partials
// (part_val/part_idx[blockIdx.x * M + i]) are stored.  Publishes them; the last
// CTA to arrive merges all CTAs' partials in CTA order and writes the tokens.
// The arrival counter wraps back to 0, ready for the next call.
template <int M, int NT, int AW>
__device__ __forceinline__ void argmax_cross_cta(const GemvArgs &a, float (&am_val)[AW][8], uint32_t (&am_idx)[AW][8],
                                                 int *s_is_last) {
    constexpr int NW = NT / 32;
    static_assert(NW <= AW, "argmax scratch too small");
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *s_is_last = (atomicInc(a.counter, gridDim.x - 1) == gridDim.x - 1);
    __syncthreads();
    if (!*s_is_last) return;
    __threadfence();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    for (int i = 0; i < M; ++i) {
        float v = -INFINITY;
        uint32_t ix = 0;
        for (int c = threadIdx.x; c < static_cast<int>(gridDim.x); c += NT) {
            const float cv = __ldcg(a.part_val + static_cast<int64_t>(c) * M + i);
            const uint32_t ci = __ldcg(a.part_idx + static_cast<int64_t>(c) * M + i);
            if (argmax_better(cv, ci, v, ix)) {
                v = cv;
                ix = ci;
            }
        }
        warp_argmax_all(v, ix);
        __syncthreads();
        if (lane == 0) {
            am_val[warp][0] = v;
            am_idx[warp][0] = ix;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            float bv = -INFINITY;
            uint32_t bi = 0;
            for (int w2 = 0; w2 < NW; ++w2)
                if (argmax_better(am_val[w2][0], am_idx[w2][0], bv, bi)) {
                    bv = am_val[w2][0];
                    bi = am_idx[w2][0];
                }
            a.tokens[i] = bi;
        }
    }
}

template <int M, int FMT, bool ARGMAX>
__global__ void __launch_bounds__(kThreads, (M <= 4 ? 2 : 1)) stream_gemv_kernel(const GemvArgs a) {
    constexpr int MP = pow2_ceil(M);
    constexpr int LOG_MP = ilog2(MP);
    constexpr int RT = 8 / MP;  // rows per lane batch; RT * MP == 8 slots
    constexpr int BPW = Fmt<FMT>::kBytesPerWeight;

    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full[kMaxStages];
    __shared__ unsigned int consumed[kMaxStages];
    __shared__ float red[2][kWarps][kMaxRowBatches][8];
    __shared__ float am_val[kAmWarps][8];
    __shared__ uint32_t am_idx[kAmWarps][8];
    __shared__ int s_is_last;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int wt_log2 = a.team_warps_log2;
    const int team_warps = 1 << wt_log2;
    const int team = warp >> wt_log2;
    const int wit = warp & (team_warps - 1);
    const int team_threads = team_warps * 32;
    const int tt = wit * 32 + lane;
    const int perm = (((lane >> 4) & 1) << 2) | (((lane >> 3) & 1) << 1) | ((lane >> 2) & 1);
    const int prt = perm >> LOG_MP;
    const int pi = perm & (MP - 1);
    const int rb = a.rb;
    const int team_rows = rb * RT;

    const int64_t g0 = static_cast<int64_t>(blockIdx.x) * a.n_groups / gridDim.x;
    const int64_t g1 = static_cast<int64_t>(blockIdx.x + 1) * a.n_groups / gridDim.x;
    const int64_t n_my = g1 - g0;
    const int64_t units = n_my * a.panels;
    const int stages = a.stages;
    uint8_t *stage_base = smem;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            consumed[s] = 0;
        }
        mbar_init_fence();
    }
    __syncthreads();

    const uint64_t policy = l2_policy_evict_first();
    const int64_t first = units < stages ? units : stages;
    // e4m3 weights are never outputs of the preceding kernel on the stream (a
    // documented contract of the e4m3 entry points), so the first stages'
    // weight copies start before the grid dependency wait: with programmatic
    // dependent launch they overlap the tail of the previous call.  bf16
    // weights can be the preceding dequant kernel's output (the NVFP4 expert
    // scratch), so they are only prefetched into L2 (coherent) before it.
    constexpr bool kEarlyWeights = FMT == kE4M3;
    if (tid == 0) {
        const int64_t pf0 = kEarlyWeights ? first : 0;
        const int64_t pf_end = kEarlyWeights ? (units < 2 * first ? units : 2 * first) : first;
        if (kEarlyWeights)
            for (int64_t u = 0; u < first; ++u)
                issue_unit<FMT>(a, u, n_my, g0, smem_addr(stage_base + u * a.stage_bytes),
                                smem_addr(&full[u]), policy, false);
        if (a.l2_prefetch)
            for (int64_t u = pf0; u < pf_end; ++u) issue_unit<FMT>(a, u, n_my, g0, 0, 0, policy, true);
    }
    // Everything below may read what the previous grid wrote (x, scales, bf16
    // weights), or overwrite what it reads (y).
    grid_dependency_wait();
    grid_launch_dependents();
    if (!kEarlyWeights && tid == 0) {
        for (int64_t u = 0; u < first; ++u)
            issue_unit<FMT>(a, u, n_my, g0, smem_addr(stage_base + u * a.stage_bytes),
                            smem_addr(&full[u]), policy, false);
    }

    float best_v = -INFINITY;
    uint32_t best_i = 0;
    float2 xr[MP][8];
    int cur_panel = -1;
    int64_t cur_rblk = -1;
    bool aborted = false;
    int64_t failed_unit = 0;
    int buf = 0;

    for (int64_t u = 0; u < units; ++u) {
        const int s = static_cast<int>(u % stages);
        const int panel = static_cast<int>(u / n_my);
        const int64_t row0 = (g0 + u % n_my) * a.stage_rows;
        const int64_t pc64 = a.cols - static_cast<int64_t>(panel) * a.panel_cols;
        const int pc = pc64 < a.panel_cols ? static_cast<int>(pc64) : a.panel_cols;
        const int pwb = pc * BPW;
        const int64_t rblk = row0 >> 7;
        if (panel != cur_panel || rblk != cur_rblk) {
            load_x_regs<M, FMT>(a, panel, pwb, rblk, tt, team_threads, pi, xr);
            cur_panel = panel;
            cur_rblk = rblk;
        }
        // Warp-uniform: the compute below holds warp-wide shuffles.
        const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait_limit(smem_addr(&full[s]), static_cast<uint32_t>((u / stages) & 1),
                                                                a.wait_limit_ns));
        if (ok) {
            const uint8_t *st = stage_base + static_cast<size_t>(s) * a.stage_bytes;
            if (pwb == kMaxPanelCols * BPW)
                team_stage_compute<M, FMT, true>(st, pwb, rb, team, team_rows, tt, team_threads, prt, lane,
                                                 xr, red[buf][warp]);
            else
                team_stage_compute<M, FMT, false>(st, pwb, rb, team, team_rows, tt, team_threads, prt, lane,
                                                  xr, red[buf][warp]);
        }
        // The last warp to finish reading stage s refills it, unless some
        // warp's wait timed out (its copy may still be landing in stage s):
        // a failed warp adds 1 to the high half of the arrival word.
        if (lane == 0) {
            const unsigned int inc = ok ? 1u : 0x10001u;
            const unsigned int total = atomicAdd(&consumed[s], inc) + inc;
            if ((total & 0xFFFFu) == kWarps) {
                consumed[s] = 0;
                if ((total >> 16) == 0 && u + stages < units)
                    issue_unit<FMT>(a, u + stages, n_my, g0,
                                    smem_addr(stage_base + static_cast<size_t>(s) * a.stage_bytes),
                                    smem_addr(&full[s]), policy, false);
            }
        }
        // Publishes red[buf]; agrees on an abort if any thread timed out.
        if (__syncthreads_or(!ok)) {
            aborted = true;
            failed_unit = u;
            break;
        }

        // Cross-warp sum, output write and argmax tracking.  Output slot o =
        // (b, v) goes to team thread o mod team_threads; team_threads is a
        // multiple of 8, so a thread's activation row (v & (MP-1)) is fixed.
        for (int o = tt; o < rb * 8; o += team_threads) {
            const int b = o >> 3;
            const int v = o & 7;
            const int rt = v >> LOG_MP;
            const int i = v & (MP - 1);
            const int64_t row = row0 + team * team_rows + b * RT + rt;
            if (i < M && row < a.rows) {
                float val = 0.f;
                for (int w2 = 0; w2 < team_warps; ++w2) val += red[buf][team * team_warps + w2][b][v];
                float *yp = a.y ? a.y + static_cast<int64_t>(i) * a.rows + row : nullptr;
                if (a.panels > 1) {
                    if (panel > 0) val += *yp;
                    *yp = val;
                } else if (yp) {
                    *yp = val;
                }
                if (ARGMAX && panel == a.panels - 1) {
                    if (argmax_better(val, static_cast<uint32_t>(row), best_v, best_i)) {
                        best_v = val;
                        best_i = static_cast<uint32_t>(row);
                    }
                }
            }
        }
        buf ^= 1;
    }

    if (aborted) {
        // Units up to failed_unit + stages - 1 have been issued (a failed warp
        // stops the refill of failed_unit + stages); let those copies land
        // before the shared memory is released (each wait bounded by the fixed
        // limit), then report.
        const int64_t issued_end = failed_unit + stages < units ? failed_unit + stages : units;
        for (int64_t u = failed_unit; u < issued_end; ++u)
            (void)mbar_wait_bounded(smem_addr(&full[u % stages]), static_cast<uint32_t>((u / stages) & 1));
        if (tid == 0) atomicOr(a.status, 1u);
    }

    if constexpr (ARGMAX) {
        // CTA merge: finalize thread tt handles activation row (tt & 7) & (MP-1).
        warp_argmax_merge<MP>(best_v, best_i);
        if (lane < MP) {
            am_val[warp][lane] = best_v;
            am_idx[warp][lane] = best_i;
        }
        __syncthreads();
        if (tid < M) {
            float bv = -INFINITY;
            uint32_t bi = 0;
            for (int w2 = 0; w2 < kWarps; ++w2)
                if (argmax_better(am_val[w2][tid], am_idx[w2][tid], bv, bi)) {
                    bv = am_val[w2][tid];
                    bi = am_idx[w2][tid];
                }
            __stcg(a.part_val + static_cast<int64_t>(blockIdx.x) * M + tid, bv);
            __stcg(a.part_idx + static_cast<int64_t>(blockIdx.x) * M + tid, bi);
        }
        argmax_cross_cta<M, kThreads>(a, am_val, am_idx, &s_is_last);
    }
}

}  // namespace fp8blk
