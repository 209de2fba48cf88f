// rowwarp_gemv.cuh -- the single-activation-row (m = 1) decode GEMV: the
// greedy decode step's dense linears and vocab head ("Struct Dsv4Gpu" page,
// decode_step_greedy; "Module dsv4_gpu" page, struct Fp8Dense).
//
// With one activation row, x for 128 columns fits in a lane's registers, so a
// warp can own whole rows of a <= 4096-column panel: lane l holds the 16-byte
// chunks l, l + 32, ... of every row.  Each warp streams its own contiguous
// run of rows through a private ring of shared-memory stages filled by 1-D
// bulk copies (issued by its lane 0) on per-stage mbarriers, decodes in
// registers, accumulates with scalar FMAs and reduces rows two at a time with
// a fixed 5-level xor butterfly.  Warps never wait for one another inside the
// main loop: no cross-warp reduction, no CTA barrier, nothing but the warp's
// own weight stream.  Results are deterministic; identical rows give
// bit-identical outputs.
#pragma once

#include "stream_gemv.cuh"

namespace fp8blk {

constexpr int kRowWarps = 4;  // independent row streams per CTA
constexpr int kRowThreads = kRowWarps * 32;

// x for this lane's chunks of the panel, times each chunk's block scale.
template <int FMT>
__device__ __forceinline__ void rowwarp_load_x(const GemvArgs &a, int panel, int pwb, int64_t rblk,
                                               int lane, float2 (&xr)[64]) {
    constexpr int BPW = Fmt<FMT>::kBytesPerWeight;
    constexpr int CPL = 8 * BPW;        // chunks per lane in a full panel
    constexpr int CPC = 16 / BPW;       // columns per chunk
    constexpr int PPC = CPC / 2;        // f32 pairs per chunk
    const int64_t gcols = (a.cols + 127) / 128;
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const int chunk = k * 32 + lane;
        const bool ok = chunk * 16 < pwb;
        const int64_t c0 = static_cast<int64_t>(panel) * a.panel_cols + static_cast<int64_t>(chunk) * CPC;
        float sc = 1.f;
        if constexpr (FMT == kE4M3) {
            if (ok) sc = __ldg(a.scales + rblk * gcols + c0 / 128);
        }
#pragma unroll
        for (int q = 0; q < CPC / 4; ++q) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (ok) v = __ldg(reinterpret_cast<const float4 *>(a.x + c0) + q);
            if constexpr (FMT == kE4M3) {
                v.x *= sc;
                v.y *= sc;
                v.z *= sc;
                v.w *= sc;
            }
            xr[k * PPC + 2 * q] = make_float2(v.x, v.y);
            xr[k * PPC + 2 * q + 1] = make_float2(v.z, v.w);
        }
    }
}

// Decodes one 16-byte chunk into PPC f32 pairs.
template <int FMT>
__device__ __forceinline__ void rowwarp_decode(const uint4 &q, float2 (&w)[8 / Fmt<FMT>::kBytesPerWeight]) {
    if constexpr (FMT == kE4M3) {
        e4m3x4_to_f32(q.x, w[0], w[1]);
        e4m3x4_to_f32(q.y, w[2], w[3]);
        e4m3x4_to_f32(q.z, w[4], w[5]);
        e4m3x4_to_f32(q.w, w[6], w[7]);
    } else {
        w[0] = bf16x2_to_f32(q.x);
        w[1] = bf16x2_to_f32(q.y);
        w[2] = bf16x2_to_f32(q.z);
        w[3] = bf16x2_to_f32(q.w);
    }
}

// This lane's shares of two staged rows A and B: sums over its chunks of w * x.
// Scalar FMAs into four independent accumulators per row (measured faster
// than packed f32x2 FMAs for this decode-bound loop).  FULL: every chunk of
// the panel row is present, so no per-chunk edge test is needed.
template <int FMT, bool FULL>
__device__ __forceinline__ void rowwarp_two_rows(const uint8_t *row_a, const uint8_t *row_b, int lane,
                                                 int pwb, const float2 (&xr)[64], float &pa, float &pb) {
    constexpr int BPW = Fmt<FMT>::kBytesPerWeight;
    constexpr int CPL = 8 * BPW;
    constexpr int PPC = 8 / BPW;
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    float b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const int off = (k * 32 + lane) * 16;
        if (FULL || off < pwb) {
            const uint4 qa = *reinterpret_cast<const uint4 *>(row_a + off);
            const uint4 qb = *reinterpret_cast<const uint4 *>(row_b + off);
            float2 wa[PPC], wb[PPC];
            rowwarp_decode<FMT>(qa, wa);
            rowwarp_decode<FMT>(qb, wb);
#pragma unroll
            for (int j = 0; j < PPC; ++j) {
                const float2 xv = xr[k * PPC + j];
                a[(2 * j) & 3] = fmaf(wa[j].x, xv.x, a[(2 * j) & 3]);
                a[(2 * j + 1) & 3] = fmaf(wa[j].y, xv.y, a[(2 * j + 1) & 3]);
                b[(2 * j) & 3] = fmaf(wb[j].x, xv.x, b[(2 * j) & 3]);
                b[(2 * j + 1) & 3] = fmaf(wb[j].y, xv.y, b[(2 * j + 1) & 3]);
            }
        }
    }
    pa = (a[0] + a[1]) + (a[2] + a[3]);
    pb = (b[0] + b[1]) + (b[2] + b[3]);
}

// Warp sum of two rows at once.  Lanes with bit 4 set hold row B in slot A
// (their row addresses are swapped), so one exchange at distance 16 splits
// the rows without selects; four more levels finish.  Lanes 0-15 return row
// A's total, lanes 16-31 row B's.  Same combination tree for every row.
__device__ __forceinline__ float warp_sum_two_rows(float slot_a, float slot_b) {
    float t = slot_a + __shfl_xor_sync(0xFFFFFFFFu, slot_b, 16);
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, off);
    return t;
}

template <int FMT, bool ARGMAX>
__global__ void __launch_bounds__(kRowThreads, 2) rowwarp_gemv_kernel(const GemvArgs a) {
    constexpr int BPW = Fmt<FMT>::kBytesPerWeight;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kRowWarps][kMaxStages];
    __shared__ float am_val[kAmWarps][8];
    __shared__ uint32_t am_idx[kAmWarps][8];
    __shared__ int s_is_last;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int stages = a.stages;
    uint8_t *ring = smem + static_cast<size_t>(warp) * stages * a.stage_bytes;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kRowWarps;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * kRowWarps + warp;
    const int64_t g0 = gw * a.n_groups / nwarps;
    const int64_t g1 = (gw + 1) * a.n_groups / nwarps;
    const int64_t n_my = g1 - g0;
    const int64_t units = n_my * a.panels;
    const uint32_t bar0 = smem_addr(&bars[warp][0]);

    if (lane == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(bar0 + 8 * s, 1);
        mbar_init_fence();
    }
    __syncwarp();

    const uint64_t policy = l2_policy_evict_first();
    const int64_t first = units < stages ? units : stages;
    // e4m3 weight copies of the first stages start before the grid dependency
    // wait (e4m3 weights are never outputs of the preceding kernel); bf16
    // weights may be (the NVFP4 expert scratch), so those wait, with only a
    // coherent L2 prefetch before.  x, the scales and y are only touched after.
    constexpr bool kEarlyWeights = FMT == kE4M3;
    if (lane == 0) {
        const int64_t pf0 = kEarlyWeights ? first : 0;
        const int64_t pf_end = kEarlyWeights ? (units < 2 * first ? units : 2 * first) : first;
        if (kEarlyWeights)
            for (int64_t u = 0; u < first; ++u)
                issue_unit<FMT>(a, u, n_my, g0, smem_addr(ring + u * a.stage_bytes),
                                bar0 + 8 * static_cast<uint32_t>(u), policy, false);
        if (a.l2_prefetch)
            for (int64_t u = pf0; u < pf_end; ++u) issue_unit<FMT>(a, u, n_my, g0, 0, 0, policy, true);
    }
    grid_dependency_wait();
    grid_launch_dependents();
    if (!kEarlyWeights && lane == 0) {
        for (int64_t u = 0; u < first; ++u)
            issue_unit<FMT>(a, u, n_my, g0, smem_addr(ring + u * a.stage_bytes), bar0 + 8 * static_cast<uint32_t>(u),
                            policy, false);
    }
    int64_t issued_end = first;

    float2 xr[64];
    int cur_panel = -1;
    int64_t cur_rblk = -1;
    float best_v = -INFINITY;
    uint32_t best_i = 0;
    bool aborted = false;
    int64_t failed_unit = 0;

    for (int64_t u = 0; u < units; ++u) {
        const int s = static_cast<int>(u % stages);
        const int panel = static_cast<int>(u / n_my);
        const int64_t row0 = (g0 + u % n_my) * a.stage_rows;
        const int64_t nr64 = a.rows - row0 < a.stage_rows ? a.rows - row0 : a.stage_rows;
        const int nr = static_cast<int>(nr64);
        const int64_t pc64 = a.cols - static_cast<int64_t>(panel) * a.panel_cols;
        const int pc = pc64 < a.panel_cols ? static_cast<int>(pc64) : a.panel_cols;
        const int pwb = pc * BPW;
        const int64_t rblk = row0 >> 7;
        if (panel != cur_panel || rblk != cur_rblk) {
            rowwarp_load_x<FMT>(a, panel, pwb, rblk, lane, xr);
            cur_panel = panel;
            cur_rblk = rblk;
        }
        const bool ok = mbar_wait_limit(bar0 + 8 * s, static_cast<uint32_t>((u / stages) & 1), a.wait_limit_ns);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
            aborted = true;
            failed_unit = u;
            break;
        }
        const uint8_t *st = ring + static_cast<size_t>(s) * a.stage_bytes;
        const bool full_panel = pwb == kMaxPanelCols * BPW;
        const int hi = lane >> 4;  // 1: this lane handles the pair's rows swapped
        for (int r = 0; r < nr; r += 2) {
            // Rows r and r+1 (a lone last row pairs with itself; its copy is dropped).
            const int rb2 = r + 1 < nr ? r + 1 : r;
            const uint8_t *ra = st + (hi ? rb2 : r) * pwb;
            const uint8_t *rbp = st + (hi ? r : rb2) * pwb;
            float pa, pb;
            if (full_panel)
                rowwarp_two_rows<FMT, true>(ra, rbp, lane, pwb, xr, pa, pb);
            else
                rowwarp_two_rows<FMT, false>(ra, rbp, lane, pwb, xr, pa, pb);
            const float total = warp_sum_two_rows(pa, pb);  // lanes 0-15: row r, 16-31: row rb2
            if ((lane & 15) == 0 && (hi == 0 || rb2 != r)) {
                const int64_t row = row0 + (hi ? rb2 : r);
                float val = total;
                if (a.panels > 1) {
                    float *yp = a.y + row;
                    if (panel > 0) val += *yp;
                    *yp = val;
                } else if (a.y) {
                    a.y[row] = val;
                }
                if (ARGMAX && panel == a.panels - 1 &&
                    argmax_better(val, static_cast<uint32_t>(row), best_v, best_i)) {
                    best_v = val;
                    best_i = static_cast<uint32_t>(row);
                }
            }
        }
        __syncwarp();  // every lane is done reading stage s
        if (u + stages < units) {
            if (lane == 0)
                issue_unit<FMT>(a, u + stages, n_my, g0, smem_addr(ring + static_cast<size_t>(s) * a.stage_bytes),
                                bar0 + 8 * s, policy, false);
            issued_end = u + stages + 1;
        }
    }

    if (aborted) {
        // Let copies already in flight land (each wait bounded), then report.
        for (int64_t u = failed_unit; u < issued_end; ++u)
            (void)mbar_wait_bounded(bar0 + 8 * static_cast<uint32_t>(u % stages),
                                     static_cast<uint32_t>((u / stages) & 1));
        if (lane == 0) atomicOr(a.status, 1u);
    }

    if constexpr (ARGMAX) {
        {   // lanes 0 and 16 track the two row slots
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, best_v, 16);
            const uint32_t oi = __shfl_xor_sync(0xFFFFFFFFu, best_i, 16);
            if (argmax_better(ov, oi, best_v, best_i)) {
                best_v = ov;
                best_i = oi;
            }
        }
        if (lane == 0) {
            am_val[warp][0] = best_v;
            am_idx[warp][0] = best_i;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            float bv = -INFINITY;
            uint32_t bi = 0;
            for (int w2 = 0; w2 < kRowWarps; ++w2)
                if (argmax_better(am_val[w2][0], am_idx[w2][0], bv, bi)) {
                    bv = am_val[w2][0];
                    bi = am_idx[w2][0];
                }
            __stcg(a.part_val + blockIdx.x, bv);
            __stcg(a.part_idx + blockIdx.x, bi);
        }
        argmax_cross_cta<1, kRowThreads>(a, am_val, am_idx, &s_is_last);
    }
}

}  // namespace fp8blk
