// nvfp4_gemv.cuh -- routed-expert GEMV straight from NVFP4 storage, all
// active experts in one launch, expert ids and global scales read on the
// device:
//   y[k][r] = sum_c bf16( e2m1(q[e][r][c]) * e4m3(s[e][r][c/16]) * g[e] ) * x[c],
//   e = ids[k].
// Source: "Module dsv4_gpu" page, module header and enum ExpertArm (routed
// experts stay NVFP4 as stored; each activated expert's weights take the
// exact bf16 values of its dequantisation) and the header's one-launch-per-
// projection indirect expert dispatch.  The bf16 scratch round trip of the
// dequant-then-GEMV arm is skipped: every product e2m1 * e4m3 * g is exact in
// f32 (at most 6 significant bits, g a power of two), so decoding in registers
// gives the same weight values; the sum is formed as
//   g * sum_blocks e4m3(s) * sum_{16 columns} e2m1 * x      (f32).
//
// Structure follows the row-per-warp GEMV: with one activation row, x for the
// lane's 128 columns of a <= 4096-column panel lives in registers; each warp
// streams its own contiguous run of (expert, row group) units through a
// private ring of shared-memory stages filled by 1-D bulk copies (codes rows
// then scale rows) on per-stage mbarriers; rows are reduced two at a time.
// An expert id outside [0, n_experts) or a global scale that is not a power
// of two in [2^-100, 2^100] sets FP8BLK_STATUS_BAD_EXPERT and makes that
// slot's outputs NaN.
//
// The same kernel serves OCP MXFP4 experts (the MTP block's, "Module
// dsv4_gpu" page, enum ExpertKind): the same code layout, one e8m0 scale
// 2^(c-127) per 32 columns (0xFF = NaN), no global scale.
#pragma once

#include "rowwarp_gemv.cuh"

namespace fp8blk {

constexpr int kNvWarps = 4;
constexpr int kNvThreads = kNvWarps * 32;
constexpr int kNvMaxPanel = 4096;           // columns per panel
constexpr int kNvChunks = kNvMaxPanel / 1024;  // 32-column chunks of a panel per lane (x registers: 32 each)
constexpr int kNvCtasPerSm = 2;
constexpr unsigned kStatusBadExpert = 2u;   // FP8BLK_STATUS_BAD_EXPERT
constexpr int kFp4Nv = 0;                   // NVFP4: e4m3 scale per 16 columns, f32 global scale
constexpr int kFp4Mx = 1;                   // MXFP4: e8m0 scale per 32 columns

template <int FP4>
__host__ __device__ constexpr int fp4_scale_cols() { return FP4 == kFp4Mx ? 32 : 16; }

// e8m0 code -> 2^(c - 127) as f32 (c = 0 is the subnormal 2^-127), 0xFF -> NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t c) {
    return __int_as_float(c == 0u ? 0x00400000 : (c == 255u ? 0x7FC00000 : static_cast<int>(c << 23)));
}
constexpr int kNvXSmemBytes = kNvMaxPanel * 4;  // one panel of x, lane-transposed (single-panel shapes)

// Expert of slot k, or -1 when the id or its global scale is unusable.
template <int FP4>
__device__ __forceinline__ int nv_expert(const Nvfp4Args &a, int k, float *g) {
    const int e = __ldg(a.ids + k);
    if (e < 0 || e >= a.n_experts) return -1;
    if (FP4 == kFp4Mx) {
        *g = 1.f;
        return e;
    }
    const float gv = __ldg(a.gscale + e);
    int ex = 0;
    const float f = frexpf(gv, &ex);
    if (!(gv > 0.f) || f != 0.5f || ex - 1 < -100 || ex - 1 > 100) return -1;
    *g = gv;
    return e;
}

// The expert of the slot last looked up: a warp's units run through few
// slots, and each lookup is two dependent global loads.
struct NvSlot {
    int k = -1, e = -1;
    float g = 0.f;
};
template <int FP4>
__device__ __forceinline__ const NvSlot &nv_slot(const Nvfp4Args &a, int k, NvSlot &c) {
    if (k != c.k) {
        c.k = k;
        c.e = nv_expert<FP4>(a, k, &c.g);
    }
    return c;
}

// Lane 0: copy unit u (slot k, row group, panel) into a ring stage.
template <int FP4>
__device__ __forceinline__ void nv_issue(const Nvfp4Args &a, int64_t u, int64_t n_my, int64_t g0,
                                         uint32_t dst, uint32_t bar, uint64_t policy, NvSlot &cache) {
    const int panel = static_cast<int>(u / n_my);
    const int64_t gg = g0 + u % n_my;  // global group index over (slot, row group)
    const int k = static_cast<int>(gg / a.groups);
    const int64_t row0 = (gg % a.groups) * a.stage_rows;
    const int nr = static_cast<int>(a.rows - row0 < a.stage_rows ? a.rows - row0 : a.stage_rows);
    const int e = nv_slot<FP4>(a, k, cache).e;
    if (e < 0) {  // nothing to copy: complete the phase so the consumers move on
        mbar_arrive(bar);
        return;
    }
    const int64_t pc64 = a.cols - static_cast<int64_t>(panel) * a.panel_cols;
    const int pc = pc64 < a.panel_cols ? static_cast<int>(pc64) : a.panel_cols;
    constexpr int SC = fp4_scale_cols<FP4>();
    const uint32_t cb = static_cast<uint32_t>(pc / 2), sb = static_cast<uint32_t>(pc / SC);
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nr) * (cb + sb));
    const int64_t erow = static_cast<int64_t>(e) * a.rows + row0;
    const uint8_t *csrc = a.codes + erow * (a.cols / 2) + static_cast<int64_t>(panel) * (a.panel_cols / 2);
    const uint8_t *ssrc = a.scales + erow * (a.cols / SC) + static_cast<int64_t>(panel) * (a.panel_cols / SC);
    const uint32_t sdst = dst + static_cast<uint32_t>(a.stage_rows) * static_cast<uint32_t>(a.panel_cols / 2);
    if (a.panels == 1) {  // rows are contiguous: one copy each
        bulk_g2s(dst, csrc, static_cast<uint32_t>(nr) * cb, bar, policy);
        bulk_g2s(sdst, ssrc, static_cast<uint32_t>(nr) * sb, bar, policy);
    } else {
        for (int r = 0; r < nr; ++r) {
            bulk_g2s(dst + r * cb, csrc + static_cast<int64_t>(r) * (a.cols / 2), cb, bar, policy);
            bulk_g2s(sdst + r * sb, ssrc + static_cast<int64_t>(r) * (a.cols / SC), sb, bar, policy);
        }
    }
}

// x for this lane's chunks of the panel: chunk c = 32 columns, lane l holds
// chunks l, l + 32, l + 64, l + 96.
__device__ __forceinline__ void nv_load_x(const Nvfp4Args &a, int panel, int pc, int lane, float (&xr)[32 * kNvChunks]) {
#pragma unroll
    for (int j = 0; j < kNvChunks; ++j) {
        const int chunk = j * 32 + lane;
        const bool ok = chunk * 32 < pc;
        const int64_t c0 = static_cast<int64_t>(panel) * a.panel_cols + static_cast<int64_t>(chunk) * 32;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 v = ok ? __ldg(reinterpret_cast<const float4 *>(a.x + c0) + q) : make_float4(0.f, 0.f, 0.f, 0.f);
            xr[j * 32 + 4 * q] = v.x;
            xr[j * 32 + 4 * q + 1] = v.y;
            xr[j * 32 + 4 * q + 2] = v.z;
            xr[j * 32 + 4 * q + 3] = v.w;
        }
    }
}

// Single-panel shapes: the CTA loads x once (coalesced, every load in flight
// at once) into shared memory in lane-transposed float4 order,
// xT[(j * 8 + q) * 32 + l] = x4[(j * 32 + l) * 8 + q], so that each warp
// fills its registers with conflict-free 16-byte reads.
constexpr int kNvXPerThread = kNvMaxPanel / 4 / kNvThreads;
__device__ __forceinline__ void nv_stage_x_load(const Nvfp4Args &a, float4 (&v)[kNvXPerThread]) {
    const int n4 = static_cast<int>(a.cols / 4);
#pragma unroll
    for (int t = 0; t < kNvXPerThread; ++t) {
        const int i = static_cast<int>(threadIdx.x) + t * kNvThreads;
        v[t] = i < n4 ? __ldg(reinterpret_cast<const float4 *>(a.x) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}
__device__ __forceinline__ void nv_stage_x_store(const float4 (&v)[kNvXPerThread], float4 *xT) {
#pragma unroll
    for (int t = 0; t < kNvXPerThread; ++t) {
        const int i = static_cast<int>(threadIdx.x) + t * kNvThreads;
        const int chunk = i >> 3, q = i & 7;
        xT[((chunk >> 5) * 8 + q) * 32 + (chunk & 31)] = v[t];
    }
}

__device__ __forceinline__ void nv_load_x_smem(const float4 *xT, int lane, float (&xr)[32 * kNvChunks]) {
#pragma unroll
    for (int j = 0; j < kNvChunks; ++j)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 v = xT[(j * 8 + q) * 32 + lane];
            xr[j * 32 + 4 * q] = v.x;
            xr[j * 32 + 4 * q + 1] = v.y;
            xr[j * 32 + 4 * q + 2] = v.z;
            xr[j * 32 + 4 * q + 3] = v.w;
        }
}

// Sum over one 16-column block (two code words) of e2m1 * x, f32.
__device__ __forceinline__ float nv_block16(uint32_t w0, uint32_t w1, const float *xb) {
    uint32_t h[8];
    e2m1x8_to_f16x2(w0, h);
    e2m1x8_to_f16x2(w1, h + 4);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h[k]));
        s0 = fmaf(f.x, xb[2 * k], s0);
        s1 = fmaf(f.y, xb[2 * k + 1], s1);
    }
    return s0 + s1;
}

// This lane's share of one staged row: sum over its chunks of the chunk's
// block scale(s) times the sums of e2m1 * x.
template <int FP4, bool FULL>
__device__ __forceinline__ float nv_row(const uint8_t *crow, const uint8_t *srow, int lane, int pc,
                                        const float (&xr)[32 * kNvChunks]) {
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kNvChunks; ++j) {
        const int chunk = j * 32 + lane;
        if (FULL || chunk * 32 < pc) {
            const uint4 q = *reinterpret_cast<const uint4 *>(crow + chunk * 16);
            if (FP4 == kFp4Mx) {  // one e8m0 scale for the chunk's 32 columns
                const float s = e8m0_to_f32(srow[chunk]);
                acc = fmaf(s, nv_block16(q.x, q.y, &xr[j * 32]) + nv_block16(q.z, q.w, &xr[j * 32 + 16]), acc);
            } else {  // two e4m3 scales, one per 16 columns
                const uint32_t sc = *reinterpret_cast<const unsigned short *>(srow + chunk * 2);
                const float2 s = e4m3x2_to_f32(sc);
                acc = fmaf(s.x, nv_block16(q.x, q.y, &xr[j * 32]), acc);
                acc = fmaf(s.y, nv_block16(q.z, q.w, &xr[j * 32 + 16]), acc);
            }
        }
    }
    return acc;
}

template <int FP4>
__global__ void __launch_bounds__(kNvThreads, kNvCtasPerSm) fp4_expert_gemv_kernel(const Nvfp4Args a) {
    constexpr int SC = fp4_scale_cols<FP4>();
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kNvWarps][kMaxStages];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int stages = a.stages;
    const bool x_in_smem = a.panels == 1;
    float4 *xT = reinterpret_cast<float4 *>(smem);  // single-panel shapes only
    uint8_t *ring = smem + (x_in_smem ? kNvXSmemBytes : 0) + static_cast<size_t>(warp) * stages * a.stage_bytes;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kNvWarps;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * kNvWarps + warp;
    const int64_t total_groups = a.groups * a.n_active;
    const int64_t g0 = gw * total_groups / nwarps;
    const int64_t g1 = (gw + 1) * total_groups / nwarps;
    const int64_t n_my = g1 - g0;
    const int64_t units = n_my * a.panels;
    const uint32_t bar0 = smem_addr(&bars[warp][0]);
    if (lane == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(bar0 + 8 * s, 1);
        mbar_init_fence();
    }
    __syncwarp();

    // The ids, scales and x may be outputs of the preceding kernel.
    grid_dependency_wait();
    grid_launch_dependents();
    // x loads first: they are in flight while lane 0 looks the experts up
    // (dependent loads) and issues the first ring.
    float4 xv[kNvXPerThread];
    if (x_in_smem) nv_stage_x_load(a, xv);
    const uint64_t policy = l2_policy_evict_first();
    const int64_t first = units < stages ? units : stages;
    NvSlot issue_slot, use_slot;
    if (lane == 0)
        for (int64_t u = 0; u < first; ++u)
            nv_issue<FP4>(a, u, n_my, g0, smem_addr(ring + u * a.stage_bytes), bar0 + 8 * static_cast<uint32_t>(u),
                          policy, issue_slot);
    int64_t issued_end = first;

    float xr[32 * kNvChunks];
    int cur_panel = -1;
    if (x_in_smem) {  // uniform over the CTA
        nv_stage_x_store(xv, xT);
        __syncthreads();
        nv_load_x_smem(xT, lane, xr);
        cur_panel = 0;
    }
    bool aborted = false;
    int64_t failed_unit = 0;
    for (int64_t u = 0; u < units; ++u) {
        const int s = static_cast<int>(u % stages);
        const int panel = static_cast<int>(u / n_my);
        const int64_t gg = g0 + u % n_my;
        const int k = static_cast<int>(gg / a.groups);
        const int64_t row0 = (gg % a.groups) * a.stage_rows;
        const int nr = static_cast<int>(a.rows - row0 < a.stage_rows ? a.rows - row0 : a.stage_rows);
        const int64_t pc64 = a.cols - static_cast<int64_t>(panel) * a.panel_cols;
        const int pc = pc64 < a.panel_cols ? static_cast<int>(pc64) : a.panel_cols;
        if (panel != cur_panel) {
            nv_load_x(a, panel, pc, lane, xr);
            cur_panel = panel;
        }
        const NvSlot &sl = nv_slot<FP4>(a, k, use_slot);
        const int e = sl.e;
        const float g = sl.g;
        const bool ok = mbar_wait_limit(bar0 + 8 * s, static_cast<uint32_t>((u / stages) & 1), a.wait_limit_ns);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
            aborted = true;
            failed_unit = u;
            break;
        }
        const uint8_t *st = ring + static_cast<size_t>(s) * a.stage_bytes;
        const uint8_t *sst = st + a.stage_rows * (a.panel_cols / 2);
        const bool full = pc == kNvMaxPanel;
        const int hi = lane >> 4;  // 1: this lane handles the pair's rows swapped
        for (int r = 0; r < nr; r += 2) {
            const int rb2 = r + 1 < nr ? r + 1 : r;
            const int ra = hi ? rb2 : r, rb = hi ? r : rb2;
            float pa = 0.f, pb = 0.f;
            if (e >= 0) {
                if (full) {
                    pa = nv_row<FP4, true>(st + ra * (pc / 2), sst + ra * (pc / SC), lane, pc, xr);
                    pb = nv_row<FP4, true>(st + rb * (pc / 2), sst + rb * (pc / SC), lane, pc, xr);
                } else {
                    pa = nv_row<FP4, false>(st + ra * (pc / 2), sst + ra * (pc / SC), lane, pc, xr);
                    pb = nv_row<FP4, false>(st + rb * (pc / 2), sst + rb * (pc / SC), lane, pc, xr);
                }
            }
            const float total = warp_sum_two_rows(pa, pb);  // lanes 0-15: row r, 16-31: row rb2
            if ((lane & 15) == 0 && (hi == 0 || rb2 != r)) {
                const int64_t row = row0 + (hi ? rb2 : r);
                float *yp = a.y + static_cast<int64_t>(k) * a.rows + row;
                float val = e >= 0 ? total * g : __int_as_float(0x7FC00000);
                if (a.panels > 1 && panel > 0) val += *yp;
                *yp = val;
            }
        }
        if (e < 0 && lane == 0 && panel == 0 && row0 == 0) atomicOr(a.status, kStatusBadExpert);
        __syncwarp();  // every lane is done reading stage s
        if (u + stages < units) {
            if (lane == 0)
                nv_issue<FP4>(a, u + stages, n_my, g0, smem_addr(ring + static_cast<size_t>(s) * a.stage_bytes),
                              bar0 + 8 * s, policy, issue_slot);
            issued_end = u + stages + 1;
        }
    }

    if (aborted) {
        // Let copies already in flight land (each wait bounded), then report.
        for (int64_t u = failed_unit; u < issued_end; ++u)
            (void)mbar_wait_bounded(bar0 + 8 * static_cast<uint32_t>(u % stages), static_cast<uint32_t>((u / stages) & 1));
        if (lane == 0) atomicOr(a.status, 1u);
    }
}

}  // namespace fp8blk
