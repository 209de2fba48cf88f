// launch.h -- host-side planning and launch entry points shared by the
// libfp8blk translation units (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "rowwarp_gemv.cuh"
#include "stream_gemv.cuh"
#include "tc8_gemv.cuh"

namespace fp8blk {

// Launch-shape knobs.  Results do not depend on them (each output's
// reduction order is fixed by the column panel layout alone); only speed does.
struct Tuning {
    int target_stage_bytes = 32 * 1024;  // bytes of weights per pipeline stage
    int ctas_per_sm = 0;                 // 0 = 2 for m <= 4, 1 for m > 4
    int use_pdl = 1;                     // programmatic dependent launch
    int l2_prefetch = 1;                 // L2 prefetch of the first stages before the PDL wait
    int64_t tc_l2_prefetch = 192 * 1024; // tensor-core kernel: bytes of each CTA's first rows prefetched
    int max_stages = kMaxStages;
    int m1_kernel = 0;                   // m = 1: 0 = by size, 1 = row-per-warp, 2 = team
    int tc_min_m = 1;                    // tensor-core kernel for m >= this (9 = never)
    int64_t tc_min_bytes = 0;            // ... and at least this many weight bytes (0 = by m, below)
    int64_t m1_rowwarp_min_bytes = 96ll << 20;  // by size: row-per-warp from this many weight bytes
    uint64_t wait_limit_ns = kWaitLimitNs;      // consumer waits of the CUDA-core kernels
    int fp4_kernel = 0;                  // NVFP4 experts: 0 = by shape, 1 = CUDA cores, 2 = tensor cores
};
Tuning &tuning();

struct DeviceInfo {
    int sms = 0;
    int smem_per_sm = 0;      // bytes
    int smem_per_block = 0;   // opt-in maximum, bytes
    unsigned int *status = nullptr;  // device address of the status word
};
// Default weight-byte threshold of the tensor-core kernel by activation rows
// (measured crossovers against the CUDA-core kernels at 4096 columns; below
// them the tensor-core kernel's per-tile set-up and the tile count's
// quantisation over the SMs cost more than it saves).
inline int64_t tc_default_min_bytes(int m) {
    return m >= 5 ? (24ll << 20) : (m >= 3 ? (32ll << 20) : (48ll << 20));
}

// Per-device facts, queried once per device (current device).
cudaError_t current_device_info(DeviceInfo *out);

// Geometry of one streaming-GEMV launch (see GemvArgs).
enum PlanKind : int { kTeamKernel = 0, kRowWarpKernel = 1, kTensorCoreKernel = 2 };
struct Plan {
    int kind = kTeamKernel;  // m = 1 uses the row-per-warp kernel
    int panels = 1;
    int panel_cols = 0;
    int team_warps_log2 = 0;
    int rb = 1;
    int stage_rows = 0;
    int stage_bytes = 0;
    int stages = 2;
    int ctas_per_sm = 1;
    int64_t n_groups = 0;
};
constexpr int kStaticSmemReserve = 6 * 1024;  // red/argmax buffers + slack
constexpr int kMaxGrid = 1024;               // bound on CTAs (argmax partials)

// Plans a launch of m rows over a [rows, cols] matrix of bpw-byte weights.
Plan make_plan(int m, int64_t rows, int64_t cols, int bpw, const DeviceInfo &dev);

// Fill GemvArgs geometry from a plan.
void apply_plan(const Plan &p, GemvArgs *a);

// Tensor map of an e4m3 weight matrix for the tensor-core kernel: 2-D,
// {cols, rows}, boxes of box_rows rows x 128 bytes, 128-byte swizzle, zeros
// out of range.  Cached per (pointer, shape, box height).
cudaError_t weight_tensor_map(const uint8_t *w, int64_t rows, int64_t cols, int box_rows, CUtensorMap *out);
// FP4 codes [total_rows, cols] e2m1 (boxes of box_rows x 128 codes, each 8
// code bytes landing in a 16-byte shared-memory chunk, 128-byte swizzle) and
// scales [total_rows, cols / scale_block] bytes (box_rows x 16-byte boxes)
// for the tensor-core FP4 kernel, which copies 256 columns per stage.
constexpr int kF4StageColsHost = 256;
cudaError_t nvfp4_tensor_maps(const uint8_t *codes, const uint8_t *scales, int64_t total_rows, int64_t cols,
                              int scale_block, int box_rows, CUtensorMap *cmap, CUtensorMap *smap);

// Kernel launches (defined in gemv_e4m3.cu / gemv_bf16.cu / nvfp4_dequant.cu /
// gemv_tc.cu).
cudaError_t launch_gemv_tc(const GemvArgs &a, const Plan &p, int m, bool argmax, const DeviceInfo &dev,
                           cudaStream_t stream);
cudaError_t launch_gemv_e4m3(const GemvArgs &a, const Plan &p, int m, bool argmax,
                             const DeviceInfo &dev, cudaStream_t stream);
cudaError_t launch_gemv_bf16(const GemvArgs &a, const Plan &p, int m, const DeviceInfo &dev,
                             cudaStream_t stream);
cudaError_t launch_nvfp4_dequant(const uint8_t *codes, const uint8_t *scales, float g,
                                 uint16_t *out, int64_t rows, int64_t cols,
                                 const DeviceInfo &dev, cudaStream_t stream);

// Resident CTAs per SM of `kernel` with `smem` dynamic shared memory on the
// current device.  Raises the kernel's dynamic-smem limit first; both answers
// are cached per (kernel, device, smem), so steady-state launches (and stream
// capture) make no attribute or occupancy calls.
cudaError_t kernel_occupancy(const void *kernel, int threads, size_t smem, int *per_sm);

// One-launch NVFP4 routed-expert GEMV (kernel in nvfp4_gemv.cuh, launch in
// nvfp4_gemv.cu, which plans the panels, stages and grid itself).
struct Nvfp4Args {
    const uint8_t *codes;    // [n_experts, rows, cols / 2]
    const uint8_t *scales;   // NVFP4: e4m3 [n_experts, rows, cols / 16]; MXFP4: e8m0 [.., cols / 32]
    const float *gscale;     // [n_experts], device (NVFP4 only)
    const int32_t *ids;      // [n_active], device
    const float *x;          // [cols]
    float *y;                // [n_active, rows]
    unsigned int *status;
    int n_experts, n_active;
    int64_t rows, cols;
    int panels, panel_cols;  // panel_cols = cols (one panel) or 4096
    int stage_rows;          // R rows per stage
    int stage_bytes;         // R * (panel_cols / 2 + panel_cols / scale_cols)
    int stages;
    int64_t groups;          // row groups per expert: ceil(rows / R)
    uint64_t wait_limit_ns;  // consumer-side weight-tile wait limit
};
cudaError_t launch_fp4_expert_gemv(Nvfp4Args a, bool mxfp4, const DeviceInfo &dev, cudaStream_t stream);

// Dynamic shared memory of a planned launch.
inline size_t plan_smem_bytes(const Plan &p) {
    if (p.kind == kTensorCoreKernel) return kT8SmemBytes;
    if (p.kind == kRowWarpKernel) return static_cast<size_t>(kRowWarps) * p.stages * p.stage_bytes;
    return static_cast<size_t>(p.stages) * p.stage_bytes;
}

// Shared launcher: grid from occupancy, dynamic smem attribute, optional PDL.
template <typename Kernel>
cudaError_t launch_stream_kernel(Kernel kernel, const GemvArgs &a, const Plan &p,
                                 const DeviceInfo &dev, cudaStream_t stream) {
    const int threads = p.kind == kRowWarpKernel ? kRowThreads : kThreads;
    const size_t smem = plan_smem_bytes(p);
    int per_sm = 0;
    cudaError_t err = kernel_occupancy(reinterpret_cast<const void *>(kernel), threads, smem, &per_sm);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    if (per_sm > p.ctas_per_sm) per_sm = p.ctas_per_sm;
    const int64_t work_ctas = p.kind == kRowWarpKernel ? (p.n_groups + kRowWarps - 1) / kRowWarps : p.n_groups;
    int64_t grid = static_cast<int64_t>(dev.sms) * per_sm;
    if (grid > work_ctas) grid = work_ctas;
    if (grid > kMaxGrid) grid = kMaxGrid;
    if (grid < 1) grid = 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = tuning().use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace fp8blk
