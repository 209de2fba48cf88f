// nvfp4_gemv.cu -- plan and launch of the one-launch FP4 (NVFP4 / MXFP4)
// routed-expert GEMV (nvfp4_gemv.cuh).
#include "launch.h"
#include "nvfp4_gemv.cuh"

namespace fp8blk {

constexpr int kNvStageTarget = 16384;  // bytes of two stages (R rows each) the row count aims at

cudaError_t launch_fp4_expert_gemv(Nvfp4Args a, bool mxfp4, const DeviceInfo &dev, cudaStream_t stream) {
    a.panels = static_cast<int>((a.cols + kNvMaxPanel - 1) / kNvMaxPanel);
    a.panel_cols = a.panels == 1 ? static_cast<int>(a.cols) : kNvMaxPanel;
    const int row_bytes = a.panel_cols / 2 + a.panel_cols / (mxfp4 ? 32 : 16);
    // Stages of about 8 KiB (R rows), fewer rows while there are fewer row
    // groups than warps or while two stages per warp do not fit beside x in
    // the CTA's share of the SM (kNvCtasPerSm CTAs per SM).
    const int ctas_per_sm = kNvCtasPerSm;
    const int x_bytes = a.panels == 1 ? kNvXSmemBytes : 0;  // x staged once per CTA
    int per_cta = dev.smem_per_sm / ctas_per_sm - 1024 - kStaticSmemReserve;
    const int block_cap = dev.smem_per_block - kStaticSmemReserve;
    if (per_cta > block_cap) per_cta = block_cap;
    const int per_warp = (per_cta - x_bytes) / kNvWarps;
    int rw = 1;
    while (rw < 8 && 2 * rw * row_bytes <= kNvStageTarget) rw *= 2;
    while (rw > 1 && per_warp / (rw * row_bytes) < 2) rw /= 2;
    const int64_t warps = static_cast<int64_t>(dev.sms) * ctas_per_sm * kNvWarps;
    while (rw > 1 && (a.rows + rw - 1) / rw * a.n_active < warps) rw /= 2;
    a.stage_rows = rw;
    a.stage_bytes = rw * row_bytes;
    a.groups = (a.rows + rw - 1) / rw;
    int stages = per_warp / a.stage_bytes;
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return cudaErrorInvalidConfiguration;
    a.stages = stages;
    const size_t smem = static_cast<size_t>(x_bytes) + static_cast<size_t>(kNvWarps) * stages * a.stage_bytes;
    int per_sm = 0;
    const void *kernel = mxfp4 ? reinterpret_cast<const void *>(fp4_expert_gemv_kernel<kFp4Mx>)
                               : reinterpret_cast<const void *>(fp4_expert_gemv_kernel<kFp4Nv>);
    cudaError_t err = kernel_occupancy(kernel, kNvThreads, smem, &per_sm);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int64_t total_groups = a.groups * a.n_active;
    int64_t grid = (total_groups + kNvWarps - 1) / kNvWarps;
    const int64_t cap = static_cast<int64_t>(dev.sms) * (per_sm < ctas_per_sm ? per_sm : ctas_per_sm);
    if (grid > cap) grid = cap;
    if (grid > kMaxGrid) grid = kMaxGrid;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kNvThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = tuning().use_pdl ? 1 : 0;
    return mxfp4 ? cudaLaunchKernelEx(&cfg, fp4_expert_gemv_kernel<kFp4Mx>, a)
                 : cudaLaunchKernelEx(&cfg, fp4_expert_gemv_kernel<kFp4Nv>, a);
}

}  // namespace fp8blk
