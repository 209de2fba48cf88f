// nvfp4_gemv.cu -- plan and launch of the one-launch FP4 (NVFP4 / MXFP4)
// routed-expert GEMV (nvfp4_gemv.cuh).
#include "launch.h"
#include "fp4tc_gemv.cuh"
#include "nvfp4_gemv.cuh"

namespace fp8blk {

constexpr int kNvStageTarget = 16384;  // bytes of two stages (R rows each) the row count aims at

// Rows per unit for the tensor-core FP4 kernel: the smallest multiple of 8
// (at most 128) whose units, n_active x ceil(rows / R), fit one per SM.
static int f4_slab_rows(const Nvfp4Args &a, const DeviceInfo &dev) {
    for (int r = 8; r < 128; r += 8)
        if (static_cast<int64_t>(a.n_active) * ((a.rows + r - 1) / r) <= dev.sms) return r;
    return 128;
}

// FP4 experts on the tensor cores: one CTA per SM over contiguous ranges of
// (slot, slab) units.
template <int FP4>
static cudaError_t launch_fp4tc(const Nvfp4Args &a, const DeviceInfo &dev, cudaStream_t stream) {
    F4Args f = {};
    f.nv = a;
    f.slab_rows = f4_slab_rows(a, dev);
    f.raw_stages = f4_raw_stages(a.cols, f.slab_rows, dev.smem_per_block - kStaticSmemReserve);
    if (f.raw_stages < kF4MinRawStages) return cudaErrorInvalidConfiguration;
    f.n_slabs = (a.rows + f.slab_rows - 1) / f.slab_rows;
    f.units = f.n_slabs * a.n_active;
    CUtensorMap cmap, smap;
    cudaError_t err = nvfp4_tensor_maps(a.codes, a.scales, static_cast<int64_t>(a.n_experts) * a.rows, a.cols,
                                        fp4_scale_cols<FP4>(), f.slab_rows, &cmap, &smap);
    if (err != cudaSuccess) return err;
    const size_t smem = f4_smem_bytes(a.cols, f.raw_stages, f.slab_rows);
    int per_sm = 0;
    err = kernel_occupancy(reinterpret_cast<const void *>(fp4tc_gemv_kernel<FP4>), kF4Threads, smem, &per_sm);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int64_t grid = dev.sms;
    if (grid > f.units) grid = f.units;
    if (grid > kMaxGrid) grid = kMaxGrid;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kF4Threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = tuning().use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, fp4tc_gemv_kernel<FP4>, cmap, smap, f);
}

// By shape, FP4 experts take the tensor cores from this many active rows
// (n_active x rows) on.  The tensor-core kernel costs about 0.5 us per
// 256-column stage however short its slab, so below it the CUDA-core kernel
// is faster (2048 x 4096 experts, us, tensor vs CUDA cores: NVFP4 4 active
// about 12.3 vs 9.2, 6 active 12.2 vs 12.5, 64 active 60.1 vs 86.3; MXFP4
// 6 active 11.9 vs 12.8).
constexpr int64_t kF4TcMinActiveRows = 12288;

// FP4 experts take the tensor cores when chosen (by shape or pinned) and
// the codes start on a 32-byte boundary (the packed-code TMA type), the slab
// rows fit 32-bit TMA coordinates over the experts' stacked rows, and B plus
// a minimal ring fit in shared memory.
static bool fp4_use_tensor_cores(const Nvfp4Args &a, const DeviceInfo &dev) {
    if (tuning().fp4_kernel == 1) return false;
    if (tuning().fp4_kernel == 0 && static_cast<int64_t>(a.n_active) * a.rows < kF4TcMinActiveRows) return false;
    return (reinterpret_cast<uintptr_t>(a.codes) & 31u) == 0 &&
           static_cast<int64_t>(a.n_experts) * a.rows + 128 <= (1ll << 31) - 1 &&
           f4_raw_stages(a.cols, f4_slab_rows(a, dev), dev.smem_per_block - kStaticSmemReserve) >= kF4MinRawStages;
}

cudaError_t launch_fp4_expert_gemv(Nvfp4Args a, bool mxfp4, const DeviceInfo &dev, cudaStream_t stream) {
    if (fp4_use_tensor_cores(a, dev))
        return mxfp4 ? launch_fp4tc<kFp4Mx>(a, dev, stream) : launch_fp4tc<kFp4Nv>(a, dev, stream);
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
