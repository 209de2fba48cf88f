// gemv_tc.cu -- instantiations and launch of the tensor-core batched-verify
// GEMV (tc_gemv.cuh), m = 2..8, with and without the fused argmax.
#include "launch.h"

namespace fp8blk {

template <bool ARGMAX>
static cudaError_t launch_tc(const GemvArgs &a, const Plan &p, int m, const DeviceInfo &dev, cudaStream_t stream) {
    CUtensorMap map_big, map_small, map_x;
    cudaError_t err = weight_tensor_map(a.w, a.rows, a.cols, kTcM, &map_big);
    if (err == cudaSuccess) err = weight_tensor_map(a.w, a.rows, a.cols, kTcSmallBoxRows, &map_small);
    if (err == cudaSuccess) err = activation_tensor_map(a.x, m, a.cols, kTcXCols, &map_x);
    if (err != cudaSuccess) return err;
    const size_t smem = kTcSmemBytes;
    int per_sm = 0;
    err = kernel_occupancy(reinterpret_cast<const void *>(tc_gemv_kernel<ARGMAX>), kTcThreads, smem, &per_sm);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    TcArgs t = {};
    t.scales = a.scales;
    t.x = a.x;
    t.y = a.y;
    t.tokens = a.tokens;
    t.part_val = a.part_val;
    t.part_idx = a.part_idx;
    t.counter = a.counter;
    t.status = a.status;
    t.w = a.w;
    t.rows = a.rows;
    t.cols = a.cols;
    t.m = m;
    t.panels = p.panels;
    t.panel_cols = p.panel_cols;
    t.n_units8 = p.n_groups;
    int64_t grid = dev.sms;
    if (grid > t.n_units8) grid = t.n_units8;
    if (grid > kMaxGrid) grid = kMaxGrid;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = tuning().use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, tc_gemv_kernel<ARGMAX>, map_big, map_small, map_x, t);
}

cudaError_t launch_gemv_tc(const GemvArgs &a, const Plan &p, int m, bool argmax, const DeviceInfo &dev,
                           cudaStream_t stream) {
    return argmax ? launch_tc<true>(a, p, m, dev, stream) : launch_tc<false>(a, p, m, dev, stream);
}

}  // namespace fp8blk
