// gemv_tc.cu -- instantiations and launch of the tensor-core e4m3 GEMV
// (tc8_gemv.cuh): weight codes straight from TMA into kind::f8f6f4 MMAs, with
// and without the fused argmax.
#include "launch.h"

namespace fp8blk {

template <bool ARGMAX>
static cudaError_t launch_tc8(const GemvArgs &a, const Plan &p, int m, const DeviceInfo &dev, cudaStream_t stream) {
    CUtensorMap map;
    cudaError_t err = weight_tensor_map(a.w, a.rows, a.cols, 128, &map);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = kernel_occupancy(reinterpret_cast<const void *>(tc8_gemv_kernel<ARGMAX>), kT8Threads, kT8SmemBytes, &per_sm);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    T8Args t = {};
    t.w = a.w;
    t.scales = a.scales;
    t.x = a.x;
    t.y = a.y;
    t.tokens = a.tokens;
    t.part_val = a.part_val;
    t.part_idx = a.part_idx;
    t.counter = a.counter;
    t.status = a.status;
    t.rows = a.rows;
    t.cols = a.cols;
    t.m = m;
    t.n_tiles = p.n_groups;
    t.l2_prefetch = tuning().l2_prefetch ? tuning().tc_l2_prefetch : 0;
    int64_t grid = dev.sms;
    if (grid > t.n_tiles) grid = t.n_tiles;
    if (grid > kMaxGrid) grid = kMaxGrid;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kT8Threads);
    cfg.dynamicSmemBytes = kT8SmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = tuning().use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, tc8_gemv_kernel<ARGMAX>, map, t);
}

cudaError_t launch_gemv_tc(const GemvArgs &a, const Plan &p, int m, bool argmax, const DeviceInfo &dev,
                           cudaStream_t stream) {
    return argmax ? launch_tc8<true>(a, p, m, dev, stream) : launch_tc8<false>(a, p, m, dev, stream);
}

}  // namespace fp8blk
