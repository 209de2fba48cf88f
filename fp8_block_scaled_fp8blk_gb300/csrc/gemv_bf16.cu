// gemv_bf16.cu -- instantiations of the streaming GEMV for bf16 weights (the
// dequantised NVFP4 expert scratch): row-per-warp for large m = 1 matrices,
// the team kernel otherwise.
#include "launch.h"

namespace fp8blk {

cudaError_t launch_gemv_bf16(const GemvArgs &a, const Plan &p, int m, const DeviceInfo &dev,
                             cudaStream_t stream) {
    if (p.kind == kRowWarpKernel) return launch_stream_kernel(rowwarp_gemv_kernel<kBF16, false>, a, p, dev, stream);
    switch (m) {
        case 1: return launch_stream_kernel(stream_gemv_kernel<1, kBF16, false>, a, p, dev, stream);
        case 2: return launch_stream_kernel(stream_gemv_kernel<2, kBF16, false>, a, p, dev, stream);
        case 3: return launch_stream_kernel(stream_gemv_kernel<3, kBF16, false>, a, p, dev, stream);
        case 4: return launch_stream_kernel(stream_gemv_kernel<4, kBF16, false>, a, p, dev, stream);
        case 5: return launch_stream_kernel(stream_gemv_kernel<5, kBF16, false>, a, p, dev, stream);
        case 6: return launch_stream_kernel(stream_gemv_kernel<6, kBF16, false>, a, p, dev, stream);
        case 7: return launch_stream_kernel(stream_gemv_kernel<7, kBF16, false>, a, p, dev, stream);
        case 8: return launch_stream_kernel(stream_gemv_kernel<8, kBF16, false>, a, p, dev, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fp8blk
