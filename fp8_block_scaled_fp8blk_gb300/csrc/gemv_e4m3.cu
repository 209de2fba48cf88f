// gemv_e4m3.cu -- instantiations of the streaming GEMV for e4m3 weights with
// 128x128 f32 block scales, m = 1..8, with and without the fused argmax.
#include "launch.h"

namespace fp8blk {

template <int M>
static cudaError_t launch_m(const GemvArgs &a, const Plan &p, bool argmax, const DeviceInfo &dev,
                            cudaStream_t stream) {
    if (argmax) return launch_stream_kernel(stream_gemv_kernel<M, kE4M3, true>, a, p, dev, stream);
    return launch_stream_kernel(stream_gemv_kernel<M, kE4M3, false>, a, p, dev, stream);
}

cudaError_t launch_gemv_e4m3(const GemvArgs &a, const Plan &p, int m, bool argmax,
                             const DeviceInfo &dev, cudaStream_t stream) {
    if (p.kind == kTensorCoreKernel) return launch_gemv_tc(a, p, m, argmax, dev, stream);
    if (p.kind == kRowWarpKernel) {
        if (argmax) return launch_stream_kernel(rowwarp_gemv_kernel<kE4M3, true>, a, p, dev, stream);
        return launch_stream_kernel(rowwarp_gemv_kernel<kE4M3, false>, a, p, dev, stream);
    }
    switch (m) {
        case 1: return launch_m<1>(a, p, argmax, dev, stream);
        case 2: return launch_m<2>(a, p, argmax, dev, stream);
        case 3: return launch_m<3>(a, p, argmax, dev, stream);
        case 4: return launch_m<4>(a, p, argmax, dev, stream);
        case 5: return launch_m<5>(a, p, argmax, dev, stream);
        case 6: return launch_m<6>(a, p, argmax, dev, stream);
        case 7: return launch_m<7>(a, p, argmax, dev, stream);
        case 8: return launch_m<8>(a, p, argmax, dev, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fp8blk
