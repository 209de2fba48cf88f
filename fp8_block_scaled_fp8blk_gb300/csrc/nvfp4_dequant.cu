// nvfp4_dequant.cu -- one NVFP4 routed expert to bf16, exactly:
//   out[r][c] = bf16( e2m1(q[r][c]) * e4m3(s[r][c/16]) * g ).
// Source: "Module dsv4_gpu" page, module header and enum ExpertArm: routed
// experts stay NVFP4 as stored; each activated expert is dequantised into a
// reused bf16 scratch, exact in bf16.  Layout readings: two codes per byte,
// column 2j in the low nibble; one e4m3 scale per 16 consecutive columns.
//
// The product e2m1 * (e4m3 * g) has at most 6 significant bits; with g a power
// of two in [2^-100, 2^100] (checked on the host) every step is exact in f32
// and the result is a bf16 value, so the final round-to-nearest is exact.
#include "launch.h"

namespace fp8blk {

__global__ void __launch_bounds__(256) nvfp4_dequant_kernel(const uint8_t *__restrict__ codes,
                                                            const uint8_t *__restrict__ scales,
                                                            float g, uint16_t *__restrict__ out,
                                                            int64_t rows, int64_t cols) {
    // The scratch may still be read by the previous grid (the GEMV of the
    // previous expert): wait before writing it.
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t groups_per_row = cols / 32;  // 32 columns = 16 code bytes, 2 scales
    const int64_t total = rows * groups_per_row;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += stride) {
        const int64_t r = t / groups_per_row;
        const int64_t q = t - r * groups_per_row;
        const uint4 c = __ldcs(reinterpret_cast<const uint4 *>(codes + r * (cols / 2) + q * 16));
        const uint16_t sc = __ldcs(reinterpret_cast<const unsigned short *>(scales + r * (cols / 16) + q * 2));
        float2 s = e4m3x2_to_f32(sc);
        s.x *= g;
        s.y *= g;
        const uint32_t words[4] = {c.x, c.y, c.z, c.w};
        uint4 *dst = reinterpret_cast<uint4 *>(out + r * cols + q * 32);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float sv = w < 2 ? s.x : s.y;
            uint32_t h[4];
            e2m1x8_to_f16x2(words[w], h);
            uint32_t o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h[k]));
                o[k] = pack_bf16x2(f.x * sv, f.y * sv);
            }
            dst[w] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

cudaError_t launch_nvfp4_dequant(const uint8_t *codes, const uint8_t *scales, float g,
                                 uint16_t *out, int64_t rows, int64_t cols,
                                 const DeviceInfo &dev, cudaStream_t stream) {
    const int64_t total = rows * (cols / 32);
    int64_t grid = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(dev.sms) * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = tuning().use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, nvfp4_dequant_kernel, codes, scales, g, out, rows, cols);
}

}  // namespace fp8blk
