// noalloc.cu -- fp8blk_gemv_argmax_noalloc: the fused GEMV + greedy argmax
// for callers that cannot allocate device memory.
//
// fp8blk_gemv_argmax needs a small caller-owned workspace (an arrival counter
// and per-CTA partial maxima).  Some callers have no way to provide one: code
// running while a CUDA graph is being captured (cudaMalloc is not allowed
// then), serving loops that must never call cudaMalloc/cudaFree because those
// calls synchronize the device, and plain C hosts or plugins that live inside
// another framework's memory manager and own no allocator of their own.  This
// entry point gives them the same computation with the workspace placed in a
// fixed-size array in the library's own device memory instead.
//
// The array below is a host-side stand-in in host code: kernels must be given
// its device address, which cudaGetSymbolAddress returns for the current
// device.  That lookup is done once per device, on the first call made with
// that device current.
#include <mutex>

#include "fp8blk.h"
#include "launch.h"

namespace {

// Counter (16 B) + 1024 CTAs x 8 rows x (f32 value + u32 index) = 65,552 B,
// rounded up to a multiple of 256.  Every GPU that loads the library holds it
// until the process exits.
constexpr size_t kNoAllocScratchBytes = 65792;
static_assert(kNoAllocScratchBytes % 256 == 0, "scratch size must stay 256-byte granular");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr size_t kCounterBytes = 16;

// Device address of g_noalloc_scratch on the current device, looked up once
// per device.  Returns cudaSuccess and sets *out, or the lookup's error.
cudaError_t scratch_address(unsigned char **out) {
    static std::mutex mu;
    static unsigned char *addr[128] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        unsigned char *ptr = nullptr;
        err = cudaGetSymbolAddress(reinterpret_cast<void **>(&ptr), g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        addr[dev] = ptr;
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" size_t fp8blk_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int fp8blk_gemv_argmax_noalloc(const uint8_t *w_codes, const float *scales,
                                          const float *x, float *logits, uint32_t *tokens, int m,
                                          int64_t rows, int64_t cols, void *stream) {
    if (!w_codes || !scales || !x || !tokens) return FP8BLK_EINVAL;
    if (m < 1 || m > FP8BLK_MAX_M || rows < 1 || cols < 16 || cols % 16 != 0) return FP8BLK_EINVAL;
    if (rows > (int64_t(1) << 31) - 1 || cols > (int64_t(1) << 31) - 1) return FP8BLK_ERANGE;
    // The workspace fp8blk_gemv_argmax asks for this shape (counter, per-CTA
    // partials, and a panel accumulator when rows are wider than one panel);
    // shapes that need more than the fixed array are refused.
    const size_t need = fp8blk_gemv_argmax_ws_bytes(m, rows, cols);
    if (need == 0) return FP8BLK_EINVAL;
    if (need > kNoAllocScratchBytes) return FP8BLK_ERANGE;
    unsigned char *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) {
        (void)cudaGetLastError();
        return FP8BLK_ECUDA;
    }
    // The array keeps the previous call's contents: the arrival counter must
    // start at zero, so clear it in stream order (no allocation involved).
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, kCounterBytes, s) != cudaSuccess) {
        (void)cudaGetLastError();
        return FP8BLK_ECUDA;
    }
    // Hand the scratch to the existing entry point as its workspace: `need`
    // is that entry point's own answer for this shape, at most the array.
    return fp8blk_gemv_argmax(w_codes, scales, x, logits, tokens, scratch, need, m, rows, cols, stream);
}
