// abi.cu -- the extern "C" entry points of libfp8blk (declared in fp8blk.h):
// host-side argument checks, launch planning, and the device status word.
// Nothing here allocates device memory or synchronizes, except
// fp8blk_device_status, which is documented to synchronize.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "fp8blk.h"
#include "launch.h"

// Device status word (FP8BLK_STATUS_* bits), one per device context.
__device__ unsigned int g_fp8blk_status = 0;

namespace fp8blk {

Tuning &tuning() {
    static Tuning t;
    return t;
}

cudaError_t current_device_info(DeviceInfo *out) {
    static std::mutex mu;
    static DeviceInfo cache[128];
    static bool have[128] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        DeviceInfo d;
        err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (err == cudaSuccess)
            err = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (err == cudaSuccess)
            err = cudaDeviceGetAttribute(&d.smem_per_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        void *status = nullptr;
        if (err == cudaSuccess) err = cudaGetSymbolAddress(&status, g_fp8blk_status);
        if (err != cudaSuccess) return err;
        d.status = static_cast<unsigned int *>(status);
        cache[dev] = d;
        have[dev] = true;
    }
    *out = cache[dev];
    return cudaSuccess;
}

cudaError_t kernel_occupancy(const void *kernel, int threads, size_t smem, int *per_sm) {
    // The dynamic-smem limit is one value per (kernel, device): only ever
    // raise it, so a smaller request never undercuts a cached larger one.
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, size_t> limit;
    static std::map<std::tuple<const void *, int, size_t>, int> cache;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(mu);
    size_t &lim = limit[std::make_pair(kernel, dev)];
    if (smem > lim) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (err != cudaSuccess) return err;
        lim = smem;
    }
    const auto key = std::make_tuple(kernel, dev, smem);
    auto it = cache.find(key);
    if (it != cache.end()) {
        *per_sm = it->second;
        return cudaSuccess;
    }
    int n = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem);
    if (err != cudaSuccess) return err;
    cache[key] = n;
    *per_sm = n;
    return cudaSuccess;
}

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
}  // namespace

static EncodeTiledFn encode_tiled_fn(cudaError_t *err) {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        *err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
        if (*err == cudaSuccess && (!f || q != cudaDriverEntryPointSuccess)) *err = cudaErrorNotSupported;
        if (*err != cudaSuccess) return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    *err = cudaSuccess;
    return fn;
}

namespace {
struct MapEntry {
    const void *ptr;
    int64_t rows, cols;
    int box_rows, box_cols, dtype, swizzle;
    CUtensorMap map;
};
std::mutex g_map_mu;
MapEntry g_maps[128];
int g_map_next = 0;

// Encodes (or finds) a 2-D tensor map of a rows x cols row-major array whose
// rows are row_bytes apart.
cudaError_t tensor_map_2d(const void *ptr, int64_t rows, int64_t cols, int64_t row_bytes, CUtensorMapDataType dtype,
                          int box_rows, int box_cols, CUtensorMapSwizzle swizzle, CUtensorMap *out) {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (const MapEntry &e : g_maps)
        if (e.ptr == ptr && e.rows == rows && e.cols == cols && e.box_rows == box_rows && e.box_cols == box_cols &&
            e.dtype == static_cast<int>(dtype) && e.swizzle == static_cast<int>(swizzle)) {
            *out = e.map;
            return cudaSuccess;
        }
    cudaError_t err;
    EncodeTiledFn fn = encode_tiled_fn(&err);
    if (!fn) return err;
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = fn(&map, dtype, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    g_maps[g_map_next] = MapEntry{ptr, rows, cols, box_rows, box_cols, static_cast<int>(dtype), static_cast<int>(swizzle), map};
    g_map_next = (g_map_next + 1) % 128;
    *out = map;
    return cudaSuccess;
}
}  // namespace

cudaError_t weight_tensor_map(const uint8_t *w, int64_t rows, int64_t cols, int box_rows, CUtensorMap *out) {
    return tensor_map_2d(w, rows, cols, cols, CU_TENSOR_MAP_DATA_TYPE_UINT8, box_rows, kT8Kb, CU_TENSOR_MAP_SWIZZLE_128B,
                         out);
}

cudaError_t nvfp4_tensor_maps(const uint8_t *codes, const uint8_t *scales, int64_t total_rows, int64_t cols,
                              int scale_block, int box_rows, CUtensorMap *cmap, CUtensorMap *smap) {
    const cudaError_t err = tensor_map_2d(codes, total_rows, cols, cols / 2, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B,
                                          box_rows, 128, CU_TENSOR_MAP_SWIZZLE_128B, cmap);
    if (err != cudaSuccess) return err;
    return tensor_map_2d(scales, total_rows, cols / scale_block, cols / scale_block, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                         box_rows, 16, CU_TENSOR_MAP_SWIZZLE_NONE, smap);
}

static int pow2_floor(int v) {
    int p = 1;
    while (2 * p <= v) p *= 2;
    return p;
}

Plan make_plan(int m, int64_t rows, int64_t cols, int bpw, const DeviceInfo &dev) {
    const Tuning &t = tuning();
    Plan p;
    const int mp = pow2_ceil(m);
    const int rt = 8 / mp;
    // Column panels of at most kMaxPanelCols, equal widths rounded to 16.
    const int64_t panels0 = (cols + kMaxPanelCols - 1) / kMaxPanelCols;
    const int64_t per = (cols + panels0 - 1) / panels0;
    p.panel_cols = static_cast<int>((per + 15) / 16 * 16);
    p.panels = static_cast<int>((cols + p.panel_cols - 1) / p.panel_cols);
    const int64_t tc_bytes = t.tc_min_bytes > 0 ? t.tc_min_bytes : tc_default_min_bytes(m);
    // m = 1 forced onto a CUDA-core kernel (fp8blk_set_m1_kernel) skips the tensor cores.
    const bool m1_forced = m == 1 && t.m1_kernel != 0;
    if (bpw == 1 && !m1_forced && t.tc_min_m <= FP8BLK_MAX_M && m >= t.tc_min_m && cols >= kT8Kb &&
        cols <= static_cast<int64_t>(kT8MaxKb) * kT8Kb && rows * cols >= tc_bytes) {
        // Tensor-core kernel: one CTA per SM over whole 128-row tiles (one
        // scale row block each), every K-block of a row in one pass.
        p.kind = kTensorCoreKernel;
        p.panels = 1;
        p.panel_cols = static_cast<int>(cols);
        p.team_warps_log2 = 0;
        p.rb = 1;
        p.stage_rows = 128;
        p.stage_bytes = kT8StageBytes;
        p.stages = kT8Stages;
        p.ctas_per_sm = 1;
        p.n_groups = (rows + 127) / 128;
        return p;
    }
    const bool use_rowwarp =
        m == 1 && (t.m1_kernel == 1 ||
                   (t.m1_kernel == 0 && rows * cols * bpw >= t.m1_rowwarp_min_bytes));
    if (use_rowwarp) {
        // Row-per-warp kernel: each warp streams whole panel rows through a
        // private ring; stages of about target/4 bytes, shrunk while there
        // are fewer row groups than warps.
        p.kind = kRowWarpKernel;
        p.team_warps_log2 = 0;
        p.rb = 1;
        p.ctas_per_sm = t.ctas_per_sm > 0 ? t.ctas_per_sm : 2;
        const int panel_bytes = p.panel_cols * bpw;
        int rw = pow2_floor(std::max(1, (t.target_stage_bytes / 4) / panel_bytes));
        if (rw > 8) rw = 8;
        const int64_t warps = static_cast<int64_t>(dev.sms) * p.ctas_per_sm * kRowWarps;
        while (rw > 1 && (rows + rw - 1) / rw < warps) rw /= 2;
        int per_warp = 0;
        for (;;) {  // fewer CTAs per SM until two one-row stages per warp fit
            per_warp = dev.smem_per_sm / p.ctas_per_sm - 1024 - kStaticSmemReserve;
            const int block_cap = dev.smem_per_block - kStaticSmemReserve;
            if (per_warp > block_cap) per_warp = block_cap;
            per_warp /= kRowWarps;
            if (2 * panel_bytes <= per_warp || p.ctas_per_sm == 1) break;
            --p.ctas_per_sm;
        }
        while (rw > 1 && 2 * rw * panel_bytes > per_warp) rw /= 2;
        p.stage_rows = rw;
        p.stage_bytes = rw * panel_bytes;
        int stages = per_warp / p.stage_bytes;
        if (stages > t.max_stages) stages = t.max_stages;
        if (stages > kMaxStages) stages = kMaxStages;
        if (stages < 2) stages = 2;
        p.stages = stages;
        p.n_groups = (rows + rw - 1) / rw;
        return p;
    }
    // One thread per 16 columns; a team is the power-of-two warp count that
    // covers a panel row; the CTA's 8 warps form 8 / team_warps teams.
    const int need_threads = (p.panel_cols + 15) / 16;
    int team_warps = pow2_ceil((need_threads + 31) / 32);
    if (team_warps > kWarps) team_warps = kWarps;
    p.team_warps_log2 = ilog2(team_warps);
    const int teams = kWarps / team_warps;
    const int panel_bytes = p.panel_cols * bpw;
    p.ctas_per_sm = t.ctas_per_sm > 0 ? t.ctas_per_sm : (m <= 4 ? 2 : 1);
    for (;;) {
        int budget = dev.smem_per_sm / p.ctas_per_sm - 1024 - kStaticSmemReserve;
        const int block_cap = dev.smem_per_block - kStaticSmemReserve;
        if (budget > block_cap) budget = block_cap;
        budget -= kMaxStages * static_cast<int>(sizeof(uint64_t));
        int rb = t.target_stage_bytes / (teams * rt * panel_bytes);
        if (rb < 1) rb = 1;
        if (rb > kMaxRowBatches) rb = kMaxRowBatches;
        rb = pow2_floor(rb);
        while (rb > 1 && teams * rb * rt > 128) rb /= 2;
        while (rb > 1 && 2 * teams * rb * rt * panel_bytes > budget) rb /= 2;
        const int stage_bytes = teams * rb * rt * panel_bytes;
        if (2 * stage_bytes > budget && p.ctas_per_sm > 1) {
            --p.ctas_per_sm;
            continue;
        }
        p.rb = rb;
        p.stage_rows = teams * rb * rt;
        p.stage_bytes = stage_bytes;
        int stages = budget / stage_bytes;
        if (stages > t.max_stages) stages = t.max_stages;
        if (stages > kMaxStages) stages = kMaxStages;
        if (stages < 2) stages = 2;
        p.stages = stages;
        break;
    }
    p.n_groups = (rows + p.stage_rows - 1) / p.stage_rows;
    return p;
}

void apply_plan(const Plan &p, GemvArgs *a) {
    a->n_groups = p.n_groups;
    a->panels = p.panels;
    a->panel_cols = p.panel_cols;
    a->team_warps_log2 = p.team_warps_log2;
    a->rb = p.rb;
    a->stages = p.stages;
    a->stage_bytes = p.stage_bytes;
    a->stage_rows = p.stage_rows;
    a->l2_prefetch = tuning().l2_prefetch;
    a->wait_limit_ns = tuning().wait_limit_ns;
}

}  // namespace fp8blk

using namespace fp8blk;

namespace {

constexpr int64_t kMaxIndex = (int64_t(1) << 31) - 1;

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return FP8BLK_OK;
    (void)cudaGetLastError();  // do not leave a non-sticky launch error behind
    return FP8BLK_ECUDA;
}

int check_gemv_shape(int m, int64_t rows, int64_t cols) {
    if (m < 1 || m > FP8BLK_MAX_M || rows < 1 || cols < 16 || cols % 16 != 0) return FP8BLK_EINVAL;
    if (rows > kMaxIndex || cols > kMaxIndex) return FP8BLK_ERANGE;
    return FP8BLK_OK;
}

// A finite nonzero power of two in [2^-100, 2^100]: every NVFP4 product is
// then exact in f32 and bf16.
bool exact_global_scale(float g) {
    if (!std::isfinite(g) || g == 0.0f) return false;
    int e = 0;
    const float f = std::frexp(std::fabs(g), &e);
    return f == 0.5f && e - 1 >= -100 && e - 1 <= 100;
}

size_t argmax_ws_layout(int m, int64_t rows, int64_t cols, size_t *part_val_off,
                        size_t *part_idx_off, size_t *acc_off) {
    const size_t pv = 16;
    const size_t pi = pv + static_cast<size_t>(kMaxGrid) * m * sizeof(float);
    const size_t acc = pi + static_cast<size_t>(kMaxGrid) * m * sizeof(uint32_t);
    size_t total = acc;
    if (cols > kMaxPanelCols) total += static_cast<size_t>(m) * static_cast<size_t>(rows) * sizeof(float);
    if (part_val_off) *part_val_off = pv;
    if (part_idx_off) *part_idx_off = pi;
    if (acc_off) *acc_off = acc;
    return (total + 15) / 16 * 16;
}

}  // namespace

extern "C" {

int fp8blk_abi_version(void) { return 1; }

const char *fp8blk_strerror(int code) {
    switch (code) {
        case FP8BLK_OK: return "ok";
        case FP8BLK_EINVAL: return "invalid argument";
        case FP8BLK_EALIGN: return "misaligned pointer";
        case FP8BLK_ESCALE: return "refused scale (e8m0 0xFF or inexact NVFP4 global scale)";
        case FP8BLK_EWS: return "workspace missing or too small";
        case FP8BLK_ECUDA: return "CUDA runtime error";
        case FP8BLK_ERANGE: return "size out of supported range";
        default: return "unknown error";
    }
}

int fp8blk_scales_from_e8m0(const uint8_t *codes, size_t n, float *out, size_t *bad_index) {
    if (n == 0) return FP8BLK_OK;
    if (!codes || !out) return FP8BLK_EINVAL;
    for (size_t k = 0; k < n; ++k) {
        const int c = codes[k];
        if (c == 0xFF) {
            if (bad_index) *bad_index = k;
            return FP8BLK_ESCALE;
        }
        out[k] = std::ldexp(1.0f, c - 127);
    }
    return FP8BLK_OK;
}

int fp8blk_gemv(const uint8_t *w_codes, const float *scales, const float *x, float *y, int m,
                int64_t rows, int64_t cols, void *stream) {
    if (!w_codes || !scales || !x || !y) return FP8BLK_EINVAL;
    int rc = check_gemv_shape(m, rows, cols);
    if (rc != FP8BLK_OK) return rc;
    if (!aligned(w_codes, 16) || !aligned(x, 16) || !aligned(scales, 4) || !aligned(y, 4))
        return FP8BLK_EALIGN;
    DeviceInfo dev;
    if (current_device_info(&dev) != cudaSuccess) return from_cuda(cudaErrorUnknown);
    const Plan p = make_plan(m, rows, cols, 1, dev);
    GemvArgs a = {};
    a.w = w_codes;
    a.scales = scales;
    a.x = x;
    a.y = y;
    a.status = dev.status;
    a.rows = rows;
    a.cols = cols;
    apply_plan(p, &a);
    return from_cuda(launch_gemv_e4m3(a, p, m, false, dev, static_cast<cudaStream_t>(stream)));
}

size_t fp8blk_gemv_argmax_ws_bytes(int m, int64_t rows, int64_t cols) {
    if (check_gemv_shape(m, rows, cols) != FP8BLK_OK) return 0;
    return argmax_ws_layout(m, rows, cols, nullptr, nullptr, nullptr);
}

int fp8blk_gemv_argmax(const uint8_t *w_codes, const float *scales, const float *x,
                       float *logits, uint32_t *tokens, void *ws, size_t ws_bytes, int m,
                       int64_t rows, int64_t cols, void *stream) {
    if (!w_codes || !scales || !x || !tokens) return FP8BLK_EINVAL;
    int rc = check_gemv_shape(m, rows, cols);
    if (rc != FP8BLK_OK) return rc;
    if (!aligned(w_codes, 16) || !aligned(x, 16) || !aligned(scales, 4) || !aligned(tokens, 4) ||
        (logits && !aligned(logits, 4)))
        return FP8BLK_EALIGN;
    size_t pv_off = 0, pi_off = 0, acc_off = 0;
    const size_t need = argmax_ws_layout(m, rows, cols, &pv_off, &pi_off, &acc_off);
    if (!ws || ws_bytes < need) return FP8BLK_EWS;
    if (!aligned(ws, 16)) return FP8BLK_EALIGN;
    DeviceInfo dev;
    if (current_device_info(&dev) != cudaSuccess) return from_cuda(cudaErrorUnknown);
    const Plan p = make_plan(m, rows, cols, 1, dev);
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    GemvArgs a = {};
    a.w = w_codes;
    a.scales = scales;
    a.x = x;
    a.y = logits ? logits : (p.panels > 1 ? reinterpret_cast<float *>(wsb + acc_off) : nullptr);
    a.tokens = tokens;
    a.counter = reinterpret_cast<uint32_t *>(wsb);
    a.part_val = reinterpret_cast<float *>(wsb + pv_off);
    a.part_idx = reinterpret_cast<uint32_t *>(wsb + pi_off);
    a.status = dev.status;
    a.rows = rows;
    a.cols = cols;
    apply_plan(p, &a);
    return from_cuda(launch_gemv_e4m3(a, p, m, true, dev, static_cast<cudaStream_t>(stream)));
}

int fp8blk_bf16_gemv(const uint16_t *w_bf16, const float *x, float *y, int m, int64_t rows,
                     int64_t cols, void *stream) {
    if (!w_bf16 || !x || !y) return FP8BLK_EINVAL;
    int rc = check_gemv_shape(m, rows, cols);
    if (rc != FP8BLK_OK) return rc;
    if (!aligned(w_bf16, 16) || !aligned(x, 16) || !aligned(y, 4)) return FP8BLK_EALIGN;
    DeviceInfo dev;
    if (current_device_info(&dev) != cudaSuccess) return from_cuda(cudaErrorUnknown);
    const Plan p = make_plan(m, rows, cols, 2, dev);
    GemvArgs a = {};
    a.w = reinterpret_cast<const uint8_t *>(w_bf16);
    a.x = x;
    a.y = y;
    a.status = dev.status;
    a.rows = rows;
    a.cols = cols;
    apply_plan(p, &a);
    return from_cuda(launch_gemv_bf16(a, p, m, dev, static_cast<cudaStream_t>(stream)));
}

static int check_nvfp4(const uint8_t *codes, const uint8_t *scales, const float *gscale_host,
                       int n_experts, int64_t rows, int64_t cols) {
    if (!codes || !scales || !gscale_host || n_experts < 1) return FP8BLK_EINVAL;
    if (rows < 1 || cols < 32 || cols % 32 != 0) return FP8BLK_EINVAL;
    if (rows > kMaxIndex || cols > kMaxIndex) return FP8BLK_ERANGE;
    if (!aligned(codes, 16) || !aligned(scales, 2)) return FP8BLK_EALIGN;
    return FP8BLK_OK;
}

int nvfp4_expert_dequant(const uint8_t *codes, const uint8_t *scales, const float *gscale_host,
                         int n_experts, int expert_id, uint16_t *out, int64_t rows, int64_t cols,
                         void *stream) {
    int rc = check_nvfp4(codes, scales, gscale_host, n_experts, rows, cols);
    if (rc != FP8BLK_OK) return rc;
    if (!out || expert_id < 0 || expert_id >= n_experts) return FP8BLK_EINVAL;
    if (!aligned(out, 16)) return FP8BLK_EALIGN;
    const float g = gscale_host[expert_id];
    if (!exact_global_scale(g)) return FP8BLK_ESCALE;
    DeviceInfo dev;
    if (current_device_info(&dev) != cudaSuccess) return from_cuda(cudaErrorUnknown);
    const int64_t e = expert_id;
    return from_cuda(launch_nvfp4_dequant(codes + e * rows * (cols / 2), scales + e * rows * (cols / 16),
                                          g, out, rows, cols, dev, static_cast<cudaStream_t>(stream)));
}

int nvfp4_expert_dequant_gemv(const uint8_t *codes, const uint8_t *scales,
                              const float *gscale_host, int n_experts, const int32_t *ids_host,
                              int n_active, const float *x, float *y, uint16_t *bf16_scratch,
                              int64_t rows, int64_t cols, void *stream) {
    int rc = check_nvfp4(codes, scales, gscale_host, n_experts, rows, cols);
    if (rc != FP8BLK_OK) return rc;
    if (!ids_host || n_active < 1 || n_active > n_experts || !x || !y || !bf16_scratch)
        return FP8BLK_EINVAL;
    if (!aligned(x, 16) || !aligned(y, 4) || !aligned(bf16_scratch, 16)) return FP8BLK_EALIGN;
    for (int k = 0; k < n_active; ++k) {
        const int e = ids_host[k];
        if (e < 0 || e >= n_experts) return FP8BLK_EINVAL;
        for (int q = 0; q < k; ++q)
            if (ids_host[q] == e) return FP8BLK_EINVAL;
        if (!exact_global_scale(gscale_host[e])) return FP8BLK_ESCALE;
    }
    DeviceInfo dev;
    if (current_device_info(&dev) != cudaSuccess) return from_cuda(cudaErrorUnknown);
    const Plan p = make_plan(1, rows, cols, 2, dev);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int k = 0; k < n_active; ++k) {
        const int64_t e = ids_host[k];
        cudaError_t err = launch_nvfp4_dequant(codes + e * rows * (cols / 2), scales + e * rows * (cols / 16),
                                               gscale_host[e], bf16_scratch, rows, cols, dev, s);
        if (err != cudaSuccess) return from_cuda(err);
        GemvArgs a = {};
        a.w = reinterpret_cast<const uint8_t *>(bf16_scratch);
        a.x = x;
        a.y = y + k * rows;
        a.status = dev.status;
        a.rows = rows;
        a.cols = cols;
        apply_plan(p, &a);
        err = launch_gemv_bf16(a, p, 1, dev, s);
        if (err != cudaSuccess) return from_cuda(err);
    }
    return FP8BLK_OK;
}

int nvfp4_expert_gemv(const uint8_t *codes, const uint8_t *scales, const float *gscale, int n_experts,
                      const int32_t *ids, int n_active, const float *x, float *y, int64_t rows, int64_t cols,
                      void *stream) {
    if (!codes || !scales || !gscale || !ids || !x || !y || n_experts < 1) return FP8BLK_EINVAL;
    if (n_active < 1 || n_active > 65536 || rows < 1 || cols < 256 || cols % 256 != 0) return FP8BLK_EINVAL;
    if (rows > kMaxIndex || cols > kMaxIndex) return FP8BLK_ERANGE;
    if (!aligned(codes, 16) || !aligned(scales, 16) || !aligned(gscale, 4) || !aligned(ids, 4) || !aligned(x, 16) ||
        !aligned(y, 4))
        return FP8BLK_EALIGN;
    DeviceInfo dev;
    if (current_device_info(&dev) != cudaSuccess) return from_cuda(cudaErrorUnknown);
    Nvfp4Args a = {};
    a.codes = codes;
    a.scales = scales;
    a.gscale = gscale;
    a.ids = ids;
    a.x = x;
    a.y = y;
    a.status = dev.status;
    a.n_experts = n_experts;
    a.n_active = n_active;
    a.rows = rows;
    a.cols = cols;
    a.wait_limit_ns = tuning().wait_limit_ns;
    return from_cuda(launch_fp4_expert_gemv(a, false, dev, static_cast<cudaStream_t>(stream)));
}

int mxfp4_expert_gemv(const uint8_t *codes, const uint8_t *scales, int n_experts, const int32_t *ids,
                      int n_active, const float *x, float *y, int64_t rows, int64_t cols, void *stream) {
    if (!codes || !scales || !ids || !x || !y || n_experts < 1) return FP8BLK_EINVAL;
    if (n_active < 1 || n_active > 65536 || rows < 1 || cols < 512 || cols % 512 != 0) return FP8BLK_EINVAL;
    if (rows > kMaxIndex || cols > kMaxIndex) return FP8BLK_ERANGE;
    if (!aligned(codes, 16) || !aligned(scales, 16) || !aligned(ids, 4) || !aligned(x, 16) || !aligned(y, 4))
        return FP8BLK_EALIGN;
    DeviceInfo dev;
    if (current_device_info(&dev) != cudaSuccess) return from_cuda(cudaErrorUnknown);
    Nvfp4Args a = {};
    a.codes = codes;
    a.scales = scales;
    a.ids = ids;
    a.x = x;
    a.y = y;
    a.status = dev.status;
    a.n_experts = n_experts;
    a.n_active = n_active;
    a.rows = rows;
    a.cols = cols;
    a.wait_limit_ns = tuning().wait_limit_ns;
    return from_cuda(launch_fp4_expert_gemv(a, true, dev, static_cast<cudaStream_t>(stream)));
}

int fp8blk_set_launch_tuning(int target_stage_bytes, int ctas_per_sm, int use_pdl, int l2_prefetch,
                             int max_stages) {
    if (target_stage_bytes < 0 || ctas_per_sm < 0 || ctas_per_sm > 4 || max_stages < 0 ||
        max_stages == 1 || max_stages > kMaxStages)
        return FP8BLK_EINVAL;
    Tuning &t = tuning();
    t.target_stage_bytes = target_stage_bytes ? target_stage_bytes : 32 * 1024;
    t.ctas_per_sm = ctas_per_sm;
    t.use_pdl = use_pdl != 0;
    t.l2_prefetch = l2_prefetch != 0;
    t.max_stages = max_stages ? max_stages : kMaxStages;
    return FP8BLK_OK;
}

int fp8blk_set_wait_limit(int64_t limit_ns) {
    if (limit_ns < 0 || limit_ns > FP8BLK_WAIT_LIMIT_DEFAULT_NS) return FP8BLK_EINVAL;
    tuning().wait_limit_ns = static_cast<uint64_t>(limit_ns);
    return FP8BLK_OK;
}

int fp8blk_set_tensor_core_min_m(int min_m, int64_t min_bytes) {
    if (min_m != 0 && (min_m < 1 || min_m > FP8BLK_MAX_M + 1)) return FP8BLK_EINVAL;
    if (min_bytes < 0) return FP8BLK_EINVAL;
    tuning().tc_min_m = min_m == 0 ? Tuning().tc_min_m : min_m;
    tuning().tc_min_bytes = min_bytes == 0 ? Tuning().tc_min_bytes : min_bytes;
    return FP8BLK_OK;
}

int fp8blk_set_fp4_kernel(int choice) {
    if (choice < 0 || choice > 2) return FP8BLK_EINVAL;
    tuning().fp4_kernel = choice;
    return FP8BLK_OK;
}

int fp8blk_set_m1_kernel(int choice, int64_t rowwarp_min_bytes) {
    if (choice < 0 || choice > 2 || rowwarp_min_bytes < 0) return FP8BLK_EINVAL;
    tuning().m1_kernel = choice;
    tuning().m1_rowwarp_min_bytes = rowwarp_min_bytes ? rowwarp_min_bytes : (96ll << 20);
    return FP8BLK_OK;
}

int fp8blk_plan_query(int m, int64_t rows, int64_t cols, int bytes_per_weight, int sms,
                      int smem_per_sm, int smem_per_block, int64_t *out) {
    if (!out || (bytes_per_weight != 1 && bytes_per_weight != 2) || sms < 1 ||
        smem_per_sm < 64 * 1024 || smem_per_block < 64 * 1024)
        return FP8BLK_EINVAL;
    const int rc = check_gemv_shape(m, rows, cols);
    if (rc != FP8BLK_OK) return rc;
    DeviceInfo dev;
    dev.sms = sms;
    dev.smem_per_sm = smem_per_sm;
    dev.smem_per_block = smem_per_block;
    const Plan p = make_plan(m, rows, cols, bytes_per_weight, dev);
    const int team_warps = 1 << p.team_warps_log2;
    out[0] = p.panels;
    out[1] = p.panel_cols;
    out[2] = p.kind == kTeamKernel ? team_warps : 1;
    out[3] = p.kind == kRowWarpKernel ? kRowWarps : (p.kind == kTensorCoreKernel ? kT8BWarps : kWarps / team_warps);
    out[4] = p.rb;
    out[5] = p.kind == kTeamKernel ? 8 / pow2_ceil(m) : 1;
    out[6] = p.stage_rows;
    out[7] = p.stage_bytes;
    out[8] = p.stages;
    out[9] = p.ctas_per_sm;
    out[10] = p.n_groups;
    out[11] = static_cast<int64_t>(plan_smem_bytes(p));
    out[12] = p.kind;
    return FP8BLK_OK;
}

int fp8blk_device_status(uint32_t *status_out, int clear) {
    if (!status_out) return FP8BLK_EINVAL;
    cudaError_t err = cudaDeviceSynchronize();
    unsigned int v = 0;
    if (err == cudaSuccess) err = cudaMemcpyFromSymbol(&v, g_fp8blk_status, sizeof(v));
    if (err == cudaSuccess && clear) {
        const unsigned int zero = 0;
        err = cudaMemcpyToSymbol(g_fp8blk_status, &zero, sizeof(zero));
    }
    if (err != cudaSuccess) return from_cuda(err);
    *status_out = v;
    return FP8BLK_OK;
}

}  // extern "C"
