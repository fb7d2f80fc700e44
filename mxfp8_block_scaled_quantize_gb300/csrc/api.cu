// C ABI of libtemx.so: argument validation, device checks, tensor-map
// encoding and status reporting.  The kernels live in quantize.cu / gemm.cu.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "ptx.cuh"
#include "temx_internal.h"

namespace temx {

// Device status word: kernels record a bounded wait that gave up here.
__device__ unsigned int g_device_status = 0;

namespace {

// Failure-detection self-test: one thread waits on an mbarrier that never
// completes; the bounded wait gives up after `limit_ns` and records a timeout.
__global__ void selftest_timeout_kernel(unsigned int* status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbarrier_init();
    mbar_wait(b, 0, status, limit_ns);     // phase 0 never completes: nothing arrives
}

thread_local char t_last_error[512] = "";

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];     // 0 = not queried yet
int g_arch[kMaxDevices];         // major * 10 + minor
unsigned int* g_status_ptr[kMaxDevices];
std::mutex g_dev_mutex;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

te_mx_status get_encode(EncodeTiledFn* fn) {
    std::call_once(g_encode_once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                        cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!g_encode)
        return set_error(TE_MX_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)",
                         cudaGetErrorString(g_encode_err));
    *fn = g_encode;
    return TE_MX_OK;
}

// Current device must be sm_103 (the library is built for sm_103a only).
te_mx_status check_device(int* dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return set_error(TE_MX_ERR_CUDA, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_sm_count[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_status(e, "cudaDeviceGetAttribute");
        g_arch[dev] = major * 10 + minor;
        void* sp = nullptr;
        if (g_arch[dev] == 103 && (e = cudaGetSymbolAddress(&sp, g_device_status)) != cudaSuccess)
            return cuda_status(e, "cudaGetSymbolAddress(status word)");
        g_status_ptr[dev] = static_cast<unsigned int*>(sp);
        g_sm_count[dev] = sms;
    }
    if (g_arch[dev] != 103)
        return set_error(TE_MX_ERR_ARCH, "device %d is sm_%d; libtemx is built for sm_103a only", dev, g_arch[dev]);
    if (dev_out) *dev_out = dev;
    return TE_MX_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

te_mx_status set_error(te_mx_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
    return st;
}

void clear_error() { t_last_error[0] = '\0'; }

te_mx_status cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return TE_MX_OK;
    if (e == cudaErrorNoKernelImageForDevice)
        return set_error(TE_MX_ERR_ARCH, "%s: %s", what, cudaGetErrorString(e));
    return set_error(TE_MX_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

te_mx_status device_sm_count(int* sms) {
    int dev = 0;
    te_mx_status st = check_device(&dev);
    if (st != TE_MX_OK) return st;
    *sms = g_sm_count[dev];
    return TE_MX_OK;
}

te_mx_status device_status_ptr(unsigned int** ptr) {
    int dev = 0;
    te_mx_status st = check_device(&dev);
    if (st != TE_MX_OK) return st;
    *ptr = g_status_ptr[dev];
    return TE_MX_OK;
}

te_mx_status encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                                  uint64_t dim0, uint64_t dim1, uint64_t stride1_bytes,
                                  uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn;
    te_mx_status st = get_encode(&fn);
    if (st != TE_MX_OK) return st;
    const cuuint64_t dims[2] = {dim0, dim1};
    const cuuint64_t strides[1] = {stride1_bytes};
    const cuuint32_t box[2] = {box0, box1};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(TE_MX_ERR_CUDA, "cuTensorMapEncodeTiled(2d) failed with %d (dims %llu x %llu, stride %llu)",
                         int(r), (unsigned long long)dim0, (unsigned long long)dim1,
                         (unsigned long long)stride1_bytes);
    return TE_MX_OK;
}

te_mx_status encode_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                                  uint64_t dim0, uint64_t dim1, uint64_t dim2,
                                  uint64_t stride1_bytes, uint64_t stride2_bytes,
                                  uint32_t box0, uint32_t box1, uint32_t box2,
                                  CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn;
    te_mx_status st = get_encode(&fn);
    if (st != TE_MX_OK) return st;
    const cuuint64_t dims[3] = {dim0, dim1, dim2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {box0, box1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(TE_MX_ERR_CUDA, "cuTensorMapEncodeTiled(3d) failed with %d", int(r));
    return TE_MX_OK;
}

cudaError_t set_smem_attribute_once(const void* kernel, int bytes) {
    struct Entry { const void* fn; int dev; int bytes; };
    static Entry done[128];
    static int n_done = 0;
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
        if (done[i].fn == kernel && done[i].dev == dev && done[i].bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && n_done < 128) done[n_done++] = Entry{kernel, dev, bytes};
    return e;
}

te_mx_status validate_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                     uint8_t* q_row, uint8_t* s_row, int64_t ld_s_row,
                                     uint8_t* q_col, uint8_t* s_col, int64_t ld_s_col, bool dbias) {
    if (rows < 0 || cols < 0) return set_error(TE_MX_ERR_INVALID_ARG, "negative size %lld x %lld", (long long)rows, (long long)cols);
    if ((q_row == nullptr) != (s_row == nullptr))
        return set_error(TE_MX_ERR_INVALID_ARG, "q_row and s_row must both be given or both be NULL");
    if ((q_col == nullptr) != (s_col == nullptr))
        return set_error(TE_MX_ERR_INVALID_ARG, "q_col and s_col must both be given or both be NULL");
    if (rows == 0 || cols == 0 || (!q_row && !q_col && !dbias)) return TE_MX_OK;
    if (!x) return set_error(TE_MX_ERR_INVALID_ARG, "x is NULL");
    if (cols % 32) return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "cols=%lld is not a multiple of 32", (long long)cols);
    if (q_col && rows % 32)
        return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "column-wise output needs rows %% 32 == 0 (rows=%lld)", (long long)rows);
    if (rows > (int64_t(1) << 31) - 64 || cols > (int64_t(1) << 31) - 64)
        return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "a dimension exceeds 2^31 - 64");
    if (ld_x < cols || ld_x % 8) return set_error(TE_MX_ERR_MISALIGNED, "ld_x=%lld must be >= cols and a multiple of 8", (long long)ld_x);
    if (!aligned(x, 16)) return set_error(TE_MX_ERR_MISALIGNED, "x is not 16-byte aligned");
    if (q_row) {
        if (!aligned(q_row, 16)) return set_error(TE_MX_ERR_MISALIGNED, "q_row is not 16-byte aligned");
        if (ld_s_row % 16 || ld_s_row < cols / 32)
            return set_error(TE_MX_ERR_MISALIGNED, "ld_s_row=%lld must be a multiple of 16 and >= cols/32", (long long)ld_s_row);
    }
    if (q_col) {
        if (!aligned(q_col, 16)) return set_error(TE_MX_ERR_MISALIGNED, "q_col is not 16-byte aligned");
        if (ld_s_col % 16 || ld_s_col < rows / 32)
            return set_error(TE_MX_ERR_MISALIGNED, "ld_s_col=%lld must be a multiple of 16 and >= rows/32", (long long)ld_s_col);
    }
    return check_device(nullptr);
}

}  // namespace temx

using namespace temx;

extern "C" {

size_t te_mx_scale_pitch(int64_t k) {
    if (k <= 0) return 0;
    const int64_t blocks = (k + 31) / 32;
    return size_t((blocks + 15) / 16 * 16);
}

const char* te_mx_last_error(void) { return t_last_error; }

const char* te_mx_version(void) { return "temx 0.1 (sm_103a)"; }

te_mx_status te_mx_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                            uint8_t* q_row, uint8_t* s_row, int64_t ld_s_row,
                            uint8_t* q_col, uint8_t* s_col, int64_t ld_s_col, void* stream) {
    t_last_error[0] = '\0';
    te_mx_status st = validate_quantize(x, rows, cols, ld_x, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col, false);
    if (st != TE_MX_OK || rows == 0 || cols == 0 || (!q_row && !q_col)) return st;
    QuantizeArgs a{x, rows, cols, ld_x, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col, nullptr, nullptr};
    return quantize_launch(a, static_cast<cudaStream_t>(stream));
}

te_mx_status te_mx_block_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int32_t block_2d,
                                  uint8_t* q_row, uint8_t* s_row, int64_t ld_s_row,
                                  uint8_t* q_col, uint8_t* s_col, int64_t ld_s_col, void* stream) {
    t_last_error[0] = '\0';
    if (block_2d != 0 && block_2d != 1) return set_error(TE_MX_ERR_INVALID_ARG, "block_2d=%d must be 0 or 1", int(block_2d));
    te_mx_status st = validate_quantize(x, rows, cols, ld_x, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col, false);
    if (st != TE_MX_OK || rows == 0 || cols == 0 || (!q_row && !q_col)) return st;
    QuantizeArgs a{x, rows, cols, ld_x, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col, nullptr, nullptr};
    return block_quantize_launch(a, block_2d == 1, false, static_cast<cudaStream_t>(stream));
}

int64_t te_mx_block_scale_pitch_fp32(int64_t n) {
    if (n <= 0) return 0;
    return ((n + 127) / 128 + 3) / 4 * 4;
}

te_mx_status te_mx_block_quantize_fp32(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int32_t block_2d,
                                       uint8_t* q_row, float* s_row, int64_t ld_s_row,
                                       uint8_t* q_col, float* s_col, int64_t ld_s_col, void* stream) {
    t_last_error[0] = '\0';
    if (block_2d != 0 && block_2d != 1) return set_error(TE_MX_ERR_INVALID_ARG, "block_2d=%d must be 0 or 1", int(block_2d));
    // the code / shape / device checks of te_mx_quantize (MX scale pitches that pass stand in for the fp32 ones)
    uint8_t* sr = reinterpret_cast<uint8_t*>(s_row);
    uint8_t* sc = reinterpret_cast<uint8_t*>(s_col);
    if (rows > 0 && cols > 0) {
        if (q_row && s_row) {
            if (!aligned(s_row, 16)) return set_error(TE_MX_ERR_MISALIGNED, "s_row is not 16-byte aligned");
            if (ld_s_row % 4 || ld_s_row < (cols + 127) / 128)
                return set_error(TE_MX_ERR_MISALIGNED, "ld_s_row=%lld must be a multiple of 4 and >= ceil(cols/128)",
                                 (long long)ld_s_row);
        }
        if (q_col && s_col) {
            if (!aligned(s_col, 16)) return set_error(TE_MX_ERR_MISALIGNED, "s_col is not 16-byte aligned");
            if (ld_s_col % 4 || ld_s_col < (rows + 127) / 128)
                return set_error(TE_MX_ERR_MISALIGNED, "ld_s_col=%lld must be a multiple of 4 and >= ceil(rows/128)",
                                 (long long)ld_s_col);
        }
    }
    te_mx_status st = validate_quantize(x, rows, cols, ld_x, q_row, sr, int64_t(te_mx_scale_pitch(cols)), q_col, sc,
                                        int64_t(te_mx_scale_pitch(rows)), false);
    if (st != TE_MX_OK || rows == 0 || cols == 0 || (!q_row && !q_col)) return st;
    QuantizeArgs a{x, rows, cols, ld_x, q_row, sr, ld_s_row, q_col, sc, ld_s_col, nullptr, nullptr};
    return block_quantize_launch(a, block_2d == 1, true, static_cast<cudaStream_t>(stream));
}

te_mx_status te_mx_layernorm_quantize(const void* x, int64_t rows, int64_t hidden, int64_t ld_x,
                                      const void* gamma, const void* beta, float eps,
                                      uint8_t* q_row, uint8_t* s_row, int64_t ld_s_row,
                                      uint8_t* q_col, uint8_t* s_col, int64_t ld_s_col,
                                      float* mu, float* rsigma, void* stream) {
    t_last_error[0] = '\0';
    const bool work = rows > 0 && hidden > 0;
    if (work) {
        if (!gamma || !beta) return set_error(TE_MX_ERR_INVALID_ARG, "gamma and beta are required");
        if (!mu || !rsigma) return set_error(TE_MX_ERR_INVALID_ARG, "mu and rsigma are required");
        if (!(eps > 0.0f) || !std::isfinite(eps))
            return set_error(TE_MX_ERR_INVALID_ARG, "eps must be positive and finite");
        if (hidden > ln_quantize_max_hidden())
            return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "hidden=%lld exceeds %lld", (long long)hidden,
                             (long long)ln_quantize_max_hidden());
        if (!aligned(gamma, 4) || !aligned(beta, 4))
            return set_error(TE_MX_ERR_MISALIGNED, "gamma/beta not 4-byte aligned");
        if (!aligned(mu, 4) || !aligned(rsigma, 4)) return set_error(TE_MX_ERR_MISALIGNED, "mu/rsigma not 4-byte aligned");
    }
    te_mx_status st = validate_quantize(x, rows, hidden, ld_x, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col, true);
    if (st != TE_MX_OK || !work) return st;
    LnQuantizeArgs a{x, rows, hidden, ld_x, gamma, beta, eps, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col,
                     mu, rsigma};
    return ln_quantize_launch(a, static_cast<cudaStream_t>(stream));
}

int64_t te_mx_grouped_code_width(int64_t total_m, int32_t num_groups) {
    if (total_m < 0 || num_groups < 0) return 0;
    return grouped_code_width(total_m, num_groups);
}

int64_t te_mx_grouped_scale_width(int64_t total_m, int32_t num_groups) {
    if (total_m < 0 || num_groups < 0) return 0;
    const int64_t w = grouped_scale_width(total_m, num_groups);
    return w < 16 ? 16 : w;
}

te_mx_status te_mx_quantize_colwise_grouped(const void* x, int64_t total_m, int64_t cols, int64_t ld_x,
                                            int32_t num_groups, const int32_t* group_m,
                                            uint8_t* q, int64_t ld_q, uint8_t* s, int64_t ld_s, void* stream) {
    t_last_error[0] = '\0';
    if (num_groups < 1 || num_groups > 1024)
        return set_error(TE_MX_ERR_INVALID_ARG, "num_groups=%d must be in [1, 1024]", int(num_groups));
    if (!group_m || !q || !s) return set_error(TE_MX_ERR_INVALID_ARG, "group_m, q and s are required");
    if (total_m < 0 || cols < 0) return set_error(TE_MX_ERR_INVALID_ARG, "negative size");
    if (cols % 32) return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "cols=%lld is not a multiple of 32", (long long)cols);
    if (total_m > (int64_t(1) << 31) - 1024 || cols > (int64_t(1) << 31) - 64)
        return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "a dimension exceeds 2^31");
    if (ld_q % 16 || ld_q <= 0 || ld_s % 16 || ld_s <= 0)
        return set_error(TE_MX_ERR_MISALIGNED, "ld_q=%lld and ld_s=%lld must be positive multiples of 16",
                         (long long)ld_q, (long long)ld_s);
    if (cols == 0) return check_device(nullptr);
    if (total_m > 0 && (!x || ld_x < cols || ld_x % 8 || !aligned(x, 16)))
        return set_error(TE_MX_ERR_MISALIGNED, "x must be 16-byte aligned with ld_x >= cols, ld_x %% 8 == 0");
    if (!aligned(q, 16)) return set_error(TE_MX_ERR_MISALIGNED, "q is not 16-byte aligned");
    te_mx_status st = check_device(nullptr);
    if (st != TE_MX_OK) return st;
    GroupedColwiseArgs a{x, total_m, cols, ld_x > 0 ? ld_x : cols, num_groups, group_m, q, ld_q, s, ld_s};
    return grouped_colwise_launch(a, static_cast<cudaStream_t>(stream));
}

te_mx_status te_mx_grouped_gemm_wgrad(int32_t num_groups, const int32_t* group_m, int64_t total_m,
                                      const uint8_t* dY, const uint8_t* s_dY, const uint8_t* X, const uint8_t* s_X,
                                      int64_t M, int64_t N, int64_t ld_q, int64_t ld_s, int32_t accumulate,
                                      void* D, void* stream) {
    t_last_error[0] = '\0';
    if (num_groups < 1 || num_groups > 1024)
        return set_error(TE_MX_ERR_INVALID_ARG, "num_groups=%d must be in [1, 1024]", int(num_groups));
    if (!group_m || !dY || !s_dY || !X || !s_X || !D)
        return set_error(TE_MX_ERR_INVALID_ARG, "group_m, dY, s_dY, X, s_X and D are required");
    if (accumulate != 0 && accumulate != 1) return set_error(TE_MX_ERR_INVALID_ARG, "accumulate must be 0 or 1");
    if (total_m < 0 || M < 0 || N < 0) return set_error(TE_MX_ERR_INVALID_ARG, "negative size");
    if (N % 16) return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "N=%lld is not a multiple of 16", (long long)N);
    if (int64_t(num_groups) * M >= (int64_t(1) << 31) || N > (int64_t(1) << 31) - 256)
        return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "num_groups * M or N exceeds 2^31");
    if (ld_q % 16 || ld_q <= 0 || ld_s % 16 || ld_s < 16)
        return set_error(TE_MX_ERR_MISALIGNED, "ld_q=%lld must be a positive multiple of 16 and ld_s=%lld a "
                         "multiple of 16 >= 16", (long long)ld_q, (long long)ld_s);
    if (!aligned(dY, 16) || !aligned(X, 16) || !aligned(D, 16))
        return set_error(TE_MX_ERR_MISALIGNED, "dY, X and D must be 16-byte aligned");
    te_mx_status st = check_device(nullptr);
    if (st != TE_MX_OK || M == 0 || N == 0) return st;
    GemmArgs a{};
    a.A = dY; a.sA = s_dY; a.ld_sA = ld_s;
    a.B = X; a.sB = s_X; a.ld_sB = ld_s;
    a.M = M; a.N = N; a.K = 0;
    a.D = D;
    a.groups = num_groups;
    a.group_m = group_m;
    a.wgrad = true;
    a.acc_f32 = accumulate == 1;
    a.ld_code = ld_q;
    a.total_m = total_m;
    return gemm_launch(a, static_cast<cudaStream_t>(stream));
}

size_t te_mx_quantize_dbias_workspace_size(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    return size_t((rows + kDbiasBandRows - 1) / kDbiasBandRows) * size_t(cols) * sizeof(float);
}

te_mx_status te_mx_quantize_dbias(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                  uint8_t* q_row, uint8_t* s_row, int64_t ld_s_row,
                                  uint8_t* q_col, uint8_t* s_col, int64_t ld_s_col,
                                  void* dbias, void* workspace, size_t workspace_bytes, void* stream) {
    clear_error();
    if (!dbias) return set_error(TE_MX_ERR_INVALID_ARG, "dbias is NULL");
    te_mx_status st = validate_quantize(x, rows, cols, ld_x, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col, true);
    if (st != TE_MX_OK || rows == 0 || cols == 0) return st;
    if (!aligned(dbias, 16)) return set_error(TE_MX_ERR_MISALIGNED, "dbias is not 16-byte aligned");
    const size_t need = te_mx_quantize_dbias_workspace_size(rows, cols);
    if (!workspace || workspace_bytes < need)
        return set_error(TE_MX_ERR_WORKSPACE_TOO_SMALL, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
    if (!aligned(workspace, 16)) return set_error(TE_MX_ERR_MISALIGNED, "workspace is not 16-byte aligned");
    QuantizeArgs a{x, rows, cols, ld_x, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col,
                   static_cast<uint16_t*>(dbias), static_cast<float*>(workspace)};
    return quantize_launch(a, static_cast<cudaStream_t>(stream));
}

static te_mx_status validate_gemm_common(const uint8_t* A, const uint8_t* sA, int64_t ld_sA,
                                         const uint8_t* B, const uint8_t* sB, int64_t ld_sB,
                                         int64_t N, int64_t K, const void* bias, int32_t epi,
                                         void* D, void* aux) {
    if (epi < TE_MX_EPI_NONE || epi > TE_MX_EPI_ACCUMULATE_F32)
        return set_error(TE_MX_ERR_INVALID_ARG, "unknown epilogue %d", epi);
    if (epi == TE_MX_EPI_ACCUMULATE_F32 && (bias || aux))
        return set_error(TE_MX_ERR_INVALID_ARG, "the accumulating epilogue takes no bias and no aux");
    if (!A || !sA || !B || !sB || !D) return set_error(TE_MX_ERR_INVALID_ARG, "A, sA, B, sB and D are required");
    const bool has_bias = epi == TE_MX_EPI_BIAS || epi == TE_MX_EPI_BIAS_GELU_AUX;
    const bool gelu = epi == TE_MX_EPI_GELU_AUX || epi == TE_MX_EPI_BIAS_GELU_AUX || epi == TE_MX_EPI_DGELU;
    if (has_bias && !bias) return set_error(TE_MX_ERR_INVALID_ARG, "bias epilogue without a bias pointer");
    if (gelu && !aux) return set_error(TE_MX_ERR_INVALID_ARG, "GELU epilogue without an aux pointer");
    if (epi == TE_MX_EPI_DGELU && bias) return set_error(TE_MX_ERR_INVALID_ARG, "DGELU epilogue takes no bias");
    if (K < 128 || K % 128) return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "K=%lld must be a positive multiple of 128", (long long)K);
    if (N < 16 || N % 16) return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "N=%lld must be a positive multiple of 16", (long long)N);
    if (K > (int64_t(1) << 30) || N > (int64_t(1) << 30)) return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "N or K too large");
    if (ld_sA % 16 || ld_sA < K / 32 || ld_sB % 16 || ld_sB < K / 32)
        return set_error(TE_MX_ERR_MISALIGNED, "scale pitches must be multiples of 16 and >= K/32");
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sA, 16) || !aligned(sB, 16) || !aligned(D, 16) ||
        (gelu && !aligned(aux, 16)) || (has_bias && !aligned(bias, 16)))
        return set_error(TE_MX_ERR_MISALIGNED, "A, B, sA, sB, D, aux and bias must be 16-byte aligned");
    return TE_MX_OK;
}

te_mx_status te_mx_gemm(const uint8_t* A, const uint8_t* sA, int64_t ld_sA,
                        const uint8_t* B, const uint8_t* sB, int64_t ld_sB,
                        int64_t M, int64_t N, int64_t K, const void* bias, int32_t epilogue,
                        void* D, void* aux, void* workspace, size_t workspace_bytes, void* stream) {
    (void)workspace; (void)workspace_bytes;
    t_last_error[0] = '\0';
    if (M < 0) return set_error(TE_MX_ERR_INVALID_ARG, "negative M");
    if (M == 0) return TE_MX_OK;
    if (M > (int64_t(1) << 31) - 256) return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "M too large");
    te_mx_status st = validate_gemm_common(A, sA, ld_sA, B, sB, ld_sB, N, K, bias, epilogue, D, aux);
    if (st != TE_MX_OK) return st;
    if ((st = check_device(nullptr)) != TE_MX_OK) return st;
    GemmArgs a{};
    a.A = A; a.sA = sA; a.ld_sA = ld_sA; a.B = B; a.sB = sB; a.ld_sB = ld_sB;
    a.M = M; a.N = N; a.K = K; a.bias = bias;
    a.has_bias = epilogue == TE_MX_EPI_BIAS || epilogue == TE_MX_EPI_BIAS_GELU_AUX;
    a.gelu = epilogue == TE_MX_EPI_GELU_AUX || epilogue == TE_MX_EPI_BIAS_GELU_AUX;
    a.dgelu = epilogue == TE_MX_EPI_DGELU;
    a.acc_f32 = epilogue == TE_MX_EPI_ACCUMULATE_F32;
    a.D = D; a.aux = aux; a.groups = 0; a.group_m = nullptr;
    return gemm_launch(a, static_cast<cudaStream_t>(stream));
}

te_mx_status te_mx_gemm_fp32_scales(const uint8_t* A, const float* sA, int64_t ld_sA,
                                    const uint8_t* B, const float* sB, int64_t ld_sB, int32_t b_blocks_2d,
                                    int64_t M, int64_t N, int64_t K, const void* bias, int32_t epilogue,
                                    void* D, void* aux, void* stream) {
    t_last_error[0] = '\0';
    if (M < 0) return set_error(TE_MX_ERR_INVALID_ARG, "negative M");
    if (M == 0) return TE_MX_OK;
    if (M > (int64_t(1) << 31) - 256) return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "M too large");
    if (b_blocks_2d != 0 && b_blocks_2d != 1)
        return set_error(TE_MX_ERR_INVALID_ARG, "b_blocks_2d=%d must be 0 or 1", int(b_blocks_2d));
    if (epilogue == TE_MX_EPI_ACCUMULATE_F32)
        return set_error(TE_MX_ERR_INVALID_ARG, "the accumulating epilogue is not offered with FP32 scales");
    // the MX checks with stand-in scale pitches, then the FP32 scale rules
    const int64_t mx_pitch = int64_t(te_mx_scale_pitch(K));
    te_mx_status st = validate_gemm_common(A, reinterpret_cast<const uint8_t*>(sA), mx_pitch, B,
                                           reinterpret_cast<const uint8_t*>(sB), mx_pitch, N, K, bias, epilogue, D, aux);
    if (st != TE_MX_OK) return st;
    if (ld_sA % 4 || ld_sA < K / 128 || ld_sB % 4 || ld_sB < K / 128)
        return set_error(TE_MX_ERR_MISALIGNED, "FP32 scale pitches must be multiples of 4 and >= K/128");
    if ((st = check_device(nullptr)) != TE_MX_OK) return st;
    GemmArgs a{};
    a.A = A; a.sA = reinterpret_cast<const uint8_t*>(sA); a.ld_sA = ld_sA;
    a.B = B; a.sB = reinterpret_cast<const uint8_t*>(sB); a.ld_sB = ld_sB;
    a.M = M; a.N = N; a.K = K; a.bias = bias;
    a.has_bias = epilogue == TE_MX_EPI_BIAS || epilogue == TE_MX_EPI_BIAS_GELU_AUX;
    a.gelu = epilogue == TE_MX_EPI_GELU_AUX || epilogue == TE_MX_EPI_BIAS_GELU_AUX;
    a.dgelu = epilogue == TE_MX_EPI_DGELU;
    a.D = D; a.aux = aux; a.groups = 0; a.group_m = nullptr;
    a.f32_scales = true;
    a.b_2d = b_blocks_2d == 1;
    return gemm_launch(a, static_cast<cudaStream_t>(stream));
}

te_mx_status te_mx_grouped_gemm(int32_t num_groups, const int32_t* group_m, int64_t total_m,
                                const uint8_t* X, const uint8_t* sX, int64_t ld_sX,
                                const uint8_t* W, const uint8_t* sW, int64_t ld_sW,
                                int64_t N, int64_t K, const void* bias, int32_t epilogue,
                                void* D, void* aux, void* workspace, size_t workspace_bytes,
                                void* stream) {
    (void)workspace; (void)workspace_bytes;
    t_last_error[0] = '\0';
    if (num_groups < 1 || num_groups > 1024) return set_error(TE_MX_ERR_INVALID_ARG, "num_groups=%d must be in [1, 1024]", num_groups);
    if (!group_m) return set_error(TE_MX_ERR_INVALID_ARG, "group_m is NULL");
    if (!aligned(group_m, 4)) return set_error(TE_MX_ERR_MISALIGNED, "group_m is not 4-byte aligned");
    if (total_m < 0) return set_error(TE_MX_ERR_INVALID_ARG, "negative total_m");
    if (total_m == 0) return TE_MX_OK;
    if (total_m > (int64_t(1) << 31) - 256) return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "total_m too large");
    if (epilogue == TE_MX_EPI_ACCUMULATE_F32)
        return set_error(TE_MX_ERR_INVALID_ARG, "the accumulating epilogue is for te_mx_gemm and the wgrad GEMM");
    te_mx_status st = validate_gemm_common(X, sX, ld_sX, W, sW, ld_sW, N, K, bias, epilogue, D, aux);
    if (st != TE_MX_OK) return st;
    if (int64_t(num_groups) * N > (int64_t(1) << 31) - 256) return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "G*N too large");
    if ((st = check_device(nullptr)) != TE_MX_OK) return st;
    GemmArgs a{};
    a.A = X; a.sA = sX; a.ld_sA = ld_sX; a.B = W; a.sB = sW; a.ld_sB = ld_sW;
    a.M = total_m; a.N = N; a.K = K; a.bias = bias;
    a.has_bias = epilogue == TE_MX_EPI_BIAS || epilogue == TE_MX_EPI_BIAS_GELU_AUX;
    a.gelu = epilogue == TE_MX_EPI_GELU_AUX || epilogue == TE_MX_EPI_BIAS_GELU_AUX;
    a.dgelu = epilogue == TE_MX_EPI_DGELU;
    a.D = D; a.aux = aux; a.groups = num_groups; a.group_m = group_m;
    return gemm_launch(a, static_cast<cudaStream_t>(stream));
}

size_t te_mx_gemm_workspace_size(int64_t, int64_t, int64_t, int32_t) { return 0; }

te_mx_status te_mx_selftest_timeout(uint32_t limit_us, void* stream) {
    t_last_error[0] = '\0';
    if (limit_us < 1 || limit_us > 2000000u)
        return set_error(TE_MX_ERR_INVALID_ARG, "limit_us=%u must be in [1, 2000000]", limit_us);
    unsigned int* status = nullptr;
    te_mx_status st = device_status_ptr(&status);
    if (st != TE_MX_OK) return st;
    selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        status, static_cast<unsigned long long>(limit_us) * 1000ull);
    return cuda_status(cudaGetLastError(), "selftest kernel launch");
}

te_mx_status te_mx_device_status(void) {
    t_last_error[0] = '\0';
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_status(e, "cudaDeviceSynchronize");
    unsigned int v = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v));
    if (e != cudaSuccess) return cuda_status(e, "reading the device status word");
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_status(e, "clearing the device status word");
    if (v == kStatusTimeout) return set_error(TE_MX_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait");
    if (v == kStatusBadArg) return set_error(TE_MX_ERR_INVALID_ARG, "a kernel rejected device-side arguments (group sizes)");
    return TE_MX_OK;
}

}  // extern "C"
