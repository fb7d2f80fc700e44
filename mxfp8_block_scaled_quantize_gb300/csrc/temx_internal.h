// Private interface between the C ABI (api.cu) and the kernel launchers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/temx.h"

namespace temx {

struct QuantizeArgs {
    const void* x;
    int64_t rows, cols, ld_x;
    uint8_t* q_row;
    uint8_t* s_row;
    int64_t ld_s_row;
    uint8_t* q_col;
    uint8_t* s_col;
    int64_t ld_s_col;
    uint16_t* dbias;         // bf16 [cols] or null (no bias gradient)
    float* partial;          // fp32 [ceil(rows/64) x cols] band sums (with dbias)
};

constexpr int64_t kDbiasBandRows = 64;     // rows per partial column sum

struct GemmArgs {
    const uint8_t* A;        // dense: [M x K]; grouped: X [total_m x K]
    const uint8_t* sA;
    int64_t ld_sA;
    const uint8_t* B;        // dense: [N x K]; grouped: W [G x N x K]
    const uint8_t* sB;
    int64_t ld_sB;
    int64_t M, N, K;         // grouped: M = total_m
    const void* bias;        // bf16 [N] (grouped: [G x N]) or null
    bool has_bias, gelu, dgelu;
    bool acc_f32;            // D is fp32 in/out: D = D + A B^T (no bias / GELU)
    void* D;
    void* aux;
    int32_t groups;          // 0: dense GEMM
    const int32_t* group_m;  // device int32 [groups] (grouped only)
    // Grouped wgrad (dW_e = dY_e^T X_e): A = column-wise dY [M x ld_code], B =
    // column-wise X [N x ld_code] in the per-expert padded layout, group_m the
    // experts' token counts, D = [groups x M x N]; K is unused.
    bool wgrad;
    int64_t ld_code;         // code row pitch (token capacity)
    int64_t total_m;         // bound on the sum of the token counts
    // Float8BlockScaling with FP32 scales (dense): sA [M x ld_sA] and sB
    // [N x ld_sB] fp32, one scale per row and 128 K (pitches in elements);
    // b_2d: sB constant over 128-row blocks (128x128 weight blocks).
    bool f32_scales;
    bool b_2d;
};

te_mx_status quantize_launch(const QuantizeArgs& a, cudaStream_t stream);

struct LnQuantizeArgs {
    const void* x;           // bf16 [rows x hidden], pitch ld_x
    int64_t rows, hidden, ld_x;
    const void* gamma;       // bf16 [hidden]
    const void* beta;        // bf16 [hidden]
    float eps;
    uint8_t* q_row; uint8_t* s_row; int64_t ld_s_row;
    uint8_t* q_col; uint8_t* s_col; int64_t ld_s_col;
    float* mu;               // fp32 [rows]
    float* rsigma;           // fp32 [rows]
};
te_mx_status ln_quantize_launch(const LnQuantizeArgs& a, cudaStream_t stream);

struct GroupedColwiseArgs {
    const void* x;           // bf16 [total_m x cols], pitch ld_x (token-major)
    int64_t total_m, cols, ld_x;
    int32_t groups;
    const int32_t* group_m;  // device int32 [groups]
    uint8_t* q;              // [cols x ld_q]
    int64_t ld_q;
    uint8_t* s;              // [cols x ld_s]
    int64_t ld_s;
};
te_mx_status grouped_colwise_launch(const GroupedColwiseArgs& a, cudaStream_t stream);
int64_t grouped_code_width(int64_t total_m, int32_t groups);    // an upper bound of sum round_up(m_e, 128)
int64_t grouped_scale_width(int64_t total_m, int32_t groups);   // an upper bound of sum round_up(Kp_e / 32, 16)
int64_t ln_quantize_max_hidden();
// Float8BlockScaling quantisation; `partial`/`dbias` unused.  fp32_scales:
// s_row / s_col hold fp32 scales (pitches in elements), else E8M0 bytes.
te_mx_status block_quantize_launch(const QuantizeArgs& a, bool block_2d, bool fp32_scales, cudaStream_t stream);
te_mx_status gemm_launch(const GemmArgs& a, cudaStream_t stream);

// Helpers implemented in api.cu.
// Raise a kernel's dynamic shared memory limit to `bytes` on the current
// device, once per (kernel, device); later calls return at once.
cudaError_t set_smem_attribute_once(const void* kernel, int bytes);
te_mx_status set_error(te_mx_status st, const char* fmt, ...);
void clear_error();
// Host-side argument checks of te_mx_quantize (+ the current device's arch).
te_mx_status validate_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                               uint8_t* q_row, uint8_t* s_row, int64_t ld_s_row,
                               uint8_t* q_col, uint8_t* s_col, int64_t ld_s_col, bool dbias);
te_mx_status cuda_status(cudaError_t e, const char* what);
te_mx_status device_sm_count(int* sms);
te_mx_status device_status_ptr(unsigned int** ptr);   // this device's status word
te_mx_status encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                                  uint64_t dim0, uint64_t dim1, uint64_t stride1_bytes,
                                  uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle);
te_mx_status encode_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                                  uint64_t dim0, uint64_t dim1, uint64_t dim2,
                                  uint64_t stride1_bytes, uint64_t stride2_bytes,
                                  uint32_t box0, uint32_t box1, uint32_t box2,
                                  CUtensorMapSwizzle swizzle);

}  // namespace temx
