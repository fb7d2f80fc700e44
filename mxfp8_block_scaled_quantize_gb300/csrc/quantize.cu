// MXFP8 quantiser: bf16 -> E4M3 codes + E8M0 block scales, row-wise and
// column-wise (transposed) in one pass over HBM.
//
// Definition (MXFP8 1D scaling, "HipKittens MXFP8 GEMM Support" PR review;
// OCP MX v1.0 FP32 -> MX conversion): for each block of 32 elements,
//   s = max(exponent_field(amax) - 8, 0)       (= floor(log2 amax) - 8 + 127,
//                                                clamped at 2^-127; 0 for amax 0)
//   q = E4M3_rn_satfinite(x * 2^(127 - s))
// and a block holding NaN/inf gets s = 0xFF, q = 0x7F.
//
// Work decomposition.  The input is cut into units of 32 rows x 64 columns
// (4 KB of bf16).  Every warp runs its own pipeline: lane 0 keeps
// kStages units in flight with TMA (128-byte swizzle, so both the row reads
// and the column reads below are bank-conflict free), and the warp consumes
// them in order.  Per unit:
//   row-wise:    lane r owns row r: two 32-element blocks, 2 x 32 bytes of
//                codes and 2 scale bytes;
//   column-wise: lane l owns columns 2l, 2l+1: one 32-row block each, stored
//                as 32 contiguous bytes of the transposed copy plus one scale
//                byte each.
// Warps never wait on each other, so there is no CTA-wide barrier.
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "temx_internal.h"

namespace temx {

namespace {

constexpr int kRows = 32;                    // unit height (= one column-wise block)
constexpr int kCols = 64;                    // unit width in bf16 (= 128-byte swizzle row)
constexpr int kUnitBytes = kRows * kCols * 2;
constexpr int kWarps = 16;
constexpr int kStages = 3;
constexpr int kSmemBytes = kWarps * kStages * kUnitBytes + 1024;

struct QuantizeParams {
    int64_t rows, cols;
    uint8_t* q_row;
    uint8_t* s_row;
    int64_t ld_s_row;
    uint8_t* q_col;
    uint8_t* s_col;
    int64_t ld_s_col;
    int64_t col_units;     // ceil(cols / 64)
    int64_t units;         // ceil(rows / 32) * col_units
    unsigned int* status;  // device status word
};

// E8M0 byte from |amax| as bf16 bits: exponent field - 8, floored at 0;
// 0xFF for NaN/inf.
__device__ __forceinline__ uint32_t scale_byte(uint32_t amax_bits) {
    const uint32_t ef = amax_bits >> 7;
    if (ef == 0xFFu) return 0xFFu;
    return ef > 8u ? ef - 8u : 0u;
}

// 2^(127 - s) as fp32 (s <= 246 for finite blocks, so always a normal number).
__device__ __forceinline__ float inv_scale(uint32_t s) {
    return __uint_as_float((254u - s) << 23);
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Two fp32 -> two E4M3 bytes (round to nearest even, saturate): `lo` in the
// low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Four consecutive bf16 (two words) -> four E4M3 bytes in one word.
__device__ __forceinline__ uint32_t quant4(uint32_t w0, uint32_t w1, float m) {
    const uint32_t a = cvt_e4m3x2(__fmul_rn(bf16_lo(w0), m), __fmul_rn(bf16_hi(w0), m));
    const uint32_t b = cvt_e4m3x2(__fmul_rn(bf16_lo(w1), m), __fmul_rn(bf16_hi(w1), m));
    return a | (b << 16);
}

// Row-wise blocks of one unit: lane = row within the unit.
__device__ __forceinline__ void unit_rowwise(const uint8_t* tile, int lane, int64_t r, int64_t c0,
                                             const QuantizeParams& p) {
    uint32_t w[32];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 v = *reinterpret_cast<const uint4*>(tile + lane * 128 + ((j ^ (lane & 7)) << 4));
        w[4 * j + 0] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
    }
    uint32_t sb[2];
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        uint32_t m2 = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) m2 = max_u16x2(m2, w[16 * blk + i] & 0x7FFF7FFFu);
        const uint32_t amax = max(m2 & 0xFFFFu, m2 >> 16);
        sb[blk] = scale_byte(amax);
        const float m = inv_scale(sb[blk]);
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = quant4(w[16 * blk + 2 * i], w[16 * blk + 2 * i + 1], m);
        if (sb[blk] == 0xFFu) {
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = 0x7F7F7F7Fu;
        }
        const int64_t c = c0 + 32 * blk;
        if (r < p.rows && c < p.cols) {
            uint8_t* dst = p.q_row + r * p.cols + c;
            st_global_v4(dst, o[0], o[1], o[2], o[3]);
            st_global_v4(dst + 16, o[4], o[5], o[6], o[7]);
        }
    }
    if (r < p.rows) {
        uint8_t* ds = p.s_row + r * p.ld_s_row + (c0 >> 5);
        if (c0 + 32 < p.cols) st_global_u16(ds, sb[0] | (sb[1] << 8));
        else st_global_u8(ds, sb[0]);
    }
}

// Column-wise blocks of one unit: lane l owns columns 2l and 2l+1.
__device__ __forceinline__ void unit_colwise(const uint8_t* tile, int lane, int64_t r0, int64_t c0,
                                             const QuantizeParams& p) {
    uint32_t w[32];
    const int chunk = lane >> 2, in_chunk = (lane & 3) << 2;
#pragma unroll
    for (int r = 0; r < 32; ++r)
        w[r] = *reinterpret_cast<const uint32_t*>(tile + r * 128 + ((chunk ^ (r & 7)) << 4) + in_chunk);
    uint32_t m2 = 0;
#pragma unroll
    for (int r = 0; r < 32; ++r) m2 = max_u16x2(m2, w[r] & 0x7FFF7FFFu);
    const uint32_t s_lo = scale_byte(m2 & 0xFFFFu), s_hi = scale_byte(m2 >> 16);
    const float m_lo = inv_scale(s_lo), m_hi = inv_scale(s_hi);
    uint32_t o_lo[8], o_hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t a0 = w[4 * i], a1 = w[4 * i + 1], a2 = w[4 * i + 2], a3 = w[4 * i + 3];
        o_lo[i] = cvt_e4m3x2(__fmul_rn(bf16_lo(a0), m_lo), __fmul_rn(bf16_lo(a1), m_lo)) |
                  (cvt_e4m3x2(__fmul_rn(bf16_lo(a2), m_lo), __fmul_rn(bf16_lo(a3), m_lo)) << 16);
        o_hi[i] = cvt_e4m3x2(__fmul_rn(bf16_hi(a0), m_hi), __fmul_rn(bf16_hi(a1), m_hi)) |
                  (cvt_e4m3x2(__fmul_rn(bf16_hi(a2), m_hi), __fmul_rn(bf16_hi(a3), m_hi)) << 16);
    }
    if (s_lo == 0xFFu) {
#pragma unroll
        for (int i = 0; i < 8; ++i) o_lo[i] = 0x7F7F7F7Fu;
    }
    if (s_hi == 0xFFu) {
#pragma unroll
        for (int i = 0; i < 8; ++i) o_hi[i] = 0x7F7F7F7Fu;
    }
    const int64_t c = c0 + 2 * lane;
    if (c < p.cols) {   // cols % 32 == 0, so c and c + 1 are valid together
        uint8_t* d0 = p.q_col + c * p.rows + r0;
        uint8_t* d1 = d0 + p.rows;
        st_global_v4(d0, o_lo[0], o_lo[1], o_lo[2], o_lo[3]);
        st_global_v4(d0 + 16, o_lo[4], o_lo[5], o_lo[6], o_lo[7]);
        st_global_v4(d1, o_hi[0], o_hi[1], o_hi[2], o_hi[3]);
        st_global_v4(d1 + 16, o_hi[4], o_hi[5], o_hi[6], o_hi[7]);
        uint8_t* s0 = p.s_col + c * p.ld_s_col + (r0 >> 5);
        st_global_u8(s0, s_lo);
        st_global_u8(s0 + p.ld_s_col, s_hi);
    }
}

template <bool kRowwise, bool kColwise>
__global__ void __launch_bounds__(kWarps * 32, 1)
quantize_kernel(const __grid_constant__ CUtensorMap x_map, const QuantizeParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[kWarps][kStages];

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t gwarp = int64_t(blockIdx.x) * kWarps + warp;
    const int64_t nwarps = int64_t(gridDim.x) * kWarps;
    if (gwarp >= p.units) return;
    const int64_t n_mine = (p.units - gwarp + nwarps - 1) / nwarps;
    uint8_t* ring = smem + warp * (kStages * kUnitBytes);

    if (lane == 0) {
        tma_prefetch_desc(&x_map);
        for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&bars[warp][s]), 1);
        fence_mbarrier_init();
        for (int s = 0; s < kStages && s < n_mine; ++s) {
            const int64_t u = gwarp + s * nwarps;
            const uint32_t bar = smem_u32(&bars[warp][s]);
            mbar_arrive_expect_tx(bar, kUnitBytes);
            tma_load_2d(smem_u32(ring + s * kUnitBytes), &x_map, bar,
                        int32_t((u % p.col_units) * kCols), int32_t((u / p.col_units) * kRows));
        }
    }
    __syncwarp();

    for (int64_t i = 0; i < n_mine; ++i) {
        const int s = int(i % kStages);
        const uint32_t parity = uint32_t((i / kStages) & 1);
        const uint32_t bar = smem_u32(&bars[warp][s]);
        if (!mbar_wait(bar, parity, p.status)) break;
        const uint8_t* tile = ring + s * kUnitBytes;
        const int64_t u = gwarp + i * nwarps;
        const int64_t r0 = (u / p.col_units) * kRows, c0 = (u % p.col_units) * kCols;
        if (kRowwise) unit_rowwise(tile, lane, r0 + lane, c0, p);
        if (kColwise) unit_colwise(tile, lane, r0, c0, p);
        __syncwarp();
        if (lane == 0 && i + kStages < n_mine) {
            fence_proxy_async_smem();          // our generic reads before the async refill
            const int64_t un = gwarp + (i + kStages) * nwarps;
            mbar_arrive_expect_tx(bar, kUnitBytes);
            tma_load_2d(smem_u32(ring + s * kUnitBytes), &x_map, bar,
                        int32_t((un % p.col_units) * kCols), int32_t((un / p.col_units) * kRows));
        }
    }
}

template <bool R, bool C>
cudaError_t launch(const CUtensorMap& map, const QuantizeParams& p, int sms, cudaStream_t stream) {
    auto k = quantize_kernel<R, C>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t want = (p.units + kWarps - 1) / kWarps;
    const int grid = int(want < sms ? want : sms);
    k<<<grid, kWarps * 32, kSmemBytes, stream>>>(map, p);
    return cudaGetLastError();
}

}  // namespace

te_mx_status quantize_launch(const QuantizeArgs& a, cudaStream_t stream) {
    const bool rowwise = a.q_row != nullptr, colwise = a.q_col != nullptr;
    if (a.rows == 0 || a.cols == 0 || (!rowwise && !colwise)) return TE_MX_OK;

    CUtensorMap map;
    te_mx_status st = encode_tensor_map_2d(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x,
                                           uint64_t(a.cols), uint64_t(a.rows), uint64_t(a.ld_x) * 2,
                                           kCols, kRows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != TE_MX_OK) return st;

    QuantizeParams p;
    p.rows = a.rows; p.cols = a.cols;
    p.q_row = a.q_row; p.s_row = a.s_row; p.ld_s_row = a.ld_s_row;
    p.q_col = a.q_col; p.s_col = a.s_col; p.ld_s_col = a.ld_s_col;
    p.col_units = (a.cols + kCols - 1) / kCols;
    p.units = ((a.rows + kRows - 1) / kRows) * p.col_units;
    st = device_status_ptr(&p.status);
    if (st != TE_MX_OK) return st;

    int sms = 0;
    st = device_sm_count(&sms);
    if (st != TE_MX_OK) return st;
    cudaError_t e;
    if (rowwise && colwise) e = launch<true, true>(map, p, sms, stream);
    else if (rowwise) e = launch<true, false>(map, p, sms, stream);
    else e = launch<false, true>(map, p, sms, stream);
    return cuda_status(e, "quantize kernel launch");
}

}  // namespace temx
