// Float8BlockScaling quantiser with E8M0-cast scales: bf16 -> E4M3 codes with
// one power-of-two scale per 1x128 / 128x1 block (activations, gradients) or
// per 128x128 block (weights).
//
// Definition ("Blockwise FP8 GEMM support on ROCm", ROCm/TransformerEngine
// README: 1Dx2D and 1Dx1D scaling; the recipe's FP32 scale amax/448 is cast
// to E8M0 by default).  The cast is the smallest power of two not below
// amax/448, so no element saturates:
//   e = ceil(log2(amax / 448)) clamped to [-127, 127] (-127 for amax 0),
//   q = E4M3_rn_satfinite(x * 2^-e),   scale byte = e + 127,
// and a block holding NaN/inf gets scale byte 0xFF and codes 0x7F.
//
// Output layout: the MX layout of the MXFP8 quantiser (one scale byte per 32
// elements along the quantised direction), the block's scale repeated over
// its 32-element groups.  The MXFP8 GEMM then computes the block-scaled GEMM
// with no change.
//
// The README's second mode keeps the FP32 scales (kF32): per block
//   s = fl32(amax / 448)  (stored, fp32),  r = min(fl32(1 / s), FLT_MAX),
//   q = E4M3_rn_satfinite(fl32(x * r)),
// s = r = 1 for amax 0, s = NaN and codes 0x7F for a non-finite block; one
// fp32 scale per block and row of each copy ([rows][ceil(cols / 128)] and
// [cols][ceil(rows / 128)], a 128x128 block's scale repeated over its rows).
//
// Work decomposition.  A CTA owns 128 x 128 tiles (two 64-column TMA boxes,
// 128-byte swizzle) in a kStages-deep ring.  Warp 8 is the producer: it loads
// tiles, and when the compute warps have staged a tile's codes it stores them
// with TMA and refills the stage.  Compute warp w reads box b = w & 1, rows
// 32 (w >> 1) .. +31:
//   row pass:    lane l reads the 64 elements of row 32 (w >> 1) + l in box b;
//   column pass: lane l reads columns 2l, 2l+1 of box b over the warp's 32 rows.
// Both keep their data in registers.  Partial maxima go to shared memory, a
// named barrier joins the eight compute warps, and each lane then combines the
// partials of its block, quantises, and writes the codes into the consumed
// tile (row codes over box 0, column codes over box 1).
#include <cuda_runtime.h>

#include "e4m3.cuh"
#include "ptx.cuh"
#include "temx_internal.h"

namespace temx {

namespace {

constexpr int kEdge = 128;                          // block edge: 1x128, 128x1 or 128x128 elements
constexpr int kBoxCols = 64;                        // TMA box width: 64 bf16 = one 128-byte swizzle row
constexpr int kBoxBytes = kEdge * kBoxCols * 2;     // 16 KB
constexpr int kTileBytes = 2 * kBoxBytes;           // 128 x 128 bf16
constexpr int kComputeWarps = 8;
constexpr int kThreads = (kComputeWarps + 1) * 32;
constexpr int kStages = 3;
constexpr int kCtasPerSm = 2;
constexpr int kSmemBytes = kStages * kTileBytes + 1024;

struct BlockParams {
    int64_t rows, cols;
    uint8_t* s_row;        // E8M0 bytes, or fp32 scales (kF32) at this address
    int64_t ld_s_row;      // bytes, or fp32 elements (kF32)
    uint8_t* s_col;
    int64_t ld_s_col;
    int64_t col_tiles;     // ceil(cols / 128)
    int64_t tiles;         // ceil(rows / 128) * col_tiles
    unsigned int* status;  // device status word
};

struct BlockShared {
    uint64_t full[kStages];                  // tile landed (TMA transaction count)
    uint64_t staged[kStages];                // the compute warps staged the tile's codes
    uint32_t row_amax[2][2][kEdge];          // [tile parity][box][row]: half-row maxima
    uint32_t col_amax[2][4][kBoxCols];       // [tile parity][row quarter][box * 32 + lane]: column-pair maxima
    uint32_t warp_amax[2][kComputeWarps];    // [tile parity][warp]: 128x128 block partials
    int abort;
};

// E8M0 byte of the block scale 2^ceil(log2(amax / 448)), from |amax| as bf16
// bits.  With amax = 1.m * 2^E: 448 * 2^(E-8) = 1.75 * 2^E covers amax unless
// m > 0.75 (mantissa field > 96), which needs one binade more.  Floored at
// 2^-127 (also for zero and subnormal amax); 0xFF for NaN/inf.
__device__ __forceinline__ uint32_t block_scale_byte(uint32_t amax_bits) {
    const uint32_t ef = amax_bits >> 7;
    if (ef == 0xFFu) return 0xFFu;
    const int e = int(ef) - 8 + ((amax_bits & 0x7Fu) > 96u ? 1 : 0);
    return e > 0 ? uint32_t(e) : 0u;
}

// A block's quantisation: multiplier m (x * m is rounded to E4M3), whether
// the block is non-finite, and what is stored (E8M0 byte, or fp32 scale s).
struct BlockScale {
    float m;
    bool bad;
    uint32_t byte;
    float s;
};
template <bool kF32>
__device__ __forceinline__ BlockScale block_scale(uint32_t amax_bits) {
    BlockScale b;
    if constexpr (kF32) {
        b.bad = (amax_bits >> 7) == 0xFFu;
        b.byte = 0;
        if (b.bad) {
            b.s = b.m = __uint_as_float(0x7FC00000u);
        } else if (amax_bits == 0) {
            b.s = b.m = 1.0f;
        } else {
            b.s = __fdiv_rn(__uint_as_float(amax_bits << 16), 448.0f);
            b.m = fminf(__frcp_rn(b.s), 3.40282347e38f);
        }
    } else {
        b.byte = block_scale_byte(amax_bits);
        b.bad = b.byte == 0xFFu;
        b.m = inv_scale(b.byte);
        b.s = 0.0f;
    }
    return b;
}

// The eight compute warps only (the producer warp does not take part).
__device__ __forceinline__ void compute_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kComputeWarps * 32) : "memory");
}

// `n` (1..4) copies of scale byte `sb` at `p`; one 32-bit store when aligned.
__device__ __forceinline__ void put_scales(uint8_t* p, uint32_t sb, int64_t n) {
    if (n >= 4 && (reinterpret_cast<uintptr_t>(p) & 3) == 0) {
        asm volatile("st.global.b32 [%0], %1;" ::"l"(p), "r"(sb * 0x01010101u) : "memory");
    } else {
        for (int64_t k = 0; k < n && k < 4; ++k) st_global_u8(p + k, sb);
    }
}

template <bool kRowwise, bool kColwise, bool k2d, bool kF32>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
block_quantize_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap qrow_map,
                      const __grid_constant__ CUtensorMap qcol_map, const BlockParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ BlockShared sh;

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n_mine = (p.tiles - blockIdx.x + gridDim.x - 1) / gridDim.x;   // grid <= tiles: >= 1
    volatile int* abort_flag = &sh.abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&sh.full[s]), 1);
            mbar_init(smem_u32(&sh.staged[s]), kComputeWarps);
        }
        sh.abort = 0;
        fence_mbarrier_init();
    }
    __syncthreads();

    auto tile_origin = [&](int64_t i, int32_t& r0, int32_t& c0) {
        const int64_t t = int64_t(blockIdx.x) + i * gridDim.x;
        r0 = int32_t((t / p.col_tiles) * kEdge);
        c0 = int32_t((t % p.col_tiles) * kEdge);
    };

    if (warp == kComputeWarps) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        tma_prefetch_desc(&x_map);
        if (kRowwise) tma_prefetch_desc(&qrow_map);
        if (kColwise) tma_prefetch_desc(&qcol_map);
        auto load = [&](int64_t i) {
            int32_t r0, c0;
            tile_origin(i, r0, c0);
            const int s = int(i % kStages);
            const uint32_t bar = smem_u32(&sh.full[s]);
            const uint32_t dst = ring + s * kTileBytes;
            mbar_arrive_expect_tx(bar, kTileBytes);          // out-of-range boxes still count in full
            tma_load_2d(dst, &x_map, bar, c0, r0);
            tma_load_2d(dst + kBoxBytes, &x_map, bar, c0 + kBoxCols, r0);
        };
        for (int64_t i = 0; i < kStages && i < n_mine; ++i) load(i);
        int64_t i = 0;
        for (; i < n_mine; ++i) {
            const int s = int(i % kStages);
            if (!mbar_wait(smem_u32(&sh.staged[s]), uint32_t((i / kStages) & 1), p.status) || *abort_flag) break;
            int32_t r0, c0;
            tile_origin(i, r0, c0);
            const uint32_t tile = ring + s * kTileBytes;
            if (kRowwise) tma_store_2d(&qrow_map, tile, c0, r0);
            if (kColwise) tma_store_2d(&qcol_map, tile + kBoxBytes, r0, c0);
            bulk_commit();
            if (i + kStages < n_mine) {
                bulk_wait_read_all();                          // the stores have read the stage: refill it
                load(i + kStages);
            }
        }
        if (i < n_mine) {
            // Gave up: let the loads still in flight land before the CTA exits.
            for (int64_t j = i; j < i + kStages && j < n_mine; ++j)
                mbar_wait(smem_u32(&sh.full[j % kStages]), uint32_t((j / kStages) & 1), p.status);
        }
        bulk_wait_all();
        return;
    }

    // ---------------------------------------------------------------- compute
    const int b = warp & 1, g = warp >> 1;
    const int row = 32 * g + lane;                     // tile row of the row pass
    for (int64_t i = 0; i < n_mine; ++i) {
        const int s = int(i % kStages);
        const int buf = int(i & 1);
        const bool ok = mbar_wait(smem_u32(&sh.full[s]), uint32_t((i / kStages) & 1), p.status);
        if (!ok) *abort_flag = 1;
        const uint32_t tile = ring + s * kTileBytes;
        const uint32_t box = tile + b * kBoxBytes;
        int32_t r0, c0;
        tile_origin(i, r0, c0);

        uint32_t wr[32], wc[32];
        uint32_t row_part = 0, col_part = 0;
        if (ok) {
            if (kRowwise || (k2d && !kColwise)) {
                const int sw = row & 7;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 v = lds128(box + row * 128 + ((j ^ sw) << 4));
                    wr[4 * j + 0] = v.x; wr[4 * j + 1] = v.y; wr[4 * j + 2] = v.z; wr[4 * j + 3] = v.w;
                }
                const uint32_t m2 = amax_words<32>(wr);
                row_part = max(m2 & 0xFFFFu, m2 >> 16);
            }
            if (kColwise) {
                const uint32_t base = box + (32 * g) * 128 + ((lane & 3) << 2);
                const int chunk = lane >> 2;
#pragma unroll
                for (int r = 0; r < 32; ++r) wc[r] = lds32(base + r * 128 + ((chunk ^ (r & 7)) << 4));
                col_part = amax_words<32>(wc);
            }
        }
        if (k2d) {
            uint32_t t = (kRowwise || !kColwise) ? row_part : max(col_part & 0xFFFFu, col_part >> 16);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) t = max(t, __shfl_xor_sync(0xFFFFFFFFu, t, o));
            if (lane == 0) sh.warp_amax[buf][warp] = t;
        } else {
            if (kRowwise) sh.row_amax[buf][b][row] = row_part;
            if (kColwise) sh.col_amax[buf][g][b * 32 + lane] = col_part;
        }
        compute_sync();                                // partials visible; every lane has read the tile
        if (*abort_flag) break;                        // the same decision in every compute warp

        uint32_t blk = 0;
        if (k2d) {
#pragma unroll
            for (int w = 0; w < kComputeWarps; ++w) blk = max(blk, sh.warp_amax[buf][w]);
        }
        if (kRowwise) {
            const uint32_t a = k2d ? blk : max(sh.row_amax[buf][0][row], sh.row_amax[buf][1][row]);
            const BlockScale bs = block_scale<kF32>(a);
            const int sw = row & 7;
#pragma unroll
            for (int j = 0; j < 4; ++j) {                // 16 codes per chunk, chunks 4b .. 4b+3 of the row
                uint32_t c[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) c[q] = quant4(wr[8 * j + 2 * q], wr[8 * j + 2 * q + 1], bs.m);
                if (bs.bad) c[0] = c[1] = c[2] = c[3] = 0x7F7F7F7Fu;
                sts128(tile + row * 128 + (((4 * b + j) ^ sw) << 4), c[0], c[1], c[2], c[3]);
            }
            const int64_t r = int64_t(r0) + row;
            if (b == 0 && r < p.rows) {
                if constexpr (kF32)
                    reinterpret_cast<float*>(p.s_row)[r * p.ld_s_row + c0 / kEdge] = bs.s;
                else
                    put_scales(p.s_row + r * p.ld_s_row + (c0 >> 5), bs.byte, (p.cols - c0) >> 5);
            }
        }
        if (kColwise) {
            uint32_t a2;
            if (k2d) {
                a2 = blk | (blk << 16);
            } else {
                a2 = max_u16x2(max_u16x2(sh.col_amax[buf][0][b * 32 + lane], sh.col_amax[buf][1][b * 32 + lane]),
                               max_u16x2(sh.col_amax[buf][2][b * 32 + lane], sh.col_amax[buf][3][b * 32 + lane]));
            }
            const BlockScale b_lo = block_scale<kF32>(a2 & 0xFFFFu), b_hi = block_scale<kF32>(a2 >> 16);
            const float m_lo = b_lo.m, m_hi = b_hi.m;
            uint32_t lo[8], hi[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t a0 = wc[4 * k], a1 = wc[4 * k + 1], a2w = wc[4 * k + 2], a3 = wc[4 * k + 3];
                lo[k] = cvt_e4m3x2(__fmul_rn(bf16_lo(a0), m_lo), __fmul_rn(bf16_lo(a1), m_lo)) |
                        (cvt_e4m3x2(__fmul_rn(bf16_lo(a2w), m_lo), __fmul_rn(bf16_lo(a3), m_lo)) << 16);
                hi[k] = cvt_e4m3x2(__fmul_rn(bf16_hi(a0), m_hi), __fmul_rn(bf16_hi(a1), m_hi)) |
                        (cvt_e4m3x2(__fmul_rn(bf16_hi(a2w), m_hi), __fmul_rn(bf16_hi(a3), m_hi)) << 16);
            }
            if (b_lo.bad) {
#pragma unroll
                for (int k = 0; k < 8; ++k) lo[k] = 0x7F7F7F7Fu;
            }
            if (b_hi.bad) {
#pragma unroll
                for (int k = 0; k < 8; ++k) hi[k] = 0x7F7F7F7Fu;
            }
            // Column C of the tile is row C of the column-code tile; this
            // lane's 32 rows are its chunks 2g and 2g+1.
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int C = b * kBoxCols + 2 * lane + j;
                const uint32_t* w = j ? hi : lo;
#pragma unroll
                for (int t = 0; t < 2; ++t)
                    sts128(tile + kBoxBytes + C * 128 + (((2 * g + t) ^ (C & 7)) << 4), w[4 * t], w[4 * t + 1],
                           w[4 * t + 2], w[4 * t + 3]);
                const int64_t c = int64_t(c0) + C;
                if (g == 0 && c < p.cols) {
                    if constexpr (kF32)
                        reinterpret_cast<float*>(p.s_col)[c * p.ld_s_col + r0 / kEdge] = j ? b_hi.s : b_lo.s;
                    else
                        put_scales(p.s_col + c * p.ld_s_col + (r0 >> 5), j ? b_hi.byte : b_lo.byte,
                                   (p.rows - r0 + 31) >> 5);
                }
            }
        }
        fence_proxy_async_smem();                      // the staged codes are read by the TMA engine
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.staged[s]));
    }
}

template <bool R, bool C, bool D2, bool F32>
cudaError_t launch(const CUtensorMap& xm, const CUtensorMap& qr, const CUtensorMap& qc, const BlockParams& p,
                   int sms, cudaStream_t stream) {
    auto k = block_quantize_kernel<R, C, D2, F32>;
    cudaError_t e = set_smem_attribute_once(reinterpret_cast<const void*>(k), kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t cap = int64_t(kCtasPerSm) * sms;
    const int grid = int(p.tiles < cap ? p.tiles : cap);
    k<<<grid, kThreads, kSmemBytes, stream>>>(xm, qr, qc, p);
    return cudaGetLastError();
}

template <bool F32>
cudaError_t launch_all(bool rowwise, bool colwise, bool block_2d, const CUtensorMap& xm, const CUtensorMap& qr,
                       const CUtensorMap& qc, const BlockParams& p, int sms, cudaStream_t stream) {
    if (block_2d) {
        if (rowwise && colwise) return launch<true, true, true, F32>(xm, qr, qc, p, sms, stream);
        if (rowwise) return launch<true, false, true, F32>(xm, qr, qc, p, sms, stream);
        return launch<false, true, true, F32>(xm, qr, qc, p, sms, stream);
    }
    if (rowwise && colwise) return launch<true, true, false, F32>(xm, qr, qc, p, sms, stream);
    if (rowwise) return launch<true, false, false, F32>(xm, qr, qc, p, sms, stream);
    return launch<false, true, false, F32>(xm, qr, qc, p, sms, stream);
}

}  // namespace

te_mx_status block_quantize_launch(const QuantizeArgs& a, bool block_2d, bool fp32_scales, cudaStream_t stream) {
    const bool rowwise = a.q_row != nullptr, colwise = a.q_col != nullptr;
    if (a.rows == 0 || a.cols == 0 || (!rowwise && !colwise)) return TE_MX_OK;

    CUtensorMap xm, qr, qc;
    te_mx_status st = encode_tensor_map_2d(&xm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, uint64_t(a.cols),
                                           uint64_t(a.rows), uint64_t(a.ld_x) * 2, kBoxCols, kEdge,
                                           CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != TE_MX_OK) return st;
    qr = xm;
    qc = xm;
    if (rowwise && (st = encode_tensor_map_2d(&qr, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.q_row, uint64_t(a.cols),
                                              uint64_t(a.rows), uint64_t(a.cols), kEdge, kEdge,
                                              CU_TENSOR_MAP_SWIZZLE_128B)) != TE_MX_OK) return st;
    if (colwise && (st = encode_tensor_map_2d(&qc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.q_col, uint64_t(a.rows),
                                              uint64_t(a.cols), uint64_t(a.rows), kEdge, kEdge,
                                              CU_TENSOR_MAP_SWIZZLE_128B)) != TE_MX_OK) return st;

    BlockParams p;
    p.rows = a.rows; p.cols = a.cols;
    p.s_row = a.s_row; p.ld_s_row = a.ld_s_row;
    p.s_col = a.s_col; p.ld_s_col = a.ld_s_col;
    p.col_tiles = (a.cols + kEdge - 1) / kEdge;
    p.tiles = ((a.rows + kEdge - 1) / kEdge) * p.col_tiles;
    if ((st = device_status_ptr(&p.status)) != TE_MX_OK) return st;
    int sms = 0;
    if ((st = device_sm_count(&sms)) != TE_MX_OK) return st;

    const cudaError_t e = fp32_scales ? launch_all<true>(rowwise, colwise, block_2d, xm, qr, qc, p, sms, stream)
                                      : launch_all<false>(rowwise, colwise, block_2d, xm, qr, qc, p, sms, stream);
    return cuda_status(e, "block quantize kernel launch");
}

}  // namespace temx
