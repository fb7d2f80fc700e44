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
// Work decomposition.  The input is cut into units of 64 rows x 64 columns
// (8 KB of bf16), and units into strips of 8 along a band (64 x 512).  The
// CTAs walk the strips with stride gridDim.x, so the strips in flight are
// contiguous in memory; warp w of a CTA takes unit w of each strip.  Every
// warp runs its own pipeline over a kStages-deep ring: lane 0 loads units
// with TMA (128-byte swizzle, so both the row reads and the column reads below
// are bank-conflict free) and the whole warp consumes them:
//   column-wise: lane l owns columns 2l and 2l+1 (two 32-row blocks each);
//   row-wise:    lane l owns rows l and l+32 (two 32-column blocks each).
// Once every lane has read the unit, the codes (64 x 64 bytes per orientation)
// are written into the same 8 KB of shared memory with a 64-byte swizzle and
// leave with two TMA tensor stores, so global writes are whole lines instead
// of 32 scattered sectors per instruction.  The row-wise scale bytes of a
// strip (8 units x 2 per row) meet in shared memory and leave as one 16-byte
// store per row after a barrier of the CTA's warps (per-unit stores of 2
// bytes into each of 64 rows cost ~10 % of the kernel's time); column-wise
// scale bytes (2 per column per unit) are stored directly.
#include <cuda_bf16.h>
#include <mutex>
#include <cuda_runtime.h>

#include "e4m3.cuh"
#include "ptx.cuh"
#include "temx_internal.h"
#include "units.cuh"

namespace temx {

namespace {

constexpr int kRows = 64;                    // unit height (two column-wise blocks)
constexpr int kCols = 64;                    // unit width in bf16 (= 128-byte swizzle row)
constexpr int kUnitBytes = kRows * kCols * 2;
constexpr int kWarps = 8;                    // = units per strip: 8 x 2 scale bytes = 16 per row
constexpr int kStages = 3;
constexpr int kSmemBytes = kWarps * kStages * kUnitBytes + 1024;
static_assert(kRows == kDbiasBandRows, "bias-gradient bands are the unit rows");

struct QuantizeParams {
    int64_t rows, cols;
    uint8_t* s_row;
    int64_t ld_s_row;
    uint8_t* s_col;
    int64_t ld_s_col;
    int64_t col_units;     // ceil(cols / 64)
    int64_t units;         // ceil(rows / 64) * col_units
    float* partial;        // bias gradient: fp32 [ceil(rows/64) x cols] band sums
    unsigned int* status;  // device status word
};

// E8M0 byte from |amax| as bf16 bits: exponent field - 8, floored at 0;
// 0xFF for NaN/inf.
__device__ __forceinline__ uint32_t scale_byte(uint32_t amax_bits) {
    const uint32_t ef = amax_bits >> 7;
    if (ef == 0xFFu) return 0xFFu;
    return ef > 8u ? ef - 8u : 0u;
}

// One row of a unit (64 bf16 at shared address `row_addr`, 128-byte swizzle
// phase `sw`): two row-wise blocks -> codes[2][8] words, scale bytes sb[2].
__device__ __forceinline__ void row_blocks(uint32_t row_addr, int sw, uint32_t (&codes)[2][8], uint32_t (&sb)[2]) {
    uint32_t w[32];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 v = lds128(row_addr + ((j ^ sw) << 4));
        w[4 * j + 0] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
    }
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        const uint32_t m2 = amax_words<16>(w + 16 * blk);
        sb[blk] = scale_byte(max(m2 & 0xFFFFu, m2 >> 16));
        const float m = inv_scale(sb[blk]);
#pragma unroll
        for (int i = 0; i < 8; ++i) codes[blk][i] = quant4(w[16 * blk + 2 * i], w[16 * blk + 2 * i + 1], m);
        if (sb[blk] == 0xFFu) {
#pragma unroll
            for (int i = 0; i < 8; ++i) codes[blk][i] = 0x7F7F7F7Fu;
        }
    }
}

// Columns 2l and 2l+1 over the 32 rows from `row0` (a multiple of 8):
// codes lo[8] / hi[8] (32 bytes each, rows in order) and their scale bytes.
__device__ __forceinline__ void col_blocks(uint32_t tile, int row0, int lane, uint32_t (&lo)[8], uint32_t (&hi)[8],
                                           uint32_t& s_lo, uint32_t& s_hi, float& sum_lo, float& sum_hi) {
    uint32_t w[32];
    const uint32_t base = tile + row0 * 128 + ((lane & 3) << 2);
    const int chunk = lane >> 2;
#pragma unroll
    for (int r = 0; r < 32; ++r) w[r] = lds32(base + r * 128 + ((chunk ^ (r & 7)) << 4));
#pragma unroll
    for (int r = 0; r < 32; ++r) {                  // column sums for the bias gradient (row order)
        sum_lo += bf16_lo(w[r]);
        sum_hi += bf16_hi(w[r]);
    }
    const uint32_t m2 = amax_words<32>(w);
    s_lo = scale_byte(m2 & 0xFFFFu);
    s_hi = scale_byte(m2 >> 16);
    const float m_lo = inv_scale(s_lo), m_hi = inv_scale(s_hi);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t a0 = w[4 * i], a1 = w[4 * i + 1], a2 = w[4 * i + 2], a3 = w[4 * i + 3];
        lo[i] = cvt_e4m3x2(__fmul_rn(bf16_lo(a0), m_lo), __fmul_rn(bf16_lo(a1), m_lo)) |
                (cvt_e4m3x2(__fmul_rn(bf16_lo(a2), m_lo), __fmul_rn(bf16_lo(a3), m_lo)) << 16);
        hi[i] = cvt_e4m3x2(__fmul_rn(bf16_hi(a0), m_hi), __fmul_rn(bf16_hi(a1), m_hi)) |
                (cvt_e4m3x2(__fmul_rn(bf16_hi(a2), m_hi), __fmul_rn(bf16_hi(a3), m_hi)) << 16);
    }
    if (s_lo == 0xFFu) {
#pragma unroll
        for (int i = 0; i < 8; ++i) lo[i] = 0x7F7F7F7Fu;
    }
    if (s_hi == 0xFFu) {
#pragma unroll
        for (int i = 0; i < 8; ++i) hi[i] = 0x7F7F7F7Fu;
    }
}

// Column sums (columns 2l, 2l+1, all 64 rows of the unit, row order) without
// quantising, for a bias gradient without a column-wise copy.
__device__ __forceinline__ void col_sums(uint32_t tile, int lane, float& sum_lo, float& sum_hi) {
    const uint32_t base = tile + ((lane & 3) << 2);
    const int chunk = lane >> 2;
#pragma unroll 8
    for (int r = 0; r < 64; ++r) {
        const uint32_t w = lds32(base + r * 128 + ((chunk ^ (r & 7)) << 4));
        sum_lo += bf16_lo(w);
        sum_hi += bf16_hi(w);
    }
}

__device__ __forceinline__ void sts16(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b16 [%0], %1;" :: "r"(addr), "h"(static_cast<uint16_t>(v)) : "memory");
}

// Barrier `id` over `n` threads (whole warps) of the CTA.
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t n) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}

// Byte offset of 16-byte chunk c of 64-byte row r in a 64-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw64(int r, int c) { return uint32_t(r * 64 + ((c ^ ((r >> 1) & 3)) << 4)); }

template <bool kRowwise, bool kColwise, bool kDbias>
__global__ void __launch_bounds__(kWarps * 32, 1)
quantize_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap qrow_map,
                const __grid_constant__ CUtensorMap qcol_map, const QuantizeParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[kWarps][kStages];
    // row-wise scale bytes of a strip (64 rows x 16 bytes), double-buffered by round
    __shared__ __align__(16) uint8_t row_scales[2][kRows][16];
    // bias-gradient band sums of a strip (8 units x 64 columns), double-buffered by round
    __shared__ __align__(16) float part_stage[2][kWarps * kCols];

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    grid_dependency_wait();              // launched as a programmatic dependent: no global access before this
    grid_launch_dependents();
    // The CTAs walk strips of kWarps units along a band (64 rows x 512 columns)
    // with stride gridDim.x, so that the strips in flight are contiguous in
    // memory; warp w takes unit w of each strip (or none past the band's end).
    const int64_t strips_per_band = (p.col_units + kWarps - 1) / kWarps;
    const int64_t n_strips = ((p.rows + kRows - 1) / kRows) * strips_per_band;
    if (int64_t(blockIdx.x) >= n_strips) return;                         // (uniform over the CTA)
    const int64_t n_mine = (n_strips - blockIdx.x + gridDim.x - 1) / gridDim.x;
    const uint32_t ring = smem_u32(smem + warp * (kStages * kUnitBytes));
    // (band, strip) of this round and of the next load (lane 0)
    const UnitWalk walk(gridDim.x, strips_per_band);
    int32_t band, strip;
    walk.start(blockIdx.x, band, strip);
    int32_t lband = band, lstrip = strip;
    auto unit_col = [&](int32_t st) { return st * kWarps + warp; };       // this warp's column unit
    // lane 0: load this warp's unit of the round (or, past the band's end,
    // complete the stage's barrier without data)
    auto load = [&](uint32_t bar, uint32_t dst, int32_t b, int32_t st) {
        if (unit_col(st) < p.col_units) {
            mbar_arrive_expect_tx(bar, kUnitBytes);
            tma_load_2d(dst, &x_map, bar, unit_col(st) * kCols, b * kRows);
        } else {
            mbar_arrive(bar);
        }
    };

    if (lane == 0) {
        tma_prefetch_desc(&x_map);
        if (kRowwise) tma_prefetch_desc(&qrow_map);
        if (kColwise) tma_prefetch_desc(&qcol_map);
        for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&bars[warp][s]), 1);
        fence_mbarrier_init();
        for (int s = 0; s < kStages && s < n_mine; ++s) {
            load(smem_u32(&bars[warp][s]), ring + s * kUnitBytes, lband, lstrip);
            walk.step(lband, lstrip);
        }
    }
    __syncwarp();

    int s = 0;
    uint32_t parity = 0;
    bool ok = true;                      // false once a wait gave up: the warp then only keeps the barriers
    for (int64_t i = 0; i < n_mine; ++i) {
        const uint32_t bar = smem_u32(&bars[warp][s]);
        const int32_t col = unit_col(strip);
        const bool mine = col < p.col_units;
        if (ok && !__all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, p.status))) {
            ok = false;
            if (lane == 0)                       // gave up: let this warp's loads still in flight land
                for (int64_t j = i; j < i + kStages && j < n_mine; ++j)
                    mbar_wait(smem_u32(&bars[warp][j % kStages]), uint32_t((j / kStages) & 1), p.status);
        }
        const uint32_t tile = ring + s * kUnitBytes;
        const int64_t r0 = int64_t(band) * kRows, c0 = int64_t(col) * kCols;
        if (ok && mine) {
            uint32_t cc[2][2][8];             // column codes [half][column 2l / 2l+1][words]
            uint32_t rc[2][2][8];             // row codes [row l / l+32][block][words]
            float sum_lo = 0.0f, sum_hi = 0.0f;               // bias-gradient band sums
            if (kColwise) {
                const bool second = r0 + 32 < p.rows;          // rows % 32 == 0 here
                uint32_t s_lo[2] = {0, 0}, s_hi[2] = {0, 0};
                col_blocks(tile, 0, lane, cc[0][0], cc[0][1], s_lo[0], s_hi[0], sum_lo, sum_hi);
                col_blocks(tile, 32, lane, cc[1][0], cc[1][1], s_lo[1], s_hi[1], sum_lo, sum_hi);
                const int64_t c = c0 + 2 * lane;
                if (c < p.cols) {                              // cols % 32 == 0: c + 1 valid too
                    uint8_t* sp = p.s_col + c * p.ld_s_col + (r0 >> 5);
                    if (second) {
                        st_global_u16(sp, s_lo[0] | (s_lo[1] << 8));
                        st_global_u16(sp + p.ld_s_col, s_hi[0] | (s_hi[1] << 8));
                    } else {
                        st_global_u8(sp, s_lo[0]);
                        st_global_u8(sp + p.ld_s_col, s_hi[0]);
                    }
                }
            }
            if (kDbias) {
                if (!kColwise) col_sums(tile, lane, sum_lo, sum_hi);
                // (rows past the end were loaded as 0; columns past the end are not copied out)
                *reinterpret_cast<float2*>(&part_stage[i & 1][warp * kCols + 2 * lane]) = make_float2(sum_lo, sum_hi);
            }
            if (kRowwise) {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    uint32_t sb[2];
                    row_blocks(tile + (lane + 32 * rr) * 128, lane & 7, rc[rr], sb);
                    // this unit's two scale bytes at byte 2 warp of the strip's rows
                    sts16(smem_u32(&row_scales[i & 1][lane + 32 * rr][2 * warp]), sb[0] | (sb[1] << 8));
                }
            }
            __syncwarp();                     // every lane has read the unit: reuse it for the codes
            if (kRowwise) {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int r = lane + 32 * rr;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t* w = rc[rr][c >> 1] + 4 * (c & 1);
                        sts128(tile + sw64(r, c), w[0], w[1], w[2], w[3]);
                    }
                }
            }
            if (kColwise) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int cl = 2 * lane + j;
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            const uint32_t* w = cc[h][j] + 4 * t;
                            sts128(tile + 4096 + sw64(cl, 2 * h + t), w[0], w[1], w[2], w[3]);
                        }
                }
            }
            fence_proxy_async_smem();         // make the staged codes visible to the TMA engine
            __syncwarp();
            if (lane == 0) {
                if (kRowwise) tma_store_2d(&qrow_map, tile, int32_t(c0), int32_t(r0));
                if (kColwise) tma_store_2d(&qcol_map, tile + 4096, int32_t(r0), int32_t(c0));
                bulk_commit();             // (an empty group when only the bias gradient is produced)
            }
        }
        const bool refill = ok && i + kStages < n_mine;
        if (refill && lane == 0) {
            bulk_wait_read_all();         // the stores have read the tile: refill it
            load(bar, tile, lband, lstrip);
            walk.step(lband, lstrip);
        }
        // warp 2 copies a strip's band sums out after the barrier below; the copy
        // of round i - 1 must have read its staging area before the barrier of
        // round i, after which the warps write it again (a refill waited for it)
        if (kDbias && warp == 2 && lane == 0 && !refill) bulk_wait_read_all();
        __syncwarp();
        if (kRowwise || kDbias) {
            named_barrier_sync(1, kWarps * 32);
            if (kRowwise && warp < 2) {
                // the strip's row scales: 16 bytes per row, one store per row (warps 0-1,
                // lane = row); a strip cut by the band's end writes its bytes one by one
                const int rl = warp * 32 + lane;
                const int64_t r = r0 + rl;
                const int64_t first = int64_t(strip) * kWarps * 2;             // the strip's first scale byte
                const int64_t valid = (p.cols + 31) / 32 - first;               // scale bytes of the row left
                if (r < p.rows) {
                    uint8_t* sp = p.s_row + r * p.ld_s_row + first;
                    const uint4 v = lds128(smem_u32(&row_scales[i & 1][rl][0]));
                    if (valid >= 16) {
                        st_global_v4(sp, v.x, v.y, v.z, v.w);
                    } else {
                        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            if (k < valid) st_global_u8(sp + k, (w4[k >> 2] >> (8 * (k & 3))) & 0xFFu);
                    }
                }
            }
            if (kDbias && warp == 2 && lane == 0) {
                // the strip's band sums: one bulk copy of its (at most 512) columns
                const int64_t cs = int64_t(strip) * kWarps * kCols;
                const int64_t n = p.cols - cs < kWarps * kCols ? p.cols - cs : kWarps * kCols;   // a multiple of 32
                float* dst = p.partial + int64_t(band) * p.cols + cs;
                asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                             :: "l"(dst), "r"(smem_u32(&part_stage[i & 1][0])), "r"(uint32_t(n) * 4u) : "memory");
                bulk_commit();
            }
        }
        walk.step(band, strip);
        if (++s == kStages) {
            s = 0;
            parity ^= 1u;
        }
    }
    if (lane == 0) bulk_wait_all();
}

// Bias gradient, second pass: dbias[c] = bf16(sum over the bands of
// partial[b][c]).  A block owns 32 columns (lane = column, coalesced loads);
// warp w sums bands w, w + 8, w + 16, ... in order, then the 8 warp sums are
// added in warp order: a fixed order, so the result is deterministic.
constexpr int kReduceWarps = 8;
__global__ void __launch_bounds__(kReduceWarps * 32)
dbias_reduce_kernel(const float* __restrict__ partial, int64_t bands, int64_t cols, uint16_t* __restrict__ dbias) {
    __shared__ float part[kReduceWarps][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c = int64_t(blockIdx.x) * 32 + lane;
    float acc = 0.0f;
    if (c < cols)
        for (int64_t b = warp; b < bands; b += kReduceWarps) acc += partial[b * cols + c];
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && c < cols) {
        float sum = part[0][lane];
#pragma unroll
        for (int w = 1; w < kReduceWarps; ++w) sum += part[w][lane];
        const __nv_bfloat16 h = __float2bfloat16_rn(sum);
        dbias[c] = *reinterpret_cast<const uint16_t*>(&h);
    }
}

template <bool R, bool C, bool D>
cudaError_t launch(const CUtensorMap& xm, const CUtensorMap& qr, const CUtensorMap& qc, const QuantizeParams& p,
                   int sms, cudaStream_t stream) {
    auto k = quantize_kernel<R, C, D>;
    cudaError_t e = set_smem_attribute_once(reinterpret_cast<const void*>(k), kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t want = ((p.rows + kRows - 1) / kRows) * ((p.col_units + kWarps - 1) / kWarps);   // strips
    const int grid = int(want < sms ? want : sms);
    // programmatic dependent launch: the CTAs may start while the previous
    // kernel in the stream finishes (the kernel waits before touching memory)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, xm, qr, qc, p);
}

}  // namespace

te_mx_status quantize_launch(const QuantizeArgs& a, cudaStream_t stream) {
    const bool rowwise = a.q_row != nullptr, colwise = a.q_col != nullptr, dbias = a.dbias != nullptr;
    if (a.rows == 0 || a.cols == 0 || (!rowwise && !colwise && !dbias)) return TE_MX_OK;

    CUtensorMap xm, qr, qc;
    te_mx_status st = encode_tensor_map_2d(&xm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x,
                                           uint64_t(a.cols), uint64_t(a.rows), uint64_t(a.ld_x) * 2,
                                           kCols, kRows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != TE_MX_OK) return st;
    qr = xm;
    qc = xm;
    if (rowwise && (st = encode_tensor_map_2d(&qr, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.q_row, uint64_t(a.cols),
                                              uint64_t(a.rows), uint64_t(a.cols), kCols, kRows,
                                              CU_TENSOR_MAP_SWIZZLE_64B)) != TE_MX_OK) return st;
    if (colwise && (st = encode_tensor_map_2d(&qc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.q_col, uint64_t(a.rows),
                                              uint64_t(a.cols), uint64_t(a.rows), kRows, kCols,
                                              CU_TENSOR_MAP_SWIZZLE_64B)) != TE_MX_OK) return st;

    QuantizeParams p;
    p.rows = a.rows; p.cols = a.cols;
    p.s_row = a.s_row; p.ld_s_row = a.ld_s_row;
    p.s_col = a.s_col; p.ld_s_col = a.ld_s_col;
    p.col_units = (a.cols + kCols - 1) / kCols;
    p.units = ((a.rows + kRows - 1) / kRows) * p.col_units;
    p.partial = a.partial;
    st = device_status_ptr(&p.status);
    if (st != TE_MX_OK) return st;

    int sms = 0;
    st = device_sm_count(&sms);
    if (st != TE_MX_OK) return st;
    cudaError_t e;
    if (!dbias) {
        if (rowwise && colwise) e = launch<true, true, false>(xm, qr, qc, p, sms, stream);
        else if (rowwise) e = launch<true, false, false>(xm, qr, qc, p, sms, stream);
        else e = launch<false, true, false>(xm, qr, qc, p, sms, stream);
    } else {
        if (rowwise && colwise) e = launch<true, true, true>(xm, qr, qc, p, sms, stream);
        else if (rowwise) e = launch<true, false, true>(xm, qr, qc, p, sms, stream);
        else if (colwise) e = launch<false, true, true>(xm, qr, qc, p, sms, stream);
        else e = launch<false, false, true>(xm, qr, qc, p, sms, stream);
        if (e == cudaSuccess) {
            const int64_t bands = (a.rows + kDbiasBandRows - 1) / kDbiasBandRows;
            dbias_reduce_kernel<<<unsigned((a.cols + 31) / 32), kReduceWarps * 32, 0, stream>>>(a.partial, bands,
                                                                                                a.cols, a.dbias);
            e = cudaGetLastError();
        }
    }
    return cuda_status(e, "quantize kernel launch");
}

}  // namespace temx

// ---------------------------------------------------------------------------
// Allocation-free bias-gradient quantisation (te_mx_quantize_dbias_noalloc).
// The band sums live in this file-scope device array instead of a caller
// workspace.  Host code must not hand `g_noalloc_scratch` itself to a kernel
// (in host code that name is only a stand-in for the device symbol); its
// device address is looked up once per device with cudaGetSymbolAddress.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = TE_MX_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kNoAllocMaxDevices = 64;
float* g_noalloc_ptr[kNoAllocMaxDevices];     // per-device address, null until looked up
std::mutex g_noalloc_mutex;

// The scratch address on the current device (looked up on first use).
te_mx_status noalloc_scratch(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return temx::cuda_status(e, "cudaGetDevice");
    if (dev < 0 || dev >= kNoAllocMaxDevices)
        return temx::set_error(TE_MX_ERR_CUDA, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return temx::cuda_status(e, "cudaGetSymbolAddress(no-alloc scratch)");
        g_noalloc_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return TE_MX_OK;
}

}  // namespace

extern "C" te_mx_status te_mx_quantize_dbias_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                                     uint8_t* q_row, uint8_t* s_row, int64_t ld_s_row,
                                                     uint8_t* q_col, uint8_t* s_col, int64_t ld_s_col,
                                                     void* dbias, void* stream) {
    using namespace temx;
    clear_error();
    if (!dbias) return set_error(TE_MX_ERR_INVALID_ARG, "dbias is NULL");
    te_mx_status st = validate_quantize(x, rows, cols, ld_x, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col, true);
    if (st != TE_MX_OK || rows == 0 || cols == 0) return st;
    if (reinterpret_cast<uintptr_t>(dbias) % 16) return set_error(TE_MX_ERR_MISALIGNED, "dbias is not 16-byte aligned");
    const size_t need = te_mx_quantize_dbias_workspace_size(rows, cols);
    if (need > kNoAllocScratchBytes)
        return set_error(TE_MX_ERR_WORKSPACE_TOO_SMALL,
                         "%lld x %lld needs %zu bytes of bias-gradient scratch; the built-in scratch holds %zu "
                         "(use te_mx_quantize_dbias with a workspace)",
                         (long long)rows, (long long)cols, need, kNoAllocScratchBytes);
    float* scratch = nullptr;
    if ((st = noalloc_scratch(&scratch)) != TE_MX_OK) return st;
    QuantizeArgs a{x, rows, cols, ld_x, q_row, s_row, ld_s_row, q_col, s_col, ld_s_col,
                   static_cast<uint16_t*>(dbias), scratch};
    return quantize_launch(a, static_cast<cudaStream_t>(stream));
}
