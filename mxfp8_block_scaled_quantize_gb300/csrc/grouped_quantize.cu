// Per-expert column-wise MXFP8 quantisation: the operands of the grouped
// wgrad GEMM dW_e = dY_e^T X_e of a MoE layer (one launch over the experts,
// "Single-Launch Grouped GEMM Backends on ROCm", ROCm/TransformerEngine
// README).
//
// Expert e owns rows [R_e, R_e + m_e) of the token-major input x [T x C].  Its
// column-wise copy is blocked along tokens (32 per E8M0 scale, the MXFP8 rule
// of te_mx_quantize) and zero-padded to Kp_e = round_up(m_e, 128) tokens, so
// no block crosses an expert boundary and the GEMM's 128-token K-steps stay
// inside one expert:
//   q[c][P_e + t] = E4M3 code of x[R_e + t][c]   (t < m_e; 0 for m_e <= t < Kp_e)
//   s[c][Q_e + b] = E8M0 scale of tokens 32b .. 32b + 31 of expert e
//   P_e = sum_{e' < e} Kp_e',  Q_e = sum_{e' < e} round_up(Kp_e' / 32, 16)
// Expert sizes are read on the device.
//
// Work decomposition.  A unit is 64 padded tokens (two blocks; Kp_e is a
// multiple of 128, so a unit never crosses an expert) times 64 columns, and a
// strip is up to 8 consecutive units of one expert (512 tokens) in one column
// unit.  The CTAs walk the strips, column units fastest, with stride
// gridDim.x; warp w of a CTA takes unit w of each strip and runs its own TMA
// pipeline (like the MXFP8 quantiser): 64 x 64 bf16 in, lane l quantises
// columns 2l, 2l+1 over both blocks (tokens past the expert's end masked to
// 0), the codes are staged in the consumed buffer (64 columns x 64 bytes,
// 64-byte swizzle) and leave with one TMA store.  A strip's scale bytes (16
// per column, 16-byte aligned: an expert's scales start on a 16-byte
// boundary) meet in shared memory and leave as one 16-byte store per column
// after a barrier of the CTA's warps, instead of 4 single-byte stores per
// column and unit.
#include <cuda_runtime.h>

#include "e4m3.cuh"
#include "ptx.cuh"
#include "temx_internal.h"
#include "units.cuh"

namespace temx {

namespace {

constexpr int kRows = 64;                        // tokens per unit (two blocks)
constexpr int kCols = 64;                        // columns per unit (128 bytes of bf16)
constexpr int kUnitBytes = kRows * kCols * 2;
constexpr int kWarps = 8;                        // = units per strip (8 x 2 scale bytes = 16 per column)
constexpr int kStages = 3;
constexpr int kMaxGroups = 1024;
constexpr int kSmem = kWarps * kStages * kUnitBytes + 1024;

struct GroupedParams {
    int64_t total_m, cols;
    int32_t groups;
    const int32_t* group_m;  // device
    uint8_t* s;
    int64_t ld_q, ld_s;      // code / scale row pitch = capacities
    int64_t col_units;       // ceil(cols / 64)
    unsigned int* status;
};

struct GroupTable {
    int32_t blk[kMaxGroups + 1];     // padded 64-token units before expert g (= P_g / 64)
    int32_t row[kMaxGroups + 1];     // input rows before expert g (= R_g)
    int32_t sc[kMaxGroups + 1];      // scale columns before expert g (= Q_g)
    int32_t strip[kMaxGroups + 1];   // strips (8 units each, per column unit) before expert g
    int32_t bad;
};

// Prefix sums of the expert sizes (one warp).  A negative size, a sum above
// total_m or a layout wider than the given pitches sets the status word and
// the kernel writes nothing.
__device__ void build_table(const GroupedParams& p, GroupTable& t, int lane) {
    const int G = p.groups;
    const int per = (G + 31) / 32;
    const int lo = min(G, lane * per), hi = min(G, lo + per);
    bool bad = false;
    int64_t rows = 0, blks = 0, scs = 0, strips = 0;
    for (int g = lo; g < hi; ++g) {
        const int64_t m = p.group_m[g];
        bad |= m < 0;
        const int64_t mm = m < 0 ? 0 : m;
        const int64_t kb = (mm + 127) / 128 * 4;                       // Kp / 32
        rows += mm;
        blks += kb / 2;
        scs += (kb + 15) / 16 * 16;
        strips += (kb / 2 + kWarps - 1) / kWarps;
    }
    int64_t r_in = rows, b_in = blks, s_in = scs, t_in = strips;
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t r = __shfl_up_sync(0xFFFFFFFFu, r_in, o), b = __shfl_up_sync(0xFFFFFFFFu, b_in, o),
                      s = __shfl_up_sync(0xFFFFFFFFu, s_in, o), q = __shfl_up_sync(0xFFFFFFFFu, t_in, o);
        if (lane >= o) { r_in += r; b_in += b; s_in += s; t_in += q; }
    }
    int64_t r0 = r_in - rows, b0 = b_in - blks, s0 = s_in - scs, t0 = t_in - strips;
    for (int g = lo; g < hi; ++g) {
        t.row[g] = int32_t(r0);
        t.blk[g] = int32_t(b0);
        t.sc[g] = int32_t(s0);
        t.strip[g] = int32_t(t0);
        const int64_t m = p.group_m[g] < 0 ? 0 : p.group_m[g];
        const int64_t kb = (m + 127) / 128 * 4;
        r0 += m;
        b0 += kb / 2;
        s0 += (kb + 15) / 16 * 16;
        t0 += (kb / 2 + kWarps - 1) / kWarps;
    }
    const int64_t rt = __shfl_sync(0xFFFFFFFFu, r_in, 31), bt = __shfl_sync(0xFFFFFFFFu, b_in, 31),
                  st = __shfl_sync(0xFFFFFFFFu, s_in, 31), tt = __shfl_sync(0xFFFFFFFFu, t_in, 31);
    bad = __any_sync(0xFFFFFFFFu, bad);
    if (lane == 0) {
        t.row[G] = int32_t(rt);
        t.blk[G] = int32_t(bt);
        t.sc[G] = int32_t(st);
        t.strip[G] = int32_t(tt);
        bad |= rt > p.total_m || bt * kRows > p.ld_q || st > p.ld_s;
        t.bad = bad ? 1 : 0;
        if (bad && blockIdx.x == 0) set_device_status(p.status, kStatusBadArg);
    }
}

__device__ __forceinline__ void sts16(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b16 [%0], %1;" :: "r"(addr), "h"(static_cast<uint16_t>(v)) : "memory");
}

// Barrier `id` over `n` threads (whole warps) of the CTA.
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t n) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}

__global__ void __launch_bounds__(kWarps * 32, 1)
grouped_colwise_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap q_map,
                       const GroupedParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[kWarps][kStages];
    __shared__ GroupTable tab;
    // a strip's scale bytes (64 columns x 16 bytes), double-buffered by round
    __shared__ __align__(16) uint8_t strip_scales[2][kCols][16];

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) build_table(p, tab, lane);
    __syncthreads();
    if (tab.bad) return;

    const int64_t n_strips = int64_t(tab.strip[p.groups]) * p.col_units;
    if (int64_t(blockIdx.x) >= n_strips) return;                          // (uniform over the CTA)
    const int64_t n_mine = (n_strips - blockIdx.x + gridDim.x - 1) / gridDim.x;
    const uint32_t ring = smem_u32(smem + warp * (kStages * kUnitBytes));

    // The strips of this CTA as (strip row, column unit), walked without
    // dividing; the expert of a strip row is found from a lower bound that
    // only moves forward (a CTA's strips only move forward).
    const UnitWalk walk(gridDim.x, p.col_units);
    int32_t srow, col;
    walk.start(blockIdx.x, srow, col);
    int32_t lsrow = srow, lcol = col, load_hint = 0;   // lane 0: the loads run kStages strips ahead
    // lane 0: load this warp's unit of a strip (or, past the expert's units,
    // complete the stage's barrier without data)
    auto load = [&](uint32_t dst, uint32_t bar) {
        while (tab.strip[load_hint + 1] <= lsrow) ++load_hint;        // lsrow < tab.strip[groups]
        const int32_t g = load_hint;
        const int32_t u = (lsrow - tab.strip[g]) * kWarps + warp;     // the unit within the expert
        if (tab.blk[g] + u < tab.blk[g + 1]) {
            mbar_arrive_expect_tx(bar, kUnitBytes);
            tma_load_2d(dst, &x_map, bar, lcol * kCols, tab.row[g] + u * kRows);   // rows past the expert: masked
        } else {
            mbar_arrive(bar);
        }
        walk.step(lsrow, lcol);
    };

    if (lane == 0) {
        tma_prefetch_desc(&x_map);
        tma_prefetch_desc(&q_map);
        for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&bars[warp][s]), 1);
        fence_mbarrier_init();
        for (int s = 0; s < kStages && s < n_mine; ++s) load(ring + s * kUnitBytes, smem_u32(&bars[warp][s]));
    }
    __syncwarp();

    int32_t g = 0;
    int s = 0;
    uint32_t parity = 0;
    bool ok = true;                              // false once a wait gave up: the warp then only keeps the barriers
    for (int64_t i = 0; i < n_mine; ++i) {
        const uint32_t bar = smem_u32(&bars[warp][s]);
        while (tab.strip[g + 1] <= srow) ++g;    // srow < tab.strip[groups]: stops at an expert
        const int32_t j = srow - tab.strip[g];                          // strip within the expert
        const int32_t units_g = tab.blk[g + 1] - tab.blk[g];
        const int32_t u = j * kWarps + warp;                             // this warp's unit within the expert
        const bool mine = u < units_g;
        const int32_t blk = tab.blk[g] + u;
        const int64_t c0 = int64_t(col) * kCols;
        const int32_t m = tab.row[g + 1] - tab.row[g];
        const int32_t valid = m - u * kRows;                             // tokens of the expert in this unit
        if (ok && !__all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, p.status))) {
            ok = false;
            if (lane == 0)                       // gave up: let this warp's loads still in flight land
                for (int64_t k = i; k < i + kStages && k < n_mine; ++k)
                    mbar_wait(smem_u32(&bars[warp][k % kStages]), uint32_t((k / kStages) & 1), p.status);
        }
        const uint32_t unit = ring + s * kUnitBytes;
        if (ok && mine) {
            // columns 2 lane, 2 lane + 1 over the unit's two 32-token blocks
            // (128-byte swizzle on the way in, 64-byte swizzle for the codes)
            uint32_t lo[2][8], hi[2][8], s_lo[2], s_hi[2];
            const uint32_t base = unit + ((lane & 3) << 2);
            const int ch = lane >> 2;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t w[32];
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    const uint32_t v = lds32(base + (32 * h + r) * 128 + ((ch ^ (r & 7)) << 4));
                    w[r] = 32 * h + r < valid ? v : 0u;
                }
                const uint32_t m2 = amax_words<32>(w);
                const uint32_t ef_lo = (m2 & 0xFFFFu) >> 7, ef_hi = m2 >> 23;
                s_lo[h] = ef_lo == 0xFFu ? 0xFFu : (ef_lo > 8u ? ef_lo - 8u : 0u);
                s_hi[h] = ef_hi == 0xFFu ? 0xFFu : (ef_hi > 8u ? ef_hi - 8u : 0u);
                const float k_lo = inv_scale(s_lo[h]), k_hi = inv_scale(s_hi[h]);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint32_t a0 = w[4 * q], a1 = w[4 * q + 1], a2 = w[4 * q + 2], a3 = w[4 * q + 3];
                    lo[h][q] = cvt_e4m3x2(__fmul_rn(bf16_lo(a0), k_lo), __fmul_rn(bf16_lo(a1), k_lo)) |
                               (cvt_e4m3x2(__fmul_rn(bf16_lo(a2), k_lo), __fmul_rn(bf16_lo(a3), k_lo)) << 16);
                    hi[h][q] = cvt_e4m3x2(__fmul_rn(bf16_hi(a0), k_hi), __fmul_rn(bf16_hi(a1), k_hi)) |
                               (cvt_e4m3x2(__fmul_rn(bf16_hi(a2), k_hi), __fmul_rn(bf16_hi(a3), k_hi)) << 16);
                }
                if (s_lo[h] == 0xFFu) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) lo[h][q] = 0x7F7F7F7Fu;
                }
                if (s_hi[h] == 0xFFu) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) hi[h][q] = 0x7F7F7F7Fu;
                }
            }
            __syncwarp();                        // every lane has read the unit: reuse it for the codes
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {     // column 2 lane + jj: 64 bytes, chunk 2h + t of its row
                const int cl = 2 * lane + jj;
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const uint32_t* w = (jj ? hi[h] : lo[h]) + 4 * t;
                        sts128(unit + uint32_t(cl * 64 + (((2 * h + t) ^ ((cl >> 1) & 3)) << 4)), w[0], w[1], w[2],
                               w[3]);
                    }
            }
            // this unit's scale bytes at bytes 2 warp, 2 warp + 1 of the strip's columns
            sts16(smem_u32(&strip_scales[i & 1][2 * lane][2 * warp]), s_lo[0] | (s_lo[1] << 8));
            sts16(smem_u32(&strip_scales[i & 1][2 * lane + 1][2 * warp]), s_hi[0] | (s_hi[1] << 8));
            fence_proxy_async_smem();            // make the staged codes visible to the TMA engine
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(&q_map, unit, blk * kRows, int32_t(c0));
                bulk_commit();
            }
        }
        if (ok && lane == 0 && i + kStages < n_mine) {
            bulk_wait_read_all();                // the store has read the unit: refill it
            load(unit, bar);
        }
        __syncwarp();
        // the strip's scale bytes: 16 per column at a 16-byte boundary, one
        // store per column (warps 0-1, lane = column); the last strip of an
        // expert may hold fewer units
        named_barrier_sync(1, kWarps * 32);
        if (warp < 2) {
            const int cl = warp * 32 + lane;
            const int64_t c = c0 + cl;
            const int32_t nb = 2 * min(kWarps, units_g - j * kWarps);    // scale bytes of the strip
            if (c < p.cols) {
                uint8_t* sp = p.s + c * p.ld_s + tab.sc[g] + 16 * j;
                const uint4 v = lds128(smem_u32(&strip_scales[i & 1][cl][0]));
                if (nb == 16) {
                    st_global_v4(sp, v.x, v.y, v.z, v.w);
                } else {
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        if (k < nb) st_global_u8(sp + k, (w4[k >> 2] >> (8 * (k & 3))) & 0xFFu);
                }
            }
        }
        walk.step(srow, col);
        if (++s == kStages) {
            s = 0;
            parity ^= 1u;
        }
    }
    if (lane == 0) bulk_wait_all();
}

}  // namespace

int64_t grouped_code_width(int64_t total_m, int32_t groups) {
    return (total_m + 127 * int64_t(groups) + 15) / 16 * 16;
}
int64_t grouped_scale_width(int64_t total_m, int32_t groups) {
    return ((total_m + 127 * int64_t(groups)) / 32 + 12 * int64_t(groups) + 15) / 16 * 16;
}

te_mx_status grouped_colwise_launch(const GroupedColwiseArgs& a, cudaStream_t stream) {
    CUtensorMap xm, qm;
    te_mx_status st = encode_tensor_map_2d(&xm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, uint64_t(a.cols),
                                           uint64_t(a.total_m), uint64_t(a.ld_x) * 2, kCols, kRows,
                                           CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != TE_MX_OK) return st;
    if ((st = encode_tensor_map_2d(&qm, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.q, uint64_t(a.ld_q), uint64_t(a.cols),
                                   uint64_t(a.ld_q), kRows, kCols, CU_TENSOR_MAP_SWIZZLE_64B)) != TE_MX_OK)
        return st;
    GroupedParams p;
    p.total_m = a.total_m; p.cols = a.cols;
    p.groups = a.groups; p.group_m = a.group_m;
    p.s = a.s; p.ld_q = a.ld_q; p.ld_s = a.ld_s;
    p.col_units = (a.cols + kCols - 1) / kCols;
    if ((st = device_status_ptr(&p.status)) != TE_MX_OK) return st;
    int sms = 0;
    if ((st = device_sm_count(&sms)) != TE_MX_OK) return st;
    cudaError_t e = set_smem_attribute_once(reinterpret_cast<const void*>(grouped_colwise_kernel), kSmem);
    if (e == cudaSuccess) {
        // a bound on the strips: units / 8 plus one partial strip per expert, per column unit
        const int64_t bound = ((grouped_code_width(a.total_m, a.groups) + kRows - 1) / kRows / kWarps + a.groups) *
                              p.col_units;
        const int64_t want = bound;
        const int grid = int(want < sms ? (want > 0 ? want : 1) : sms);
        grouped_colwise_kernel<<<grid, kWarps * 32, kSmem, stream>>>(xm, qm, p);
        e = cudaGetLastError();
    }
    return cuda_status(e, "grouped column-wise quantize kernel launch");
}

}  // namespace temx
