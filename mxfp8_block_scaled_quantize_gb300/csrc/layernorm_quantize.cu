// LayerNorm fused with MXFP8 quantisation: the input of LayerNormLinear /
// LayerNormMLP goes from bf16 x to E4M3 codes + E8M0 scales (row-wise and
// column-wise) without writing the normalised bf16 tensor.
//
// Definition (te.LayerNorm as the drop-in of torch.nn.LayerNorm, leeroopedia
// "FP8 Training Quickstart"; parameters 'scale' and 'bias' and epsilon 1e-5,
// TE "Getting Started" JAX page; fused LayerNorm + Linear modules on both
// pages), over each row of H elements:
//   mu = sum(x) / H,  var = sum((x - mu)^2) / H,  rsigma = 1 / sqrt(var + eps),
//   y = (x - mu) * rsigma * gamma + beta,
// then y is MXFP8-quantised exactly as te_mx_quantize quantises its input
// (blocks of 32, scale byte = max(exponent field(amax) - 8, 0), E4M3 RNE
// satfinite, 0xFF / 0x7F for non-finite blocks).  Everything is fp32:
//   mu     = fl(S / H), S a sum of the row (at most 64 additions on the
//            path of any element),
//   var    = fl(S2 / H), S2 a sum of the squares of fl(x - mu) (the same
//            depth; each square rounded on its own or fused into the
//            addition that accumulates it),
//   rsigma = fl(1 / fl(sqrt(fl(var + eps)))),
//   y      = fma(fl(fl(x - mu) * rsigma), gamma, beta).
//
// Two launches.  ln_stats_kernel: persistent; four warps per row (one for
// rows under 2048 elements), each warp's part of the row copied into shared
// memory (two buffers per warp, so the next copy overlaps this row's sums)
// and read there twice; writes mu and rsigma.
// ln_apply_kernel: every warp runs its own TMA pipeline over units of 32 rows
// x 64 columns (like the MXFP8 quantiser), normalises each unit with the row
// statistics and gamma / beta, quantises it, stages the codes in the unit's
// own buffer and writes them with TMA stores.  Both orientations evaluate y
// once per element (lane = 2 columns x 32 rows: column blocks are lane-local,
// row blocks are reduced through a transposed scratch); one orientation alone
// uses its natural layout (row-wise: lane = row).  No CTA-wide barrier, no
// cluster.  The apply kernel reads x again: from L2 when the activation is
// well under the L2 size, from DRAM for one the size of L2 (measured: a
// 117 MB activation is re-read from DRAM).
#include <cuda_runtime.h>

#include "e4m3.cuh"
#include "ptx.cuh"
#include "temx_internal.h"
#include "units.cuh"

namespace temx {

namespace {

constexpr int kUnitRows = 32;                    // rows per unit (one column-wise block)
constexpr int kUnitCols = 64;                    // columns per unit (128 bytes of bf16)
constexpr int kUnitBytes = kUnitRows * kUnitCols * 2;
constexpr int kApplyWarps = 16;
constexpr int kApplyStages = 3;
// Per warp: the unit ring and two side areas (this unit's and the next one's)
// with the row statistics (mu, mu, rsigma, rsigma per row) and gamma / beta
// of the unit's columns in fp32.
constexpr int kSideBytes = kUnitRows * 16 + 2 * kUnitCols * 4;
constexpr int kWarpBytes = kApplyStages * kUnitBytes + 2 * kSideBytes;
constexpr int kApplySmem = kApplyWarps * kWarpBytes + 1024;
constexpr int kStatsMaxWarps = 32;               // warps per statistics CTA, at most
constexpr int kStatsSmem = 220 * 1024;           // two row buffers per warp
constexpr int kStatsAcc = 8;                     // independent accumulators per lane
constexpr int kStatsParts = 4;                   // warps per row (long rows)

struct ApplyParams {
    int64_t rows, hidden;
    const float* mu;
    const float* rsigma;
    const uint16_t* gamma;
    const uint16_t* beta;
    uint8_t* s_row;
    int64_t ld_s_row;
    uint8_t* s_col;
    int64_t ld_s_col;
    int64_t col_units;     // ceil(hidden / 64)
    int64_t units;         // ceil(rows / 32) * col_units
    unsigned int* status;
};

// Packed fp32 pairs (Blackwell f32x2 arithmetic; each half rounds as the
// scalar operation would).
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float lo2(uint64_t v) { return __uint_as_float(uint32_t(v)); }
__device__ __forceinline__ float hi2(uint64_t v) { return __uint_as_float(uint32_t(v >> 32)); }
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// A bf16 pair (one 32-bit word) as an fp32 pair (exact).
__device__ __forceinline__ uint64_t bf2(uint32_t w) { return pack2(bf16_lo(w), bf16_hi(w)); }
// max(|a|, |b|) in magnitude (the sign bit is meaningless); NaN if either is NaN.
__device__ __forceinline__ float maxabs(float a, float b) {
    float d;
    asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ uint64_t lds64(uint32_t addr) {
    uint64_t v;
    asm volatile("ld.shared.b64 %0, [%1];" : "=l"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void lds128x2(uint32_t addr, uint64_t& a, uint64_t& b) {
    asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(addr));
}
__device__ __forceinline__ void sts64(uint32_t addr, uint64_t v) {
    asm volatile("st.shared.b64 [%0], %1;" :: "r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ void sts16(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b16 [%0], %1;" :: "r"(addr), "h"(static_cast<uint16_t>(v)) : "memory");
}

// Pairwise sum of n fp32 pairs (log2 n levels), then the two halves: a tree of
// depth log2(n) + 1 over 2n values.
template <int kN>
__device__ __forceinline__ float tree2(uint64_t (&v)[kN]) {
#pragma unroll
    for (int s = kN / 2; s >= 1; s >>= 1)
#pragma unroll
        for (int i = 0; i < s; ++i) v[i] = add2(v[i], v[i + s]);
    return __fadd_rn(lo2(v[0]), hi2(v[0]));
}

// E8M0 byte of an MX block from |amax| as fp32 bits (exponent field - 8,
// floored at 0; 0xFF for NaN/inf).
__device__ __forceinline__ uint32_t mx_scale_byte_f32(float amax) {
    const uint32_t ef = (__float_as_uint(amax) & 0x7FFFFFFFu) >> 23;
    if (ef == 0xFFu) return 0xFFu;
    return ef > 8u ? ef - 8u : 0u;
}

// Byte offset of 16-byte chunk c of 64-byte row r in a 64-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw64(int r, int c) { return uint32_t(r * 64 + ((c ^ ((r >> 1) & 3)) << 4)); }


// ---------------------------------------------------------------- statistics

// fl(x + c) and fl(x - c) for the bf16 x in the low / high half of a word
// (mixed-precision add / sub: one rounding of the exact result, as the fp32
// operation on the exactly widened x).
__device__ __forceinline__ float addb_lo(uint32_t w, float c) {
    float d;
    asm("{.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.bf16 %0, l, %2;\n\t}" : "=f"(d) : "r"(w), "f"(c));
    return d;
}
__device__ __forceinline__ float addb_hi(uint32_t w, float c) {
    float d;
    asm("{.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.bf16 %0, h, %2;\n\t}" : "=f"(d) : "r"(w), "f"(c));
    return d;
}
// (fl(lo - c), fl(hi - c)) of a bf16 pair as an fp32 pair.
__device__ __forceinline__ uint64_t subb2(uint32_t w, float c) {
    float a, b;
    asm("{.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tsub.rn.f32.bf16 %0, l, %3;\n\tsub.rn.f32.bf16 %1, h, %3;\n\t}"
        : "=f"(a), "=f"(b) : "r"(w), "f"(c));
    return pack2(a, b);
}
// Warp sum in a fixed butterfly order (every lane gets the same value).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Each row part is copied into shared memory with one bulk asynchronous copy,
// so both passes read it there and x is read from HBM once.  Longest chain of
// additions for rows of at most 32768 elements (four parts of 1024 vectors, 32
// per lane, 4 per accumulator): 8 x 4 + 3 + 5 + 2 = 42 for the sum, 4 x 4 +
// 3 + 1 + 5 + 2 = 27 for the squares; rows under 2048 elements (one warp, at
// most 8 vectors per lane): 8 + 3 + 5 = 16.
// L2 cache policies: the statistics kernel's copies ask to keep x in L2 for
// the apply kernel (evict last), which then reads it for the last time
// (evict first).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy) : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* desc, uint32_t bar, int32_t x,
                                                 int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(desc)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// One part of a row (nvec 16-byte vectors at shared address `row`): the sum
// of its elements (kSquares false) or of their squared deviations from mu.
// Lane l takes vectors l, l + 32, ... into kStatsAcc accumulators in turn.
// Sums: every element is added to its accumulator in order (8 additions per
// vector).  Squares: (x - mu) in pairs, each pair accumulated by a fused
// multiply-add into a pair accumulator (4 per vector).  Then the
// accumulators pairwise (3 levels; squares: + the two halves) and the lanes
// by a butterfly (5).
template <bool kSquares>
__device__ __forceinline__ float row_pass(uint32_t row, int nvec, int lane, float mu) {
    if constexpr (!kSquares) {
        float acc[kStatsAcc];
#pragma unroll
        for (int a = 0; a < kStatsAcc; ++a) acc[a] = 0.0f;
        for (int v = lane; v < nvec; v += 32 * kStatsAcc) {
#pragma unroll
            for (int a = 0; a < kStatsAcc; ++a)
                if (v + 32 * a < nvec) {
                    const uint4 x = lds128(row + (v + 32 * a) * 16);
                    float t = acc[a];
                    t = addb_hi(x.x, addb_lo(x.x, t));
                    t = addb_hi(x.y, addb_lo(x.y, t));
                    t = addb_hi(x.z, addb_lo(x.z, t));
                    acc[a] = addb_hi(x.w, addb_lo(x.w, t));
                }
        }
#pragma unroll
        for (int w = kStatsAcc / 2; w >= 1; w >>= 1)
#pragma unroll
            for (int a = 0; a < w; ++a) acc[a] = __fadd_rn(acc[a], acc[a + w]);
        return warp_sum(acc[0]);
    } else {
        uint64_t acc[kStatsAcc];
#pragma unroll
        for (int a = 0; a < kStatsAcc; ++a) acc[a] = 0;
        for (int v = lane; v < nvec; v += 32 * kStatsAcc) {
#pragma unroll
            for (int a = 0; a < kStatsAcc; ++a)
                if (v + 32 * a < nvec) {
                    const uint4 x = lds128(row + (v + 32 * a) * 16);
                    const uint64_t d0 = subb2(x.x, mu), d1 = subb2(x.y, mu), d2 = subb2(x.z, mu), d3 = subb2(x.w, mu);
                    acc[a] = fma2(d3, d3, fma2(d2, d2, fma2(d1, d1, fma2(d0, d0, acc[a]))));
                }
        }
#pragma unroll
        for (int w = kStatsAcc / 2; w >= 1; w >>= 1)
#pragma unroll
            for (int a = 0; a < w; ++a) acc[a] = add2(acc[a], acc[a + w]);
        return warp_sum(__fadd_rn(lo2(acc[0]), hi2(acc[0])));
    }
}

// Barrier over the `n` threads of one row group (named barrier `id`) that
// also returns the AND of `ok` over them.
__device__ __forceinline__ bool group_and(bool ok, int id, int n) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"(uint32_t(ok)), "r"(id), "r"(n) : "memory");
    return r != 0;
}
__device__ __forceinline__ void group_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void group_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" :: "r"(id), "r"(n) : "memory");
}

// Persistent.  A row is shared by a group of kStatsParts warps (or taken by
// one warp when rows are short), warp p of the group taking the p-th
// contiguous part of it; group g of the grid takes rows g, g + G, g + 2G, ...
// (G groups in the grid).  Each warp copies its part through two buffers, so
// the next row's copy is in flight while this row is summed.  The parts' sums
// meet in shared memory behind the group's named barriers and are added in a
// fixed order: barrier g (every warp waits; it also ANDs the copy waits, so a
// group gives up together) for the sum, barrier 8 + g for the squares (only
// part 0 waits: it alone finishes the row).  The copies carry an evict-last
// hint for the apply kernel's second read of x.
__global__ void __launch_bounds__(kStatsMaxWarps * 32)
ln_stats_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t hidden, int64_t ld_x, float eps,
                float* __restrict__ mu_out, float* __restrict__ rs_out, int parts, unsigned int* status) {
    extern __shared__ __align__(16) uint8_t rowbuf[];
    __shared__ __align__(8) uint64_t bars[kStatsMaxWarps][2];
    // [group * parts + part][S of even rows, S of odd rows, S2]: part 0 may
    // still read a row's S when the other parts write the next row's
    __shared__ float part_sum[kStatsMaxWarps][3];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int groups = int(blockDim.x >> 5) / parts;
    const int g = warp / parts, part = warp % parts;
    const int64_t gg = int64_t(blockIdx.x) * groups + g, ngroups = int64_t(gridDim.x) * groups;
    if (gg >= rows) return;                                // the whole group leaves
    const int64_t n_mine = (rows - gg + ngroups - 1) / ngroups;
    const int64_t part_elems = hidden / parts;             // a multiple of 8
    const uint32_t bytes = uint32_t(part_elems) * 2;
    const uint32_t buf = smem_u32(rowbuf) + uint32_t(warp) * 2 * bytes;
    const uint16_t* src = x + part * part_elems;
    const uint64_t policy = l2_policy_evict_last();
    // the apply kernel may be scheduled as these CTAs retire (it waits for
    // this grid's completion before reading its results)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (lane == 0) {
        mbar_init(smem_u32(&bars[warp][0]), 1);
        mbar_init(smem_u32(&bars[warp][1]), 1);
        fence_mbarrier_init();
        for (int s = 0; s < 2 && s < n_mine; ++s) {
            const uint32_t bar = smem_u32(&bars[warp][s]);
            mbar_arrive_expect_tx(bar, bytes);
            bulk_load(buf + s * bytes, src + (gg + s * ngroups) * ld_x, bytes, bar, policy);
        }
    }
    __syncwarp();
    const int nvec = int(part_elems / 8);
    const float h = float(hidden);
    const int nthreads = parts * 32;
    const int w0 = g * parts;
    for (int64_t i = 0; i < n_mine; ++i) {
        const int s = int(i & 1);
        const uint32_t bar = smem_u32(&bars[warp][s]);
        bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar, uint32_t((i >> 1) & 1), status));
        const uint32_t row = buf + s * bytes;
        float sum = row_pass<false>(row, nvec, lane, 0.0f);   // reads garbage (in bounds) if a copy timed out
        if (parts > 1) {
            if (lane == 0) part_sum[warp][s] = sum;
            ok = group_and(ok, g, nthreads);
            sum = __fadd_rn(__fadd_rn(part_sum[w0][s], part_sum[w0 + 1][s]),
                            __fadd_rn(part_sum[w0 + 2][s], part_sum[w0 + 3][s]));
        }
        if (!ok) {
            // Gave up (the whole group): let this warp's copies still in flight land before leaving.
            if (lane == 0)
                for (int64_t j = i; j < i + 2 && j < n_mine; ++j)
                    mbar_wait(smem_u32(&bars[warp][j & 1]), uint32_t((j >> 1) & 1), status);
            return;
        }
        const float mu = __fdiv_rn(sum, h);
        float sq = row_pass<true>(row, nvec, lane, mu);
        // row_pass ends in a butterfly over every lane: the buffer has been read
        if (lane == 0 && i + 2 < n_mine) {
            mbar_arrive_expect_tx(bar, bytes);
            bulk_load(row, src + (gg + (i + 2) * ngroups) * ld_x, bytes, bar, policy);
        }
        if (parts > 1) {
            if (lane == 0) part_sum[warp][2] = sq;
            if (part != 0) {
                group_arrive(8 + g, nthreads);
                continue;
            }
            group_sync(8 + g, nthreads);
            sq = __fadd_rn(__fadd_rn(part_sum[w0][2], part_sum[w0 + 1][2]),
                           __fadd_rn(part_sum[w0 + 2][2], part_sum[w0 + 3][2]));
        }
        if (lane == 0) {
            const float rs = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(sq, h), eps)));
            const int64_t r = gg + i * ngroups;
            mu_out[r] = mu;
            rs_out[r] = rs;
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------- normalise + quantise

// One unit (32 rows x 64 columns at shared address `unit`, 128-byte swizzle):
// normalise with the row statistics at `stat` and gamma / beta at `gf` /
// `bf`, quantise row- and/or column-wise, stage the codes in the unit buffer
// (row codes: 64-byte swizzle over its first 2 KB; column codes: 64 columns x
// 32 bytes over the second 2 KB) and write scale bytes.
template <bool kRowwise, bool kColwise>
__device__ __forceinline__ void quantize_unit(const ApplyParams& p, uint32_t unit, int64_t r0, int64_t c0, int lane,
                                              uint32_t stat, uint32_t gaddr, uint32_t baddr) {
    const int valid = p.hidden - c0 < kUnitCols ? int(p.hidden - c0) : kUnitCols;
    uint32_t rc[2][8];                           // row codes: row `lane`, two 32-column blocks
    uint32_t sr[2] = {0, 0};
    if (kRowwise) {
        uint64_t mm, rr;
        lds128x2(stat + lane * 16, mm, rr);
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
            uint64_t y[16];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int q = blk * 4 + t;                         // 16-byte chunk of the row (8 columns)
                const uint4 x = lds128(unit + lane * 128 + ((q ^ (lane & 7)) << 4));
                uint64_t g0, g1, g2, g3, b0, b1, b2, b3;
                lds128x2(gaddr + q * 32, g0, g1);
                lds128x2(gaddr + q * 32 + 16, g2, g3);
                lds128x2(baddr + q * 32, b0, b1);
                lds128x2(baddr + q * 32 + 16, b2, b3);
                y[4 * t + 0] = fma2(mul2(sub2(bf2(x.x), mm), rr), g0, b0);
                y[4 * t + 1] = fma2(mul2(sub2(bf2(x.y), mm), rr), g1, b1);
                y[4 * t + 2] = fma2(mul2(sub2(bf2(x.z), mm), rr), g2, b2);
                y[4 * t + 3] = fma2(mul2(sub2(bf2(x.w), mm), rr), g3, b3);
            }
            float mx[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) mx[i] = maxabs(lo2(y[i]), hi2(y[i]));
#pragma unroll
            for (int s2 = 8; s2 >= 1; s2 >>= 1)
#pragma unroll
                for (int i = 0; i < s2; ++i) mx[i] = maxabs(mx[i], mx[i + s2]);
            sr[blk] = mx_scale_byte_f32(mx[0]);
            const float m = inv_scale(sr[blk]);
            const uint64_t m2 = pack2(m, m);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint64_t a = mul2(y[2 * i], m2), b = mul2(y[2 * i + 1], m2);
                rc[blk][i] = cvt_e4m3x2(lo2(a), hi2(a)) | (cvt_e4m3x2(lo2(b), hi2(b)) << 16);
            }
            if (sr[blk] == 0xFFu) {
#pragma unroll
                for (int i = 0; i < 8; ++i) rc[blk][i] = 0x7F7F7F7Fu;
            }
        }
    }
    uint32_t cc_lo[8], cc_hi[8];                 // column codes: columns 2 lane, 2 lane + 1, rows 0..31
    uint32_t s_lo = 0, s_hi = 0;
    if (kColwise) {
        const uint64_t g2 = lds64(gaddr + lane * 8), b2 = lds64(baddr + lane * 8);
        const uint32_t cbase = unit + ((lane & 3) << 2);
        const int ch = lane >> 2;
        uint64_t y[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const uint32_t x = lds32(cbase + r * 128 + ((ch ^ (r & 7)) << 4));
            uint64_t mu2, rs2;
            lds128x2(stat + r * 16, mu2, rs2);
            y[r] = fma2(mul2(sub2(bf2(x), mu2), rs2), g2, b2);
        }
        float ml[16], mh[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            ml[i] = maxabs(lo2(y[2 * i]), lo2(y[2 * i + 1]));
            mh[i] = maxabs(hi2(y[2 * i]), hi2(y[2 * i + 1]));
        }
#pragma unroll
        for (int s2 = 8; s2 >= 1; s2 >>= 1)
#pragma unroll
            for (int i = 0; i < s2; ++i) {
                ml[i] = maxabs(ml[i], ml[i + s2]);
                mh[i] = maxabs(mh[i], mh[i + s2]);
            }
        s_lo = mx_scale_byte_f32(ml[0]);
        s_hi = mx_scale_byte_f32(mh[0]);
        const uint64_t m2 = pack2(inv_scale(s_lo), inv_scale(s_hi));
#pragma unroll
        for (int r = 0; r < 32; ++r) y[r] = mul2(y[r], m2);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            cc_lo[i] = cvt_e4m3x2(lo2(y[4 * i]), lo2(y[4 * i + 1])) |
                       (cvt_e4m3x2(lo2(y[4 * i + 2]), lo2(y[4 * i + 3])) << 16);
            cc_hi[i] = cvt_e4m3x2(hi2(y[4 * i]), hi2(y[4 * i + 1])) |
                       (cvt_e4m3x2(hi2(y[4 * i + 2]), hi2(y[4 * i + 3])) << 16);
        }
        if (s_lo == 0xFFu) {
#pragma unroll
            for (int i = 0; i < 8; ++i) cc_lo[i] = 0x7F7F7F7Fu;
        }
        if (s_hi == 0xFFu) {
#pragma unroll
            for (int i = 0; i < 8; ++i) cc_hi[i] = 0x7F7F7F7Fu;
        }
    }
    __syncwarp();                                // every lane has read the unit: reuse it for the codes
    if (kRowwise) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t* w = rc[c >> 1] + 4 * (c & 1);
            sts128(unit + sw64(lane, c), w[0], w[1], w[2], w[3]);
        }
        const int64_t r = r0 + lane;
        if (r < p.rows) {
            uint8_t* sp = p.s_row + r * p.ld_s_row + (c0 >> 5);
            if (valid > 32) st_global_u16(sp, sr[0] | (sr[1] << 8));
            else st_global_u8(sp, sr[0]);
        }
    }
    if (kColwise) {
        const uint32_t cb = unit + 2048 + lane * 64;        // column 2 lane, then 2 lane + 1: 32 bytes each
        sts128(cb, cc_lo[0], cc_lo[1], cc_lo[2], cc_lo[3]);
        sts128(cb + 16, cc_lo[4], cc_lo[5], cc_lo[6], cc_lo[7]);
        sts128(cb + 32, cc_hi[0], cc_hi[1], cc_hi[2], cc_hi[3]);
        sts128(cb + 48, cc_hi[4], cc_hi[5], cc_hi[6], cc_hi[7]);
        if (2 * lane < valid) {                               // valid is a multiple of 32
            uint8_t* sp = p.s_col + (c0 + 2 * lane) * p.ld_s_col + (r0 >> 5);
            st_global_u8(sp, s_lo);
            st_global_u8(sp + p.ld_s_col, s_hi);
        }
    }
}

// Both orientations from one evaluation of y per element.  Lane l holds
// columns 2l (lo) and 2l + 1 (hi) of all 32 rows as fp32 pairs of consecutive
// rows, ylo[k] = (y[2k][2l], y[2k+1][2l]) and yhi[k] likewise, so the column
// blocks are lane-local and the statistics of a row pair are one load.  A row
// block spans 16 lanes: every lane writes its per-row-pair maxima into the
// consumed unit (a 16 x 32 scratch of fp32 pairs, 16-byte chunks XOR-swizzled
// by row pair), lane (p, b) = (l & 15, l >> 4) reduces rows 2p and 2p + 1 of
// block b, and the row scales come back through the statistics area of the
// side data, [block][row] in fp32.  Row codes are staged one 16-bit pair per
// lane and row, column codes as in the column-wise path.  The side data's
// statistics are (mu[2k], mu[2k+1], rsigma[2k], rsigma[2k+1]) per row pair.
__device__ __forceinline__ void quantize_unit_both(const ApplyParams& p, uint32_t unit, int64_t r0, int64_t c0,
                                                   int lane, uint32_t stat, uint32_t gaddr, uint32_t baddr) {
    const int valid = p.hidden - c0 < kUnitCols ? int(p.hidden - c0) : kUnitCols;
    uint64_t ylo[16], yhi[16];
    {
        const uint64_t g2 = lds64(gaddr + lane * 8), b2 = lds64(baddr + lane * 8);
        const uint64_t glo = pack2(lo2(g2), lo2(g2)), ghi = pack2(hi2(g2), hi2(g2));
        const uint64_t blo = pack2(lo2(b2), lo2(b2)), bhi = pack2(hi2(b2), hi2(b2));
        const uint32_t cbase = unit + ((lane & 3) << 2);
        const int ch = lane >> 2;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int r = 2 * k;
            const uint32_t w0 = lds32(cbase + r * 128 + ((ch ^ (r & 7)) << 4));
            const uint32_t w1 = lds32(cbase + (r + 1) * 128 + ((ch ^ ((r + 1) & 7)) << 4));
            uint64_t mu2, rs2;
            lds128x2(stat + k * 16, mu2, rs2);
            ylo[k] = fma2(mul2(sub2(pack2(bf16_lo(w0), bf16_lo(w1)), mu2), rs2), glo, blo);
            yhi[k] = fma2(mul2(sub2(pack2(bf16_hi(w0), bf16_hi(w1)), mu2), rs2), ghi, bhi);
        }
    }
    __syncwarp();                                // every lane has read x and the statistics
    // per-row-pair maxima of this lane's two columns: scratch [pair k][lane l]
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const uint64_t m = pack2(maxabs(lo2(ylo[k]), lo2(yhi[k])), maxabs(hi2(ylo[k]), hi2(yhi[k])));
        sts64(unit + k * 256 + (lane >> 4) * 128 + ((((lane >> 1) & 7) ^ (k & 7)) << 4) + (lane & 1) * 8, m);
    }
    __syncwarp();
    const int pr = lane & 15, blk = lane >> 4;   // rows 2 pr, 2 pr + 1 of row block blk
    float ta[16], tb[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint64_t u, v;
        lds128x2(unit + pr * 256 + blk * 128 + ((j ^ (pr & 7)) << 4), u, v);
        ta[2 * j] = lo2(u); tb[2 * j] = hi2(u);
        ta[2 * j + 1] = lo2(v); tb[2 * j + 1] = hi2(v);
    }
#pragma unroll
    for (int s2 = 8; s2 >= 1; s2 >>= 1)
#pragma unroll
        for (int i = 0; i < s2; ++i) {
            ta[i] = maxabs(ta[i], ta[i + s2]);
            tb[i] = maxabs(tb[i], tb[i + s2]);
        }
    const uint32_t sa = mx_scale_byte_f32(ta[0]), sb = mx_scale_byte_f32(tb[0]);
    {
        // row 2 pr (lanes of block 0) / 2 pr + 1 (block 1): both blocks' bytes
        const uint32_t mine = sa | (sb << 8);
        const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, mine, 16);
        const int64_t r = r0 + 2 * pr + blk;
        if (r < p.rows) {
            uint8_t* sp = p.s_row + r * p.ld_s_row + (c0 >> 5);
            const uint32_t b0 = blk ? (other >> 8) : (mine & 0xFFu);      // block 0's byte of row r
            const uint32_t b1 = blk ? (mine >> 8) : (other & 0xFFu);      // block 1's byte of row r
            if (valid > 32) st_global_u16(sp, b0 | (b1 << 8));
            else st_global_u8(sp, b0);
        }
        sts64(stat + blk * 128 + pr * 8, pack2(inv_scale(sa), inv_scale(sb)));   // -inf for a non-finite block
    }
    const bool nonfinite = __any_sync(0xFFFFFFFFu, sa == 0xFFu || sb == 0xFFu);
    __syncwarp();                                // row scales visible; the scratch is consumed
    {
        const uint32_t ms = stat + (lane >> 4) * 128;      // this lane's row block
        const uint32_t rcode = unit + (lane & 7) * 2;
        const int rch = lane >> 3;
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
            uint64_t m_a, m_b;                   // (m[2k], m[2k+1]), (m[2k+2], m[2k+3])
            lds128x2(ms + k * 8, m_a, m_b);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const uint64_t m2 = t ? m_b : m_a;
                const int r = 2 * (k + t);
                const uint64_t a = mul2(ylo[k + t], m2), b = mul2(yhi[k + t], m2);
                uint32_t c_even = cvt_e4m3x2(lo2(a), lo2(b)), c_odd = cvt_e4m3x2(hi2(a), hi2(b));
                if (nonfinite) {
                    if (__float_as_uint(lo2(m2)) == 0xFF800000u) c_even = 0x7F7Fu;
                    if (__float_as_uint(hi2(m2)) == 0xFF800000u) c_odd = 0x7F7Fu;
                }
                sts16(rcode + r * 64 + ((rch ^ ((r >> 1) & 3)) << 4), c_even);
                sts16(rcode + (r + 1) * 64 + ((rch ^ (((r + 1) >> 1) & 3)) << 4), c_odd);
            }
        }
    }
    // column blocks: lane-local
    float ml[16], mh[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        ml[k] = maxabs(lo2(ylo[k]), hi2(ylo[k]));
        mh[k] = maxabs(lo2(yhi[k]), hi2(yhi[k]));
    }
#pragma unroll
    for (int s2 = 8; s2 >= 1; s2 >>= 1)
#pragma unroll
        for (int i = 0; i < s2; ++i) {
            ml[i] = maxabs(ml[i], ml[i + s2]);
            mh[i] = maxabs(mh[i], mh[i + s2]);
        }
    const uint32_t s_lo = mx_scale_byte_f32(ml[0]), s_hi = mx_scale_byte_f32(mh[0]);
    const float il = inv_scale(s_lo), ih = inv_scale(s_hi);
    const uint64_t ml2 = pack2(il, il), mh2 = pack2(ih, ih);
    uint32_t cc_lo[8], cc_hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint64_t a = mul2(ylo[2 * i], ml2), b = mul2(ylo[2 * i + 1], ml2);
        const uint64_t c = mul2(yhi[2 * i], mh2), d = mul2(yhi[2 * i + 1], mh2);
        cc_lo[i] = cvt_e4m3x2(lo2(a), hi2(a)) | (cvt_e4m3x2(lo2(b), hi2(b)) << 16);
        cc_hi[i] = cvt_e4m3x2(lo2(c), hi2(c)) | (cvt_e4m3x2(lo2(d), hi2(d)) << 16);
    }
    if (s_lo == 0xFFu) {
#pragma unroll
        for (int i = 0; i < 8; ++i) cc_lo[i] = 0x7F7F7F7Fu;
    }
    if (s_hi == 0xFFu) {
#pragma unroll
        for (int i = 0; i < 8; ++i) cc_hi[i] = 0x7F7F7F7Fu;
    }
    const uint32_t cb = unit + 2048 + lane * 64;            // column 2 lane, then 2 lane + 1: 32 bytes each
    sts128(cb, cc_lo[0], cc_lo[1], cc_lo[2], cc_lo[3]);
    sts128(cb + 16, cc_lo[4], cc_lo[5], cc_lo[6], cc_lo[7]);
    sts128(cb + 32, cc_hi[0], cc_hi[1], cc_hi[2], cc_hi[3]);
    sts128(cb + 48, cc_hi[4], cc_hi[5], cc_hi[6], cc_hi[7]);
    if (2 * lane < valid) {                                   // valid is a multiple of 32
        uint8_t* sp = p.s_col + (c0 + 2 * lane) * p.ld_s_col + (r0 >> 5);
        st_global_u8(sp, s_lo);
        st_global_u8(sp + p.ld_s_col, s_hi);
    }
}

template <bool kRowwise, bool kColwise>
__global__ void __launch_bounds__(kApplyWarps * 32, 1)
ln_apply_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap qrow_map,
                const __grid_constant__ CUtensorMap qcol_map, const ApplyParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[kApplyWarps][kApplyStages];

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t gwarp = int64_t(blockIdx.x) * kApplyWarps + warp;
    const int64_t nwarps = int64_t(gridDim.x) * kApplyWarps;
    if (gwarp >= p.units) return;
    const int64_t n_mine = (p.units - gwarp + nwarps - 1) / nwarps;
    const uint32_t ring = smem_u32(smem + warp * (kApplyStages * kUnitBytes));
    // two side areas per warp (this unit's, the next unit's): stat [32][4], gamma [64], beta [64]
    uint8_t* side = smem + kApplyWarps * kApplyStages * kUnitBytes + warp * (2 * kSideBytes);
    // (band, column unit) of this unit, of the next one and of the next load
    const UnitWalk walk(nwarps, p.col_units);
    int32_t band, col;
    walk.start(gwarp, band, col);
    int32_t nband = band, ncol = col;
    walk.step(nband, ncol);
    auto load_side = [&](int32_t b, int32_t c, float& m, float& rs, uint32_t& g2, uint32_t& b2) {
        const int64_t r = int64_t(b) * kUnitRows + lane, cc = int64_t(c) * kUnitCols + 2 * lane;
        m = r < p.rows ? p.mu[r] : 0.0f;
        rs = r < p.rows ? p.rsigma[r] : 0.0f;
        g2 = cc < p.hidden ? *reinterpret_cast<const uint32_t*>(p.gamma + cc) : 0u;
        b2 = cc < p.hidden ? *reinterpret_cast<const uint32_t*>(p.beta + cc) : 0u;
    };
    auto store_side = [&](uint8_t* area, float m, float rs, uint32_t g2, uint32_t b2) {
        if constexpr (kRowwise && kColwise) {          // (mu, mu', rsigma, rsigma') per row pair
            float* pair = reinterpret_cast<float*>(area) + (lane >> 1) * 4 + (lane & 1);
            pair[0] = m;
            pair[2] = rs;
        } else {
            reinterpret_cast<float4*>(area)[lane] = make_float4(m, m, rs, rs);
        }
        reinterpret_cast<float2*>(area + kUnitRows * 16)[lane] = make_float2(bf16_lo(g2), bf16_hi(g2));
        reinterpret_cast<float2*>(area + kUnitRows * 16 + kUnitCols * 4)[lane] = make_float2(bf16_lo(b2), bf16_hi(b2));
    };

    const uint64_t policy = l2_policy_evict_first();
    int32_t lband = band, lcol = col;                  // next unit to load (lane 0)
    if (lane == 0) {
        tma_prefetch_desc(&x_map);
        if (kRowwise) tma_prefetch_desc(&qrow_map);
        if (kColwise) tma_prefetch_desc(&qcol_map);
        for (int s = 0; s < kApplyStages; ++s) mbar_init(smem_u32(&bars[warp][s]), 1);
        fence_mbarrier_init();
        for (int s = 0; s < kApplyStages && s < n_mine; ++s) {
            const uint32_t bar = smem_u32(&bars[warp][s]);
            mbar_arrive_expect_tx(bar, kUnitBytes);
            tma_load_2d_hint(ring + s * kUnitBytes, &x_map, bar, lcol * kUnitCols, lband * kUnitRows, policy);
            walk.step(lband, lcol);
        }
    }
    // mu / rsigma come from the statistics kernel, launched just before this
    // one as its programmatic dependent: wait for it to complete (x itself
    // was complete before the statistics kernel started).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    {
        float m, rs;
        uint32_t g2, b2;
        load_side(band, col, m, rs, g2, b2);
        store_side(side, m, rs, g2, b2);
    }
    __syncwarp();

    int s = 0;
    uint32_t phase = 0;
    for (int64_t i = 0; i < n_mine; ++i) {
        const uint32_t bar = smem_u32(&bars[warp][s]);
        const int64_t r0 = int64_t(band) * kUnitRows, c0 = int64_t(col) * kUnitCols;
        // the next unit's statistics and gamma / beta, loaded now, stored after this unit
        float nm = 0.0f, nrs = 0.0f;
        uint32_t ng = 0, nb = 0;
        if (i + 1 < n_mine) load_side(nband, ncol, nm, nrs, ng, nb);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar, phase, p.status))) {
            // Gave up: let this warp's loads still in flight land before leaving.
            if (lane == 0)
                for (int64_t j = i; j < i + kApplyStages && j < n_mine; ++j)
                    mbar_wait(smem_u32(&bars[warp][j % kApplyStages]), uint32_t((j / kApplyStages) & 1), p.status);
            break;
        }
        const uint32_t unit = ring + s * kUnitBytes;
        const uint32_t sb = smem_u32(side) + uint32_t(i & 1) * kSideBytes;
        if constexpr (kRowwise && kColwise)
            quantize_unit_both(p, unit, r0, c0, lane, sb, sb + kUnitRows * 16, sb + kUnitRows * 16 + kUnitCols * 4);
        else
            quantize_unit<kRowwise, kColwise>(p, unit, r0, c0, lane, sb, sb + kUnitRows * 16,
                                              sb + kUnitRows * 16 + kUnitCols * 4);
        if (i + 1 < n_mine) store_side(side + ((i + 1) & 1) * kSideBytes, nm, nrs, ng, nb);
        fence_proxy_async_smem();                // make the staged codes visible to the TMA engine
        __syncwarp();
        if (lane == 0) {
            if (kRowwise) tma_store_2d(&qrow_map, unit, int32_t(c0), int32_t(r0));
            if (kColwise) tma_store_2d(&qcol_map, unit + 2048, int32_t(r0), int32_t(c0));
            bulk_commit();
            if (i + kApplyStages < n_mine) {
                bulk_wait_read_all();            // the stores have read the unit: refill it
                mbar_arrive_expect_tx(bar, kUnitBytes);
                tma_load_2d_hint(unit, &x_map, bar, lcol * kUnitCols, lband * kUnitRows, policy);
                walk.step(lband, lcol);
            }
        }
        __syncwarp();
        band = nband;
        col = ncol;
        walk.step(nband, ncol);
        if (++s == kApplyStages) {
            s = 0;
            phase ^= 1u;
        }
    }
    if (lane == 0) bulk_wait_all();
}

template <bool R, bool C>
cudaError_t launch_apply(const CUtensorMap& xm, const CUtensorMap& qr, const CUtensorMap& qc, const ApplyParams& p,
                         int sms, cudaStream_t stream) {
    auto kern = ln_apply_kernel<R, C>;
    cudaError_t e = set_smem_attribute_once(reinterpret_cast<const void*>(kern), kApplySmem);
    if (e != cudaSuccess) return e;
    const int64_t want = (p.units + kApplyWarps - 1) / kApplyWarps;
    const int grid = int(want < sms ? want : sms);
    // Programmatic dependent launch: the CTAs may start (and load x) as the
    // statistics kernel's CTAs retire; they wait for its results before
    // reading mu / rsigma.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kApplyWarps * 32);
    cfg.dynamicSmemBytes = kApplySmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, xm, qr, qc, p);
}

}  // namespace

int64_t ln_quantize_max_hidden() { return 32768; }   // keeps the longest chain of additions at 42

te_mx_status ln_quantize_launch(const LnQuantizeArgs& a, cudaStream_t stream) {
    const bool rowwise = a.q_row != nullptr, colwise = a.q_col != nullptr;
    if (a.rows == 0 || a.hidden == 0) return TE_MX_OK;

    unsigned int* status = nullptr;
    te_mx_status st = device_status_ptr(&status);
    if (st != TE_MX_OK) return st;
    int sms = 0;
    if ((st = device_sm_count(&sms)) != TE_MX_OK) return st;
    // statistics: one CTA per SM with as many row groups as two row buffers
    // each allow; rows of 2048 elements or more are shared by four warps (at
    // most 8 groups, barriers 0..15), shorter rows take one warp each (at
    // most 32 groups)
    const int64_t buf_bytes = 2 * a.hidden * 2;
    const int64_t fit = kStatsSmem / buf_bytes;
    const int parts = a.hidden >= 2048 ? kStatsParts : 1;
    const int64_t cap = kStatsMaxWarps / parts;
    const int groups = int(fit < cap ? fit : cap);
    const size_t stats_smem = size_t(groups) * size_t(buf_bytes);
    cudaError_t e = set_smem_attribute_once(reinterpret_cast<const void*>(ln_stats_kernel), kStatsSmem);
    if (e != cudaSuccess) return cuda_status(e, "layernorm statistics kernel attributes");
    const int64_t want = (a.rows + groups - 1) / groups;
    const int64_t blocks = want < int64_t(sms) ? want : int64_t(sms);
    ln_stats_kernel<<<unsigned(blocks), groups * parts * 32, stats_smem, stream>>>(
        static_cast<const uint16_t*>(a.x), a.rows, a.hidden, a.ld_x, a.eps, a.mu, a.rsigma, parts, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e, "layernorm statistics kernel launch");
    if (!rowwise && !colwise) return TE_MX_OK;

    CUtensorMap xm, qr, qc;
    if ((st = encode_tensor_map_2d(&xm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, uint64_t(a.hidden),
                                   uint64_t(a.rows), uint64_t(a.ld_x) * 2, kUnitCols, kUnitRows,
                                   CU_TENSOR_MAP_SWIZZLE_128B)) != TE_MX_OK) return st;
    qr = xm;
    qc = xm;
    if (rowwise && (st = encode_tensor_map_2d(&qr, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.q_row, uint64_t(a.hidden),
                                              uint64_t(a.rows), uint64_t(a.hidden), kUnitCols, kUnitRows,
                                              CU_TENSOR_MAP_SWIZZLE_64B)) != TE_MX_OK) return st;
    if (colwise && (st = encode_tensor_map_2d(&qc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.q_col, uint64_t(a.rows),
                                              uint64_t(a.hidden), uint64_t(a.rows), kUnitRows, kUnitCols,
                                              CU_TENSOR_MAP_SWIZZLE_NONE)) != TE_MX_OK) return st;
    ApplyParams p;
    p.rows = a.rows; p.hidden = a.hidden;
    p.mu = a.mu; p.rsigma = a.rsigma;
    p.gamma = static_cast<const uint16_t*>(a.gamma);
    p.beta = static_cast<const uint16_t*>(a.beta);
    p.s_row = a.s_row; p.ld_s_row = a.ld_s_row;
    p.s_col = a.s_col; p.ld_s_col = a.ld_s_col;
    p.col_units = (a.hidden + kUnitCols - 1) / kUnitCols;
    p.units = ((a.rows + kUnitRows - 1) / kUnitRows) * p.col_units;
    p.status = status;
    if (rowwise && colwise) e = launch_apply<true, true>(xm, qr, qc, p, sms, stream);
    else if (colwise) e = launch_apply<false, true>(xm, qr, qc, p, sms, stream);
    else e = launch_apply<true, false>(xm, qr, qc, p, sms, stream);
    return cuda_status(e, "layernorm quantize kernel launch");
}

}  // namespace temx
