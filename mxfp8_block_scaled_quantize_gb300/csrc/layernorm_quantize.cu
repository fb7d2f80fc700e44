// LayerNorm fused with MXFP8 quantisation: the input of LayerNormLinear /
// LayerNormMLP goes from bf16 x to E4M3 codes + E8M0 scales (row-wise and
// column-wise) in one pass over HBM, without writing the normalised bf16
// tensor.
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
//   mu     = fl(S / H), S a tree sum of the row (depth <= 64 additions),
//   var    = fl(S2 / H), S2 a tree sum of fl(fl(x - mu)^2),
//   rsigma = fl(1 / fl(sqrt(fl(var + eps)))),
//   y      = fma(fl(fl(x - mu) * rsigma), gamma, beta).
//
// Work decomposition.  A cluster of k CTAs (k = 1, 2, 4 or 8) owns a band of
// 32 rows; CTA rank q holds chunks [q cpc, (q+1) cpc) of 64 columns in shared
// memory (TMA, 128-byte swizzle, one mbarrier per chunk), and warp w works on
// its chunks w, w + 8, ...  Pass 1: lane l sums row l of each chunk (a
// 6-level tree per chunk), warps and then CTAs are combined in a fixed order
// (CTA partials are read over distributed shared memory), so every CTA of the
// cluster derives the same mu.  Pass 2 does the same for the squared
// deviations.  Pass 3 quantises each chunk both ways from the shared-memory
// copy (row-wise: lane = row; column-wise: lane = 2 columns x 32 rows, so one
// column block per lane), stages the codes in the chunk's own buffer and
// writes them with TMA stores.
#include <cuda_runtime.h>

#include "e4m3.cuh"
#include "ptx.cuh"
#include "temx_internal.h"

namespace temx {

namespace {

constexpr int kBand = 32;                        // rows per cluster (one column-wise block)
constexpr int kChunkCols = 64;                   // columns per chunk (128 bytes of bf16)
constexpr int kChunkBytes = kBand * kChunkCols * 2;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxChunks = 48;                   // per CTA: 192 KB of shared memory
constexpr int kMaxCluster = 8;

struct LnParams {
    int64_t rows, hidden;
    float eps;
    const uint16_t* gamma;
    const uint16_t* beta;
    uint8_t* s_row;
    int64_t ld_s_row;
    uint8_t* s_col;
    int64_t ld_s_col;
    float* mu;
    float* rsigma;
    int nch;               // chunks per row: ceil(hidden / 64)
    int cpc;               // chunks per CTA
    unsigned int* status;
};

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t cluster_addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
    return v;
}

// Pairwise sum of 64 floats (six levels of additions).
__device__ __forceinline__ float tree64(float (&v)[64]) {
#pragma unroll
    for (int s = 32; s >= 1; s >>= 1)
#pragma unroll
        for (int i = 0; i < s; ++i) v[i] = __fadd_rn(v[i], v[i + s]);
    return v[0];
}

// The 64 bf16 of row `r` of a chunk (128-byte swizzle) as 32 words.
__device__ __forceinline__ void load_row(uint32_t chunk, int r, uint32_t (&w)[32]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 v = lds128(chunk + r * 128 + ((j ^ (r & 7)) << 4));
        w[4 * j + 0] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
    }
}

__device__ __forceinline__ float ln_y(float x, float mu, float rs, float g, float b) {
    return __fmaf_rn(__fmul_rn(__fsub_rn(x, mu), rs), g, b);
}

// E8M0 byte of an MX block from |amax| as fp32 bits (exponent field - 8,
// floored at 0; 0xFF for NaN/inf).
__device__ __forceinline__ uint32_t mx_scale_byte_f32(uint32_t amax_bits) {
    const uint32_t ef = amax_bits >> 23;
    if (ef == 0xFFu) return 0xFFu;
    return ef > 8u ? ef - 8u : 0u;
}

// Byte offset of 16-byte chunk c of 64-byte row r in a 64-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw64(int r, int c) { return uint32_t(r * 64 + ((c ^ ((r >> 1) & 3)) << 4)); }

template <bool kRowwise, bool kColwise>
__global__ void __launch_bounds__(kThreads, 2)
ln_quantize_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap qrow_map,
                   const __grid_constant__ CUtensorMap qcol_map, const LnParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[kMaxChunks];
    __shared__ float wsum[kWarps][kBand];
    __shared__ float part[2][kBand];             // this CTA's partial sums, read by the whole cluster
    __shared__ float mu_s[kBand], rs_s[kBand];
    __shared__ int abort_flag;

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t base = smem_u32(smem);
    uint16_t* g_s = reinterpret_cast<uint16_t*>(smem + p.cpc * kChunkBytes);   // gamma of this CTA's columns
    uint16_t* b_s = g_s + p.cpc * kChunkCols;                                    // beta
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank(), k = cluster_nctarank();
    const int64_t r0 = int64_t(blockIdx.x / k) * kBand;
    const int chunk0 = int(rank) * p.cpc;
    const int my_n = max(0, min(p.cpc, p.nch - chunk0));
    const float h = float(p.hidden);
    volatile int* abort_v = &abort_flag;

    if (tid == 0) {
        for (int j = 0; j < my_n; ++j) mbar_init(smem_u32(&bars[j]), 1);
        abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    if (tid == 0) {
        tma_prefetch_desc(&x_map);
        for (int j = 0; j < my_n; ++j) {
            const uint32_t bar = smem_u32(&bars[j]);
            mbar_arrive_expect_tx(bar, kChunkBytes);
            tma_load_2d(base + j * kChunkBytes, &x_map, bar, (chunk0 + j) * kChunkCols, int32_t(r0));
        }
    }
    for (int i = tid; i < my_n * kChunkCols; i += kThreads) {
        const int64_t c = int64_t(chunk0) * kChunkCols + i;
        g_s[i] = c < p.hidden ? p.gamma[c] : uint16_t(0);
        b_s[i] = c < p.hidden ? p.beta[c] : uint16_t(0);
    }

    // ---------------------------------------------------------------- pass 1: row sums
    float acc = 0.0f;
    for (int j = warp; j < my_n; j += kWarps) {
        if (!mbar_wait(smem_u32(&bars[j]), 0, p.status)) {
            *abort_v = 1;
            break;
        }
        uint32_t w[32];
        load_row(base + j * kChunkBytes, lane, w);
        float v[64];
#pragma unroll
        for (int i = 0; i < 32; ++i) { v[2 * i] = bf16_lo(w[i]); v[2 * i + 1] = bf16_hi(w[i]); }
        acc = __fadd_rn(acc, tree64(v));         // columns past the row end were loaded as 0
    }
    wsum[warp][lane] = acc;
    __syncthreads();                             // also publishes gamma/beta
    if (warp == 0) {
        float s = wsum[0][lane];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) s = __fadd_rn(s, wsum[w][lane]);
        part[0][lane] = s;
    }
    cluster_sync();
    if (warp == 0) {
        float s = 0.0f;
        for (uint32_t q = 0; q < k; ++q) s = __fadd_rn(s, ld_cluster_f32(mapa_shared(smem_u32(&part[0][lane]), q)));
        mu_s[lane] = __fdiv_rn(s, h);
    }
    __syncthreads();

    // ---------------------------------------------------------------- pass 2: squared deviations
    const float mu_l = mu_s[lane];
    acc = 0.0f;
    if (!*abort_v) {
        for (int j = warp; j < my_n; j += kWarps) {
            uint32_t w[32];
            load_row(base + j * kChunkBytes, lane, w);
            const int64_t left = p.hidden - int64_t(chunk0 + j) * kChunkCols;
            const int valid = left < kChunkCols ? int(left) : kChunkCols;
            float v[64];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float d0 = __fsub_rn(bf16_lo(w[i]), mu_l), d1 = __fsub_rn(bf16_hi(w[i]), mu_l);
                v[2 * i] = 2 * i < valid ? __fmul_rn(d0, d0) : 0.0f;
                v[2 * i + 1] = 2 * i + 1 < valid ? __fmul_rn(d1, d1) : 0.0f;
            }
            acc = __fadd_rn(acc, tree64(v));
        }
    }
    wsum[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {
        float s = wsum[0][lane];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) s = __fadd_rn(s, wsum[w][lane]);
        part[1][lane] = s;
    }
    cluster_sync();
    if (warp == 0) {
        float s = 0.0f;
        for (uint32_t q = 0; q < k; ++q) s = __fadd_rn(s, ld_cluster_f32(mapa_shared(smem_u32(&part[1][lane]), q)));
        const float var = __fdiv_rn(s, h);
        const float rs = __frcp_rn(__fsqrt_rn(__fadd_rn(var, p.eps)));
        rs_s[lane] = rs;
        const int64_t r = r0 + lane;
        if (rank == 0 && r < p.rows) {
            if (p.mu) p.mu[r] = mu_l;
            if (p.rsigma) p.rsigma[r] = rs;
        }
    }
    cluster_arrive_release();                    // done reading the other CTAs' shared memory
    __syncthreads();

    // ---------------------------------------------------------------- pass 3: normalise + quantise
    if (!*abort_v) {
        const float rs_l = rs_s[lane];
        for (int j = warp; j < my_n; j += kWarps) {
            const uint32_t chunk = base + j * kChunkBytes;
            const int64_t c0 = int64_t(chunk0 + j) * kChunkCols;
            const int valid = p.hidden - c0 < kChunkCols ? int(p.hidden - c0) : kChunkCols;
            const uint32_t gb = smem_u32(g_s + j * kChunkCols), bb = smem_u32(b_s + j * kChunkCols);
            uint32_t rc[2][8];                   // row codes: row `lane`, two 32-column blocks
            uint32_t sr[2];
            if (kRowwise) {
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    float y[32];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int cc = blk * 4 + t;                  // 16-byte chunk of the row (8 columns)
                        const uint4 xv = lds128(chunk + lane * 128 + ((cc ^ (lane & 7)) << 4));
                        const uint4 gv = lds128(gb + cc * 16), bv = lds128(bb + cc * 16);
                        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
                        const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            y[8 * t + 2 * i] = ln_y(bf16_lo(xw[i]), mu_l, rs_l, bf16_lo(gw[i]), bf16_lo(bw[i]));
                            y[8 * t + 2 * i + 1] = ln_y(bf16_hi(xw[i]), mu_l, rs_l, bf16_hi(gw[i]), bf16_hi(bw[i]));
                        }
                    }
                    uint32_t am = 0;
#pragma unroll
                    for (int i = 0; i < 32; ++i) am = max(am, __float_as_uint(y[i]) & 0x7FFFFFFFu);
                    sr[blk] = mx_scale_byte_f32(am);
                    const float m = inv_scale(sr[blk]);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        rc[blk][i] = cvt_e4m3x2(__fmul_rn(y[4 * i], m), __fmul_rn(y[4 * i + 1], m)) |
                                     (cvt_e4m3x2(__fmul_rn(y[4 * i + 2], m), __fmul_rn(y[4 * i + 3], m)) << 16);
                    if (sr[blk] == 0xFFu) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) rc[blk][i] = 0x7F7F7F7Fu;
                    }
                }
            }
            uint32_t cc_lo[8], cc_hi[8];         // column codes: columns 2 lane, 2 lane + 1, rows 0..31
            uint32_t s_lo = 0, s_hi = 0;
            if (kColwise) {
                const uint32_t g2 = lds32(gb + lane * 4), b2 = lds32(bb + lane * 4);
                const float g_lo = bf16_lo(g2), g_hi = bf16_hi(g2), b_lo = bf16_lo(b2), b_hi = bf16_hi(b2);
                const uint32_t cbase = chunk + ((lane & 3) << 2);
                const int ch = lane >> 2;
                uint32_t xw[32];
#pragma unroll
                for (int r = 0; r < 32; ++r) xw[r] = lds32(cbase + r * 128 + ((ch ^ (r & 7)) << 4));
                uint32_t am_lo = 0, am_hi = 0;
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    const float mu_r = mu_s[r], rs_r = rs_s[r];
                    am_lo = max(am_lo, __float_as_uint(ln_y(bf16_lo(xw[r]), mu_r, rs_r, g_lo, b_lo)) & 0x7FFFFFFFu);
                    am_hi = max(am_hi, __float_as_uint(ln_y(bf16_hi(xw[r]), mu_r, rs_r, g_hi, b_hi)) & 0x7FFFFFFFu);
                }
                s_lo = mx_scale_byte_f32(am_lo);
                s_hi = mx_scale_byte_f32(am_hi);
                const float m_lo = inv_scale(s_lo), m_hi = inv_scale(s_hi);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float ylo[4], yhi[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int r = 4 * i + t;
                        const float mu_r = mu_s[r], rs_r = rs_s[r];
                        ylo[t] = __fmul_rn(ln_y(bf16_lo(xw[r]), mu_r, rs_r, g_lo, b_lo), m_lo);
                        yhi[t] = __fmul_rn(ln_y(bf16_hi(xw[r]), mu_r, rs_r, g_hi, b_hi), m_hi);
                    }
                    cc_lo[i] = cvt_e4m3x2(ylo[0], ylo[1]) | (cvt_e4m3x2(ylo[2], ylo[3]) << 16);
                    cc_hi[i] = cvt_e4m3x2(yhi[0], yhi[1]) | (cvt_e4m3x2(yhi[2], yhi[3]) << 16);
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
            __syncwarp();                        // every lane has read the chunk: reuse it for the codes
            if (kRowwise) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t* w = rc[c >> 1] + 4 * (c & 1);
                    sts128(chunk + sw64(lane, c), w[0], w[1], w[2], w[3]);
                }
                const int64_t r = r0 + lane;
                if (r < p.rows) {
                    uint8_t* sp = p.s_row + r * p.ld_s_row + (c0 >> 5);
                    if (valid > 32) st_global_u16(sp, sr[0] | (sr[1] << 8));
                    else st_global_u8(sp, sr[0]);
                }
            }
            if (kColwise) {
                const uint32_t cb = chunk + 2048 + lane * 64;   // column 2 lane, then 2 lane + 1: 32 bytes each
                sts128(cb, cc_lo[0], cc_lo[1], cc_lo[2], cc_lo[3]);
                sts128(cb + 16, cc_lo[4], cc_lo[5], cc_lo[6], cc_lo[7]);
                sts128(cb + 32, cc_hi[0], cc_hi[1], cc_hi[2], cc_hi[3]);
                sts128(cb + 48, cc_hi[4], cc_hi[5], cc_hi[6], cc_hi[7]);
                if (2 * lane < valid) {                           // valid is a multiple of 32
                    uint8_t* sp = p.s_col + (c0 + 2 * lane) * p.ld_s_col + (r0 >> 5);
                    st_global_u8(sp, s_lo);
                    st_global_u8(sp + p.ld_s_col, s_hi);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (kRowwise) tma_store_2d(&qrow_map, chunk, int32_t(c0), int32_t(r0));
                if (kColwise) tma_store_2d(&qcol_map, chunk + 2048, int32_t(r0), int32_t(c0));
                bulk_commit();
            }
        }
        if (lane == 0) bulk_wait_all();
    } else if (tid == 0) {
        // Gave up: let the loads still in flight land before the CTA exits.
        for (int j = 0; j < my_n; ++j) mbar_wait(smem_u32(&bars[j]), 0, p.status);
    }
    cluster_wait_acquire();                      // no CTA leaves while another may read its partials
}

template <bool R, bool C>
cudaError_t launch(const CUtensorMap& xm, const CUtensorMap& qr, const CUtensorMap& qc, const LnParams& p,
                   int k, int64_t bands, size_t smem, cudaStream_t stream) {
    auto kern = ln_quantize_kernel<R, C>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(bands * k), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(k);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, xm, qr, qc, p);
}

}  // namespace

int64_t ln_quantize_max_hidden() { return int64_t(kMaxCluster) * kMaxChunks * kChunkCols; }

te_mx_status ln_quantize_launch(const LnQuantizeArgs& a, cudaStream_t stream) {
    const bool rowwise = a.q_row != nullptr, colwise = a.q_col != nullptr;
    if (a.rows == 0 || a.hidden == 0 || (!rowwise && !colwise && !a.mu && !a.rsigma)) return TE_MX_OK;

    int sms = 0;
    te_mx_status st = device_sm_count(&sms);
    if (st != TE_MX_OK) return st;
    const int64_t bands = (a.rows + kBand - 1) / kBand;
    const int nch = int((a.hidden + kChunkCols - 1) / kChunkCols);
    // Cluster size: at most 16 chunks (64 KB) per CTA when possible, and at
    // least two CTAs per SM when the band count allows it.
    int k = 1;
    while (k < kMaxCluster && 2 * k <= nch &&
           ((nch + k - 1) / k > 16 || bands * k < 2 * int64_t(sms)))
        k *= 2;
    const int cpc = (nch + k - 1) / k;
    if (cpc > kMaxChunks)
        return set_error(TE_MX_ERR_UNSUPPORTED_SHAPE, "hidden=%lld exceeds the largest supported %lld",
                         (long long)a.hidden, (long long)ln_quantize_max_hidden());

    CUtensorMap xm, qr, qc;
    if ((st = encode_tensor_map_2d(&xm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, uint64_t(a.hidden),
                                   uint64_t(a.rows), uint64_t(a.ld_x) * 2, kChunkCols, kBand,
                                   CU_TENSOR_MAP_SWIZZLE_128B)) != TE_MX_OK) return st;
    qr = xm;
    qc = xm;
    if (rowwise && (st = encode_tensor_map_2d(&qr, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.q_row, uint64_t(a.hidden),
                                              uint64_t(a.rows), uint64_t(a.hidden), kChunkCols, kBand,
                                              CU_TENSOR_MAP_SWIZZLE_64B)) != TE_MX_OK) return st;
    if (colwise && (st = encode_tensor_map_2d(&qc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.q_col, uint64_t(a.rows),
                                              uint64_t(a.hidden), uint64_t(a.rows), kBand, kChunkCols,
                                              CU_TENSOR_MAP_SWIZZLE_NONE)) != TE_MX_OK) return st;

    LnParams p;
    p.rows = a.rows; p.hidden = a.hidden; p.eps = a.eps;
    p.gamma = static_cast<const uint16_t*>(a.gamma);
    p.beta = static_cast<const uint16_t*>(a.beta);
    p.s_row = a.s_row; p.ld_s_row = a.ld_s_row;
    p.s_col = a.s_col; p.ld_s_col = a.ld_s_col;
    p.mu = a.mu; p.rsigma = a.rsigma;
    p.nch = nch; p.cpc = cpc;
    if ((st = device_status_ptr(&p.status)) != TE_MX_OK) return st;
    const size_t smem = size_t(cpc) * (kChunkBytes + 2 * kChunkCols * 2) + 1024;

    cudaError_t e;
    if (rowwise && colwise) e = launch<true, true>(xm, qr, qc, p, k, bands, smem, stream);
    else if (colwise) e = launch<false, true>(xm, qr, qc, p, k, bands, smem, stream);
    else if (rowwise) e = launch<true, false>(xm, qr, qc, p, k, bands, smem, stream);
    else e = launch<false, false>(xm, qr, qc, p, k, bands, smem, stream);    // statistics only
    return cuda_status(e, "layernorm quantize kernel launch");
}

}  // namespace temx
