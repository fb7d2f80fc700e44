// MXFP8 TN GEMM (dense and grouped) on tcgen05 block-scaled tensor cores.
//
// Computes, per output tile, acc = sum_k (A q_k 2^sA) (B q_k 2^sB) with
// tcgen05.mma.kind::mxf8f6f4.block_scale (E4M3 x E4M3, UE8M0 scale per 32 K),
// fp32 accumulator in Tensor Memory, then the epilogue (bias, GELU-tanh with
// the pre-activation written to AUX) in registers.  Definitions: MXFP8 GEMM
// with BIAS and GELU AUX epilogues, TN layout, K % 128 ("HipKittens MXFP8
// GEMM Support", ROCm/TransformerEngine PR #566); single-launch grouped GEMM
// for MoE experts (ROCm/TransformerEngine README, "Single-Launch Grouped GEMM
// Backends on ROCm").
//
// Kernel structure (one persistent CTA per SM, 10 warps):
//   warp 0      TMA producer: A/B tiles (128-byte swizzle) and, every 4th
//               K-step, the row-major scale tiles, into a kStages-deep ring;
//   warp 1      TMEM owner and MMA issuer: turns each raw scale tile into the
//               scale-factor layout in shared memory (an in-place 4x4 word
//               transpose), copies it to TMEM with tcgen05.cp and issues 4
//               block-scaled MMAs (K = 32 each) per 128-wide K-step;
//   warps 2..9  epilogue: each takes one 32-lane quarter x 128 columns of the
//               128 x 256 accumulator into registers, releases TMEM at once
//               (so the next tile's MMAs overlap this tile's epilogue), then
//               applies bias / GELU and stores bf16 D (and AUX).
// Every mbarrier wait is bounded; a wait that gives up aborts the CTA cleanly
// and sets the device status word.
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "temx_internal.h"

namespace temx {

namespace {

constexpr int kBM = 128;                 // tile rows (TMEM lanes)
constexpr int kBN = 256;                 // tile columns (accumulator columns)
constexpr int kBK = 128;                 // K per pipeline stage (bytes of E4M3)
constexpr int kStages = 4;
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kGroupM = 16;              // m-tiles per raster band (L2 reuse of B)
constexpr int kMaxGroups = 1024;

constexpr int kABytes = kBM * kBK;       // 16 KB
constexpr int kBBytes = kBN * kBK;       // 32 KB
constexpr int kSFABytes = kBM * 16;      // 128 rows x 16 scale bytes (4 K-steps)
constexpr int kSFBBytes = kBN * 16;
constexpr int kStageBytes = kABytes + kBBytes + kSFABytes + kSFBBytes;   // 55296
constexpr int kSmemDyn = kStages * kStageBytes + 1024;

// TMEM columns: accumulator [0, 256); scale-factor slots from 256, 8 slots of
// 12 columns (4 for A's 128 rows, 8 for B's 256 rows).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 256;
constexpr uint32_t kSfSlotCols = 12;
constexpr uint32_t kSfSlots = 8;

// Instruction descriptor, kind::mxf8f6f4 with block scaling: E4M3 A and B
// (format 0), both K-major, N >> 3 at bit 17, UE8M0 scales (bit 23),
// M >> 4 at bit 24; scale-factor byte ids at bits 4..5 (B) and 29..30 (A).
constexpr uint32_t kIdescBase = (uint32_t(kBN >> 3) << 17) | (1u << 23) | (uint32_t(kBM >> 4) << 24);
__device__ __forceinline__ uint32_t idesc_for(uint32_t sf_id) {
    return kIdescBase | (sf_id << 4) | (sf_id << 29);
}

struct GemmParams {
    int64_t M;               // dense: rows of A/D; grouped: total_m (rows of X/D)
    int32_t N, K;
    int32_t k_iters;         // K / 128
    int32_t n_tiles;         // ceil(N / 256)
    int32_t m_tiles;         // dense: ceil(M / 128)
    int64_t total_tiles;     // dense only
    int32_t groups;          // 0: dense
    const int32_t* group_m;  // device
    const uint16_t* bias;    // bf16 bits, [N] or [G x N]
    uint16_t* D;
    uint16_t* aux;
    bool has_bias, gelu;
    unsigned int* status;
};

__device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

struct Tile {
    int32_t a_row;           // first A row (TMA coordinate)
    int32_t row_end;         // rows >= row_end are not stored
    int32_t n0;              // first output column
    int32_t b_row;           // first B row (TMA coordinate)
    int32_t group;           // bias / B group
};

// Shared state besides the stage ring.
struct __align__(16) SharedState {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tmem_full;
    uint64_t tmem_empty;
    uint32_t tmem_base;
    int32_t abort;
    int64_t grouped_tiles;                 // total tiles of a grouped launch
    int32_t row_start[kMaxGroups + 1];     // grouped: first row of each group
    int32_t tile_start[kMaxGroups + 1];    // grouped: first linear tile of each group
};

// Linear tile index -> tile.  Dense: bands of kGroupM m-tiles, n-major inside
// a band, so the CTAs running at one time share a few A row-bands and B
// column-bands in L2.  Grouped: group-major, then n-major over the group's
// m-tiles.  `hint` carries the group found last time (tiles increase).
__device__ __forceinline__ Tile map_tile(const GemmParams& p, const SharedState& sh, int64_t t, int32_t& hint) {
    Tile tl;
    if (p.groups == 0) {
        const int64_t per_band = int64_t(kGroupM) * p.n_tiles;
        const int64_t band = t / per_band;
        const int32_t first_m = int32_t(band * kGroupM);
        const int32_t gm = min(p.m_tiles - first_m, kGroupM);
        const int64_t local = t - band * per_band;
        const int32_t mt = first_m + int32_t(local % gm);
        const int32_t nt = int32_t(local / gm);
        tl.a_row = mt * kBM;
        tl.row_end = int32_t(imin64(p.M, int64_t(tl.a_row) + kBM));
        tl.n0 = nt * kBN;
        tl.b_row = tl.n0;
        tl.group = 0;
    } else {
        int32_t g = hint;
        while (int64_t(sh.tile_start[g + 1]) <= t) ++g;
        hint = g;
        const int32_t local = int32_t(t - sh.tile_start[g]);
        const int32_t rows = sh.row_start[g + 1] - sh.row_start[g];
        const int32_t mtg = (rows + kBM - 1) / kBM;
        const int32_t mt = local % mtg, nt = local / mtg;
        tl.a_row = sh.row_start[g] + mt * kBM;
        tl.row_end = min(sh.row_start[g + 1], tl.a_row + kBM);
        tl.n0 = nt * kBN;
        tl.b_row = g * p.N + tl.n0;
        tl.group = g;
    }
    return tl;
}

// Grouped launch: prefix sums of the device group sizes (one warp).  Group g
// owns rows [row_start[g], row_start[g+1]) and linear tiles [tile_start[g],
// tile_start[g+1]).  Sizes are clamped so that no group reaches past total_m;
// a negative size or a sum above total_m sets the status word.
__device__ void group_prefix(const GemmParams& p, SharedState& sh, int lane) {
    const int G = p.groups;
    const int per = (G + 31) / 32;
    const int lo = min(G, lane * per), hi = min(G, lo + per);
    bool bad = false;
    int64_t rsum = 0;
    for (int g = lo; g < hi; ++g) {
        const int32_t m = p.group_m[g];
        bad |= m < 0;
        rsum += max(m, 0);
    }
    int64_t rincl = rsum;
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t v = __shfl_up_sync(0xFFFFFFFFu, rincl, o);
        if (lane >= o) rincl += v;
    }
    int64_t row = rincl - rsum, tsum = 0;
    for (int g = lo; g < hi; ++g) {
        const int32_t m = max(p.group_m[g], 0);
        const int64_t start = imin64(row, p.M), end = imin64(row + m, p.M);
        sh.row_start[g] = int32_t(start);
        tsum += (end - start + kBM - 1) / kBM * p.n_tiles;
        row += m;
    }
    if (hi == G && lo < hi) sh.row_start[G] = int32_t(imin64(row, p.M));
    bad |= (lane == 31) && rincl > p.M;
    int64_t tincl = tsum;
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t v = __shfl_up_sync(0xFFFFFFFFu, tincl, o);
        if (lane >= o) tincl += v;
    }
    int64_t t0 = tincl - tsum;
    row = rincl - rsum;
    for (int g = lo; g < hi; ++g) {
        const int32_t m = max(p.group_m[g], 0);
        const int64_t start = imin64(row, p.M), end = imin64(row + m, p.M);
        sh.tile_start[g] = int32_t(t0);
        t0 += (end - start + kBM - 1) / kBM * p.n_tiles;
        row += m;
    }
    if (lane == 31) {
        sh.tile_start[G] = int32_t(tincl);
        sh.grouped_tiles = tincl;
    }
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) set_device_status(p.status, kStatusBadArg);
}

// Bounded mbarrier wait that also returns false once another role aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, SharedState& sh,
                                              unsigned int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    volatile int32_t* abort_flag = &sh.abort;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            set_device_status(status, kStatusTimeout);
            *abort_flag = 1;
            return false;
        }
    }
}

// Raw scale tile (row r: 16 bytes = 4 words, word c = the 4 scale bytes of
// K-step c) -> scale-factor layout for tcgen05.cp 32x128b: for each 128-row
// atom and K-step c, 512 bytes where byte j*16 + i*4 + b is scale byte b of
// row 32i + j.  In place; the whole warp reads before anyone writes.
__device__ __forceinline__ void sf_to_tmem_layout(uint8_t* sf, int atoms, int lane) {
    uint4 v[3][4];
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        if (a < atoms) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                v[a][i] = *reinterpret_cast<const uint4*>(sf + a * 2048 + (32 * i + lane) * 16);
        }
    }
    __syncwarp();
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        if (a < atoms) {
            uint8_t* base = sf + a * 2048 + lane * 16;
            *reinterpret_cast<uint4*>(base + 0 * 512) = make_uint4(v[a][0].x, v[a][1].x, v[a][2].x, v[a][3].x);
            *reinterpret_cast<uint4*>(base + 1 * 512) = make_uint4(v[a][0].y, v[a][1].y, v[a][2].y, v[a][3].y);
            *reinterpret_cast<uint4*>(base + 2 * 512) = make_uint4(v[a][0].z, v[a][1].z, v[a][2].z, v[a][3].z);
            *reinterpret_cast<uint4*>(base + 3 * 512) = make_uint4(v[a][0].w, v[a][1].w, v[a][2].w, v[a][3].w);
        }
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// GELU, tanh form: 0.5 x (1 + tanh u) with u = sqrt(2/pi) (x + 0.044715 x^3),
// evaluated as the algebraically equal x / (1 + exp(-2u)), which keeps its
// relative accuracy for large negative x (no 1 + tanh cancellation).
__device__ __forceinline__ float gelu_tanh_f(float x) {
    constexpr float kTwoC0 = 2.0f * 0.7978845608028654f;          // 2 sqrt(2/pi)
    constexpr float kTwoC1 = 2.0f * 0.7978845608028654f * 0.044715f;
    constexpr float kLog2e = 1.4426950408889634f;
    const float two_u = x * fmaf(x * x, kTwoC1, kTwoC0);
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-two_u * kLog2e));
    return __fdividef(x, 1.0f + e);
}

// 16 accumulator columns of one row -> bias / GELU -> bf16 stores.
__device__ __forceinline__ void store_chunk(const uint32_t* acc, const GemmParams& p, const uint16_t* bias,
                                            int64_t row, int32_t n) {
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(acc[i]);
    if (p.has_bias) {
        const uint4 b0 = __ldg(reinterpret_cast<const uint4*>(bias + n));
        const uint4 b1 = __ldg(reinterpret_cast<const uint4*>(bias + n + 8));
        const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] += __uint_as_float(bw[i] << 16);
            v[2 * i + 1] += __uint_as_float(bw[i] & 0xFFFF0000u);
        }
    }
    const int64_t off = row * p.N + n;
    uint32_t o[8];
    if (p.gelu) {
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
        st_global_v4(p.aux + off, o[0], o[1], o[2], o[3]);
        st_global_v4(p.aux + off + 8, o[4], o[5], o[6], o[7]);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = gelu_tanh_f(v[i]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    st_global_v4(p.D + off, o[0], o[1], o[2], o[3]);
    st_global_v4(p.D + off + 8, o[4], o[5], o[6], o[7]);
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
            const __grid_constant__ CUtensorMap map_sfa, const __grid_constant__ CUtensorMap map_sfb,
            const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ SharedState sh;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&sh.full[s]), 1);
            mbar_init(smem_u32(&sh.empty[s]), 1);
        }
        mbar_init(smem_u32(&sh.tmem_full), 1);
        mbar_init(smem_u32(&sh.tmem_empty), kEpiWarps);
        sh.abort = 0;
        sh.grouped_tiles = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b);
        tma_prefetch_desc(&map_sfa);
        tma_prefetch_desc(&map_sfb);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&sh.tmem_base), kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    if (p.groups > 0 && warp == 2) group_prefix(p, sh, lane);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    const int64_t total = p.groups > 0 ? sh.grouped_tiles : p.total_tiles;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int32_t hint = 0;
            uint32_t stage = 0, phase = 0;
            for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
                const Tile tl = map_tile(p, sh, t, hint);
                bool ok = true;
                for (int32_t k = 0; k < p.k_iters && ok; ++k) {
                    if (!wait_or_abort(smem_u32(&sh.empty[stage]), phase ^ 1u, sh, p.status)) { ok = false; break; }
                    uint8_t* st = smem + stage * kStageBytes;
                    const uint32_t full = smem_u32(&sh.full[stage]);
                    const bool sf = (k & 3) == 0;
                    mbar_arrive_expect_tx(full, kABytes + kBBytes + (sf ? kSFABytes + kSFBBytes : 0));
                    tma_load_2d(smem_u32(st), &map_a, full, k * kBK, tl.a_row);
                    tma_load_2d(smem_u32(st + kABytes), &map_b, full, k * kBK, tl.b_row);
                    if (sf) {
                        tma_load_2d(smem_u32(st + kABytes + kBBytes), &map_sfa, full, k * 4, tl.a_row);
                        tma_load_2d(smem_u32(st + kABytes + kBBytes + kSFABytes), &map_sfb, full, k * 4, tl.b_row);
                    }
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        uint32_t stage = 0, phase = 0, gk = 0;
        int32_t local = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x, ++local) {
            if (local > 0) {
                if (!wait_or_abort(smem_u32(&sh.tmem_empty), uint32_t(local - 1) & 1u, sh, p.status)) break;
                tc_fence_after();
            }
            for (int32_t k = 0; k < p.k_iters; ++k) {
                if (!wait_or_abort(smem_u32(&sh.full[stage]), phase, sh, p.status)) { ok = false; break; }
                uint8_t* st = smem + stage * kStageBytes;
                uint8_t* sfa = st + kABytes + kBBytes;
                if ((k & 3) == 0) {
                    sf_to_tmem_layout(sfa, 3, lane);          // A atom + 2 B atoms (contiguous)
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tc_fence_after();
                        const int nchunks = min(4, p.k_iters - k);
                        for (int c = 0; c < nchunks; ++c) {
                            const uint32_t col = tmem + kSfCol0 + ((gk + c) % kSfSlots) * kSfSlotCols;
                            tc_cp_32x128b_warpx4(col + 0, smem_desc(smem_u32(sfa + c * 512), 0, 128, 0));
                            tc_cp_32x128b_warpx4(col + 4, smem_desc(smem_u32(sfa + 2048 + c * 512), 0, 128, 0));
                            tc_cp_32x128b_warpx4(col + 8, smem_desc(smem_u32(sfa + 4096 + c * 512), 0, 128, 0));
                        }
                    }
                }
                if (lane == 0) {
                    tc_fence_after();
                    const uint32_t sf_col = tmem + kSfCol0 + (gk % kSfSlots) * kSfSlotCols;
                    const uint32_t a_base = smem_u32(st), b_base = smem_u32(st + kABytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        mma_mxf8(tmem, smem_desc(a_base + kk * 32, 16, 1024, 2), smem_desc(b_base + kk * 32, 16, 1024, 2),
                                 idesc_for(uint32_t(kk)), sf_col, sf_col + 4, (k | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit(smem_u32(&sh.empty[stage]));
                }
                __syncwarp();
                ++gk;
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            if (lane == 0) tc_commit(smem_u32(&sh.tmem_full));
            __syncwarp();
        }
    } else {
        // ------------------------------------------------ epilogue
        const int e = warp - 2, q = warp & 3, h = e >> 2;
        int32_t hint = 0, local = 0;
        for (int64_t t = blockIdx.x; t < total; t += gridDim.x, ++local) {
            const Tile tl = map_tile(p, sh, t, hint);
            if (!wait_or_abort(smem_u32(&sh.tmem_full), uint32_t(local) & 1u, sh, p.status)) break;
            tc_fence_after();
            uint32_t acc0[64], acc1[64];
            const uint32_t taddr = tmem + (uint32_t(32 * q) << 16) + uint32_t(128 * h);
            tmem_ld_32x32b_x64(taddr, acc0);
            tmem_ld_32x32b_x64(taddr + 64, acc1);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.tmem_empty));
            const int64_t row = int64_t(tl.a_row) + 32 * q + lane;
            if (row < tl.row_end) {
                const uint16_t* bias = p.has_bias ? p.bias + int64_t(tl.group) * p.N : nullptr;
                const int32_t nb = tl.n0 + 128 * h;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (nb + 16 * j < p.N) store_chunk(acc0 + 16 * j, p, bias, row, nb + 16 * j);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (nb + 64 + 16 * j < p.N) store_chunk(acc1 + 16 * j, p, bias, row, nb + 64 + 16 * j);
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

te_mx_status gemm_launch(const GemmArgs& a, cudaStream_t stream) {
    const bool grouped = a.groups > 0;
    const uint64_t b_rows = grouped ? uint64_t(a.groups) * uint64_t(a.N) : uint64_t(a.N);
    const uint64_t sf_cols = uint64_t(a.K / 32) < 16 ? 16 : uint64_t(a.K / 32);
    CUtensorMap ma, mb, msa, msb;
    te_mx_status st;
    if ((st = encode_tensor_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.A, uint64_t(a.K), uint64_t(a.M),
                                   uint64_t(a.K), kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B)) != TE_MX_OK) return st;
    if ((st = encode_tensor_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, uint64_t(a.K), b_rows,
                                   uint64_t(a.K), kBK, kBN, CU_TENSOR_MAP_SWIZZLE_128B)) != TE_MX_OK) return st;
    if ((st = encode_tensor_map_2d(&msa, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.sA, sf_cols, uint64_t(a.M),
                                   uint64_t(a.ld_sA), 16, kBM, CU_TENSOR_MAP_SWIZZLE_NONE)) != TE_MX_OK) return st;
    if ((st = encode_tensor_map_2d(&msb, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.sB, sf_cols, b_rows,
                                   uint64_t(a.ld_sB), 16, kBN, CU_TENSOR_MAP_SWIZZLE_NONE)) != TE_MX_OK) return st;

    GemmParams p{};
    p.M = a.M;
    p.N = int32_t(a.N);
    p.K = int32_t(a.K);
    p.k_iters = int32_t(a.K / kBK);
    p.n_tiles = int32_t((a.N + kBN - 1) / kBN);
    p.m_tiles = int32_t((a.M + kBM - 1) / kBM);
    p.total_tiles = grouped ? 0 : int64_t(p.m_tiles) * p.n_tiles;
    p.groups = a.groups;
    p.group_m = a.group_m;
    p.bias = static_cast<const uint16_t*>(a.bias);
    p.D = static_cast<uint16_t*>(a.D);
    p.aux = static_cast<uint16_t*>(a.aux);
    p.has_bias = a.has_bias;
    p.gelu = a.gelu;
    if ((st = device_status_ptr(&p.status)) != TE_MX_OK) return st;

    int sms = 0;
    if ((st = device_sm_count(&sms)) != TE_MX_OK) return st;
    int64_t grid = grouped ? sms : (p.total_tiles < sms ? p.total_tiles : sms);
    if (grid < 1) grid = 1;
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemDyn);
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(gemm)");
    gemm_kernel<<<int(grid), kThreads, kSmemDyn, stream>>>(ma, mb, msa, msb, p);
    return cuda_status(cudaGetLastError(), "gemm kernel launch");
}

}  // namespace temx
