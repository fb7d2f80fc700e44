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
// Kernel structure (persistent, one CTA per SM, 12 warps), in two shapes:
//   kPair = 1: one CTA computes a 128 x 256 tile (cta_group::1);
//   kPair = 2: a cluster of two CTAs computes a 256 x 256 tile with
//              cta_group::2 MMAs: each CTA holds 128 rows of A and 128 rows of
//              B, the even CTA issues the MMAs and each CTA's TMEM receives
//              its 128 x 256 accumulator.  Per SM this halves the B bytes a
//              K-step needs, which is what limits the single-CTA shape (the
//              ingress of an SM is ~53 B/clk; 48 KB per 512-cycle K-step does
//              not fit).
//   warp 0      TMA producer: A/B tiles (128-byte swizzle) into a kStages ring
//               (completion on the MMA CTA's barrier) and, every 4th K-step,
//               the row-major scale tiles (completion on the CTA's own barrier);
//   warps 1, 11 MMA issuers (warp 1 also owns TMEM): in the MMA CTA they take
//               alternate K-steps, one lane issuing 4 block-scaled MMAs
//               (K = 32 each) per 128-wide K-step and nothing else (a tcgen05
//               instruction costs ~80-90 issue cycles and blocks while the
//               tensor pipe is busy, so one issuer waits while the other
//               issues, and neither has slack for the scale copies); dense
//               GEMMs of fewer than 16 K-steps and the grouped wgrad use warp
//               1 alone;
//   warp 10     scale-factor warp: turns each landed scale tile into the
//               tcgen05 scale-factor layout in place (a 4x4 word transpose),
//               copies the group's scale factors into TMEM (tcgen05.cp, from the
//               MMA CTA for a pair) and commits them to the MMA warp;
//   warps 2..9  epilogue: each takes one 32-lane quarter x 128 columns of its
//               CTA's 128 x 256 accumulator into registers, releases TMEM at
//               once (so the next tile's MMAs overlap this tile's epilogue),
//               then applies bias / GELU and stores bf16 D (and AUX).
// FP32 block scales (Float8BlockScaling) use the same tiles with 12 warps in
// three warp groups: warps 0-3 producer, MMA issuer, scale warp and a second
// MMA issuer (registers lowered to 64 per thread), warps 4-11 epilogue
// (raised to 216): every K-step's product lands in one of two 256-column TMEM
// buffers and each epilogue thread adds it, scaled, to the 128 accumulator
// columns of its row that it keeps in registers.
// Every mbarrier wait is bounded; a wait that gives up aborts the CTA cleanly
// and sets the device status word.
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "tcgen05.cuh"
#include "temx_internal.h"

namespace temx {

namespace {

constexpr int kBM = 128;                 // accumulator rows per CTA (TMEM lanes)
constexpr int kBN = 256;                 // tile columns (accumulator columns)
constexpr int kBK = 128;                 // K per pipeline stage (bytes of E4M3)
constexpr int kThreads = 384;            // 12 warps
constexpr int kEpiWarps = 8;
constexpr int kGroupM = 16;              // m-tiles per raster band (L2 reuse of B)
constexpr int kMaxGroups = 1024;
constexpr int kSFABytes = kBM * 16;      // 128 rows x 16 scale bytes (4 K-steps)
constexpr int kSfRing = 3;               // scale-group slots in shared memory
constexpr int kSfAhead = 2;              // scale groups loaded ahead of the one being prepared
constexpr int kSfTmemGroups = 4;         // scale groups resident in TMEM
constexpr int kSplitMinK = 16;           // MXFP8: dense GEMMs of at least this many K-steps use both MMA issuers
constexpr int kScrBufs = 2;              // FP32 scales: K-step product buffers in TMEM (256 columns each)
// FP32 scales: registers per thread after the split (warp group 0 / 1 and 2);
// 4 x 64 + 8 x 216 = 1984 <= 12 x 168, the launch's 168 per thread
constexpr int kRegsRoles = 64;
constexpr int kRegsEpi = 216;

// kF32 (Float8BlockScaling with FP32 scales): the same 256-column tiles; the
// warp roles move so that the 8 epilogue warps form warp groups 1 and 2.
template <int kPair, bool kF32 = false>
struct Cfg {
    static constexpr int kTileM = kBM * kPair;            // rows of one (pair) tile
    static constexpr int kBN = ::temx::kBN;               // tile columns
    static constexpr int kBRows = kBN / kPair;            // B rows loaded per CTA
    static constexpr int kABytes = kBM * kBK;             // 16 KB
    static constexpr int kBBytes = kBRows * kBK;          // 32 or 16 KB
    static constexpr int kStages = kPair == 2 ? 5 : 4;
    static constexpr int kSfWarp = kF32 ? 2 : 10;         // scale-factor warp
    static constexpr int kMma2Warp = kF32 ? 3 : 11;       // second MMA issuer
    static constexpr int kEpiWarp0 = kF32 ? 4 : 2;        // first epilogue warp
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kSFBBytes = kBN * 16;            // every CTA holds all of the tile's B rows' scales
    static constexpr int kSfSlotBytes = kSFABytes + kSFBBytes;   // one scale group (4 K-steps) in the ring
    // CTA pairs stage the epilogue's bf16 rows in shared memory (4 KB per
    // epilogue warp) so that global stores are written as whole lines.
    static constexpr bool kStagedStores = kPair == 2;
    static constexpr int kEpiStageBytes = kStagedStores ? kEpiWarps * 4096 : 0;
    // ... and each epilogue warp's 128 bias values, fetched while the tile's
    // MMAs run (a global load at store time costs an L2 round trip under load)
    static constexpr int kBiasBytes = kStagedStores ? kEpiWarps * 256 : 0;
    static constexpr int kSmemDyn = kStages * kStageBytes + kSfRing * kSfSlotBytes + kEpiStageBytes + kBiasBytes + 1024;
    // Instruction descriptor, kind::mxf8f6f4 with block scaling: E4M3 A and B
    // (format 0), both K-major, N >> 3 at bit 17, UE8M0 scales (bit 23),
    // M >> 4 at bit 24; scale-factor byte ids at bits 4..5 (B) and 29..30 (A).
    static constexpr uint32_t kIdescBase =
        (uint32_t(kBN >> 3) << 17) | (1u << 23) | (uint32_t(kTileM >> 4) << 24);
    // Instruction descriptor, kind::f8f6f4 (no block scaling; FP32 scales):
    // fp32 D (bits 4..5 = 1), E4M3 A and B (formats 0), both K-major, N >> 3
    // at bit 17, M >> 4 at bit 24.
    static constexpr uint32_t kIdescF32 = (1u << 4) | (uint32_t(kBN >> 3) << 17) | (uint32_t(kTileM >> 4) << 24);
};
static_assert(Cfg<1>::kStageBytes % 1024 == 0 && Cfg<2>::kStageBytes % 1024 == 0 &&
              Cfg<1, true>::kStageBytes % 1024 == 0 && Cfg<2, true>::kStageBytes % 1024 == 0, "stage alignment");
// (the static shared state, ~8.5 KB, comes on top of the dynamic part; 227 KB per CTA in all)
static_assert(Cfg<2, true>::kSmemDyn <= 218 * 1024 && Cfg<1, true>::kSmemDyn <= 218 * 1024 &&
              Cfg<2>::kSmemDyn <= 218 * 1024 && Cfg<1>::kSmemDyn <= 218 * 1024, "shared memory");

__device__ __forceinline__ uint32_t idesc_sf(uint32_t base, uint32_t sf_id) {
    return base | (sf_id << 4) | (sf_id << 29);
}

// TMEM columns: accumulator [0, 256); scale-factor slots from 256, 16 slots
// of 12 columns (4 for A's 128 rows, 8 for B's 256 rows): K-step c of scale
// group j uses slot (j % 4) * 4 + c.  The scale-factor warp copies group j
// only after the MMAs of group j - 3 completed, so a slot is never rewritten
// while an MMA may still read it.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 256;
constexpr uint32_t kSfSlotCols = 12;
constexpr uint32_t kSfSlots = 16;
static_assert(kSfCol0 + kSfSlots * kSfSlotCols <= kTmemCols, "scale-factor slots fit in TMEM");
static_assert(kScrBufs * Cfg<2, true>::kBN <= int(kTmemCols), "FP32-scale product buffers fit in TMEM");
static_assert(4 * kRegsRoles + 8 * kRegsEpi <= 12 * 168, "FP32-scale register split");

struct GemmParams {
    int64_t M;               // dense: rows of A/D; grouped: total_m (rows of X/D)
    int32_t N, K;
    int32_t k_iters;         // K / 128
    int32_t n_tiles;         // ceil(N / 256)
    int32_t m_tiles;         // dense: ceil(M / tile rows)
    int64_t total_tiles;     // dense only
    int32_t groups;          // 0: dense
    const int32_t* group_m;  // device
    const uint16_t* bias;    // bf16 bits, [N] or [G x N]
    uint16_t* D;
    uint16_t* aux;
    bool has_bias, gelu, dgelu;          // dgelu: aux is an input (forward pre-activation)
    bool wgrad;                          // grouped wgrad: per-group K range, D = [groups x M x N]
    bool b_2d;                           // FP32 scales: B's scales constant over 128-row blocks
                                         // (next to the other flags: no other field moves)
    int64_t total_m;                     // wgrad: bound on the token counts' sum
    int64_t ld_code, ld_sfa, ld_sfb;     // wgrad: operand pitches (capacities)
    unsigned int* status;
};

__device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

struct Tile {
    int32_t a_row;           // first A row of the (pair) tile
    int32_t d_row;           // first output row (= a_row except for wgrad)
    int32_t row_end;         // output rows >= row_end are not stored
    int32_t n0;              // first output column
    int32_t b_row;           // first B row of the tile
    int32_t group;           // bias / B group
    int32_t k0, nk;          // K-steps [k0, k0 + nk) of 128
    int32_t sf0;             // first scale column (bytes, a multiple of 16)
};

// Shared state besides the stage ring.
template <int kStages>
struct __align__(16) SharedState {
    uint64_t full[kStages];                // A/B bytes landed (used in the MMA CTA)
    uint64_t empty[kStages];               // stage consumed by the MMAs (each CTA)
    uint64_t sf_full[kSfRing];             // this CTA's scale group landed in its ring slot
    uint64_t sf_ready[kSfRing];            // the group's scale factors are in TMEM (each CTA of a pair)
    uint64_t sf_peer[kSfRing];             // (MMA CTA of a pair) the peer's scale group is in copy layout
    uint64_t grp_done[kSfTmemGroups];      // (MMA CTA) the MMAs of a scale group completed
    uint64_t tmem_full;
    uint64_t tmem_empty;                   // (MMA CTA) accumulator drained by every epilogue warp of the pair
    uint64_t first_done;                   // (MMA CTA) the MMAs of a tile's first K-step completed
    // FP32-scale mode: K-step kg's product lands in TMEM buffer kg % kScrBufs
    // (columns 256 * buffer ..; the scaled accumulator lives in registers)
    uint64_t scr_full[kScrBufs];           // a product landed (each CTA)
    uint64_t scr_empty[kScrBufs];          // (MMA CTA) the epilogue warps of both CTAs read that buffer
    uint64_t sf_done[kSfRing];             // this CTA's epilogue warps are done with a scale group
    uint32_t tmem_base;
    int32_t abort;
    int64_t grouped_tiles;                 // total tiles of a grouped launch
    int32_t row_start[kMaxGroups + 1];     // grouped: first row of each group
    int32_t tile_start[kMaxGroups + 1];    // grouped: first linear tile of each group
};

// Linear tile index -> tile.  Dense: bands of kGroupM m-tiles, n-major inside
// a band, so the CTAs running at one time share a few A row-bands and B
// column-bands in L2.  Grouped: group-major, then n-major over the group's
// m-tiles.  Wgrad: group-major, every group the full M x N output over its
// own K range.  `hint` carries the group found last time (tiles increase).
template <int kTileM, int kTileN, bool kWgrad, typename SH>
__device__ __forceinline__ Tile map_tile(const GemmParams& p, const SH& sh, int64_t t, int32_t& hint) {
    Tile tl;
    tl.k0 = 0;
    tl.nk = p.k_iters;
    tl.sf0 = 0;
    if constexpr (kWgrad) {
        const int64_t per = int64_t(p.m_tiles) * p.n_tiles;
        const int32_t g = int32_t(t / per);
        const int32_t local = int32_t(t - int64_t(g) * per);
        const int32_t mt = local % p.m_tiles, nt = local / p.m_tiles;
        tl.a_row = mt * kTileM;
        tl.d_row = int32_t(int64_t(g) * p.M + tl.a_row);
        tl.row_end = int32_t(int64_t(g) * p.M + imin64(p.M, int64_t(tl.a_row) + kTileM));
        tl.n0 = nt * kTileN;
        tl.b_row = tl.n0;
        tl.group = g;
        tl.k0 = sh.row_start[g];
        tl.nk = sh.row_start[g + 1] - sh.row_start[g];
        tl.sf0 = sh.tile_start[g];
    } else if (p.groups == 0) {
        const int64_t per_band = int64_t(kGroupM) * p.n_tiles;
        const int64_t band = t / per_band;
        const int32_t first_m = int32_t(band * kGroupM);
        const int32_t gm = min(p.m_tiles - first_m, kGroupM);
        const int64_t local = t - band * per_band;
        const int32_t mt = first_m + int32_t(local % gm);
        const int32_t nt = int32_t(local / gm);
        tl.a_row = mt * kTileM;
        tl.d_row = tl.a_row;
        tl.row_end = int32_t(imin64(p.M, int64_t(tl.a_row) + kTileM));
        tl.n0 = nt * kTileN;
        tl.b_row = tl.n0;
        tl.group = 0;
    } else {
        int32_t g = hint;
        while (int64_t(sh.tile_start[g + 1]) <= t) ++g;
        hint = g;
        const int32_t local = int32_t(t - sh.tile_start[g]);
        const int32_t rows = sh.row_start[g + 1] - sh.row_start[g];
        const int32_t mtg = (rows + kTileM - 1) / kTileM;
        const int32_t mt = local % mtg, nt = local / mtg;
        tl.a_row = sh.row_start[g] + mt * kTileM;
        tl.d_row = tl.a_row;
        tl.row_end = min(sh.row_start[g + 1], tl.a_row + kTileM);
        tl.n0 = nt * kTileN;
        tl.b_row = g * p.N + tl.n0;
        tl.group = g;
    }
    return tl;
}

// Grouped launch: prefix sums of the device group sizes (one warp).  Group g
// owns rows [row_start[g], row_start[g+1]) and linear tiles [tile_start[g],
// tile_start[g+1]).  Sizes are clamped so that no group reaches past total_m;
// a negative size or a sum above total_m sets the status word.
template <int kTileM, typename SH>
__device__ void group_prefix(const GemmParams& p, SH& sh, int lane) {
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
        tsum += (end - start + kTileM - 1) / kTileM * p.n_tiles;
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
        t0 += (end - start + kTileM - 1) / kTileM * p.n_tiles;
        row += m;
    }
    if (lane == 31) {
        sh.tile_start[G] = int32_t(tincl);
        sh.grouped_tiles = tincl;
    }
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) set_device_status(p.status, kStatusBadArg);
}

// Wgrad launch (one warp): expert g's padded tokens are K-steps
// [row_start[g], row_start[g+1]) of 128, its scales start at byte
// tile_start[g] (16-byte aligned): Kp_g = round_up(m_g, 128), scale width
// round_up(Kp_g / 32, 16).  A negative size, a sum above total_m or a layout
// wider than the operand pitches sets the status word and leaves no tiles.
template <typename SH>
__device__ void wgrad_prefix(const GemmParams& p, SH& sh, int lane) {
    const int G = p.groups;
    const int per = (G + 31) / 32;
    const int lo = min(G, lane * per), hi = min(G, lo + per);
    bool bad = false;
    int64_t toks = 0, steps = 0, sfw = 0;
    for (int g = lo; g < hi; ++g) {
        const int64_t m = p.group_m[g];
        bad |= m < 0;
        const int64_t ks = (m < 0 ? 0 : m + 127) / 128;
        toks += m < 0 ? 0 : m;
        steps += ks;
        sfw += (4 * ks + 15) / 16 * 16;
    }
    int64_t t_in = toks, k_in = steps, s_in = sfw;
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t a = __shfl_up_sync(0xFFFFFFFFu, t_in, o), b = __shfl_up_sync(0xFFFFFFFFu, k_in, o),
                      c = __shfl_up_sync(0xFFFFFFFFu, s_in, o);
        if (lane >= o) { t_in += a; k_in += b; s_in += c; }
    }
    int64_t k0 = k_in - steps, s0 = s_in - sfw;
    for (int g = lo; g < hi; ++g) {
        const int64_t m = p.group_m[g];
        const int64_t ks = (m < 0 ? 0 : m + 127) / 128;
        sh.row_start[g] = int32_t(k0);
        sh.tile_start[g] = int32_t(s0);
        k0 += ks;
        s0 += (4 * ks + 15) / 16 * 16;
    }
    const int64_t tt = __shfl_sync(0xFFFFFFFFu, t_in, 31), kt = __shfl_sync(0xFFFFFFFFu, k_in, 31),
                  st = __shfl_sync(0xFFFFFFFFu, s_in, 31);
    bad = __any_sync(0xFFFFFFFFu, bad) || tt > p.total_m || kt * kBK > p.ld_code || st > p.ld_sfa || st > p.ld_sfb;
    if (lane == 0) {
        sh.row_start[G] = int32_t(kt);
        sh.tile_start[G] = int32_t(st);
        sh.grouped_tiles = bad ? 0 : int64_t(G) * p.m_tiles * p.n_tiles;
        if (bad) set_device_status(p.status, kStatusBadArg);
    }
}

// Bounded mbarrier wait that also returns false once another role aborted.
template <typename SH>
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, SH& sh,
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
__device__ __forceinline__ void sf_to_tmem_layout(uint32_t sf, int lane) {
    uint4 v[3][4];
#pragma unroll
    for (int a = 0; a < 3; ++a)
#pragma unroll
        for (int i = 0; i < 4; ++i) v[a][i] = lds128(sf + a * 2048 + (32 * i + lane) * 16);
    __syncwarp();
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        const uint32_t base = sf + a * 2048 + lane * 16;
        sts128(base + 0 * 512, v[a][0].x, v[a][1].x, v[a][2].x, v[a][3].x);
        sts128(base + 1 * 512, v[a][0].y, v[a][1].y, v[a][2].y, v[a][3].y);
        sts128(base + 2 * 512, v[a][0].z, v[a][1].z, v[a][2].z, v[a][3].z);
        sts128(base + 3 * 512, v[a][0].w, v[a][1].w, v[a][2].w, v[a][3].w);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Packed fp32 pairs (two lanes of one 64-bit register) for the f32x2 forms of
// add, sub, mul and fma, which issue two operations per instruction.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// GELU (tanh form) of two values: 0.5 x (1 + tanh u) with
// u = sqrt(2/pi) (x + 0.044715 x^3), evaluated as the algebraically equal
// x / (1 + 2^t), t = -2 log2(e) u, which keeps its relative accuracy for large
// negative x (no 1 + tanh cancellation).  The epilogue is bound by instruction
// issue, so the arithmetic runs as packed f32x2 operations (t = x (A x^2 + B)
// with the constants folded in, 1 + 2^t, the final product) around the two
// MUFU operations per value (ex2, reciprocal): 4.5 instructions per value.
__device__ __forceinline__ void gelu_tanh_f2(float& x0, float& x1) {
    constexpr float kA = -2.0f * 1.4426950408889634f * 0.7978845608028654f * 0.044715f;
    constexpr float kB = -2.0f * 1.4426950408889634f * 0.7978845608028654f;
    const uint64_t x = f2_pack(x0, x1);
    float t0, t1;
    f2_unpack(f2_mul(x, f2_fma(f2_mul(x, x), f2_pack(kA, kA), f2_pack(kB, kB))), t0, t1);
    float e0, e1;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(t0));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(t1));
    float d0, d1;
    f2_unpack(f2_add(f2_pack(e0, e1), f2_pack(1.0f, 1.0f)), d0, d1);
    float r0, r1;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(d0));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(d1));
    f2_unpack(f2_mul(x, f2_pack(r0, r1)), x0, x1);
}

// Derivative of the tanh-form GELU: with s = sigmoid(2u) = 0.5 (1 + tanh u)
// and t = 1 - s, gelu'(x) = s + 2 x s t sqrt(2/pi) (1 + 3 * 0.044715 x^2).
// t is taken as 1 - s or e s (e = exp(-2u)), whichever does not cancel.
__device__ __forceinline__ float dgelu_tanh_f(float x) {
    constexpr float kC0 = 0.7978845608028654f;                     // sqrt(2/pi)
    constexpr float kTwoC0 = 2.0f * kC0;
    constexpr float kTwoC1 = 2.0f * kC0 * 0.044715f;
    constexpr float kThreeC1 = 3.0f * 0.044715f;
    constexpr float kLog2e = 1.4426950408889634f;
    const float x2 = x * x;
    const float two_u = x * fmaf(x2, kTwoC1, kTwoC0);
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-two_u * kLog2e));
    const float sg = __fdividef(1.0f, 1.0f + e);
    const float t = e > 1.0f ? 1.0f - sg : e * sg;
    return fmaf(2.0f * x * sg * t * kC0, fmaf(kThreeC1, x2, 1.0f), sg);
}

// Multiply 8 consecutive values by gelu' of 8 bf16 pre-activations (one uint4).
__device__ __forceinline__ void apply_dgelu8(float* v, uint4 w) {
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] *= dgelu_tanh_f(__uint_as_float(ww[i] << 16));
        v[2 * i + 1] *= dgelu_tanh_f(__uint_as_float(ww[i] & 0xFFFF0000u));
    }
}

// 16 accumulator columns of one row -> bias / GELU -> bf16 stores.
template <bool kAcc>
__device__ __forceinline__ void store_chunk(const uint32_t* acc, const GemmParams& p, const uint16_t* bias,
                                            int64_t row, int32_t n) {
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(acc[i]);
    if constexpr (kAcc) {                        // D (fp32) += acc, one rounding per element
        float4* d = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.D) + row * p.N + n);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 o = d[q];
            d[q] = make_float4(__fadd_rn(o.x, v[4 * q]), __fadd_rn(o.y, v[4 * q + 1]), __fadd_rn(o.z, v[4 * q + 2]),
                               __fadd_rn(o.w, v[4 * q + 3]));
        }
        return;
    }
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
    if (p.dgelu) {
        apply_dgelu8(v, __ldg(reinterpret_cast<const uint4*>(p.aux + off)));
        apply_dgelu8(v + 8, __ldg(reinterpret_cast<const uint4*>(p.aux + off + 8)));
    }
    if (p.gelu) {
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
        st_global_v4(p.aux + off, o[0], o[1], o[2], o[3]);
        st_global_v4(p.aux + off + 8, o[4], o[5], o[6], o[7]);
#pragma unroll
        for (int i = 0; i < 16; i += 2) gelu_tanh_f2(v[i], v[i + 1]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    st_global_v4(p.D + off, o[0], o[1], o[2], o[3]);
    st_global_v4(p.D + off + 8, o[4], o[5], o[6], o[7]);
}

// 64 accumulator columns of one row per lane (32 rows per warp) -> bias /
// GELU -> bf16, written as whole 128-byte lines: each lane puts its row's 128
// bytes into the warp's staging tile (16-byte chunks XOR-swizzled by row, so
// neither the writes nor the reads conflict), then every store instruction
// writes 4 complete rows.
// `bias_sm` is the shared-memory address of column n's bf16 bias (the warp's
// slice, copied there beforehand).
template <bool kAcc>
__device__ __forceinline__ void store_64_staged(uint32_t* acc, const GemmParams& p, uint32_t bias_sm,
                                                int64_t row0, int64_t row_end, int32_t n, uint32_t stage,
                                                int lane, const CUtensorMap* map_d, const CUtensorMap* map_aux,
                                                bool tma) {
    float* v = reinterpret_cast<float*>(acc);
    if constexpr (kAcc) {
        // D (fp32) += acc: each lane reads, adds and writes its own row, 16
        // bytes at a time (whole 32-byte sectors).
        const int64_t row = row0 + lane;
        if (row < row_end) {
            float4* d = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.D) + row * p.N + n);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                if (n + 4 * q < p.N) {
                    const float4 o = d[q];
                    d[q] = make_float4(__fadd_rn(o.x, v[4 * q]), __fadd_rn(o.y, v[4 * q + 1]),
                                       __fadd_rn(o.z, v[4 * q + 2]), __fadd_rn(o.w, v[4 * q + 3]));
                }
            }
        }
        return;
    }
    if (p.has_bias) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            if (n + 8 * c < p.N) {
                const uint4 b = lds128(bias_sm + 16 * c);
                const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {          // bf16 -> fp32 is a 16-bit shift; one packed add per pair
                    const uint64_t sum = f2_add(f2_pack(v[8 * c + 2 * i], v[8 * c + 2 * i + 1]),
                                                f2_pack(__uint_as_float(bw[i] << 16), __uint_as_float(bw[i] & 0xFFFF0000u)));
                    f2_unpack(sum, v[8 * c + 2 * i], v[8 * c + 2 * i + 1]);
                }
            }
        }
    }
    // the staging tile is free once this warp's previous TMA store has read it
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
    if (p.dgelu) {
        // the forward pre-activation rows come in as whole lines through the
        // staging tile, then each lane takes its own row
        const int c = lane & 7;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + (lane >> 3);
            uint4 w = make_uint4(0, 0, 0, 0);
            if (row0 + r < row_end && n + 8 * c < p.N)
                w = __ldg(reinterpret_cast<const uint4*>(p.aux + (row0 + r) * p.N + n + 8 * c));
            sts128(stage + r * 128 + ((c ^ (r & 7)) << 4), w.x, w.y, w.z, w.w);
        }
        __syncwarp();
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) apply_dgelu8(v + 8 * cc, lds128(stage + lane * 128 + ((cc ^ (lane & 7)) << 4)));
        __syncwarp();
    }
    const int passes = p.gelu ? 2 : 1;
    for (int pass = 0; pass < passes; ++pass) {
        const bool is_aux = p.gelu && pass == 0;
        if (p.gelu && pass == 1) {
#pragma unroll
            for (int i = 0; i < 64; i += 2) gelu_tanh_f2(v[i], v[i + 1]);
            // the AUX store issued before the GELU has read the staging tile by now
            if (tma && lane == 0) bulk_wait_read_all();
            __syncwarp();
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint32_t w0 = pack_bf16x2(v[8 * c + 0], v[8 * c + 1]), w1 = pack_bf16x2(v[8 * c + 2], v[8 * c + 3]);
            const uint32_t w2 = pack_bf16x2(v[8 * c + 4], v[8 * c + 5]), w3 = pack_bf16x2(v[8 * c + 6], v[8 * c + 7]);
            sts128(stage + lane * 128 + ((c ^ (lane & 7)) << 4), w0, w1, w2, w3);
        }
        if (tma) {
            // the staging tile is the 128-byte-swizzled 32 x 64 box of the
            // output's tensor map: one asynchronous store; the warp goes on
            // and waits only before it writes the tile again
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                // (evict-first for the dense GEMMs; the grouped forward GEMM's
                // outputs keep the default policy: with the hint, the MXFP8
                // quantisation launched after it measured slower)
                if (p.groups > 0 && !p.wgrad) tma_store_2d(is_aux ? map_aux : map_d, stage, n, int32_t(row0));
                else tma_store_2d_evict_first(is_aux ? map_aux : map_d, stage, n, int32_t(row0));
                bulk_commit();
            }
            __syncwarp();
            continue;
        }
        __syncwarp();
        uint16_t* out = is_aux ? p.aux : p.D;
        const int c = lane & 7;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + (lane >> 3);
            const uint4 w = lds128(stage + r * 128 + ((c ^ (r & 7)) << 4));
            if (row0 + r < row_end && n + 8 * c < p.N)
                st_global_v4(out + (row0 + r) * p.N + n + 8 * c, w.x, w.y, w.z, w.w);
        }
        __syncwarp();
    }
}

// FP32 scales: acc[j] += v[j] * (sA sB) for 64 columns of one row.  2D weight
// blocks: one factor f = sA sB for all of them, acc = fma(v, f, acc);
// otherwise sB per column from the [4 K-steps][256 columns] shared table at
// sbt: acc = fma(v sB, sA, acc).  Packed pairs (f32x2: each half rounds as the
// scalar mul / fma does).
__device__ __forceinline__ void scale_accumulate_64(uint32_t (&acc)[64], const uint32_t (&v)[64], bool b_2d, float f,
                                                    float sa, uint32_t sbt) {
    if (b_2d) {
#pragma unroll
        for (int j = 0; j < 64; j += 2) {
            uint64_t a2, v2, f2;
            asm("mov.b64 %0, {%1, %2};" : "=l"(a2) : "r"(acc[j]), "r"(acc[j + 1]));
            asm("mov.b64 %0, {%1, %2};" : "=l"(v2) : "r"(v[j]), "r"(v[j + 1]));
            asm("mov.b64 %0, {%1, %1};" : "=l"(f2) : "r"(__float_as_uint(f)));
            asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a2) : "l"(v2), "l"(f2));
            asm("mov.b64 {%0, %1}, %2;" : "=r"(acc[j]), "=r"(acc[j + 1]) : "l"(a2));
        }
    } else {
        uint64_t sa2;
        asm("mov.b64 %0, {%1, %1};" : "=l"(sa2) : "r"(__float_as_uint(sa)));
#pragma unroll
        for (int j4 = 0; j4 < 16; ++j4) {
            const uint4 w = lds128(sbt + 16 * j4);
#pragma unroll
            for (int i = 0; i < 4; i += 2) {
                const int j = 4 * j4 + i;
                uint64_t a2, v2, s2;
                asm("mov.b64 %0, {%1, %2};" : "=l"(a2) : "r"(acc[j]), "r"(acc[j + 1]));
                asm("mov.b64 %0, {%1, %2};" : "=l"(v2) : "r"(v[j]), "r"(v[j + 1]));
                asm("mov.b64 %0, {%1, %2};" : "=l"(s2) : "r"(i == 0 ? w.x : w.z), "r"(i == 0 ? w.y : w.w));
                asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(v2) : "l"(s2));
                asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a2) : "l"(v2), "l"(sa2));
                asm("mov.b64 {%0, %1}, %2;" : "=r"(acc[j]), "=r"(acc[j + 1]) : "l"(a2));
            }
        }
    }
}

// kAcc: fp32 D accumulated into; kWgrad: grouped wgrad; kF32: Float8BlockScaling
// operands with FP32 scales (dense only): every K-step's product lands in one
// of kScrBufs TMEM buffers and the epilogue warps accumulate it, scaled, in
// registers.
template <int kPair, bool kAcc, bool kWgrad, bool kF32>
__global__ void __launch_bounds__(kThreads, 1)   // 168 registers: 3 warps share a 16K-register sub-partition
gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
            const __grid_constant__ CUtensorMap map_sfa, const __grid_constant__ CUtensorMap map_sfb,
            const __grid_constant__ CUtensorMap map_d, const __grid_constant__ CUtensorMap map_aux,
            const GemmParams p) {
    using C = Cfg<kPair, kF32>;
    using SH = SharedState<C::kStages>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ SH sh;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = kPair == 2 ? cluster_ctarank() : 0u;     // 0 = the MMA CTA
    const int64_t unit = kPair == 2 ? blockIdx.x / 2 : blockIdx.x;  // cluster (pair) index
    const int64_t units = kPair == 2 ? gridDim.x / 2 : gridDim.x;
    // Barriers of the MMA CTA as seen from this CTA (cluster addresses for pairs).
    auto leader = [&](const uint64_t& bar) -> uint32_t {
        return kPair == 2 ? mapa_shared(smem_u32(&bar), 0) : smem_u32(&bar);
    };
    // MXFP8: two MMA issuers for dense GEMMs of at least kSplitMinK K-steps;
    // otherwise (short K, or the grouped wgrad's per-expert K ranges) warp 1
    // alone issues and commits, and the barriers count its arrivals only
    const bool two_issuers = !kWgrad && p.k_iters >= kSplitMinK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&sh.full[s]), kPair);
            mbar_init(smem_u32(&sh.empty[s]), 1);
        }
        for (int s = 0; s < kSfRing; ++s) {
            mbar_init(smem_u32(&sh.sf_full[s]), 1);
            mbar_init(smem_u32(&sh.sf_ready[s]), 1);
            mbar_init(smem_u32(&sh.sf_peer[s]), 1);
        }
        for (int s = 0; s < kSfTmemGroups; ++s) mbar_init(smem_u32(&sh.grp_done[s]), two_issuers ? 2 : 1);
        mbar_init(smem_u32(&sh.tmem_full), two_issuers ? 2 : 1);
        mbar_init(smem_u32(&sh.first_done), 1);
        mbar_init(smem_u32(&sh.tmem_empty), kPair * kEpiWarps);
        if constexpr (kF32) {
            for (int b = 0; b < kScrBufs; ++b) {
                mbar_init(smem_u32(&sh.scr_full[b]), 1);
                mbar_init(smem_u32(&sh.scr_empty[b]), kEpiWarps * kPair);
            }
            for (int s = 0; s < kSfRing; ++s) mbar_init(smem_u32(&sh.sf_done[s]), kEpiWarps);
        }
        sh.abort = 0;
        sh.grouped_tiles = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b);
        tma_prefetch_desc(&map_sfa);
        tma_prefetch_desc(&map_sfb);
    }
    if (warp == 1) {
        if constexpr (kPair == 2) {
            tmem_alloc_pair(smem_u32(&sh.tmem_base), kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(&sh.tmem_base), kTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
    }
    // Everything above touches only shared memory, TMEM and the kernel
    // parameters, so it overlaps the previous kernel in the stream; every
    // global-memory access comes after this wait.
    grid_dependency_wait();
    grid_launch_dependents();
    if (p.groups > 0 && warp == 2) {
        if constexpr (kWgrad) wgrad_prefix(p, sh, lane);
        else group_prefix<C::kTileM>(p, sh, lane);
    }
    __syncthreads();
    if constexpr (kPair == 2) cluster_sync();      // peer barriers initialised before any remote use
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    const int64_t total = p.groups > 0 ? sh.grouped_tiles : p.total_tiles;

    // FP32 scales: MMA issuer for the K-steps of one parity: 4 MMAs (N = 256,
    // K = 32 each) per K-step into product buffer kg % kScrBufs (= the parity),
    // once the epilogue warps of both CTAs read that buffer's previous product
    // (K-step kg - kScrBufs).  Two issuers (warps 1 and kMma2Warp) alternate
    // K-steps, so that one can wait for its operands or its buffer while the
    // other issues (a thread's tcgen05.mma issue blocks while the tensor pipe
    // is busy).  The MMAs run up to one K-step ahead of the epilogue, and on
    // into the next tile while the epilogue stores one.
    // (run by a whole warp, values warp-uniform; lane 0's tcgen05 operations
    // are predicated on)
    auto mma_f32 = [&](uint32_t par) {
        const uint32_t issue = lane == 0 ? 1u : 0u;
        uint32_t kg = 0;
        bool ok = true;
        for (int64_t t = unit; t < total && ok; t += units) {
            for (int32_t k = 0; k < p.k_iters; ++k, ++kg) {
                if ((kg & 1u) != par) continue;
                const uint32_t stage = kg % C::kStages, phase = (kg / C::kStages) & 1u;
                if (!__all_sync(0xFFFFFFFFu, wait_or_abort(smem_u32(&sh.full[stage]), phase, sh, p.status))) {
                    ok = false;
                    break;
                }
                const uint32_t buf = kg % kScrBufs, use = kg / kScrBufs;
                if (use >= 1 && !__all_sync(0xFFFFFFFFu, wait_or_abort(smem_u32(&sh.scr_empty[buf]), (use - 1) & 1u,
                                                                       sh, p.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint8_t* st = smem + stage * C::kStageBytes;
                const uint64_t a_desc = smem_desc(smem_u32(st), 16, 1024, 2);
                const uint64_t b_desc = smem_desc(smem_u32(st + C::kABytes), 16, 1024, 2);
                const uint32_t d = tmem + uint32_t(C::kBN) * buf;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    if constexpr (kPair == 2)
                        mma_f8_pair_if(d, a_desc + 2 * kk, b_desc + 2 * kk, C::kIdescF32, kk != 0 ? 1u : 0u, issue);
                    else
                        mma_f8_if(d, a_desc + 2 * kk, b_desc + 2 * kk, C::kIdescF32, kk != 0 ? 1u : 0u, issue);
                }
                if constexpr (kPair == 2) {
                    tc_commit_pair_mc_if(smem_u32(&sh.empty[stage]), 0x3, issue);
                    tc_commit_pair_mc_if(smem_u32(&sh.scr_full[buf]), 0x3, issue);
                } else {
                    tc_commit_if(smem_u32(&sh.empty[stage]), issue);
                    tc_commit_if(smem_u32(&sh.scr_full[buf]), issue);
                }
            }
        }
    };

    // MXFP8: MMA issuer for the K-steps of one parity of the global K-step
    // count: 4 block-scaled MMAs (K = 32 each) per 128-wide K-step.  Two
    // issuers (warps 1 and kMma2Warp) alternate K-steps, so that one waits for
    // its operands or blocks in a tcgen05.mma issue while the other issues.
    // MMAs of different threads may run in either order, which only reorders
    // the fp32 additions, except for a tile's first K-step, which overwrites
    // the accumulator: the issuer that does not own it waits until its MMAs
    // completed (first_done) before issuing any of the tile's MMAs.  That
    // wait costs about one K-step's latency per tile, so only dense GEMMs of
    // at least kSplitMinK K-steps use two issuers (two_issuers).  Both
    // issuers wait for the accumulator, each scale group and the operands of
    // their own K-steps, and both commit every scale group (grp_done) and
    // every tile (tmem_full), whose barriers count two arrivals.
    // (run by a whole warp, values warp-uniform; lane 0's tcgen05 operations
    // are predicated on: about 4 % fewer cycles per K-step than a loop that
    // lane 0 runs alone)
    auto mma_mx = [&](uint32_t par) {
        const uint32_t issue = lane == 0 ? 1u : 0u;
        uint32_t g = 0, grp = 0;   // global K-step and scale-group counts (both issuers' K-steps)
        int32_t local = 0;
        bool ok = true;
        auto wait = [&](const uint64_t& bar, uint32_t parity) -> bool {
            // (the lanes decide together: warp-collective tcgen05 operations follow)
            return __all_sync(0xFFFFFFFFu, wait_or_abort(smem_u32(&bar), parity, sh, p.status));
        };
        for (int64_t t = unit; t < total && ok; t += units, ++local) {
            const int32_t nk = p.k_iters;
            if (local > 0) {
                if (!wait(sh.tmem_empty, uint32_t(local - 1) & 1u)) break;
                tc_fence_after();
            }
            if ((g & 1u) != par) {               // the other issuer owns the tile's first K-step
                if (!wait(sh.first_done, uint32_t(local) & 1u)) break;
                tc_fence_after();
            }
            for (int32_t k = 0; k < nk; ++k, ++g) {
                const bool mine = (g & 1u) == par;
                const uint32_t stage = g % C::kStages, phase = (g / C::kStages) & 1u;
                // (the operands first, then a new scale group's factors, as in
                // the single-issuer loop)
                if (mine && !wait(sh.full[stage], phase)) { ok = false; break; }
                if ((k & 3) == 0) {
                    if (!wait(sh.sf_ready[grp % kSfRing], (grp / kSfRing) & 1u)) { ok = false; break; }
                    tc_fence_after();
                }
                if (mine) {
                    uint8_t* st = smem + stage * C::kStageBytes;
                    const uint32_t sf_col = tmem + kSfCol0 + ((grp % kSfTmemGroups) * 4 + uint32_t(k & 3)) * kSfSlotCols;
                    const uint64_t a_desc = smem_desc(smem_u32(st), 16, 1024, 2);
                    const uint64_t b_desc = smem_desc(smem_u32(st + C::kABytes), 16, 1024, 2);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        // +32 bytes along K inside the 128-byte swizzled row = +2 in the address field
                        const uint32_t idesc = idesc_sf(C::kIdescBase, uint32_t(kk));
                        const uint32_t acc = (k | kk) != 0 ? 1u : 0u;
                        if constexpr (kPair == 2)
                            mma_mxf8_pair_if(tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc, sf_col, sf_col + 4, acc,
                                             issue);
                        else
                            mma_mxf8_if(tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc, sf_col, sf_col + 4, acc, issue);
                    }
                    if constexpr (kPair == 2) tc_commit_pair_mc_if(smem_u32(&sh.empty[stage]), 0x3, issue);
                    else tc_commit_if(smem_u32(&sh.empty[stage]), issue);
                    if (k == 0) {
                        if constexpr (kPair == 2) tc_commit_pair_mc_if(smem_u32(&sh.first_done), 0x1, issue);
                        else tc_commit_if(smem_u32(&sh.first_done), issue);
                    }
                }
                if ((k & 3) == 3 || k == nk - 1) {             // last K-step of the scale group
                    if constexpr (kPair == 2)
                        tc_commit_pair_mc_if(smem_u32(&sh.grp_done[grp % kSfTmemGroups]), 0x1, issue);
                    else tc_commit_if(smem_u32(&sh.grp_done[grp % kSfTmemGroups]), issue);
                    ++grp;
                }
            }
            if (!ok) break;
            if constexpr (kPair == 2) tc_commit_pair_mc_if(smem_u32(&sh.tmem_full), 0x3, issue);
            else tc_commit_if(smem_u32(&sh.tmem_full), issue);
        }
    };

    // Role warps (for FP32 scales warp group 0) and epilogue warps.  With FP32
    // scales the role warp group gives registers to the epilogue warp groups,
    // whose threads hold 128 accumulator columns and a product slice each
    // (the host checked that the split fits); each side changes its count
    // first, before the warps of a group part ways.
    const bool role_warp = kF32 ? warp < 4 : (warp < 2 || warp == C::kSfWarp || warp == C::kMma2Warp);
    if (role_warp) {
        if constexpr (kF32) regs_lower<kRegsRoles>();
        if (warp == 0) {
            // ------------------------------------------------ TMA producer (every CTA)
            if (lane == 0) {
                int32_t hint = 0;
                uint32_t stage = 0, phase = 0;
                bool ok = true;
                for (int64_t t = unit; t < total && ok; t += units) {
                    const Tile tl = map_tile<C::kTileM, C::kBN, kWgrad>(p, sh, t, hint);
                    const int32_t a_row = tl.a_row + int32_t(rank) * kBM;
                    const int32_t b_row = tl.b_row + int32_t(rank) * C::kBRows;
                    for (int32_t k = 0; k < tl.nk; ++k) {
                        const int32_t kx = (tl.k0 + k) * kBK;
                        if (!wait_or_abort(smem_u32(&sh.empty[stage]), phase ^ 1u, sh, p.status)) { ok = false; break; }
                        uint8_t* st = smem + stage * C::kStageBytes;
                        const uint32_t full = leader(sh.full[stage]);
                        if constexpr (kPair == 2) {
                            if (rank == 0) mbar_arrive_expect_tx(smem_u32(&sh.full[stage]), C::kABytes + C::kBBytes);
                            else mbar_arrive_expect_tx_cluster_relaxed(full, C::kABytes + C::kBBytes);
                            tma_load_2d_pair(smem_u32(st), &map_a, full, kx, a_row);
                            tma_load_2d_pair(smem_u32(st + C::kABytes), &map_b, full, kx, b_row);
                        } else {
                            mbar_arrive_expect_tx(full, C::kABytes + C::kBBytes);
                            tma_load_2d(smem_u32(st), &map_a, full, kx, a_row);
                            tma_load_2d(smem_u32(st + C::kABytes), &map_b, full, kx, b_row);
                        }
                        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                    }
                }
            }
        } else if (warp == 1) {
            // ------------------------------------------------ MMA issuer (the MMA CTA)
            if (rank == 0 && kF32) {
                mma_f32(0u);
            } else if (rank == 0 && two_issuers) {
                mma_mx(0u);
            } else if (rank == 0) {
                // The whole warp runs the loop (its values stay warp-uniform) and
                // lane 0's tcgen05.mma / tcgen05.commit are predicated on: about 4 %
                // fewer cycles per K-step than a loop that lane 0 runs alone.
                const uint32_t issue = lane == 0 ? 1u : 0u;
                uint32_t stage = 0, phase = 0, grp = 0;   // grp: global index of the current scale group
                int32_t local = 0, hint = 0;
                bool ok = true;
                for (int64_t t = unit; t < total && ok; t += units, ++local) {
                    // K-steps of this tile (wgrad: the expert's own; 0 for an expert without tokens)
                    int32_t nk = p.k_iters;
                    if constexpr (kWgrad) nk = map_tile<C::kTileM, C::kBN, kWgrad>(p, sh, t, hint).nk;
                    if (local > 0) {
                        if (!__all_sync(0xFFFFFFFFu, wait_or_abort(smem_u32(&sh.tmem_empty), uint32_t(local - 1) & 1u, sh,
                                                                   p.status)))
                            break;
                        tc_fence_after();
                    }
                    for (int32_t k = 0; k < nk; ++k) {
                        if (!__all_sync(0xFFFFFFFFu, wait_or_abort(smem_u32(&sh.full[stage]), phase, sh, p.status))) {
                            ok = false;
                            break;
                        }
                        uint8_t* st = smem + stage * C::kStageBytes;
                        if ((k & 3) == 0) {
                            if (!__all_sync(0xFFFFFFFFu, wait_or_abort(smem_u32(&sh.sf_ready[grp % kSfRing]),
                                                                       (grp / kSfRing) & 1u, sh, p.status))) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        const uint32_t sf_col =
                            tmem + kSfCol0 + ((grp % kSfTmemGroups) * 4 + uint32_t(k & 3)) * kSfSlotCols;
                        const uint64_t a_desc = smem_desc(smem_u32(st), 16, 1024, 2);
                        const uint64_t b_desc = smem_desc(smem_u32(st + C::kABytes), 16, 1024, 2);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            // +32 bytes along K inside the 128-byte swizzled row = +2 in the address field
                            const uint32_t idesc = idesc_sf(C::kIdescBase, uint32_t(kk));
                            const uint32_t acc = (k | kk) != 0 ? 1u : 0u;
                            if constexpr (kPair == 2)
                                mma_mxf8_pair_if(tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc, sf_col, sf_col + 4, acc,
                                                 issue);
                            else
                                mma_mxf8_if(tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc, sf_col, sf_col + 4, acc, issue);
                        }
                        if constexpr (kPair == 2) tc_commit_pair_mc_if(smem_u32(&sh.empty[stage]), 0x3, issue);
                        else tc_commit_if(smem_u32(&sh.empty[stage]), issue);
                        if ((k & 3) == 3 || k == nk - 1) {             // last K-step of the scale group
                            if constexpr (kPair == 2)
                                tc_commit_pair_mc_if(smem_u32(&sh.grp_done[grp % kSfTmemGroups]), 0x1, issue);
                            else tc_commit_if(smem_u32(&sh.grp_done[grp % kSfTmemGroups]), issue);
                            ++grp;
                        }
                        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                    }
                    if (!ok) break;
                    if constexpr (kPair == 2) tc_commit_pair_mc_if(smem_u32(&sh.tmem_full), 0x3, issue);
                    else tc_commit_if(smem_u32(&sh.tmem_full), issue);
                }
            }
        } else if (warp == C::kMma2Warp) {
            if (rank == 0) {
                if constexpr (kF32) mma_f32(1u);
                else if (two_issuers) mma_mx(1u);
            }
        } else {                                   // the scale-factor warp
            // ------------------------------------------------ scale-factor layout (every CTA)
            // Scale groups (4 K-steps each, the last of a tile possibly shorter)
            // go through a kSfRing-slot ring: lane 0 loads group j + kSfAhead
            // while group j is prepared.  Group j is copied into TMEM only after
            // the MMAs of group j - 3 completed (grp_done); that keeps its TMEM
            // slots free and also means the MMA warp has passed its wait on
            // sf_ready of group j - 3, the previous user of this ring slot.  A ring
            // slot is reloaded only after the copies of its previous group landed
            // (sf_ready).  So every barrier phase here is observed by its waiter
            // before the barrier can complete again.
            uint8_t* ring = smem + C::kStages * C::kStageBytes;
            auto tile_groups = [](const Tile& t) { return (t.nk + 3) / 4; };
            int64_t lt = unit;                // next group to load: tile lt, group lg
            int32_t lg = 0, lhint = 0;
            uint32_t jl = 0;                  // its global index
            Tile ltl{};
            auto seek = [&]() {               // the first tile from lt on that has scale groups
                for (; lt < total; lt += units) {
                    ltl = map_tile<C::kTileM, C::kBN, kWgrad>(p, sh, lt, lhint);
                    if (tile_groups(ltl) > 0) break;
                }
            };
            seek();
            bool ok = true;
            auto load_next = [&]() -> bool {  // lane 0
                if (lt >= total) return true;
                const uint32_t slot = jl % kSfRing;
                // reuse a slot once its previous group is consumed: copied into
                // TMEM (MX), or read by this CTA's epilogue warps (FP32 scales)
                if (jl >= kSfRing &&
                    !wait_or_abort(smem_u32(kF32 ? &sh.sf_done[slot] : &sh.sf_ready[slot]), ((jl / kSfRing) - 1) & 1u,
                                   sh, p.status))
                    return false;
                const uint32_t bar = smem_u32(&sh.sf_full[slot]);
                const uint32_t dst = smem_u32(ring + slot * C::kSfSlotBytes);
                mbar_arrive_expect_tx(bar, kSFABytes + C::kSFBBytes);
                tma_load_2d(dst, &map_sfa, bar, ltl.sf0 + lg * 16, ltl.a_row + int32_t(rank) * kBM);
                tma_load_2d(dst + kSFABytes, &map_sfb, bar, ltl.sf0 + lg * 16, ltl.b_row);
                ++jl;
                if (++lg == tile_groups(ltl)) {
                    lg = 0;
                    lt += units;
                    seek();
                }
                return true;
            };
            if (lane == 0)
                for (int i = 0; i < kSfAhead && ok; ++i) ok = load_next();
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            uint32_t j = 0;
            int32_t chint = 0;
            for (int64_t t = unit; t < total && ok; t += units) {
                const Tile ct = map_tile<C::kTileM, C::kBN, kWgrad>(p, sh, t, chint);
                const int32_t ngroups = tile_groups(ct);
                for (int32_t g = 0; g < ngroups && ok; ++g, ++j) {
                    const uint32_t slot = j % kSfRing, bit = (j / kSfRing) & 1u;
                    if (!wait_or_abort(smem_u32(&sh.sf_full[slot]), bit, sh, p.status)) { ok = false; break; }
                    const uint32_t sf = smem_u32(ring + slot * C::kSfSlotBytes);
                    if constexpr (kF32) {
                        // B's scales [256 columns][4 K-steps] -> [4 K-steps][256 columns] (fp32), so
                        // that the epilogue reads 4 consecutive columns' scales at once; A's stay
                        // [128 rows][4 K-steps].  The whole warp reads before anyone writes.
                        static_assert(C::kBN == 256, "the transpose covers 256 B rows");
                        uint4 v[8];
    #pragma unroll
                        for (int i = 0; i < 8; ++i) v[i] = lds128(sf + kSFABytes + (128 * (i >> 2) + 4 * lane + (i & 3)) * 16);
                        __syncwarp();
    #pragma unroll
                        for (int hb = 0; hb < 2; ++hb) {       // columns 128 hb + 4 lane .. + 3
                            const uint32_t w = sf + kSFABytes + 512 * hb + 16 * lane;
                            const uint4* u = v + 4 * hb;
                            sts128(w, u[0].x, u[1].x, u[2].x, u[3].x);
                            sts128(w + 1024, u[0].y, u[1].y, u[2].y, u[3].y);
                            sts128(w + 2048, u[0].z, u[1].z, u[2].z, u[3].z);
                            sts128(w + 3072, u[0].w, u[1].w, u[2].w, u[3].w);
                        }
                        fence_proxy_async_smem();            // the slot is next written by TMA
                        __syncwarp();
                        if (lane == 0) {
                            mbar_arrive(smem_u32(&sh.sf_ready[slot]));
                            ok = load_next();
                        }
                        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                        continue;
                    }
                    sf_to_tmem_layout(sf, lane);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (kPair == 2 && rank != 0) {
                            mbar_arrive_cluster(leader(sh.sf_peer[slot]));
                        } else {
                            if (kPair == 2) ok = wait_or_abort(smem_u32(&sh.sf_peer[slot]), bit, sh, p.status);
                            if (ok && j >= 3)
                                ok = wait_or_abort(smem_u32(&sh.grp_done[(j - 3) % kSfTmemGroups]),
                                                   ((j - 3) / kSfTmemGroups) & 1u, sh, p.status);
                            if (ok) {
                                tc_fence_after();
                                const int nchunks = min(4, ct.nk - 4 * g);
                                for (int c = 0; c < nchunks; ++c) {
                                    const uint32_t col = tmem + kSfCol0 + ((j % kSfTmemGroups) * 4 + c) * kSfSlotCols;
                                    const uint64_t d0 = smem_desc(sf + c * 512, 0, 128, 0);
                                    const uint64_t d1 = smem_desc(sf + 2048 + c * 512, 0, 128, 0);
                                    const uint64_t d2 = smem_desc(sf + 4096 + c * 512, 0, 128, 0);
                                    if constexpr (kPair == 2) {
                                        tc_cp_32x128b_warpx4_pair(col + 0, d0);
                                        tc_cp_32x128b_warpx4_pair(col + 4, d1);
                                        tc_cp_32x128b_warpx4_pair(col + 8, d2);
                                    } else {
                                        tc_cp_32x128b_warpx4(col + 0, d0);
                                        tc_cp_32x128b_warpx4(col + 4, d1);
                                        tc_cp_32x128b_warpx4(col + 8, d2);
                                    }
                                }
                                // sf_ready completes once these copies landed (in both CTAs of a pair)
                                if constexpr (kPair == 2) tc_commit_pair_mc(smem_u32(&sh.sf_ready[slot]), 0x3);
                                else tc_commit(smem_u32(&sh.sf_ready[slot]));
                            }
                        }
                        if (ok) ok = load_next();
                    }
                    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                }
            }
        }
    } else {
        if constexpr (kF32) regs_raise<kRegsEpi>();
        // ------------------------------------------------ epilogue (every CTA)
        const int e = warp - C::kEpiWarp0, q = warp & 3, h = e >> 2;
        int32_t hint = 0, local = 0;
        uint32_t kg = 0, jg = 0;                 // FP32 scales: K-steps and scale groups consumed
        for (int64_t t = unit; t < total; t += units, ++local) {
            const Tile tl = map_tile<C::kTileM, C::kBN, kWgrad>(p, sh, t, hint);
            // this warp's 128 output columns; their bias is loaded now, while
            // the tile's MMAs run
            const int32_t nbw = tl.n0 + 128 * h;
            uint4 bias_pre = make_uint4(0u, 0u, 0u, 0u);
            if (C::kStagedStores && p.has_bias && lane < 16 && nbw + 8 * lane < p.N)
                bias_pre = __ldg(reinterpret_cast<const uint4*>(p.bias + int64_t(tl.group) * p.N + nbw + 8 * lane));
            uint32_t acc0[64], acc1[64];
            if constexpr (kF32) {
                // acc (registers: my row x the warp's 128 columns 128 h ..) +=
                // product(K-step) * sA[row][kb] * sB[col][kb], one K-step (128)
                // per scale block
#pragma unroll
                for (int i = 0; i < 64; ++i) acc0[i] = acc1[i] = 0u;
                uint32_t slot = 0;
                bool ok = true;
                const uint32_t lanes = uint32_t(32 * q) << 16;
                for (int32_t k = 0; k < tl.nk; ++k, ++kg) {
                    if ((k & 3) == 0) {
                        slot = jg % kSfRing;
                        // (the lanes decide together: warp-collective tcgen05 operations follow)
                        if (!__all_sync(0xFFFFFFFFu, wait_or_abort(smem_u32(&sh.sf_ready[slot]), (jg / kSfRing) & 1u,
                                                                   sh, p.status))) {
                            ok = false;
                            break;
                        }
                    }
                    const uint32_t b = kg % kScrBufs;
                    if (!__all_sync(0xFFFFFFFFu, wait_or_abort(smem_u32(&sh.scr_full[b]), (kg / kScrBufs) & 1u, sh,
                                                               p.status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t src = tmem + lanes + uint32_t(C::kBN) * b + uint32_t(128 * h);
                    uint32_t v[64];
                    tmem_ld_32x32b_x64(src, v);
                    const uint32_t sf = smem_u32(smem + C::kStages * C::kStageBytes + slot * C::kSfSlotBytes);
                    const float sa = __uint_as_float(lds32(sf + (32 * q + lane) * 16 + (k & 3) * 4));
                    // B scales of my 128 columns: [4 K-steps][256 columns] fp32
                    const uint32_t sbt = sf + kSFABytes + (k & 3) * 1024 + 512 * h;
                    // 2D weight blocks: the warp's 128 columns are one 128 x 128 block
                    const float f = p.b_2d ? sa * __uint_as_float(lds32(sbt)) : 0.0f;
                    tmem_ld_wait();
                    scale_accumulate_64(acc0, v, p.b_2d, f, sa, sbt);
                    tmem_ld_32x32b_x64(src + 64, v);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    const bool last_of_group = (k & 3) == 3 || k == tl.nk - 1;
                    if (lane == 0) {                      // the product is in registers: release its buffer
                        if constexpr (kPair == 2) mbar_arrive_cluster_relaxed(leader(sh.scr_empty[b]));
                        else mbar_arrive(smem_u32(&sh.scr_empty[b]));
                    }
                    scale_accumulate_64(acc1, v, p.b_2d, f, sa, sbt + 256);
                    __syncwarp();
                    if (lane == 0 && last_of_group) mbar_arrive(smem_u32(&sh.sf_done[slot]));   // scales read
                    if (last_of_group) ++jg;
                }
                if (!ok) break;
            } else {
            if (!__all_sync(0xFFFFFFFFu, wait_or_abort(smem_u32(&sh.tmem_full), uint32_t(local) & 1u, sh, p.status)))
                break;                           // (all lanes together: tcgen05.ld is warp-collective)
            tc_fence_after();
            if (!kWgrad || tl.nk > 0) {
                const uint32_t taddr = tmem + (uint32_t(32 * q) << 16) + uint32_t(128 * h);
                tmem_ld_32x32b_x64(taddr, acc0);
                tmem_ld_32x32b_x64(taddr + 64, acc1);
                tmem_ld_wait();
            } else {                             // no K-steps (an expert without tokens): the product is 0
#pragma unroll
                for (int i = 0; i < 64; ++i) acc0[i] = acc1[i] = 0u;
            }
            tc_fence_before();
            // Each epilogue warp releases its part of the accumulator with one
            // relaxed arrive on the MMA CTA's barrier, which completes once all
            // the warps of the CTA (of both CTAs of a pair) hold their registers
            // (the reads retired at wait::ld; a release arrive would also wait
            // for this warp's earlier global stores).
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(leader(sh.tmem_empty));
            }
            const int64_t row = int64_t(tl.d_row) + int64_t(rank) * kBM + 32 * q + lane;
            if constexpr (C::kStagedStores) {
                const int64_t row0 = row - lane;
                if (row0 < tl.row_end) {             // warp-uniform: some row of this warp is stored
                    // output columns of acc0 / acc1
                    const int32_t nb0 = nbw;
                    const uint32_t epi = smem_u32(smem + C::kStages * C::kStageBytes + kSfRing * C::kSfSlotBytes);
                    const uint32_t stage = epi + uint32_t(e) * 4096u;
                    const uint32_t bias = epi + uint32_t(C::kEpiStageBytes) + uint32_t(e) * 256u;
                    if (p.has_bias) {                // (the warp read its previous tile's slice in program order)
                        if (lane < 16) sts128(bias + 16 * lane, bias_pre.x, bias_pre.y, bias_pre.z, bias_pre.w);
                        __syncwarp();
                    }
                    // TMA stores where the warp's 32 rows all belong to the tile, or run
                    // past the end of D (clipped there); per-row stores otherwise
                    const int64_t d_rows = kWgrad ? int64_t(p.groups) * p.M : p.M;
                    const bool tma = !kAcc && (row0 + 32 <= tl.row_end || tl.row_end == d_rows);
                    if (nb0 < p.N)
                        store_64_staged<kAcc>(acc0, p, bias, row0, tl.row_end, nb0, stage, lane, &map_d, &map_aux, tma);
                    if (nb0 + 64 < p.N)
                        store_64_staged<kAcc>(acc1, p, bias + 128u, row0, tl.row_end, nb0 + 64, stage, lane, &map_d,
                                              &map_aux, tma);
                }
            } else {
                // (tcgen05.ld is warp-collective: the lanes' row test guards the stores only)
                const bool live = row < tl.row_end;
                const uint16_t* bias = p.has_bias ? p.bias + int64_t(tl.group) * p.N : nullptr;
                const int32_t nb = tl.n0 + 128 * h;
                // The next tile's operands stream in while these stores go out;
                // a burst of D/AUX stores at the start of that tile slows its
                // loads, so the 8 chunks are spread over about half of the
                // tile's mainloop (~700 cycles per K-step).
                const uint32_t gap_ns = uint32_t(tl.nk) * 20u;
                if (live) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (nb + 16 * j < p.N) store_chunk<kAcc>(acc0 + 16 * j, p, bias, row, nb + 16 * j);
                        __nanosleep(gap_ns);
                    }
                }
                if (live) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (nb + 64 + 16 * j < p.N) store_chunk<kAcc>(acc1 + 16 * j, p, bias, row, nb + 64 + 16 * j);
                        if (j < 3) __nanosleep(gap_ns);
                    }
                }
            }
        }
    }

    if (C::kStagedStores && lane == 0) bulk_wait_all();   // this warp's TMA stores (epilogue warps)
    __syncthreads();
    if constexpr (kPair == 2) cluster_sync();      // no CTA leaves while its peer may still signal it
    if (warp == 1) {
        tc_fence_after();
        if constexpr (kPair == 2) tmem_dealloc_pair(tmem, kTmemCols);
        else tmem_dealloc(tmem, kTmemCols);
    }
}

template <int kPair, bool kAcc, bool kWgrad, bool kF32 = false>
te_mx_status launch_gemm(const GemmArgs& a, int sms, unsigned int* status, cudaStream_t stream) {
    using C = Cfg<kPair, kF32>;
    const bool grouped = a.groups > 0;
    const bool wg = a.wgrad;
    // Extent and pitch of the operands along the reduction axis: K for the
    // dense and grouped GEMMs, the token capacity of the padded layout for wgrad.
    const uint64_t kext = wg ? uint64_t(a.ld_code) : uint64_t(a.K);
    const uint64_t b_rows = (grouped && !wg) ? uint64_t(a.groups) * uint64_t(a.N) : uint64_t(a.N);
    // scale rows in bytes: E8M0, one per 32 K; FP32 scales, 4 bytes per 128 K
    const uint64_t sf_bytes = kF32 ? uint64_t(a.K / 128) * 4 : uint64_t(a.K / 32);
    const uint64_t sf_cols = sf_bytes < 16 ? 16 : sf_bytes;
    const uint64_t sfa_cols = wg ? uint64_t(a.ld_sA) : sf_cols, sfb_cols = wg ? uint64_t(a.ld_sB) : sf_cols;
    const uint64_t sfa_pitch = kF32 ? uint64_t(a.ld_sA) * 4 : uint64_t(a.ld_sA);
    const uint64_t sfb_pitch = kF32 ? uint64_t(a.ld_sB) * 4 : uint64_t(a.ld_sB);
    CUtensorMap ma, mb, msa, msb;
    te_mx_status st;
    if ((st = encode_tensor_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.A, kext, uint64_t(a.M),
                                   kext, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B)) != TE_MX_OK) return st;
    if ((st = encode_tensor_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, kext, b_rows,
                                   kext, kBK, C::kBRows, CU_TENSOR_MAP_SWIZZLE_128B)) != TE_MX_OK) return st;
    if ((st = encode_tensor_map_2d(&msa, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.sA, sfa_cols, uint64_t(a.M),
                                   sfa_pitch, 16, kBM, CU_TENSOR_MAP_SWIZZLE_NONE)) != TE_MX_OK) return st;
    if ((st = encode_tensor_map_2d(&msb, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.sB, sfb_cols, b_rows,
                                   sfb_pitch, 16, C::kBN, CU_TENSOR_MAP_SWIZZLE_NONE)) != TE_MX_OK) return st;
    // bf16 D and AUX as 32 x 64 boxes in the epilogue's 128-byte-swizzled
    // staging layout (CTA pairs store through them; unused otherwise)
    CUtensorMap md = ma, mx = ma;
    if (C::kStagedStores && !kAcc) {
        const uint64_t d_rows = wg ? uint64_t(a.groups) * uint64_t(a.M) : uint64_t(a.M);
        if ((st = encode_tensor_map_2d(&md, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.D, uint64_t(a.N), d_rows,
                                       uint64_t(a.N) * 2, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B)) != TE_MX_OK)
            return st;
        mx = md;
        if (a.gelu && (st = encode_tensor_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.aux, uint64_t(a.N), d_rows,
                                                 uint64_t(a.N) * 2, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B)) != TE_MX_OK)
            return st;
    }

    GemmParams p{};
    p.M = a.M;
    p.N = int32_t(a.N);
    p.K = int32_t(a.K);
    p.k_iters = wg ? 0 : int32_t(a.K / kBK);
    p.n_tiles = int32_t((a.N + C::kBN - 1) / C::kBN);
    p.m_tiles = int32_t((a.M + C::kTileM - 1) / C::kTileM);
    p.total_tiles = grouped ? 0 : int64_t(p.m_tiles) * p.n_tiles;
    p.groups = a.groups;
    p.group_m = a.group_m;
    p.bias = static_cast<const uint16_t*>(a.bias);
    p.D = static_cast<uint16_t*>(a.D);
    p.aux = static_cast<uint16_t*>(a.aux);
    p.has_bias = a.has_bias;
    p.gelu = a.gelu;
    p.dgelu = a.dgelu;
    p.wgrad = wg;
    p.total_m = a.total_m;
    p.ld_code = a.ld_code;
    p.ld_sfa = a.ld_sA;
    p.ld_sfb = a.ld_sB;
    p.b_2d = a.b_2d;
    p.status = status;

    const int64_t slots = sms / kPair;                     // CTAs (pairs) resident at once
    int64_t units = grouped ? slots : (p.total_tiles < slots ? p.total_tiles : slots);
    if (units < 1) units = 1;
    auto kern = gemm_kernel<kPair, kAcc, kWgrad, kF32>;
    cudaError_t e = set_smem_attribute_once(reinterpret_cast<const void*>(kern), C::kSmemDyn);
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(gemm)");
    if constexpr (kF32) {
        // the kernel moves registers between warp groups (setmaxnreg): the
        // block must be launched with at least the registers the split hands
        // out, or a raise would wait for ever
        cudaFuncAttributes fa{};
        if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return cuda_status(e, "cudaFuncGetAttributes(gemm)");
        if (fa.numRegs * 12 < 4 * kRegsRoles + 8 * kRegsEpi)
            return set_error(TE_MX_ERR_CUDA, "GEMM with FP32 scales built with %d registers per thread; its register "
                             "split needs %d", fa.numRegs, (4 * kRegsRoles + 8 * kRegsEpi) / 12);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(units * kPair));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemDyn;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPair;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent launch: the CTAs may start, and set up their
    // barriers and TMEM, while the previous kernel in the stream finishes
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if constexpr (kPair == 2) {
        // persistent grid: never more pairs than can be resident together (the
        // occupancy query is slow, so its answer is kept per device)
        static int max_clusters_of[64];
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_status(e, "cudaGetDevice");
        int max_clusters = dev < 64 ? __atomic_load_n(&max_clusters_of[dev], __ATOMIC_RELAXED) : 0;
        if (max_clusters == 0) {
            e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
            if (e != cudaSuccess) return cuda_status(e, "cudaOccupancyMaxActiveClusters(gemm)");
            if (max_clusters < 1) return set_error(TE_MX_ERR_CUDA, "no CTA pair of the GEMM fits on this device");
            if (dev < 64) __atomic_store_n(&max_clusters_of[dev], max_clusters, __ATOMIC_RELAXED);
        }
        if (units > max_clusters) units = max_clusters;
        cfg.gridDim = dim3(unsigned(units * kPair));
    }
    e = cudaLaunchKernelEx(&cfg, kern, ma, mb, msa, msb, md, mx, p);
    return cuda_status(e, "gemm kernel launch");
}

}  // namespace

te_mx_status gemm_launch(const GemmArgs& a, cudaStream_t stream) {
    unsigned int* status = nullptr;
    te_mx_status st = device_status_ptr(&status);
    if (st != TE_MX_OK) return st;
    int sms = 0;
    if ((st = device_sm_count(&sms)) != TE_MX_OK) return st;
    // CTA pairs whenever the rows fill a 256-row pair tile: an SM of a pair
    // loads 32 KB per K-step for the same MMA work for which a single CTA
    // loads 48 KB, and operand ingress is what bounds the mainloop, so pairs
    // are faster even when fewer tiles than pairs exist (a single-CTA split
    // would keep the same number of SMs busy).  FP32 scales: the same rule.
    const bool pair = a.wgrad ? a.M >= 256 : (a.groups > 0 ? a.M >= 256 * 8 : a.M >= 256);
    if (a.f32_scales) return pair ? launch_gemm<2, false, false, true>(a, sms, status, stream)
                                  : launch_gemm<1, false, false, true>(a, sms, status, stream);
    if (a.wgrad) {
        if (a.acc_f32) return pair ? launch_gemm<2, true, true>(a, sms, status, stream)
                                   : launch_gemm<1, true, true>(a, sms, status, stream);
        return pair ? launch_gemm<2, false, true>(a, sms, status, stream)
                    : launch_gemm<1, false, true>(a, sms, status, stream);
    }
    if (a.acc_f32) return pair ? launch_gemm<2, true, false>(a, sms, status, stream)
                               : launch_gemm<1, true, false>(a, sms, status, stream);
    return pair ? launch_gemm<2, false, false>(a, sms, status, stream)
                : launch_gemm<1, false, false>(a, sms, status, stream);
}

}  // namespace temx
