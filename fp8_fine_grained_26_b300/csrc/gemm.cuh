// gemm.cuh -- block-scaled FP8 GEMM with per-128-K promotion (dense and
// grouped-by-expert), sm_103a.
//
// What it computes ["DeepSeek-V3 Technical Report digest", section 3: all
// GEMMs in FP8, partial results promoted to FP32 every 128 accumulated
// elements; "DeepSeek-V3 training walkthrough", section 二(四): MMA
// intermediate results accumulated in FP32 registers; qqstock.cn walkthrough,
// report figure 7b]:
//     C[m][n] = sum_kb sA[kb][m] * sB(n, kb) * P_kb[m][n],
//     P_kb[m][n] = sum_{k in 128-wide slice kb} qA[m][k] * qB(n, k)   (exact FP8 products)
//
// Design (one persistent 384-thread CTA per SM; each CTA owns a 128 x 256
// FP32 output tile at a time):
//   warp 0      TMA producer: one 128-K slice of A (128x128 B) and B per
//               pipeline stage, 128-byte swizzle, STAGES-deep ring.
//   warp 1      MMA issuer: 4 x tcgen05.mma kind::f8f6f4 (K = 32 each) write a
//               FRESH FP32 partial P_kb into one of two 256-column TMEM
//               buffers (2 x 256 columns = all 512), then tcgen05.commit
//               frees the smem stage and signals the partial.
//   warps 4-11  promote / epilogue: two warpgroups, each owning 128 of the
//               256 columns; thread = tile row.  Per slice they load the
//               partial from TMEM (two 64-column tcgen05.ld 32x32b) and apply
//               acc = fma(P, sA*sB, acc) with packed f32x2 FMAs in FP32
//               registers -- the pages' promotion, on CUDA cores -- then
//               release the TMEM buffer so the MMA of slice kb+2 can start
//               while slice kb+1 is promoted.  After the last slice each
//               warpgroup rounds its 128 x 128 block to BF16 into two
//               128-row, 128-byte-swizzled staging boxes and goes on to the
//               next tile; FP32 outputs, unaligned row strides and the rows
//               of a grouped tile that reach past the expert's segment are
//               stored directly, masked.
//   warp 2      scale loader: copies each slice's row and column-block
//               scales into a shared ring ahead of the promote warps.
//   warp 3      store issuer: issues the TMA stores of the staged boxes
//               (rows >= M and columns >= N are clipped by the tensor map)
//               and hands the boxes back once the stores have read them.
// CTA pairs (PAIR, dense GEMMs of two or more M-blocks): a 2-CTA cluster
// computes a 256 x 256 tile with tcgen05 cta_group::2 MMAs (M = 256).  Each
// CTA stages only its own 128 rows of A and half (128 rows) of the B block,
// 32 KiB per stage instead of 48, and both CTAs' copies complete on the
// leader CTA's `full` barrier; the leader issues the MMAs and multicasts its
// commits to both CTAs; every promote warp of either CTA releases a TMEM
// buffer with one arrive on the leader's barrier.  Each CTA still promotes
// and stores its own 128 x 256 half.
// Every mbarrier wait is bounded (WAIT_LIMIT_NS); on expiry the kernel sets
// the device error word, stops all roles, drains its own TMA copies and MMAs,
// frees TMEM and returns.
#pragma once
#include "common.cuh"
#include "quant.cuh"            // the E4M3 encoder shared with the E4M3-output epilogue

namespace fp8bs {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr int A_STAGE_BYTES = BM * BK;                   // 16 KiB
constexpr int B_STAGE_BYTES = BN * BK;                   // 32 KiB
constexpr int EPI_BOX_BYTES = BM * 128;                 // one 128-row x 64-col BF16 output box
constexpr int GEMM_THREADS = 384;
constexpr uint32_t TMEM_COLS = 512;
constexpr int MAX_EXPERTS = 2048;
constexpr int SCALE_SLOTS = 8;                           // slices of scales staged ahead
constexpr int SCALE_SLOT_FLOATS = 132;                   // 128 row scales + 2 column-block scales (+pad)
constexpr int SCALE_SLOT_FLOATS_TOK = 384;               // weight gradient: 128 row + 256 column scales
constexpr int SCALE_LOOKAHEAD = 2;                       // loader copy groups in flight
constexpr uint64_t ABORT_GRACE_NS = 1000000;              // pair kernel: wait after an abort (1 ms)

// Shared-memory layout for S pipeline stages of BSB bytes of B each
// (offsets from a 1024-byte aligned base): operand stages, the output staging
// boxes (two 64-column halves per promote warpgroup, so a tile's stores never
// wait on each other), barriers, the scale ring and (grouped) the expert tile
// table.
template <int S, int BSB = B_STAGE_BYTES, int SSF = SCALE_SLOT_FLOATS>
struct Layout {
    static constexpr int A = 0;
    static constexpr int B = A + S * A_STAGE_BYTES;
    static constexpr int EPI = B + S * BSB;                          // [warpgroup][half] boxes
    static constexpr int BAR = EPI + 2 * 2 * EPI_BOX_BYTES;         // 8-byte barriers
    // full, empty, pfull, pempty, drain, sready, sfree, per-warpgroup epilogue pair
    static constexpr int NUM_BARS = 2 * S + 2 + 2 + 1 + 2 * SCALE_SLOTS + 4;
    static constexpr int MISC = BAR + NUM_BARS * 8;                 // tmem slot, abort flag
    static constexpr int SCALES = (MISC + 16 + 127) & ~127;         // scale ring (16-byte vector reads)
    static constexpr int TILES = SCALES + SCALE_SLOTS * SSF * 4;   // grouped: tile prefix [E+1]
    static_assert(SCALES % 16 == 0 && (SSF * 4) % 16 == 0, "scale slots must allow 16-byte reads");
    static_assert(EPI % 1024 == 0 && A % 1024 == 0 && B % 1024 == 0, "swizzled regions need 1024-byte alignment");
};

template <bool GROUPED, int S, int BSB = B_STAGE_BYTES, int SSF = SCALE_SLOT_FLOATS>
constexpr int gemm_smem_bytes()
{
    return 1024 + Layout<S, BSB, SSF>::TILES + (GROUPED ? (MAX_EXPERTS + 1) * 4 : 0);
}

struct GemmArgs {
    int64_t M;          // rows of A (grouped: M_total)
    int64_t N, K;
    int64_t ldc;
    const float *sA;    // [K/128][M]
    const float *sB;    // K-major: [ceil(N/128)][K/128] (grouped: per expert); MN-major: [K/128][N/128]
    void *C;
    const int32_t *offsets;   // grouped: [E+1]
    int E;
    int c_fp32;
    int c_tma;          // BF16 output through the C tensor map
    float *sC;          // E4M3 output: [N/128][M] scales of the 1x128 output tiles
    int num_m_blk;      // dense: ceil(M/128)
    int num_m_pair;     // dense, cluster pairs: ceil(num_m_blk / 2)
    int m_group;        // dense, cluster pairs: M-pairs per rasterisation group
    int num_n_blk;      // ceil(N/256)
    int KB;             // K/128
    int NB128;          // ceil(N/128)
    int64_t num_tiles;  // dense: num_m_blk * num_n_blk (cluster pairs: num_m_pair * num_n_blk)
    uint64_t wait_ns;   // time limit of every pipeline wait (WAIT_LIMIT_NS unless a test shortens it)
};

// tcgen05 instruction descriptor, kind::f8f6f4: D = F32 (bits 4-5 = 1),
// A = B = E4M3 (bits 7-9, 10-12 = 0), A K-major (bit 15 = 0), B K- or
// MN-major (bit 16), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n, bool b_mn_major)
{
    return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand: start
// address >> 4 (bits 0-13), leading byte offset >> 4 (16-29), stride byte
// offset >> 4 (32-45), descriptor version 1 (bit 46), swizzle mode
// 128B = 2 (bits 61-63).
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

struct Tile {
    int64_t m0;         // first row of the tile in A / C
    int64_t m_end;      // rows [m0, m_end) are stored (segment or matrix end)
    int32_t n0;         // first column
    int32_t expert;
};

template <int S, int BSB = B_STAGE_BYTES, int SSF = SCALE_SLOT_FLOATS>
struct SharedState {
    using L = Layout<S, BSB, SSF>;
    uint32_t base;      // shared address of the aligned base
    uint8_t *gbase;     // generic pointer to the same
    __device__ uint32_t bar(int i) const { return base + L::BAR + 8 * i; }
    __device__ uint32_t full(int s) const { return bar(s); }
    __device__ uint32_t empty(int s) const { return bar(S + s); }
    __device__ uint32_t pfull(int p) const { return bar(2 * S + p); }
    __device__ uint32_t pempty(int p) const { return bar(2 * S + 2 + p); }
    __device__ uint32_t drain() const { return bar(2 * S + 4); }
    __device__ uint32_t sready(int j) const { return bar(2 * S + 5 + j); }
    __device__ uint32_t sfree(int j) const { return bar(2 * S + 5 + SCALE_SLOTS + j); }
    // warpgroup wg's staging boxes are free (its issuing thread saw the last
    // stores read them) / filled (all four warps wrote and fenced)
    __device__ uint32_t epi_free(int wg) const { return bar(2 * S + 5 + 2 * SCALE_SLOTS + wg); }
    __device__ uint32_t epi_full(int wg) const { return bar(2 * S + 7 + 2 * SCALE_SLOTS + wg); }
    __device__ uint32_t epi_box(int wg, int h) const { return base + L::EPI + (2 * wg + h) * EPI_BOX_BYTES; }
    __device__ uint32_t scale_slot(int j) const { return base + L::SCALES + j * SSF * 4; }
    __device__ uint32_t a_stage(int s) const { return base + L::A + s * A_STAGE_BYTES; }
    __device__ uint32_t b_stage(int s) const { return base + L::B + s * BSB; }
    __device__ volatile uint32_t *tmem_slot() const
    {
        return reinterpret_cast<volatile uint32_t *>(gbase + L::MISC);
    }
    __device__ volatile uint32_t *abort_flag() const
    {
        return reinterpret_cast<volatile uint32_t *>(gbase + L::MISC + 4);
    }
    __device__ int32_t *tile_prefix() const
    {
        return reinterpret_cast<int32_t *>(gbase + L::TILES);
    }
};

template <int S, int BSB, int SSF, class Args>
__device__ __forceinline__ bool wait_bounded(const SharedState<S, BSB, SSF> &ss, const Args &g, uint32_t bar,
                                             uint32_t parity)
{
    return wait_bounded(bar, parity, ss.abort_flag(), g.wait_ns);
}

// A bounded wait whose outcome is the same for every lane of the warp: after a
// time-out or an abort one lane may still have seen the phase complete, and
// the warp-wide (.sync.aligned) tcgen05 loads that follow must be executed by
// all lanes or by none.
template <int S, int BSB, int SSF, class Args>
__device__ __forceinline__ bool warp_wait(const SharedState<S, BSB, SSF> &ss, const Args &g, uint32_t bar,
                                          uint32_t parity)
{
    return __all_sync(0xffffffffu, wait_bounded(ss, g, bar, parity));
}

template <bool GROUPED, int S, int BSB, int SSF>
__device__ __forceinline__ int64_t total_tiles(const GemmArgs &g, const SharedState<S, BSB, SSF> &ss)
{
    if constexpr (GROUPED)
        return ss.tile_prefix()[g.E];
    else
        return g.num_tiles;
}

template <bool GROUPED, bool PAIR, int S, int BSB, int SSF>
__device__ __forceinline__ Tile tile_at(const GemmArgs &g, const SharedState<S, BSB, SSF> &ss, int64_t t, uint32_t rank)
{
    Tile tl;
    if constexpr (GROUPED) {
        // expert e owns tiles [prefix[e], prefix[e+1]); within an expert the
        // M-blocks vary fastest so that the CTAs sharing one weight N-block
        // run together and the block is read from HBM once.
        const int32_t *pre = ss.tile_prefix();
        int lo = 0, hi = g.E;                       // find e: pre[e] <= t < pre[e+1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pre[mid] <= t) lo = mid; else hi = mid;
        }
        const int e = lo;
        const int64_t seg0 = min(max((int64_t)g.offsets[e], (int64_t)0), g.M);
        const int64_t seg1 = min(max((int64_t)g.offsets[e + 1], seg0), g.M);
        const int64_t mt = (seg1 - seg0 + BM - 1) / BM;
        const int64_t local = t - pre[e];
        const int64_t nb = local / mt;
        tl.m0 = seg0 + (local - nb * mt) * BM;
        tl.m_end = seg1;
        tl.n0 = (int32_t)(nb * BN);
        tl.expert = e;
    } else if constexpr (PAIR) {
        // work unit = one 256 x 256 tile of a CTA pair; CTA `rank` owns its
        // M-block 2 * pair + rank (a block past the last one computes on zero
        // rows and stores nothing).  Tiles are rasterised in groups of
        // m_group M-pairs: within a group the M-pairs vary fastest, then the
        // N-blocks, so the group's A rows stay in L2 while B streams once
        // per group instead of A being re-read for every N-block.
        const int64_t per_group = (int64_t)g.m_group * g.num_n_blk;
        const int64_t grp = t / per_group;
        const int64_t local = t - grp * per_group;
        const int64_t gsize = min((int64_t)g.m_group, (int64_t)g.num_m_pair - grp * g.m_group);
        const int64_t nb = local / gsize;
        tl.m0 = (2 * (grp * g.m_group + (local - nb * gsize)) + rank) * BM;
        tl.m_end = g.M;
        tl.n0 = (int32_t)(nb * BN);
        tl.expert = 0;
        (void)ss;
    } else {
        const int64_t nb = t / g.num_m_blk;
        tl.m0 = (t - nb * g.num_m_blk) * BM;
        tl.m_end = g.M;
        tl.n0 = (int32_t)(nb * BN);
        tl.expert = 0;
    }
    return tl;
}

// Whether a warpgroup's 128 x 128 output block of tile `tl` goes out through
// the staged boxes and TMA stores: a block with columns inside N and rows
// inside the tile's range, where the tensor map clips rows at M but a grouped
// tile may not write past its expert's segment.  The promote warps and the
// store issuer take the same decision from this one predicate.
__device__ __forceinline__ bool epi_uses_boxes(const GemmArgs &g, const Tile &tl, int64_t n_first)
{
    return g.c_tma && n_first < g.N && tl.m0 < tl.m_end && (tl.m0 + BM <= tl.m_end || tl.m_end == g.M);
}

// Grouped: per-expert tile counts ceil(n_e / 128) * num_n_blk, exclusive
// prefix over experts into shared memory.  Offsets are clamped into
// [0, M_total] and made nondecreasing, so malformed offsets cannot move any
// access out of bounds.
template <int S, int BSB, int SSF>
__device__ void build_tile_prefix(const GemmArgs &g, const SharedState<S, BSB, SSF> &ss)
{
    __shared__ int32_t chunk_sum[GEMM_THREADS];
    int32_t *pre = ss.tile_prefix();
    const int tid = threadIdx.x;
    const int per = (g.E + GEMM_THREADS - 1) / GEMM_THREADS;
    const int e0 = min(tid * per, g.E), e1 = min(e0 + per, g.E);
    int32_t sum = 0;
    for (int e = e0; e < e1; ++e) {
        const int64_t a = min(max((int64_t)g.offsets[e], (int64_t)0), g.M);
        const int64_t b = min(max((int64_t)g.offsets[e + 1], a), g.M);
        const int32_t c = (int32_t)((b - a + BM - 1) / BM) * g.num_n_blk;
        pre[e] = c;                                   // count, turned into a prefix below
        sum += c;
    }
    chunk_sum[tid] = sum;
    __syncthreads();
    if (tid == 0) {
        int32_t run = 0;
        for (int i = 0; i < GEMM_THREADS; ++i) {
            const int32_t c = chunk_sum[i];
            chunk_sum[i] = run;
            run += c;
        }
        pre[g.E] = run;
    }
    __syncthreads();
    int32_t run = chunk_sum[tid];
    for (int e = e0; e < e1; ++e) {
        const int32_t c = pre[e];
        pre[e] = run;
        run += c;
    }
    __syncthreads();
}

// acc[j] += P[j] * scale for 64 columns (32 column pairs), as packed f32x2
// FMAs: each lane is one correctly rounded fused multiply-add.
__device__ __forceinline__ void promote64(float2 *acc, const uint32_t (&p)[64], float scale)
{
    const float2 s2 = make_float2(scale, scale);
#pragma unroll
    for (int j = 0; j < 32; ++j)
        acc[j] = __ffma2_rn(make_float2(__uint_as_float(p[2 * j]), __uint_as_float(p[2 * j + 1])), s2,
                            acc[j]);
}

// acc[j] += P[j] * (sa * sB[j]) for 64 columns whose scales sB are 64 floats
// at shared address `sb`: per-column scales of the weight-gradient GEMM.  The
// scales are read in groups of 8 (two 16-byte loads issued together: the
// promote threads have no registers to spare), the scale pairs formed with
// packed multiplies, then packed FMAs.
__device__ __forceinline__ void promote64_cols(float2 *acc, const uint32_t (&p)[64], float sa, uint32_t sb)
{
    const float2 sa2 = make_float2(sa, sa);
#pragma unroll
    for (int grp = 0; grp < 8; ++grp) {
        float4 b[2];
#pragma unroll
        for (int i = 0; i < 2; ++i)
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(b[i].x), "=f"(b[i].y), "=f"(b[i].z), "=f"(b[i].w)
                         : "r"(sb + 16 * (2 * grp + i)));
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int c = 2 * grp + i;
            const float2 s0 = __fmul2_rn(sa2, make_float2(b[i].x, b[i].y));
            const float2 s1 = __fmul2_rn(sa2, make_float2(b[i].z, b[i].w));
            acc[2 * c] = __ffma2_rn(make_float2(__uint_as_float(p[4 * c]), __uint_as_float(p[4 * c + 1])), s0,
                                    acc[2 * c]);
            acc[2 * c + 1] = __ffma2_rn(make_float2(__uint_as_float(p[4 * c + 2]), __uint_as_float(p[4 * c + 3])),
                                        s1, acc[2 * c + 1]);
        }
    }
}

// Direct, masked stores of one thread's row segment (128 columns from n_first).
__device__ __forceinline__ void store_row_direct(const GemmArgs &g, const float2 *acc2, int64_t gm,
                                                 int64_t n_first)
{
    const bool full_cols = n_first + 128 <= g.N;
    if (g.c_fp32) {
        float *crow = reinterpret_cast<float *>(g.C) + gm * g.ldc + n_first;
        const bool vec = full_cols && ((reinterpret_cast<uintptr_t>(crow) & 15u) == 0);
        if (vec) {
#pragma unroll
            for (int j = 0; j < 64; j += 2)
                ptx::st_v4(crow + 2 * j, __float_as_uint(acc2[j].x), __float_as_uint(acc2[j].y),
                           __float_as_uint(acc2[j + 1].x), __float_as_uint(acc2[j + 1].y));
        } else {
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                if (n_first + 2 * j < g.N)
                    crow[2 * j] = acc2[j].x;
                if (n_first + 2 * j + 1 < g.N)
                    crow[2 * j + 1] = acc2[j].y;
            }
        }
    } else {
        uint16_t *crow = reinterpret_cast<uint16_t *>(g.C) + gm * g.ldc + n_first;
        const bool vec = full_cols && ((reinterpret_cast<uintptr_t>(crow) & 15u) == 0);
        if (vec) {
#pragma unroll
            for (int j = 0; j < 64; j += 4)
                ptx::st_v4(crow + 2 * j, ptx::cvt_bf16x2(acc2[j].x, acc2[j].y),
                           ptx::cvt_bf16x2(acc2[j + 1].x, acc2[j + 1].y),
                           ptx::cvt_bf16x2(acc2[j + 2].x, acc2[j + 2].y),
                           ptx::cvt_bf16x2(acc2[j + 3].x, acc2[j + 3].y));
        } else {
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const uint32_t pr = ptx::cvt_bf16x2(acc2[j].x, acc2[j].y);
                if (n_first + 2 * j < g.N)
                    crow[2 * j] = (uint16_t)(pr & 0xFFFFu);
                if (n_first + 2 * j + 1 < g.N)
                    crow[2 * j + 1] = (uint16_t)(pr >> 16);
            }
        }
    }
}

// QOUT: the epilogue writes C as E4M3 codes with one FP32 scale per 1x128
// row tile (the activation quantiser's rule applied to the BF16-rounded
// output, bit for bit) instead of BF16.  Dense only; N % 128 == 0 and a
// TMA-able code matrix are guaranteed by the host.
// TOK: the weight-gradient GEMM -- B carries one scale per row and 128-wide
// K-slice (sB [K/128][N]), like A, so each output column has its own B
// scale; dense, K-major B, BF16 or FP32 output.
// PT: per-tensor scaling, the contrast variant -- sA and sB are one scalar
// each, so there is nothing to promote per slice: the MMAs accumulate the
// whole K of a tile into one TMEM buffer (the tensor core's FP32
// accumulation), the promote warps read it once per tile and multiply by
// sA * sB; tile t uses buffer t & 1, so the next tile's MMAs overlap this
// tile's epilogue.  Dense, BF16 or FP32 output.
template <bool GROUPED, bool B_MN, bool PAIR, int STAGES, bool QOUT = false, bool TOK = false, bool PT = false>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const GemmArgs g)
{
    constexpr int BSB = PAIR ? B_STAGE_BYTES / 2 : B_STAGE_BYTES;   // pair: this CTA's half of B
    constexpr int SSF = TOK ? SCALE_SLOT_FLOATS_TOK : SCALE_SLOT_FLOATS;
    using L = Layout<STAGES, BSB, SSF>;
    extern __shared__ uint8_t smem_raw[];
    SharedState<STAGES, BSB, SSF> ss;
    {
        const uint32_t raw = ptx::smem_u32(smem_raw);
        const uint32_t aligned = (raw + 1023u) & ~1023u;
        ss.base = aligned;
        ss.gbase = smem_raw + (aligned - raw);
    }
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    ptx::grid_dep_launch();                          // the next kernel may start its own set-up

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(ss.full(s), 1);
            ptx::mbar_init(ss.empty(s), 1);
        }
        for (int p = 0; p < 2; ++p) {
            ptx::mbar_init(ss.pfull(p), 1);
            ptx::mbar_init(ss.pempty(p), PAIR ? 16 : 8);   // one arrive per promote warp (pair: of both CTAs)
        }
        ptx::mbar_init(ss.drain(), 1);
        for (int j = 0; j < SCALE_SLOTS; ++j) {
            ptx::mbar_init(ss.sready(j), 32);          // every lane of the loader warp
            ptx::mbar_init(ss.sfree(j), 256);          // every promote thread
        }
        for (int wg = 0; wg < 2; ++wg) {
            ptx::mbar_init(ss.epi_free(wg), 1);        // the store issuer (warp 3)
            ptx::mbar_init(ss.epi_full(wg), 4);        // one arrive per warp
        }
        *ss.abort_flag() = 0u;
        ptx::fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        if (g.c_tma)
            ptx::prefetch_tmap(&tmC);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            ptx::tmem_alloc_pair(ss.base + L::MISC, TMEM_COLS);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ss.base + L::MISC, TMEM_COLS);
            ptx::tmem_relinquish();
        }
    }
    // Everything above touches only this CTA's shared and tensor memory; the
    // first global reads (expert offsets, operands, scales) wait for the
    // kernels this one depends on.
    ptx::grid_dep_wait();
    if constexpr (GROUPED)
        build_tile_prefix(g, ss);                    // ends with __syncthreads
    ptx::tc_fence_before();
    if constexpr (PAIR)
        ptx::cluster_sync();                         // the peer's barriers exist before it is signalled
    else
        __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *ss.tmem_slot();
    // persistent schedule: CTA (pair: cluster) i takes work units i, i + count, ...
    const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
    const int64_t t_first = PAIR ? (int64_t)(blockIdx.x >> 1) : (int64_t)blockIdx.x;
    const int64_t t_stride = PAIR ? (int64_t)(gridDim.x >> 1) : (int64_t)gridDim.x;
    const int64_t ntiles = total_tiles<GROUPED>(g, ss);

    // Register split, one setmaxnreg per warpgroup (the same instruction for
    // its four warps): 128 x 56 + 256 x 224 = 64512 = the launch's 384 x 168.
    if (warp < 4) {
        ptx::setmaxnreg_dec<56>();
        if (warp == 0 && lane == 0) {
            // -------------------------------------------- TMA producer
            // L2 policy: A row blocks are re-read by the tiles of later
            // N-blocks (keep them); dense B column blocks are shared by the
            // concurrently running M-tiles (default policy); an expert's
            // weight slice is read once more by each later M-block of the
            // expert, which runs on a neighbouring CTA a little later (keep
            // it), and is not needed again after its last M-block (evict
            // first).
            const uint64_t keep = ptx::policy_evict_last();
            const uint64_t stream = ptx::policy_evict_first();
            // No separate L2 prefetch of the expert weights: a bulk prefetch
            // of each slice's weight box ahead of its load made the routed-
            // expert GEMM slower at every distance tried (0, 2 and 4 slices
            // ahead, or the next tile's first slices at a tile's end).
            uint32_t it = 0;
            bool ok = true;
            for (int64_t t = t_first; ok && t < ntiles; t += t_stride) {
                const Tile tl = tile_at<GROUPED, PAIR>(g, ss, t, rank);
                for (int kb = 0; kb < g.KB; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!wait_bounded(ss, g, ss.empty(s), ph ^ 1u)) { ok = false; break; }
                    const uint32_t fb = ss.full(s);
                    const uint32_t sa = ss.a_stage(s);
                    const uint32_t sb = ss.b_stage(s);
                    if constexpr (PAIR) {
                        // this CTA's A rows and its half of the B block; both
                        // CTAs' bytes complete on the leader's `full` barrier
                        const uint32_t fb0 = ptx::mapa_shared(fb, 0);
                        if (rank == 0)
                            ptx::mbar_arrive_expect_tx(fb, 2 * (A_STAGE_BYTES + BSB));
                        ptx::tma_load_2d_pair_hint(sa, &tmA, fb0, kb * BK, (int32_t)tl.m0, keep);
                        if constexpr (B_MN)
                            ptx::tma_load_2d_pair(sb, &tmB, fb0, tl.n0 + 128 * (int32_t)rank, kb * BK);
                        else
                            ptx::tma_load_2d_pair(sb, &tmB, fb0, kb * BK, tl.n0 + 128 * (int32_t)rank);
                        continue;
                    }
                    ptx::mbar_arrive_expect_tx(fb, A_STAGE_BYTES + B_STAGE_BYTES);
                    ptx::tma_load_2d_hint(sa, &tmA, fb, kb * BK, (int32_t)tl.m0, keep);
                    if constexpr (GROUPED) {
                        ptx::tma_load_3d_hint(sb, &tmB, fb, kb * BK, tl.n0, tl.expert,
                                              tl.m0 + BM < tl.m_end ? keep : stream);
                    } else if constexpr (B_MN) {
                        ptx::tma_load_2d(sb, &tmB, fb, tl.n0, kb * BK);
                        ptx::tma_load_2d(sb + B_STAGE_BYTES / 2, &tmB, fb, tl.n0 + 128, kb * BK);
                    } else {
                        ptx::tma_load_2d(sb, &tmB, fb, kb * BK, tl.n0);
                    }
                }
            }
            // Drain: every copy this thread issued must land before exit.  (A
            // pair's second CTA completes its bytes on the leader's barriers,
            // which the leader's MMA waits on before the final cluster sync.)
            const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
            if (rank == 0)
                for (uint32_t j = first; j < it; ++j)
                    wait_drain(ss.full(j % STAGES), (j / STAGES) & 1u);
        } else if (warp == 1 && lane == 0 && rank == 0) {
            // -------------------------------------------- MMA issuer (pair: leader CTA, M = 256)
            constexpr uint32_t idesc = make_idesc(PAIR ? 2 * BM : BM, BN, B_MN);
            uint32_t it = 0, pit = 0;           // pit: uses of the two TMEM buffers (per slice; PT: per tile)
            bool ok = true;
            for (int64_t t = t_first; ok && t < ntiles; t += t_stride) {
                if constexpr (PT) {
                    // the tile's buffer must have been read out by the previous tile's epilogue
                    if (!wait_bounded(ss, g, ss.pempty(pit & 1), ((pit >> 1) & 1u) ^ 1u)) { ok = false; break; }
                }
                for (int kb = 0; kb < g.KB; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    const int p = pit & 1;
                    const uint32_t pph = (pit >> 1) & 1u;
                    if (!wait_bounded(ss, g, ss.full(s), ph)) { ok = false; break; }
                    if (!PT && !wait_bounded(ss, g, ss.pempty(p), pph ^ 1u)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t d = tmem_base + (uint32_t)(p * BN);
                    const uint32_t sa = ss.a_stage(s);
                    const uint32_t sb = ss.b_stage(s);
#pragma unroll
                    for (int kk = 0; kk < BK / 32; ++kk) {
                        const uint64_t ad = make_sdesc_sw128(sa + kk * 32, 16, 1024);
                        uint64_t bd;
                        if constexpr (B_MN)
                            bd = make_sdesc_sw128(sb + kk * 32 * 128, B_STAGE_BYTES / 2, 1024);
                        else
                            bd = make_sdesc_sw128(sb + kk * 32, 16, 1024);
                        // a fresh partial per slice; PT: one accumulation over all of K
                        const uint32_t acc = (kk > 0 || (PT && kb > 0)) ? 1u : 0u;
                        if constexpr (PAIR)
                            ptx::mma_f8f6f4_pair(d, ad, bd, idesc, acc);
                        else
                            ptx::mma_f8f6f4(d, ad, bd, idesc, acc);
                    }
                    const bool publish = !PT || kb == g.KB - 1;
                    if constexpr (PAIR) {
                        // stage free and partial ready, in both CTAs
                        ptx::mma_commit_pair_mc(ss.empty(s), 0x3);
                        if (publish)
                            ptx::mma_commit_pair_mc(ss.pfull(p), 0x3);
                    } else {
                        ptx::mma_commit(ss.empty(s));
                        if (publish)
                            ptx::mma_commit(ss.pfull(p));
                    }
                    if constexpr (!PT)
                        ++pit;
                }
                if constexpr (PT)
                    ++pit;
            }
            // Drain: all MMAs this thread issued complete before TMEM is freed.
            if constexpr (PAIR)
                ptx::mma_commit_pair(ss.drain());
            else
                ptx::mma_commit(ss.drain());
            wait_drain(ss.drain(), 0);
        }
        if (warp == 2 && !PT) {
            // -------------------------------------------- scale loader
            // Stages each slice's 128 row scales sA[kb][m0 .. m0+127] and the
            // two column-block scales of the tile into a SCALE_SLOTS-deep
            // shared ring (cp.async, SCALE_LOOKAHEAD slices of copies in
            // flight), so that the promote warps never wait on global memory.
            uint32_t sit = 0, done = 0;
            bool ok = true;
            auto publish = [&](uint32_t j) {             // slice j's copies have landed
                ptx::mbar_arrive(ss.sready((int)(j % SCALE_SLOTS)));
            };
            for (int64_t t = t_first; ok && t < ntiles; t += t_stride) {
                const Tile tl = tile_at<GROUPED, PAIR>(g, ss, t, rank);
                for (int kb = 0; kb < g.KB; ++kb, ++sit) {
                    const int slot = (int)(sit % SCALE_SLOTS);
                    if (!wait_bounded(ss, g, ss.sfree(slot), ((sit / SCALE_SLOTS) & 1u) ^ 1u)) { ok = false; break; }
                    const uint32_t dst = ss.scale_slot(slot);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = lane + 32 * i;
                        const int64_t gm = tl.m0 + r;
                        const bool in = gm < tl.m_end;
                        ptx::cp_async_4(dst + 4 * r, in ? (const void *)(g.sA + (int64_t)kb * g.M + gm) : (const void *)g.sA,
                                        in ? 4u : 0u);
                    }
                    if constexpr (TOK) {
                        // the tile's 256 column scales sB[kb][n0 .. n0+255]
                        const float *src0 = g.sB + (int64_t)kb * g.N + tl.n0;
#pragma unroll 1
                        for (int i = 0; i < 8; ++i) {
                            const int c = lane + 32 * i;
                            const int64_t n = (int64_t)tl.n0 + c;
                            const bool in = n < g.N;
                            ptx::cp_async_4(dst + 4 * (128 + c), in ? (const void *)(src0 + c) : (const void *)g.sB,
                                            in ? 4u : 0u);
                        }
                    } else if (lane < 2) {
                        const int nblk = (tl.n0 >> 7) + lane;
                        const bool in = nblk < g.NB128;
                        const float *src;
                        if constexpr (GROUPED)
                            src = g.sB + ((int64_t)tl.expert * g.NB128 + nblk) * g.KB + kb;
                        else if constexpr (B_MN)
                            src = g.sB + (int64_t)kb * g.NB128 + nblk;
                        else
                            src = g.sB + (int64_t)nblk * g.KB + kb;
                        ptx::cp_async_4(dst + 4 * (128 + lane), in ? (const void *)src : (const void *)g.sB, in ? 4u : 0u);
                    }
                    ptx::cp_async_commit();
                    if (sit >= (uint32_t)SCALE_LOOKAHEAD) {
                        ptx::cp_async_wait<SCALE_LOOKAHEAD>();
                        publish(done++);
                    }
                }
            }
            ptx::cp_async_wait<0>();
            while (done < sit)
                publish(done++);
        }
        if (warp == 3 && lane == 0 && g.c_tma) {
            // -------------------------------------------- output store issuer
            // A warpgroup signals epi_full once its four warps have staged
            // their rows; this thread issues the tile's TMA stores and
            // returns the boxes (epi_free) when the stores have read them,
            // so no promote warp waits on another warp's epilogue.
            const uint64_t c_policy = ptx::policy_evict_first();   // C is written once, never re-read
            ptx::mbar_arrive(ss.epi_free(0));                      // the boxes start free
            ptx::mbar_arrive(ss.epi_free(1));
            uint32_t eit[2] = {0u, 0u};
            bool ok = true;
            for (int64_t t = t_first; ok && t < ntiles; t += t_stride) {
                const Tile tl = tile_at<GROUPED, PAIR>(g, ss, t, rank);
                for (int wg = 0; wg < 2; ++wg) {
                    const int64_t n_first = tl.n0 + wg * 128;
                    if (!epi_uses_boxes(g, tl, n_first))
                        continue;
                    if (!wait_bounded(ss, g, ss.epi_full(wg), eit[wg]++ & 1u)) { ok = false; break; }
                    ptx::tma_store_2d_hint(&tmC, ss.epi_box(wg, 0), (int32_t)n_first, (int32_t)tl.m0, c_policy);
                    if (!QOUT && n_first + 64 < g.N)       // second 64-column BF16 box exists
                        ptx::tma_store_2d_hint(&tmC, ss.epi_box(wg, 1), (int32_t)(n_first + 64), (int32_t)tl.m0,
                                               c_policy);
                    ptx::bulk_commit();
                    ptx::bulk_wait_read_all();
                    ptx::mbar_arrive(ss.epi_free(wg));
                }
            }
            ptx::bulk_wait_all();                        // every store has completed before exit
        }
        __syncwarp();
    } else {
        ptx::setmaxnreg_inc<224>();
        // ------------------------------------------------ promote + epilogue
        const int wg = (warp - 4) >> 2;              // column half
        const int quarter = warp & 3;                // TMEM lane quarter
        const int row = quarter * 32 + lane;         // tile row owned by this thread
        const int col_half = wg * 128;
        uint32_t pit = 0, eit = 0;
        bool ok = true;
        // PT: the two per-tensor scales, one product for every output
        const float pt_scale = PT ? g.sA[0] * g.sB[0] : 0.0f;
        for (int64_t t = t_first; ok && t < ntiles; t += t_stride) {
            const Tile tl = tile_at<GROUPED, PAIR>(g, ss, t, rank);
            const int64_t gm = tl.m0 + row;
            const bool row_ok = gm < tl.m_end;
            // grouped: a warp whose 32 rows all lie past the expert's segment
            // (the padding of a partial M-block) skips its TMEM reads and FMAs
            const bool warp_live = !GROUPED || tl.m0 + quarter * 32 < tl.m_end;
            float2 acc2[64];
            if constexpr (PT) {
                // the tile's whole-K accumulator, read once and scaled
                const int p = pit & 1;
                const uint32_t pph = (pit >> 1) & 1u;
                ++pit;
                if (!warp_wait(ss, g, ss.pfull(p), pph)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(p * BN + col_half);
                const float2 s2 = make_float2(pt_scale, pt_scale);
                uint32_t r[64];
                ptx::tmem_ld_32x32b_x64(taddr, r);
                ptx::tmem_ld_wait(r);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    acc2[j] = __fmul2_rn(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), s2);
                ptx::tmem_ld_32x32b_x64(taddr + 64, r);
                ptx::tmem_ld_wait(r);
                ptx::tc_fence_before();
                __syncwarp();                            // the warp's accumulator is in registers
                if constexpr (PAIR)
                    ptx::mbar_arrive_cluster_if(ptx::mapa_shared(ss.pempty(p), 0), lane == 0);
                else
                    ptx::mbar_arrive_cluster_if(ss.pempty(p), lane == 0);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    acc2[32 + j] =
                        __fmul2_rn(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), s2);
            } else {
#pragma unroll
            for (int j = 0; j < 64; ++j)
                acc2[j] = make_float2(0.0f, 0.0f);
            }
            for (int kb = 0; !PT && kb < g.KB; ++kb, ++pit) {
                // this slice's scales from the shared ring (staged by warp 2)
                const int slot = (int)(pit % SCALE_SLOTS);
                if (!warp_wait(ss, g, ss.sready(slot), (pit / SCALE_SLOTS) & 1u)) { ok = false; break; }
                float sa, sb = 1.0f;
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sa) : "r"(ss.scale_slot(slot) + 4 * row));
                if constexpr (!TOK) {
                    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sb) : "r"(ss.scale_slot(slot) + 4 * (128 + wg)));
                    ptx::mbar_arrive(ss.sfree(slot));
                }
                const float scale = sa * sb;
                // TOK: this warpgroup's 128 column scales, read during the promotion
                const uint32_t col_scales = ss.scale_slot(slot) + 4 * (128 + col_half);
                const int p = pit & 1;
                const uint32_t pph = (pit >> 1) & 1u;
                if (!warp_wait(ss, g, ss.pfull(p), pph)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                       (uint32_t)(p * BN + col_half);
                // two 64-column TMEM round trips; the buffer is released as
                // soon as the second one has landed in registers
                uint32_t r[64];
                if (warp_live) {
                    ptx::tmem_ld_32x32b_x64(taddr, r);
                    ptx::tmem_ld_wait(r);
                    if constexpr (TOK)
                        promote64_cols(acc2, r, sa, col_scales);
                    else
                        promote64(acc2, r, scale);
                    ptx::tmem_ld_32x32b_x64(taddr + 64, r);
                    ptx::tmem_ld_wait(r);
                }
                ptx::tc_fence_before();
                __syncwarp();                            // the warp's partial is in registers
                if constexpr (PAIR)
                    ptx::mbar_arrive_cluster_if(ptx::mapa_shared(ss.pempty(p), 0), lane == 0);   // the leader's MMA
                else
                    ptx::mbar_arrive_cluster_if(ss.pempty(p), lane == 0);
                if constexpr (TOK) {
                    promote64_cols(acc2 + 32, r, sa, col_scales + 4 * 64);
                    ptx::mbar_arrive(ss.sfree(slot));    // the column scales have been read
                } else if (warp_live) {
                    promote64(acc2 + 32, r, scale);
                }
            }
            if (!ok)
                break;
            // ---- epilogue: the warpgroup's rows [m0, m0 + 128), columns [n0 + col_half, +128)
            const int64_t n_first = tl.n0 + col_half;
            if (n_first >= g.N || tl.m0 >= tl.m_end)
                continue;                                // uniform over the warpgroup
            if (epi_uses_boxes(g, tl, n_first)) {
                // Stage both 64-column halves as 128-row, 128-byte-swizzled
                // boxes shared by the warpgroup's four warps; warp 3 issues
                // the TMA stores.  The hand-offs are mbarriers with bounded
                // waits, so an aborting warp cannot strand the others.
                const uint32_t ph = eit & 1u;
                ++eit;
                if constexpr (QOUT) {
                    // The thread's 128 columns are exactly one 1x128 tile of
                    // its row: round to BF16, take the amax of the magnitude
                    // bits, form the divisor and encode, as the quantiser does.
                    uint32_t w[64];
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        w[j] = ptx::cvt_bf16x2(acc2[j].x, acc2[j].y);
                    uint32_t mx = 0;
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        mx = ptx::max_u16x2(mx, w[j] & 0x7FFF7FFFu);
                    const Divisor d = make_divisor(max(mx & 0xFFFFu, mx >> 16));
                    if (row_ok)
                        g.sC[(n_first >> 7) * g.M + gm] = d.s;
                    if (!warp_wait(ss, g, ss.epi_free(wg), ph)) { ok = false; break; }
                    const uint32_t buf = ss.epi_box(wg, 0) + (uint32_t)row * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint2 lo = quant_8(make_uint4(w[8 * c], w[8 * c + 1], w[8 * c + 2], w[8 * c + 3]), d);
                        const uint2 hi = quant_8(make_uint4(w[8 * c + 4], w[8 * c + 5], w[8 * c + 6], w[8 * c + 7]), d);
                        ptx::st_shared_v4(buf + ((c ^ (lane & 7)) << 4), lo.x, lo.y, hi.x, hi.y);
                    }
                } else {
                    if (!warp_wait(ss, g, ss.epi_free(wg), ph)) { ok = false; break; }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t buf = ss.epi_box(wg, h) + (uint32_t)row * 128;
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const float2 *v = acc2 + h * 32 + c * 4;
                            ptx::st_shared_v4(buf + ((c ^ (lane & 7)) << 4),
                                              ptx::cvt_bf16x2(v[0].x, v[0].y), ptx::cvt_bf16x2(v[1].x, v[1].y),
                                              ptx::cvt_bf16x2(v[2].x, v[2].y), ptx::cvt_bf16x2(v[3].x, v[3].y));
                        }
                    }
                }
                ptx::fence_proxy_async_smem();           // the boxes are visible to the TMA stores
                __syncwarp();
                ptx::mbar_arrive_cluster_if(ss.epi_full(wg), lane == 0);
            } else if (row_ok) {
                store_row_direct(g, acc2, gm, n_first);
            }
        }
        __syncwarp();
    }

    ptx::tc_fence_before();
    if constexpr (PAIR) {
        // After an abort, the second CTA's last copies complete on the
        // leader's barriers, which no one waits for any more: give any copy
        // still in flight time to land before either CTA of the pair exits.
        __syncthreads();
        if (*ss.abort_flag()) {
            const uint64_t t0 = ptx::globaltimer_ns();
            while (ptx::globaltimer_ns() - t0 < ABORT_GRACE_NS) {
            }
        }
        ptx::cluster_sync();                         // the pair's MMAs, copies and signals are done
    } else {
        __syncthreads();
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        if constexpr (PAIR)
            ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            ptx::tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

} // namespace fp8bs
