// quant.cuh -- fine-grained FP8 quantisers (1x128 activation tiles, 128x128
// weight blocks).  ["DeepSeek-V3 training walkthrough", section 二(四), and
// "DeepSeek-V3 Technical Report digest", section 3: activations per 1x128
// tile, weights per 128x128 block.]
//
// Both kernels are HBM-bound streams: 2 bytes read + 1 byte written per
// element plus 4 bytes per scale.  They are persistent (three 256-thread CTAs
// per SM) and stream 128 x 128 BF16 units (32 KiB: 128 rows of one 128-column
// K-block) through a QSTAGES-deep ring of TMA loads in shared memory, so each
// SM keeps several units in flight while it encodes another.  A unit is one
// 128x128 weight block, or 128 activation rows x one 1x128 tile column.
// An amax is an integer max over the BF16 magnitude bits (monotone for
// finite values): a 1x128 tile's over the four lanes that hold it (two
// xor-shuffles), a weight block's over its warps and the CTA.  scale =
// amax / 448 is one IEEE division; x / scale is formed exactly (see Divisor
// below) and encoded with the hardware RNE-satfinite E4M3 conversion; codes
// are stored 8 bytes per lane in runs of 32 or 128 contiguous bytes.
#pragma once
#include "common.cuh"

namespace fp8bs {

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// BF16 magnitude bits of 8 values (16 bytes): max over the masked 16-bit
// lanes, then over the two halves.
__device__ __forceinline__ uint32_t absmax_bits8(const uint4 &v)
{
    const uint32_t m = 0x7FFF7FFFu;
    const uint32_t a = ptx::max_u16x2(ptx::max_u16x2(v.x & m, v.y & m), ptx::max_u16x2(v.z & m, v.w & m));
    return max(a & 0xFFFFu, a >> 16);
}

// Per-group divisor.  The quotient fp32(x / s) is formed with Markstein's
// correction step (P. Markstein, IBM J. Res. Dev. 34(1), 1990): with the
// correctly rounded reciprocal r = RN(1/s),
//     q0 = RN(x * r),  rem = fma(-q0, s, x),  q = copysign(fma(rem, r, q0), x),
// which an exhaustive check over every BF16 amax >= 2^-90 and every BF16
// |x| <= amax shows to equal IEEE division bit for bit (up to the sign of
// zero-encoding quotients below 2^-11).  The copysign is applied to the
// E4M3 code (x's sign bit OR-ed in), which gives the same byte.  Groups with a smaller amax use
// IEEE division; an all-zero group (s == 0) encodes x itself (a signed zero).
// Two elements are processed at once with packed f32x2 arithmetic (each lane
// rounds exactly as the scalar operation).
struct Divisor {
    float s, r;
    int mode;           // 0: s == 0, 1: IEEE division, 2: reciprocal + correction
};

__device__ __forceinline__ int divisor_mode(uint32_t amax_bits)
{
    return amax_bits == 0 ? 0 : (amax_bits >= 0x1280u ? 2 : 1);   // 0x1280 = 2^-90 in BF16
}

__device__ __forceinline__ Divisor make_divisor(uint32_t amax_bits)
{
    Divisor d;
    const float amax = __uint_as_float(amax_bits << 16);
    d.s = __fdiv_rn(amax, 448.0f);
    d.mode = divisor_mode(amax_bits);
    d.r = d.mode == 2 ? __frcp_rn(d.s) : 0.0f;
    return d;
}

__device__ __forceinline__ float quotient_slow(float x, const Divisor &d)
{
    return d.mode == 1 ? __fdiv_rn(x, d.s) : x;
}

// E4M3 codes of the 8 BF16 values in v for a divisor of mode 2
// (reciprocal + correction), as 8 bytes (element 0 lowest).
__device__ __forceinline__ uint2 quant_8_recip(const uint4 &v, const Divisor &d)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t c[4];
    {
        const float2 r2 = make_float2(d.r, d.r);
        const float2 ns2 = make_float2(-d.s, -d.s);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 x2 = make_float2(bf16lo(w[k]), bf16hi(w[k]));
            const float2 q0 = __fmul2_rn(x2, r2);
            const float2 rem = __ffma2_rn(q0, ns2, x2);             // x - q0 * s, exact
            const float2 q = __ffma2_rn(rem, r2, q0);
            c[k] = ptx::cvt_e4m3x2(q.x, q.y);
        }
        // The code must carry x's sign.  A nonzero quotient has it already,
        // and a zero quotient of a positive x is +0.  Only a negative x can
        // end at +0: x = -0, where -0 + +0 rounds to +0, or an underflow.
        // OR-ing x's sign bits (bit 7 of each BF16's high byte) into the
        // codes therefore gives every code the sign of its x.
        const uint32_t sgn0 = __byte_perm(w[0], w[1], 0x7531) & 0x80808080u;
        const uint32_t sgn1 = __byte_perm(w[2], w[3], 0x7531) & 0x80808080u;
        return make_uint2(__byte_perm(c[0], c[1], 0x5410) | sgn0, __byte_perm(c[2], c[3], 0x5410) | sgn1);
    }
}

// E4M3 codes of the 8 BF16 values in v, as 8 bytes (element 0 lowest).
__device__ __forceinline__ uint2 quant_8(const uint4 &v, const Divisor &d)
{
    if (d.mode == 2)
        return quant_8_recip(v, d);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t c[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        c[k] = ptx::cvt_e4m3x2(quotient_slow(bf16lo(w[k]), d), quotient_slow(bf16hi(w[k]), d));
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

constexpr int QSTAGES = 2;
constexpr int QUNIT_BYTES = 128 * 128 * 2;                    // 32 KiB of BF16
constexpr int QUANT_THREADS = 256;
constexpr int QSMEM_BAR = QSTAGES * QUNIT_BYTES;                // full barriers
constexpr int QSMEM_ABORT = QSMEM_BAR + 8 * QSTAGES;
constexpr int QSMEM_RED = QSMEM_ABORT + 8;                       // 2 buffers x 256 words
constexpr int QSMEM_END = QSMEM_RED + 2 * 256 * 4;
constexpr int quant_smem_bytes() { return 1024 + QSMEM_END; }

struct QRing {
    uint32_t base;
    uint8_t *gbase;
    uint64_t wait_ns;   // time limit of the ring's waits
    __device__ uint32_t stage(int s) const { return base + s * QUNIT_BYTES; }
    __device__ uint32_t full(int s) const { return base + QSMEM_BAR + 8 * s; }
    __device__ volatile uint32_t *abort() const
    {
        return reinterpret_cast<volatile uint32_t *>(gbase + QSMEM_ABORT);
    }
    __device__ uint32_t *red_u(int b) const
    {
        return reinterpret_cast<uint32_t *>(gbase + QSMEM_RED) + 256 * b;
    }
};

__device__ __forceinline__ QRing qring_setup(uint64_t wait_ns)
{
    extern __shared__ uint8_t smem_raw[];
    ptx::grid_dep_launch();                      // the next kernel may start its own set-up
    QRing r;
    r.wait_ns = wait_ns;
    const uint32_t raw = ptx::smem_u32(smem_raw);
    r.base = (raw + 1023u) & ~1023u;
    r.gbase = smem_raw + (r.base - raw);
    if (threadIdx.x == 0) {
        for (int s = 0; s < QSTAGES; ++s)
            ptx::mbar_init(r.full(s), 1);
        *r.abort() = 0u;
        ptx::fence_mbarrier_init();
    }
    __syncthreads();
    ptx::grid_dep_wait();                        // global memory only after the kernels this one depends on
    return r;
}

// Unit j of this CTA (j-th in its strided list) -> (row block, column block).
__device__ __forceinline__ void qunit(int64_t j, int64_t cols_blocks, int64_t &rb, int64_t &cb)
{
    const int64_t u = (int64_t)blockIdx.x + j * gridDim.x;
    rb = u / cols_blocks;
    cb = u - rb * cols_blocks;
}

__device__ __forceinline__ void qissue(const QRing &r, const CUtensorMap *tm, int64_t j,
                                       int64_t cols_blocks)
{
    int64_t rb, cb;
    qunit(j, cols_blocks, rb, cb);
    const int s = (int)(j % QSTAGES);
    ptx::fence_proxy_async_smem();             // earlier generic reads of the stage come first
    ptx::mbar_arrive_expect_tx(r.full(s), QUNIT_BYTES);
    ptx::tma_load_2d(r.stage(s), tm, r.full(s), (int32_t)(cb * 128), (int32_t)(rb * 128));
}

// An activation unit is staged as two 64-column boxes with the 128-byte
// swizzle (16-byte chunk c of row r of a half at r * 128 + ((c ^ (r & 7)) * 16)),
// so that the four lanes reading one row and the eight rows a warp reads at
// once fall on different banks.
__device__ __forceinline__ void qissue_act_at(const QRing &r, const CUtensorMap *tm, int64_t j, int64_t rb,
                                              int64_t cb)
{
    const int s = (int)(j % QSTAGES);
    ptx::fence_proxy_async_smem();             // earlier generic reads of the stage come first
    ptx::mbar_arrive_expect_tx(r.full(s), QUNIT_BYTES);
    ptx::tma_load_2d(r.stage(s), tm, r.full(s), (int32_t)(cb * 128), (int32_t)(rb * 128));
    ptx::tma_load_2d(r.stage(s) + QUNIT_BYTES / 2, tm, r.full(s), (int32_t)(cb * 128 + 64), (int32_t)(rb * 128));
}

__device__ __forceinline__ void qissue_act(const QRing &r, const CUtensorMap *tm, int64_t j, int64_t cols_blocks)
{
    int64_t rb, cb;
    qunit(j, cols_blocks, rb, cb);
    qissue_act_at(r, tm, j, rb, cb);
}

// Waits for unit j's stage; every thread of the CTA agrees on the outcome.
__device__ __forceinline__ bool qwait(const QRing &r, int64_t j)
{
    const int s = (int)(j % QSTAGES);
    wait_bounded(r.full(s), (uint32_t)((j / QSTAGES) & 1), r.abort(), r.wait_ns);
    __syncthreads();
    return *r.abort() == 0u;
}

// After an abort: the copies this CTA issued but never consumed must land
// before it exits.
__device__ __forceinline__ void qdrain(const QRing &r, int64_t consumed, int64_t issued)
{
    if (threadIdx.x == 0)
        for (int64_t j = consumed; j < issued; ++j)
            wait_drain(r.full((int)(j % QSTAGES)), (uint32_t)((j / QSTAGES) & 1));
}

// Activation quantiser.  Unit (mb, kb): rows [128 mb, +128) of tile column kb,
// staged swizzled (qissue_act).  A 1x128 tile is held by four adjacent lanes:
// lane quarter g (lane & 3) takes the 8-column chunks g, g + 4, g + 8, g + 12
// of the row, so the four lanes' codes of each step form one 32-byte run.
// Warp w owns rows [16 w, 16 w + 16), eight at a time (lane >> 2 within the
// eight).  The row's amax takes two xor-shuffles within the four lanes; each
// of them forms the row's divisor itself, and lane quarter 0 stores the
// scale (eight consecutive rows: one 32-byte run).  `issue_next` runs once
// the staged unit has been read (the stage is free again) and queues the
// CTA's next copy.
template <class Next>
__device__ __forceinline__ void act_unit(const QRing &r, int64_t j, int64_t mb, int64_t kb, int64_t M,
                                         uint8_t *__restrict__ q, int64_t ldq, float *__restrict__ sA,
                                         Next &&issue_next)
{
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int g = lane & 3;
    const int rsub = lane >> 2;
    const uint32_t st = r.stage((int)(j % QSTAGES));
    uint4 v[2][4];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int row = 16 * (tid >> 5) + 8 * p + rsub;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int chunk = g + 4 * c;                                  // 16-byte chunk of the 256-byte row
            const uint32_t a = st + (uint32_t)((chunk >> 3) * (QUNIT_BYTES / 2) + row * 128 +
                                               (((chunk & 7) ^ (row & 7)) << 4));
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v[p][c].x), "=r"(v[p][c].y), "=r"(v[p][c].z), "=r"(v[p][c].w) : "r"(a));
        }
    }
    __syncthreads();                                   // the stage is free again
    issue_next();
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        uint32_t a = max(max(absmax_bits8(v[p][0]), absmax_bits8(v[p][1])),
                         max(absmax_bits8(v[p][2]), absmax_bits8(v[p][3])));
        a = max(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = max(a, __shfl_xor_sync(0xffffffffu, a, 2));
        const Divisor d = make_divisor(a);
        const int64_t gm = mb * 128 + 16 * (tid >> 5) + 8 * p + rsub;
        if (gm < M) {
            if (g == 0)
                sA[kb * M + gm] = d.s;
            uint8_t *qrow = q + gm * ldq + kb * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint2 codes = quant_8(v[p][c], d);
                ptx::st_v2(qrow + (g + 4 * c) * 8, codes.x, codes.y);
            }
        }
    }
}

// Weight quantiser.  Unit (rb, cb): one 128x128 block.  Thread t owns the
// 16-byte column chunk (t & 15) of rows (t >> 4) + 16 i, i = 0..7: 64 values
// held in registers between the amax and the encode passes.
template <class Next>
__device__ __forceinline__ void w_unit(const QRing &r, int64_t j, int64_t rb, int64_t cb, int64_t R, int64_t CB,
                                       uint8_t *__restrict__ q, int64_t ldq, float *__restrict__ sW,
                                       Next &&issue_next)
{
    const int tid = threadIdx.x;
    const int chunk = tid & 15;
    const int r0 = tid >> 4;
    const uint32_t st = r.stage((int)(j % QSTAGES));
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t a = st + (uint32_t)((r0 + 16 * i) * 256 + chunk * 16);
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v[i].x), "=r"(v[i].y), "=r"(v[i].z), "=r"(v[i].w) : "r"(a));
    }
    uint32_t a = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        a = max(a, absmax_bits8(v[i]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
    uint32_t *wmax = r.red_u((int)(j & 1));
    if ((tid & 31) == 0)
        wmax[tid >> 5] = a;
    __syncthreads();                                   // stage read, warp maxima written
    issue_next();
    a = wmax[0];
#pragma unroll
    for (int i = 1; i < 8; ++i)
        a = max(a, wmax[i]);
    const Divisor d = make_divisor(a);
    const int64_t col = cb * 128 + chunk * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t row = rb * 128 + r0 + 16 * i;
        if (row < R) {
            const uint2 c = quant_8(v[i], d);
            ptx::st_v2(q + row * ldq + col, c.x, c.y);
        }
    }
    if (tid == 0)
        sW[rb * CB + cb] = d.s;
}

__global__ void __launch_bounds__(QUANT_THREADS, 3) quant_act_1x128_kernel(
    const __grid_constant__ CUtensorMap tmX, int64_t M, int64_t KB, uint8_t *__restrict__ q,
    int64_t ldq, float *__restrict__ sA, int64_t units, uint64_t wait_ns)
{
    const QRing r = qring_setup(wait_ns);
    const int tid = threadIdx.x;
    const int64_t mine = (int64_t)blockIdx.x < units ? (units - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    int64_t issued = 0;
    if (tid == 0)
        for (; issued < mine && issued < QSTAGES; ++issued)
            qissue_act(r, &tmX, issued, KB);
    int64_t j = 0;
    for (; j < mine; ++j) {
        if (!qwait(r, j))
            break;
        int64_t mb, kb;
        qunit(j, KB, mb, kb);
        act_unit(r, j, mb, kb, M, q, ldq, sA, [&] {
            if (tid == 0 && issued < mine && issued < j + 1 + QSTAGES) {
                qissue_act(r, &tmX, issued, KB);
                ++issued;
            }
        });
    }
    qdrain(r, j, issued);
}

__global__ void __launch_bounds__(QUANT_THREADS, 3) quant_w_128x128_kernel(
    const __grid_constant__ CUtensorMap tmW, int64_t R, int64_t CB, uint8_t *__restrict__ q,
    int64_t ldq, float *__restrict__ sW, int64_t units, uint64_t wait_ns)
{
    const QRing r = qring_setup(wait_ns);
    const int tid = threadIdx.x;
    const int64_t mine = (int64_t)blockIdx.x < units ? (units - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    int64_t issued = 0;
    if (tid == 0)
        for (; issued < mine && issued < QSTAGES; ++issued)
            qissue(r, &tmW, issued, CB);
    int64_t j = 0;
    for (; j < mine; ++j) {
        if (!qwait(r, j))
            break;
        int64_t rb, cb;
        qunit(j, CB, rb, cb);
        w_unit(r, j, rb, cb, R, CB, q, ldq, sW, [&] {
            if (tid == 0 && issued < mine && issued < j + 1 + QSTAGES) {
                qissue(r, &tmW, issued, CB);
                ++issued;
            }
        });
    }
    qdrain(r, j, issued);
}

// Both operands of one GEMM in one launch: the activation's 1x128 units
// (units_a of them, first) and the weight's 128x128 blocks share one unit
// list and one TMA ring, so the small, latency-bound activation pass fills
// in around the weight stream instead of competing with it as a second
// kernel.  Every unit is encoded exactly as the two kernels above encode it.
struct QuantPairArgs {
    int64_t M, KB;                       // activation: rows, 1x128 tiles per row
    uint8_t *qa;
    int64_t ldqa;
    float *sA;
    int64_t units_a;
    int64_t R, CB;                       // weight: rows, 128-column blocks
    uint8_t *qw;
    int64_t ldqw;
    float *sW;
    int64_t units;                       // activation units + weight blocks
    uint64_t wait_ns;                    // time limit of the ring's waits
};

__device__ __forceinline__ void qissue_pair(const QRing &r, const CUtensorMap *tmX, const CUtensorMap *tmW,
                                            const QuantPairArgs &a, int64_t j)
{
    const int64_t u = (int64_t)blockIdx.x + j * gridDim.x;
    int64_t rb, cb;
    if (u < a.units_a) {
        rb = u / a.KB;
        qissue_act_at(r, tmX, j, rb, u - rb * a.KB);
        return;
    }
    rb = (u - a.units_a) / a.CB;
    cb = (u - a.units_a) - rb * a.CB;
    const CUtensorMap *tm = tmW;
    const int s = (int)(j % QSTAGES);
    ptx::fence_proxy_async_smem();             // earlier generic reads of the stage come first
    ptx::mbar_arrive_expect_tx(r.full(s), QUNIT_BYTES);
    ptx::tma_load_2d(r.stage(s), tm, r.full(s), (int32_t)(cb * 128), (int32_t)(rb * 128));
}

__global__ void __launch_bounds__(QUANT_THREADS, 3) quant_act_w_kernel(
    const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const QuantPairArgs a)
{
    const QRing r = qring_setup(a.wait_ns);
    const int tid = threadIdx.x;
    const int64_t units = a.units;
    const int64_t mine = (int64_t)blockIdx.x < units ? (units - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    int64_t issued = 0;
    if (tid == 0)
        for (; issued < mine && issued < QSTAGES; ++issued)
            qissue_pair(r, &tmX, &tmW, a, issued);
    auto next = [&](int64_t j) {
        if (tid == 0 && issued < mine && issued < j + 1 + QSTAGES) {
            qissue_pair(r, &tmX, &tmW, a, issued);
            ++issued;
        }
    };
    int64_t j = 0;
    for (; j < mine; ++j) {
        if (!qwait(r, j))
            break;
        const int64_t u = (int64_t)blockIdx.x + j * gridDim.x;
        if (u < a.units_a) {
            const int64_t mb = u / a.KB;
            act_unit(r, j, mb, u - mb * a.KB, a.M, a.qa, a.ldqa, a.sA, [&] { next(j); });
        } else {
            const int64_t w = u - a.units_a;
            const int64_t rb = w / a.CB;
            w_unit(r, j, rb, w - rb * a.CB, a.R, a.CB, a.qw, a.ldqw, a.sW, [&] { next(j); });
        }
    }
    qdrain(r, j, issued);
}

// ---------------------------------------------------------------------------
// Per-tensor scaling, the contrast to the fine-grained groups: one scale for
// the whole tensor ["qqstock.cn walkthrough", FP8 section: fine-grained rather
// than per-tensor quantisation; "DeepSeek-V3 Technical Report digest",
// section 3, fine-grained quantisation bullet].  Same rules with the group
// being the tensor: s = fp32(amax / 448), q = E4M3_RNE_sat(fp32(x / s)).
//
// Divisor of a float amax: a BF16-representable amax (every amax of a BF16
// tensor is one) takes the proven reciprocal path of make_divisor; any other
// value (a caller's own history amax) uses IEEE division for every element.
__device__ __forceinline__ Divisor make_divisor_f32(float amax)
{
    const uint32_t bits = __float_as_uint(fabsf(amax));
    if ((bits & 0xFFFFu) == 0u)
        return make_divisor(bits >> 16);
    Divisor d;
    d.s = __fdiv_rn(fabsf(amax), 448.0f);
    d.mode = d.s == 0.0f ? 0 : 1;                  // a zero scale encodes x itself, as for a zero group
    d.r = 0.0f;
    return d;
}

// Pass 1 of current scaling: the amax (BF16 magnitude bits) of every 128x128
// unit of the tensor into ws[unit], through the same TMA ring as the weight
// quantiser.  Rows past R are the tensor map's zero fill and do not change a
// maximum of magnitudes.
__global__ void __launch_bounds__(QUANT_THREADS, 3) amax_units_kernel(
    const __grid_constant__ CUtensorMap tmX, int64_t CB, uint32_t *__restrict__ ws, int64_t units,
    uint64_t wait_ns)
{
    const QRing r = qring_setup(wait_ns);
    const int tid = threadIdx.x;
    const int chunk = tid & 15;
    const int r0 = tid >> 4;
    const int64_t mine = (int64_t)blockIdx.x < units ? (units - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    int64_t issued = 0;
    if (tid == 0)
        for (; issued < mine && issued < QSTAGES; ++issued)
            qissue(r, &tmX, issued, CB);
    int64_t j = 0;
    for (; j < mine; ++j) {
        if (!qwait(r, j))
            break;
        const uint32_t st = r.stage((int)(j % QSTAGES));
        uint32_t a = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint4 v;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(st + (uint32_t)((r0 + 16 * i) * 256 + chunk * 16)));
            a = max(a, absmax_bits8(v));
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
            a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
        uint32_t *wmax = r.red_u((int)(j & 1));
        if ((tid & 31) == 0)
            wmax[tid >> 5] = a;
        __syncthreads();                                   // stage read, warp maxima written
        if (tid == 0 && issued < mine && issued < j + 1 + QSTAGES) {
            qissue(r, &tmX, issued, CB);
            ++issued;
        }
        if (tid == 0) {
            uint32_t m = wmax[0];
#pragma unroll
            for (int i = 1; i < 8; ++i)
                m = max(m, wmax[i]);
            ws[(int64_t)blockIdx.x + j * gridDim.x] = m;
        }
    }
    qdrain(r, j, issued);
}

// Pass 2: one CTA reduces the unit maxima ws[0 .. U) to the tensor's amax,
// stores it as a float in ws[U] and the scale fp32(amax / 448) in *scale.
constexpr int REDUCE_THREADS = 1024;

__global__ void __launch_bounds__(REDUCE_THREADS) amax_reduce_kernel(uint32_t *__restrict__ ws, int64_t U,
                                                                    float *__restrict__ scale)
{
    __shared__ uint32_t part[REDUCE_THREADS / 32];
    uint32_t a = 0;
    for (int64_t i = threadIdx.x; i < U; i += REDUCE_THREADS)
        a = max(a, ws[i]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((threadIdx.x & 31) == 0)
        part[threadIdx.x >> 5] = a;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t m = part[0];
        for (int i = 1; i < REDUCE_THREADS / 32; ++i)
            m = max(m, part[i]);
        const float amax = __uint_as_float(m << 16);
        ws[U] = __float_as_uint(amax);
        *scale = make_divisor(m).s;
    }
}

// Every 128x128 unit encoded with ONE divisor, formed from the amax at
// *amax_src (pass 3 of current scaling: ws[U]; delayed scaling: the caller's
// history amax).  RECORD (delayed scaling): also the tensor's own amax, kept
// per thread over all its units and merged with one atomicMax per CTA into
// *amax_rec (float bits: monotone for non-negative floats), which the host
// has zeroed.  CTA 0 stores the scale.
template <bool RECORD>
__global__ void __launch_bounds__(QUANT_THREADS, 3) quant_fixed_kernel(
    const __grid_constant__ CUtensorMap tmX, int64_t R, int64_t CB, uint8_t *__restrict__ q, int64_t ldq,
    const float *__restrict__ amax_src, float *__restrict__ scale_out, uint32_t *__restrict__ amax_rec,
    int64_t units, uint64_t wait_ns)
{
    const QRing r = qring_setup(wait_ns);
    const int tid = threadIdx.x;
    const int chunk = tid & 15;
    const int r0 = tid >> 4;
    const Divisor d = make_divisor_f32(*amax_src);
    if (blockIdx.x == 0 && tid == 0)
        *scale_out = d.s;
    const int64_t mine = (int64_t)blockIdx.x < units ? (units - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    int64_t issued = 0;
    if (tid == 0)
        for (; issued < mine && issued < QSTAGES; ++issued)
            qissue(r, &tmX, issued, CB);
    uint32_t seen = 0;                                     // RECORD: max magnitude bits seen by this thread
    int64_t j = 0;
    for (; j < mine; ++j) {
        if (!qwait(r, j))
            break;
        const uint32_t st = r.stage((int)(j % QSTAGES));
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v[i].x), "=r"(v[i].y), "=r"(v[i].z), "=r"(v[i].w)
                         : "r"(st + (uint32_t)((r0 + 16 * i) * 256 + chunk * 16)));
        __syncthreads();                                   // the stage is free again
        if (tid == 0 && issued < mine && issued < j + 1 + QSTAGES) {
            qissue(r, &tmX, issued, CB);
            ++issued;
        }
        int64_t rb, cb;
        qunit(j, CB, rb, cb);
        if constexpr (RECORD) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                seen = max(seen, absmax_bits8(v[i]));      // rows past R are zero fill
        }
        const int64_t col = cb * 128 + chunk * 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t row = rb * 128 + r0 + 16 * i;
            if (row < R) {
                const uint2 c = quant_8(v[i], d);
                ptx::st_v2(q + row * ldq + col, c.x, c.y);
            }
        }
    }
    if constexpr (RECORD) {
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
            seen = max(seen, __shfl_xor_sync(0xffffffffu, seen, o));
        uint32_t *wmax = r.red_u(0);
        __syncthreads();
        if ((tid & 31) == 0)
            wmax[tid >> 5] = seen;
        __syncthreads();
        if (tid == 0) {
            uint32_t m = wmax[0];
#pragma unroll
            for (int i = 1; i < 8; ++i)
                m = max(m, wmax[i]);
            atomicMax(amax_rec, m << 16);
        }
    }
    qdrain(r, j, issued);
}

// Gather + 1x128 activation quantisation for expert dispatch: output row i
// is the quantisation of input row rows[i] (the token routed to that expert
// slot).  Quantising then gathering equals gathering then quantising, so
// the codes and scales equal fp8_quant_act_1x128 of the gathered BF16
// matrix, without materialising it.  The rows are arbitrary, so the loads
// are plain read-only 16-byte loads, kept in L2 (each token row is read once
// per routed copy); the codes are streamed out.  A warp takes one output row
// and eight consecutive 1x128 tiles, four adjacent lanes per tile (lane
// quarter g loads the tile's 16-byte chunks g, g + 4, g + 8, g + 12, all four
// before any use, and stores their codes: each step of the four lanes is one
// 32-byte run); a tile's amax takes two xor-shuffles and every lane forms its
// tile's divisor.  An index outside [0, T) is not read: the
// row encodes as zeros with a zero scale and bit 1 of the error word is set.
// (A version staging 16-row units through bulk copies into a shared-memory
// ring measured slower.)
constexpr int GATHER_THREADS = 256;
constexpr int GATHER_TILES = 8;                                  // tiles per warp task

// PACKED (expert-parallel dispatch): row i of q holds the row's K codes
// followed by its KB scales (FP32, row-major), so that one all-to-all moves a
// routed row and its scales together; sA is unused.
template <bool PACKED = false>
__global__ void __launch_bounds__(GATHER_THREADS) quant_act_gather_kernel(
    const uint16_t *__restrict__ x, int64_t T, int64_t ldx, const int32_t *__restrict__ rows, int64_t M,
    int64_t KB, uint8_t *__restrict__ q, int64_t ldq, float *__restrict__ sA)
{
    const int lane = threadIdx.x & 31;
    const int tt = lane >> 2;                                     // tile of the task
    const int g = lane & 3;                                       // lane quarter of the tile
    const uint64_t keep = ptx::policy_evict_last();
    const int64_t chunks = (KB + GATHER_TILES - 1) / GATHER_TILES;
    const int64_t warp0 = ((int64_t)blockIdx.x * GATHER_THREADS + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * GATHER_THREADS) >> 5;
    // the warp's tasks are warp0, warp0 + nwarps, ...: (row, chunk) advance
    // by a fixed step with one carry instead of a division per task
    const int64_t step_i = nwarps / chunks, step_c = nwarps - step_i * chunks;
    int64_t i = warp0 / chunks, chunk = warp0 - i * chunks;
    for (; i < M; i += step_i, chunk += step_c) {
        if (chunk >= chunks) {
            chunk -= chunks;
            if (++i >= M)
                break;
        }
        const int64_t kb = chunk * GATHER_TILES + tt;
        const int32_t src = rows[i];
        const bool valid = src >= 0 && (int64_t)src < T;
        if (!valid && lane == 0)
            atomicOr(&g_error_word, 2u);
        uint4 v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            v[c] = make_uint4(0u, 0u, 0u, 0u);
            if (valid && kb < KB)
                v[c] = ptx::ld_nc_v4_hint(x + (int64_t)src * ldx + kb * 128 + (g + 4 * c) * 8, keep);
        }
        uint32_t a = max(max(absmax_bits8(v[0]), absmax_bits8(v[1])), max(absmax_bits8(v[2]), absmax_bits8(v[3])));
        a = max(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = max(a, __shfl_xor_sync(0xffffffffu, a, 2));
        const Divisor d = make_divisor(a);
        // the usual case, every tile of the task on the reciprocal path,
        // encodes without a per-tile branch
        const bool recip = __all_sync(0xffffffffu, d.mode == 2);
        if (kb < KB) {
            uint8_t *qrow = q + i * ldq + kb * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint2 codes = recip ? quant_8_recip(v[c], d) : quant_8(v[c], d);
                ptx::st_v2_cs(qrow + (g + 4 * c) * 8, codes.x, codes.y);
            }
            if (g == 0) {
                if constexpr (PACKED)
                    reinterpret_cast<float *>(q + i * ldq + KB * 128)[kb] = d.s;
                else
                    sA[kb * M + i] = d.s;
            }
        }
    }
}

// Scatter + 1x128 activation quantisation, the dispatch written from the
// token side: token row t is read and encoded ONCE and its codes and scales
// are stored to each of its topk destination rows dest[t * topk + j].  The
// result is the gather form's (quantising before or after the copy gives the
// same bytes), with a topk-th of the loads and of the encoding work.  A warp
// task is one token row x GATHER_TILES consecutive 1x128 tiles, four lanes
// per tile, lane quarter g taking the tile's columns [32 g, 32 g + 32) (four
// 16-byte loads; its 32 codes leave as one 32-byte store per destination when
// the code matrix allows it); lane j < topk fetches destination j and the
// warp broadcasts it.  A destination outside [0, M) is skipped and sets bit 1 of the error
// word; a row named twice receives one of the tokens (unspecified which).
constexpr int SCATTER_MAX_TOPK = 32;

// PACKED (expert-parallel dispatch): each destination row holds the row's K
// codes followed by its KB scales (FP32), as in quant_act_gather_kernel.
template <bool PACKED = false>
__global__ void __launch_bounds__(GATHER_THREADS) quant_act_scatter_kernel(
    const uint16_t *__restrict__ x, int64_t T, int64_t ldx, const int32_t *__restrict__ dest, int topk, int64_t M,
    int64_t KB, uint8_t *__restrict__ q, int64_t ldq, float *__restrict__ sA)
{
    // Global memory only after the kernels this one depends on.  (Its grid is
    // larger than what fits on the GPU at once, so the next kernel is let in
    // only as blocks finish: launched earlier, its CTAs would take SMs that
    // this kernel's later blocks still need.)
    ptx::grid_dep_wait();
    const int lane = threadIdx.x & 31;
    const int tt = lane >> 2;                                     // tile of the task
    const int g = lane & 3;                                       // lane quarter of the tile: columns [32 g, +32)
    const bool st32 = ((reinterpret_cast<uintptr_t>(q) | (uintptr_t)ldq) & 31u) == 0;
    const int64_t chunks = (KB + GATHER_TILES - 1) / GATHER_TILES;
    const int64_t warp0 = ((int64_t)blockIdx.x * GATHER_THREADS + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * GATHER_THREADS) >> 5;
    const int64_t step_t = nwarps / chunks, step_c = nwarps - step_t * chunks;
    int64_t t = warp0 / chunks, chunk = warp0 - t * chunks;
    for (; t < T; t += step_t, chunk += step_c) {
        if (chunk >= chunks) {
            chunk -= chunks;
            if (++t >= T)
                break;
        }
        const int64_t kb = chunk * GATHER_TILES + tt;
        int32_t my_dst = -1;
        if (lane < topk) {
            my_dst = dest[t * topk + lane];
            if (my_dst < 0 || (int64_t)my_dst >= M) {
                if (chunk == 0)
                    atomicOr(&g_error_word, 2u);
                my_dst = -1;
            }
        }
        uint4 v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            v[c] = make_uint4(0u, 0u, 0u, 0u);
            if (kb < KB)
                v[c] = ptx::ld_nc_v4(x + t * ldx + kb * 128 + (4 * g + c) * 8);
        }
        uint32_t a = max(max(absmax_bits8(v[0]), absmax_bits8(v[1])), max(absmax_bits8(v[2]), absmax_bits8(v[3])));
        a = max(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = max(a, __shfl_xor_sync(0xffffffffu, a, 2));
        const Divisor d = make_divisor(a);
        uint32_t codes[8];                                        // the lane's 32 columns, in order
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint2 cc = quant_8(v[c], d);
            codes[2 * c] = cc.x;
            codes[2 * c + 1] = cc.y;
        }
        for (int j = 0; j < topk; ++j) {
            const int32_t row = __shfl_sync(0xffffffffu, my_dst, j);
            if (row < 0 || kb >= KB)
                continue;
            uint8_t *dst = q + (int64_t)row * ldq + kb * 128 + 32 * g;
            if (st32) {
                ptx::st_v8_cs(dst, codes);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    ptx::st_v2_cs(dst + 8 * c, codes[2 * c], codes[2 * c + 1]);
            }
            if (g == 0) {
                if constexpr (PACKED)
                    reinterpret_cast<float *>(q + (int64_t)row * ldq + KB * 128)[kb] = d.s;
                else
                    sA[kb * M + row] = d.s;
            }
        }
    }
    ptx::grid_dep_launch();
}

// Expert-parallel receive side: rows packed as [K codes | KB FP32 scales]
// arrive grouped by source rank; output row i is packed row perm[i], its
// codes into q[i] and its scales into the grouped GEMM's column layout
// sA[kb][i].  Blocks take runs of 32 output rows in turn: a block's warps copy
// the run's codes (16-byte loads and stores), then its 32 x KB scales go
// through shared memory so that each sA run of 32 rows is one 128-byte store.  An index outside
// [0, n_src) gives zero codes and scales and sets bit 1 of the error word.
constexpr int UNPACK_THREADS = 256;
constexpr int UNPACK_ROWS = 32;
constexpr int UNPACK_KB_CHUNK = 64;
constexpr int COPY_UNROLL = 8;          // 16-byte loads in flight per lane in a row copy

// One warp copies `chunks` 16-byte chunks of a row (zeros when !ok): each
// lane issues COPY_UNROLL loads before their stores, so a row is not a chain
// of dependent load -> store round trips.
__device__ __forceinline__ void warp_copy_row16(uint8_t *__restrict__ dst, const uint8_t *__restrict__ src,
                                                int64_t chunks, bool ok, int lane)
{
    int64_t c = lane;
    for (; c + 32 * (COPY_UNROLL - 1) < chunks; c += 32 * COPY_UNROLL) {
        uint4 v[COPY_UNROLL];
#pragma unroll
        for (int u = 0; u < COPY_UNROLL; ++u)
            v[u] = ok ? ptx::ld_nc_v4(src + (c + 32 * u) * 16) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < COPY_UNROLL; ++u)
            ptx::st_v4(dst + (c + 32 * u) * 16, v[u].x, v[u].y, v[u].z, v[u].w);
    }
    for (; c < chunks; c += 32) {
        const uint4 v = ok ? ptx::ld_nc_v4(src + c * 16) : make_uint4(0u, 0u, 0u, 0u);
        ptx::st_v4(dst + c * 16, v.x, v.y, v.z, v.w);
    }
}

__global__ void __launch_bounds__(UNPACK_THREADS) ep_unpack_kernel(
    const uint8_t *__restrict__ packed, int64_t ld_packed, int64_t n_src, int64_t KB, const int32_t *__restrict__ perm,
    int64_t M, uint8_t *__restrict__ q, int64_t ldq, float *__restrict__ sA)
{
    __shared__ float tile[UNPACK_KB_CHUNK][UNPACK_ROWS + 1];
    __shared__ int64_t src_row[UNPACK_ROWS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nblk = (M + UNPACK_ROWS - 1) / UNPACK_ROWS;
    const int64_t chunks = KB * 8;                                   // 16-byte chunks of codes per row
    // persistent: block b takes row blocks b, b + gridDim.x, ... so that the
    // blocks of an SM are at different phases (code copy, scale transpose)
    for (int64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
        const int64_t i0 = blk * UNPACK_ROWS;
        __syncthreads();                                             // the previous block's rows are done
        if (threadIdx.x < UNPACK_ROWS) {
            const int64_t i = i0 + threadIdx.x;
            int64_t s = -1;
            if (i < M) {
                const int32_t p = perm[i];
                if (p >= 0 && (int64_t)p < n_src)
                    s = p;
                else
                    atomicOr(&g_error_word, 2u);
            }
            src_row[threadIdx.x] = s;
        }
        __syncthreads();
        for (int r = warp; r < UNPACK_ROWS; r += UNPACK_THREADS / 32) {
            const int64_t i = i0 + r;
            if (i >= M)
                break;
            const int64_t s = src_row[r];
            warp_copy_row16(q + i * ldq, packed + (s >= 0 ? s : 0) * ld_packed, chunks, s >= 0, lane);
        }
        for (int64_t kb0 = 0; kb0 < KB; kb0 += UNPACK_KB_CHUNK) {
            const int nkb = (int)min((int64_t)UNPACK_KB_CHUNK, KB - kb0);
            __syncthreads();
            for (int e = threadIdx.x; e < UNPACK_ROWS * nkb; e += UNPACK_THREADS) {
                const int r = e / nkb, kb = e - r * nkb;
                const int64_t s = src_row[r];
                tile[kb][r] = s >= 0 ? reinterpret_cast<const float *>(packed + s * ld_packed + KB * 128)[kb0 + kb]
                                     : 0.0f;
            }
            __syncthreads();
            for (int e = threadIdx.x; e < UNPACK_ROWS * nkb; e += UNPACK_THREADS) {
                const int kb = e / UNPACK_ROWS, r = e - kb * UNPACK_ROWS;
                if (i0 + r < M)
                    sA[(kb0 + kb) * M + i0 + r] = tile[kb][r];
            }
        }
    }
}

// Row gather of byte rows: dst row i = src row rows[i] (row_bytes a multiple
// of 16, both row starts 16-byte aligned).  One warp per row, 16-byte copies.
// An index outside [0, n_src) gives a zero row and sets bit 1 of the error
// word.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint8_t *__restrict__ src, int64_t n_src,
                                                          int64_t ld_src, const int32_t *__restrict__ rows, int64_t M,
                                                          int64_t chunks, uint8_t *__restrict__ dst, int64_t ld_dst)
{
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t i = w0; i < M; i += nw) {
        const int32_t p = rows[i];
        const bool ok = p >= 0 && (int64_t)p < n_src;
        if (!ok && lane == 0)
            atomicOr(&g_error_word, 2u);
        warp_copy_row16(dst + i * ld_dst, src + (ok ? (int64_t)p : 0) * ld_src, chunks, ok, lane);
    }
}

// Token-dimension quantiser (the weight-gradient GEMM's operands): X is
// [T][F] (features contiguous); every feature column is cut into runs of 128
// tokens, each quantised with the 1x128 rule, and the codes are written
// transposed, qT[f][t], so that the GEMM reads them K(token)-major.  Unit
// (tb, fb): tokens [128 tb, +128) x features [128 fb, +128), staged through
// the same TMA ring.  Thread t holds the feature pair (2 fp, 2 fp + 1),
// fp = t % 64, for the 32 tokens of quarter t / 64 (32-bit shared loads, one
// 128-byte row segment per warp and token); the amax of each feature is the
// max over the four quarters, exchanged through shared memory.
__global__ void __launch_bounds__(QUANT_THREADS, 3) quant_tokens_1x128_kernel(
    const __grid_constant__ CUtensorMap tmX, int64_t T, int64_t F, int64_t FB, uint8_t *__restrict__ q,
    int64_t ldq, float *__restrict__ s, int64_t units, uint64_t wait_ns)
{
    const QRing r = qring_setup(wait_ns);
    const int tid = threadIdx.x;
    const int fp = tid & 63;
    const int qtr = tid >> 6;
    // a feature's 32 codes of a quarter are one whole 32-byte sector when the
    // code matrix allows 32-byte stores
    const bool st32 = ((reinterpret_cast<uintptr_t>(q) | (uintptr_t)ldq) & 31u) == 0;
    const int64_t mine = (int64_t)blockIdx.x < units ? (units - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    int64_t issued = 0;
    if (tid == 0)
        for (; issued < mine && issued < QSTAGES; ++issued)
            qissue(r, &tmX, issued, FB);
    int64_t j = 0;
    for (; j < mine; ++j) {
        if (!qwait(r, j))
            break;
        const uint32_t st = r.stage((int)(j % QSTAGES));
        uint32_t w[32];                                    // token qtr*32 + i: features (2fp | 2fp+1 << 16)
#pragma unroll
        for (int i = 0; i < 32; ++i)
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[i]) : "r"(st + (uint32_t)((qtr * 32 + i) * 256 + fp * 4)));
        uint32_t mx = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            mx = ptx::max_u16x2(mx, w[i] & 0x7FFF7FFFu);
        uint32_t *red = r.red_u((int)(j & 1));             // [4 quarters][64 feature pairs]
        red[qtr * 64 + fp] = mx;
        __syncthreads();                                   // stage read, partial maxima written
        if (tid == 0 && issued < mine && issued < j + 1 + QSTAGES) {
            qissue(r, &tmX, issued, FB);
            ++issued;
        }
        mx = ptx::max_u16x2(ptx::max_u16x2(red[fp], red[64 + fp]), ptx::max_u16x2(red[128 + fp], red[192 + fp]));
        const Divisor d0 = make_divisor(mx & 0xFFFFu);
        const Divisor d1 = make_divisor(mx >> 16);
        int64_t tb, fb;
        qunit(j, FB, tb, fb);
        const int64_t f0 = fb * 128 + 2 * fp;
        uint32_t c0[8], c1[8];                             // 32 codes of each feature
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const uint32_t *v = w + 8 * g;
            const uint4 lo = make_uint4(__byte_perm(v[0], v[1], 0x5410), __byte_perm(v[2], v[3], 0x5410),
                                        __byte_perm(v[4], v[5], 0x5410), __byte_perm(v[6], v[7], 0x5410));
            const uint4 hi = make_uint4(__byte_perm(v[0], v[1], 0x7632), __byte_perm(v[2], v[3], 0x7632),
                                        __byte_perm(v[4], v[5], 0x7632), __byte_perm(v[6], v[7], 0x7632));
            const uint2 a = quant_8(lo, d0);
            const uint2 b = quant_8(hi, d1);
            c0[2 * g] = a.x; c0[2 * g + 1] = a.y;
            c1[2 * g] = b.x; c1[2 * g + 1] = b.y;
        }
        const int64_t t0 = tb * 128 + qtr * 32;
        if (f0 < F) {
            uint8_t *dst = q + f0 * ldq + t0;
            if (st32) {
                ptx::st_v8(dst, c0);
            } else {
                ptx::st_v4(dst, c0[0], c0[1], c0[2], c0[3]);
                ptx::st_v4(dst + 16, c0[4], c0[5], c0[6], c0[7]);
            }
        }
        if (f0 + 1 < F) {
            uint8_t *dst = q + (f0 + 1) * ldq + t0;
            if (st32) {
                ptx::st_v8(dst, c1);
            } else {
                ptx::st_v4(dst, c1[0], c1[1], c1[2], c1[3]);
                ptx::st_v4(dst + 16, c1[4], c1[5], c1[6], c1[7]);
            }
        }
        if (qtr == 0) {
            float *srow = s + tb * F;
            if (f0 < F)
                srow[f0] = d0.s;
            if (f0 + 1 < F)
                srow[f0 + 1] = d1.s;
        }
    }
    qdrain(r, j, issued);
}

} // namespace fp8bs
