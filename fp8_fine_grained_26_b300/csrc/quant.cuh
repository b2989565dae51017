// quant.cuh -- fine-grained FP8 quantisers (1x128 activation tiles, 128x128
// weight blocks).  ["DeepSeek-V3 training walkthrough", section 二(四), and
// "DeepSeek-V3 Technical Report digest", section 3: activations per 1x128
// tile, weights per 128x128 block.]
//
// Both kernels are HBM-bound streams: 2 bytes read + 1 byte written per
// element plus 4 bytes per scale.  Each 1x128 tile is one 256-byte row segment,
// read by a half-warp with one 16-byte load per lane; the tile's amax is an
// integer max over the BF16 magnitude bits (monotone for finite values)
// reduced with four xor-shuffles.  scale = amax / 448 is one IEEE division;
// x / scale is formed exactly (see Divisor below) and encoded with the
// hardware RNE-satfinite E4M3 conversion; codes are stored 8 bytes per lane.
#pragma once
#include "ptx.cuh"

namespace fp8bs {

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t absmax_bits_bf16x2(uint32_t w)
{
    return max(w & 0x7FFFu, (w >> 16) & 0x7FFFu);
}

// Per-group divisor.  The quotient fp32(x / s) is formed with Markstein's
// correction step (P. Markstein, IBM J. Res. Dev. 34(1), 1990): with the
// correctly rounded reciprocal r = RN(1/s),
//     q0 = RN(x * r),  rem = fma(-q0, s, x),  q = copysign(fma(rem, r, q0), x),
// which an exhaustive check over every BF16 amax >= 2^-90 and every BF16
// |x| <= amax shows to equal IEEE division bit for bit (up to the sign of
// zero-encoding quotients below 2^-11).  Groups with a smaller amax use
// IEEE division; an all-zero group (s == 0) encodes x itself (a signed zero).
struct Divisor {
    float s, r;
    int mode;           // 0: s == 0, 1: IEEE division, 2: reciprocal + correction
};

__device__ __forceinline__ Divisor make_divisor(uint32_t amax_bits)
{
    Divisor d;
    const float amax = __uint_as_float(amax_bits << 16);
    d.s = __fdiv_rn(amax, 448.0f);
    d.mode = amax_bits == 0 ? 0 : (amax_bits >= 0x1280u ? 2 : 1);   // 0x1280 = 2^-90 in BF16
    d.r = d.mode == 2 ? __frcp_rn(d.s) : 0.0f;
    return d;
}

__device__ __forceinline__ float quotient(float x, const Divisor &d)
{
    if (d.mode == 2) {
        const float q0 = __fmul_rn(x, d.r);
        const float rem = __fmaf_rn(-q0, d.s, x);
        // the quotient of x by a positive s carries x's sign; this also keeps
        // -0 (where rem = +0 and +0 + -0 would round to +0)
        return copysignf(__fmaf_rn(rem, d.r, q0), x);
    }
    return d.mode == 1 ? __fdiv_rn(x, d.s) : x;
}

// q = E4M3(x / s) for the two BF16 values packed in `w`.
__device__ __forceinline__ uint32_t quant_pair(uint32_t w, const Divisor &d)
{
    return ptx::cvt_e4m3x2(quotient(bf16lo(w), d), quotient(bf16hi(w), d));
}

__device__ __forceinline__ uint2 quant_8(const uint4 &v, const Divisor &d)
{
    uint2 r;
    r.x = quant_pair(v.x, d) | (quant_pair(v.y, d) << 16);
    r.y = quant_pair(v.z, d) | (quant_pair(v.w, d) << 16);
    return r;
}

// One half-warp per 1x128 tile.  Tiles are numbered t = kb * M + m so that
// consecutive half-warps write consecutive scales of sA[kb][*].  The loop is
// warp-uniform (both half-warps iterate together) because of the shuffles.
__global__ void __launch_bounds__(256) quant_act_1x128_kernel(
    const uint16_t *__restrict__ x, int64_t M, int64_t KB, int64_t ldx,
    uint8_t *__restrict__ q, int64_t ldq, float *__restrict__ sA)
{
    const int lane16 = threadIdx.x & 15;
    const int half = (threadIdx.x >> 4) & 1;
    const int64_t total = M * KB;
    const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t wp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
         wp * 2 < total; wp += warps_total) {
        const int64_t t = wp * 2 + half;
        const bool valid = t < total;
        const int64_t kb = valid ? t / M : 0;
        const int64_t m = valid ? t - kb * M : 0;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (valid)
            v = ptx::ld_nc_v4(x + m * ldx + kb * 128 + lane16 * 8);
        uint32_t a = max(max(absmax_bits_bf16x2(v.x), absmax_bits_bf16x2(v.y)),
                         max(absmax_bits_bf16x2(v.z), absmax_bits_bf16x2(v.w)));
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1)
            a = max(a, __shfl_xor_sync(0xffffffffu, a, o, 16));
        const Divisor d = make_divisor(a);
        if (valid) {
            const uint2 r = quant_8(v, d);
            ptx::st_v2(q + m * ldq + kb * 128 + lane16 * 8, r.x, r.y);
            if (lane16 == 0)
                sA[kb * M + m] = d.s;
        }
    }
}

// One 256-thread CTA per 128x128 block.  Thread t owns the 16-byte column
// chunk (t & 15) of rows (t >> 4) + 16 i, i = 0..7: 64 elements held in
// registers between the amax pass and the encode pass (one HBM read).
__global__ void __launch_bounds__(256) quant_w_128x128_kernel(
    const uint16_t *__restrict__ w, int64_t R, int64_t CB, int64_t ldw,
    uint8_t *__restrict__ q, int64_t ldq, float *__restrict__ sW)
{
    __shared__ uint32_t warp_max[8];
    const int64_t blk = blockIdx.x;
    const int64_t rb = blk / CB, cb = blk - rb * CB;
    const int chunk = threadIdx.x & 15;
    const int r0 = threadIdx.x >> 4;
    const int64_t row0 = rb * 128;
    const int64_t col = cb * 128 + chunk * 8;

    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = row0 + r0 + 16 * i;
        v[i] = (r < R) ? ptx::ld_nc_v4(w + r * ldw + col) : make_uint4(0, 0, 0, 0);
    }
    uint32_t a = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        a = max(a, max(max(absmax_bits_bf16x2(v[i].x), absmax_bits_bf16x2(v[i].y)),
                       max(absmax_bits_bf16x2(v[i].z), absmax_bits_bf16x2(v[i].w))));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((threadIdx.x & 31) == 0)
        warp_max[threadIdx.x >> 5] = a;
    __syncthreads();
    a = warp_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i)
        a = max(a, warp_max[i]);
    const Divisor d = make_divisor(a);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = row0 + r0 + 16 * i;
        if (r < R) {
            const uint2 c = quant_8(v[i], d);
            ptx::st_v2(q + r * ldq + col, c.x, c.y);
        }
    }
    if (threadIdx.x == 0)
        sW[rb * CB + cb] = d.s;
}

} // namespace fp8bs
