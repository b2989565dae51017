// fp8bs.cu -- the C ABI of the library (see include/fp8bs.h): argument
// validation, TMA tensor-map encoding and kernel launches.  One translation
// unit so that the device error word is a single symbol per device.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "fp8bs.h"
#include "ptx.cuh"
#include "quant.cuh"
#include "gemm.cuh"

namespace {

using namespace fp8bs;

constexpr int kMaxDevices = 64;
static_assert(MAX_EXPERTS == FP8BS_MAX_EXPERTS, "the header's expert limit is the kernel's");

struct DeviceInfo {
    bool probed = false;
    bool is_sm103 = false;
    int num_sms = 0;
    bool attrs_set = false;
    int max_pairs = 0;      // co-resident CTA pairs of the dense GEMM
};

constexpr int PAIR_STAGES = 4;      // 4 x 32 KiB operand stages per CTA of a pair
#ifndef PAIR_M_GROUP
#define PAIR_M_GROUP 16             // M-pairs (256 rows each) per tile rasterisation group
#endif

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
// Wait limit for single-CTA kernels set by fp8bs_selftest_set_wait_limit (0:
// the default WAIT_LIMIT_NS).  CTA-pair GEMMs always use the default.
std::atomic<uint64_t> g_test_wait_ns{0};

uint64_t wait_limit_single()
{
    const uint64_t t = g_test_wait_ns.load(std::memory_order_relaxed);
    return t ? t : WAIT_LIMIT_NS;
}
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Current device, checked to be sm_103; fills `info`.
int current_device(DeviceInfo **info)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FP8BS_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.probed) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FP8BS_ERR_DEVICE;
        d.is_sm103 = (major == 10 && minor == 3);
        d.num_sms = sms;
        d.probed = true;
    }
    if (!d.is_sm103)
        return FP8BS_ERR_DEVICE;
    if (!d.attrs_set) {
        const int pair_smem = gemm_smem_bytes<false, PAIR_STAGES, B_STAGE_BYTES / 2>();
        if (cudaFuncSetAttribute(fp8_gemm_kernel<false, false, false, 3>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 gemm_smem_bytes<false, 3>()) != cudaSuccess ||
            cudaFuncSetAttribute(fp8_gemm_kernel<false, true, false, 3>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 gemm_smem_bytes<false, 3>()) != cudaSuccess ||
            cudaFuncSetAttribute(fp8_gemm_kernel<false, false, true, PAIR_STAGES>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, pair_smem) != cudaSuccess ||
            cudaFuncSetAttribute(fp8_gemm_kernel<false, true, true, PAIR_STAGES>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, pair_smem) != cudaSuccess ||
            cudaFuncSetAttribute(fp8_gemm_kernel<false, false, false, 3, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 gemm_smem_bytes<false, 3>()) != cudaSuccess ||
            cudaFuncSetAttribute(fp8_gemm_kernel<false, true, false, 3, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 gemm_smem_bytes<false, 3>()) != cudaSuccess ||
            cudaFuncSetAttribute(fp8_gemm_kernel<false, false, true, PAIR_STAGES, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, pair_smem) != cudaSuccess ||
            cudaFuncSetAttribute(fp8_gemm_kernel<false, true, true, PAIR_STAGES, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, pair_smem) != cudaSuccess ||
            cudaFuncSetAttribute(fp8_gemm_kernel<false, false, false, 3, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 gemm_smem_bytes<false, 3, B_STAGE_BYTES, SCALE_SLOT_FLOATS_TOK>()) != cudaSuccess ||
            cudaFuncSetAttribute(fp8_gemm_kernel<false, false, true, PAIR_STAGES, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 gemm_smem_bytes<false, PAIR_STAGES, B_STAGE_BYTES / 2, SCALE_SLOT_FLOATS_TOK>()) !=
                cudaSuccess ||
            cudaFuncSetAttribute(quant_tokens_1x128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 quant_smem_bytes()) != cudaSuccess ||
            cudaFuncSetAttribute(fp8_gemm_kernel<true, false, false, 3>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 gemm_smem_bytes<true, 3>()) != cudaSuccess ||
            cudaFuncSetAttribute(quant_act_1x128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 quant_smem_bytes()) != cudaSuccess ||
            cudaFuncSetAttribute(quant_w_128x128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 quant_smem_bytes()) != cudaSuccess ||
            cudaFuncSetAttribute(quant_act_w_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 quant_smem_bytes()) != cudaSuccess ||
            cudaFuncSetAttribute(amax_units_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 quant_smem_bytes()) != cudaSuccess ||
            cudaFuncSetAttribute(quant_fixed_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 quant_smem_bytes()) != cudaSuccess ||
            cudaFuncSetAttribute(quant_fixed_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 quant_smem_bytes()) != cudaSuccess ||
            cudaFuncSetAttribute(fp8_gemm_kernel<false, false, false, 3, false, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 gemm_smem_bytes<false, 3>()) != cudaSuccess ||
            cudaFuncSetAttribute(fp8_gemm_kernel<false, true, false, 3, false, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 gemm_smem_bytes<false, 3>()) != cudaSuccess ||
            cudaFuncSetAttribute(fp8_gemm_kernel<false, false, true, PAIR_STAGES, false, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, pair_smem) != cudaSuccess ||
            cudaFuncSetAttribute(fp8_gemm_kernel<false, true, true, PAIR_STAGES, false, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, pair_smem) != cudaSuccess)
            return FP8BS_ERR_LAUNCH;
        // how many CTA pairs (2-CTA clusters) fit at once
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(d.num_sms & ~1));
        cfg.blockDim = dim3(GEMM_THREADS);
        cfg.dynamicSmemBytes = pair_smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, fp8_gemm_kernel<false, false, true, PAIR_STAGES>, &cfg) != cudaSuccess)
            clusters = 0;
        cudaGetLastError();
        d.max_pairs = std::min(clusters, d.num_sms / 2);
        d.attrs_set = true;
    }
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return FP8BS_ERR_DEVICE;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *info = &d;
    return FP8BS_OK;
}

int launch_status()
{
    return cudaGetLastError() == cudaSuccess ? FP8BS_OK : FP8BS_ERR_LAUNCH;
}

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the previous kernel on the stream finishes; it runs only its on-chip
// set-up before grid_dep_wait, so stream order is kept for every access to
// global memory.  cluster > 1 also sets the cluster dimension.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, int cluster,
               Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int n = 1;
    if (cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        n = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    if (cudaLaunchKernelEx(&cfg, kernel, args...) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_LAUNCH;
    }
    return launch_status();
}

// Row-major uint8 matrix [rows][cols] (row stride ld bytes) as a 2-D tensor
// map with a box of box_cols x box_rows and 128-byte swizzle.
bool encode_2d_u8(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t ld,
                  uint32_t box_cols, uint32_t box_rows)
{
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {ld};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d_u8(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                  uint32_t b0, uint32_t b1)
{
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0, d0 * d1};
    const cuuint32_t box[3] = {b0, b1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// BF16 output [M][N] (row stride ldc elements) as a 2-D tensor map for the
// epilogue's TMA stores: 64 x 32 boxes, 128-byte swizzle.
bool encode_c_bf16(CUtensorMap *m, void *C, uint64_t N, uint64_t M, uint64_t ldc)
{
    const cuuint64_t dims[2] = {N, M};
    const cuuint64_t strides[1] = {ldc * 2};
    const cuuint32_t box[2] = {64, BM};            // one promote warpgroup's 64-column half
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// BF16 matrix [rows][cols] (row stride ld elements) as a 2-D tensor map with
// 128 x 128 boxes (no swizzle): the quantisers' unit of work.
bool encode_bf16_units(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t ld)
{
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {ld * 2};
    const cuuint32_t box[2] = {128, 128};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Activation units: two 64 x 128 boxes per unit with the 128-byte swizzle
// (the activation quantiser's conflict-free shared-memory reads).
bool encode_bf16_units_sw128(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t ld)
{
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {ld * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int c_vector_ok(const void *C, int c_dtype, int64_t ldc)
{
    const int64_t es = c_dtype == FP8BS_OUT_FP32 ? 4 : 2;
    return aligned16(C) && (ldc * es) % 16 == 0;
}

int zero_output(void *C, int c_dtype, int64_t ldc, int64_t M, int64_t N, cudaStream_t stream)
{
    const size_t es = c_dtype == FP8BS_OUT_FP32 ? 4 : 2;
    if (cudaMemset2DAsync(C, (size_t)ldc * es, 0, (size_t)N * es, (size_t)M, stream) != cudaSuccess)
        return FP8BS_ERR_LAUNCH;
    return FP8BS_OK;
}

int check_gemm_common(const void *qA, const float *sA, const void *qB, const float *sB,
                      int64_t M, int64_t N, int64_t K, void *C, int c_dtype, int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0 || K % 128 != 0)
        return FP8BS_ERR_SHAPE;
    if (c_dtype != FP8BS_OUT_BF16 && c_dtype != FP8BS_OUT_FP32)
        return FP8BS_ERR_ARG;
    if (M == 0 || N == 0)
        return FP8BS_OK;
    if (!C || (K > 0 && (!qA || !sA || !qB || !sB)))
        return FP8BS_ERR_NULL;
    if (ldc < N)
        return FP8BS_ERR_SHAPE;
    const uintptr_t es = c_dtype == FP8BS_OUT_FP32 ? 4 : 2;
    if ((reinterpret_cast<uintptr_t>(C) % es) != 0)
        return FP8BS_ERR_ALIGN;
    if (K > 0 && (!aligned16(qA) || !aligned16(qB) || !aligned4(sA) || !aligned4(sB)))
        return FP8BS_ERR_ALIGN;
    if (M > INT32_MAX || N > INT32_MAX - 2 * BN || K > INT32_MAX)
        return FP8BS_ERR_SHAPE;
    return FP8BS_OK;
}

// Dense GEMM launch after argument checks (K > 0, M > 0, N > 0).  sC != null
// selects the E4M3-output epilogue (C is then the code matrix, ldc its row
// stride in bytes).
int launch_dense(DeviceInfo *dev, const void *qA, const float *sA, const void *qB, const float *sB,
                 int64_t M, int64_t N, int64_t K, int b_major, void *C, int c_dtype, int64_t ldc,
                 float *sC, cudaStream_t stream, bool tok = false, bool pt = false)
{
    const bool qout = sC != nullptr;              // (tok implies K-major B and no qout)
    CUtensorMap tmA, tmB;
    if (!encode_2d_u8(&tmA, qA, (uint64_t)K, (uint64_t)M, (uint64_t)K, BK, BM))
        return FP8BS_ERR_ARG;
    bool ok;
    // Dense GEMMs of two or more M-blocks run on CTA pairs (256 x 256 tiles,
    // each CTA holding its 128 rows of A and half of the B block).
#ifndef FP8BS_NO_PAIR
    const bool pair = dev->max_pairs > 0 && M > BM;
#else
    const bool pair = false;
#endif
    if (b_major == FP8BS_B_KMAJOR)
        ok = encode_2d_u8(&tmB, qB, (uint64_t)K, (uint64_t)N, (uint64_t)K, BK, pair ? 128 : BN);
    else
        ok = encode_2d_u8(&tmB, qB, (uint64_t)N, (uint64_t)K, (uint64_t)N, 128, BK);
    if (!ok)
        return FP8BS_ERR_ARG;

    GemmArgs g{};
    g.M = M;
    g.N = N;
    g.K = K;
    g.ldc = ldc;
    g.sA = sA;
    g.sB = sB;
    g.C = C;
    g.sC = sC;
    g.offsets = nullptr;
    g.E = 1;
    g.c_fp32 = c_dtype == FP8BS_OUT_FP32;
    g.wait_ns = pair ? WAIT_LIMIT_NS : wait_limit_single();
    CUtensorMap tmC = tmA;                        // unused unless a TMA epilogue runs
    if (qout) {
        // [M][N] codes, 128 x 128-byte boxes: one per warpgroup and tile
        if (!encode_2d_u8(&tmC, C, (uint64_t)N, (uint64_t)M, (uint64_t)ldc, 128, BM))
            return FP8BS_ERR_ARG;
        g.c_tma = 1;
    } else {
        g.c_tma = !g.c_fp32 && c_vector_ok(C, c_dtype, ldc) &&
                  encode_c_bf16(&tmC, C, (uint64_t)N, (uint64_t)M, (uint64_t)ldc);
    }
    g.num_m_blk = (int)((M + BM - 1) / BM);
    g.num_n_blk = (int)((N + BN - 1) / BN);
    g.KB = (int)(K / BK);
    g.NB128 = (int)((N + 127) / 128);
    g.num_m_pair = (g.num_m_blk + 1) / 2;
    {
        // rasterisation groups of at most PAIR_M_GROUP M-pairs, equal-sized
        const int ngroups = (g.num_m_pair + PAIR_M_GROUP - 1) / PAIR_M_GROUP;
        g.m_group = (g.num_m_pair + ngroups - 1) / ngroups;
    }
    if (pair) {
        g.num_tiles = (int64_t)g.num_m_pair * g.num_n_blk;
        const dim3 grid2((unsigned)(2 * std::min<int64_t>(g.num_tiles, dev->max_pairs)));
        const size_t psmem = tok ? gemm_smem_bytes<false, PAIR_STAGES, B_STAGE_BYTES / 2, SCALE_SLOT_FLOATS_TOK>()
                                 : gemm_smem_bytes<false, PAIR_STAGES, B_STAGE_BYTES / 2>();
        const dim3 blk(GEMM_THREADS);
        if (tok)
            return launch_pdl(fp8_gemm_kernel<false, false, true, PAIR_STAGES, false, true>, grid2, blk, psmem, stream, 2,
                              tmA, tmB, tmC, g);
        if (pt)
            return b_major == FP8BS_B_KMAJOR
                       ? launch_pdl(fp8_gemm_kernel<false, false, true, PAIR_STAGES, false, false, true>, grid2, blk,
                                    psmem, stream, 2, tmA, tmB, tmC, g)
                       : launch_pdl(fp8_gemm_kernel<false, true, true, PAIR_STAGES, false, false, true>, grid2, blk,
                                    psmem, stream, 2, tmA, tmB, tmC, g);
        if (b_major == FP8BS_B_KMAJOR)
            return qout ? launch_pdl(fp8_gemm_kernel<false, false, true, PAIR_STAGES, true>, grid2, blk, psmem, stream, 2,
                                     tmA, tmB, tmC, g)
                        : launch_pdl(fp8_gemm_kernel<false, false, true, PAIR_STAGES>, grid2, blk, psmem, stream, 2, tmA,
                                     tmB, tmC, g);
        return qout ? launch_pdl(fp8_gemm_kernel<false, true, true, PAIR_STAGES, true>, grid2, blk, psmem, stream, 2, tmA,
                                 tmB, tmC, g)
                    : launch_pdl(fp8_gemm_kernel<false, true, true, PAIR_STAGES>, grid2, blk, psmem, stream, 2, tmA, tmB,
                                 tmC, g);
    }
    g.num_tiles = (int64_t)g.num_m_blk * g.num_n_blk;
    const dim3 grid((unsigned)std::min<int64_t>(g.num_tiles, dev->num_sms));
    const dim3 blk(GEMM_THREADS);
    const size_t smem = gemm_smem_bytes<false, 3>();
    if (tok)
        return launch_pdl(fp8_gemm_kernel<false, false, false, 3, false, true>, grid, blk,
                          (size_t)gemm_smem_bytes<false, 3, B_STAGE_BYTES, SCALE_SLOT_FLOATS_TOK>(), stream, 1, tmA, tmB,
                          tmC, g);
    if (pt)
        return b_major == FP8BS_B_KMAJOR
                   ? launch_pdl(fp8_gemm_kernel<false, false, false, 3, false, false, true>, grid, blk, smem, stream, 1,
                                tmA, tmB, tmC, g)
                   : launch_pdl(fp8_gemm_kernel<false, true, false, 3, false, false, true>, grid, blk, smem, stream, 1,
                                tmA, tmB, tmC, g);
    if (b_major == FP8BS_B_KMAJOR)
        return qout ? launch_pdl(fp8_gemm_kernel<false, false, false, 3, true>, grid, blk, smem, stream, 1, tmA, tmB, tmC, g)
                    : launch_pdl(fp8_gemm_kernel<false, false, false, 3>, grid, blk, smem, stream, 1, tmA, tmB, tmC, g);
    return qout ? launch_pdl(fp8_gemm_kernel<false, true, false, 3, true>, grid, blk, smem, stream, 1, tmA, tmB, tmC, g)
                : launch_pdl(fp8_gemm_kernel<false, true, false, 3>, grid, blk, smem, stream, 1, tmA, tmB, tmC, g);
}

} // namespace

namespace fp8bs {

// One warp; lane 0 waits on a fresh mbarrier that nothing arrives at, with the
// pipelines' bounded wait and the given limit.
__global__ void selftest_wait_kernel(uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    const uint32_t b = ptx::smem_u32(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        abort_flag = 0u;
        ptx::fence_mbarrier_init();
    }
    __syncwarp();
    if (threadIdx.x == 0)
        wait_bounded(b, 0u, &abort_flag, limit_ns);
    __syncwarp();
}

// E4M3 codes of the fp32 values with bit patterns first, first + 1, ...,
// first + n - 1, two at a time through the conversion every quantiser uses
// (ptx::cvt_e4m3x2: cvt.rn.satfinite.e4m3x2.f32).
__global__ void selftest_encode_kernel(uint32_t first, int64_t n, uint8_t *__restrict__ q)
{
    const int64_t pairs = (n + 1) / 2;
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < pairs;
         p += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = 2 * p;
        const float a = __uint_as_float(first + (uint32_t)i);
        const float b = __uint_as_float(first + (uint32_t)(i + 1));
        const uint32_t c = ptx::cvt_e4m3x2(a, b);
        q[i] = (uint8_t)(c & 0xFFu);
        if (i + 1 < n)
            q[i + 1] = (uint8_t)(c >> 8);
    }
}

// Clears the given bits of the error word, atomically with respect to kernels
// on other streams that may set bits meanwhile.
__global__ void clear_error_bits_kernel(unsigned int bits)
{
    atomicAnd(&g_error_word, ~bits);
}

} // namespace fp8bs

extern "C" {

int fp8_quant_act_1x128(const void *x_bf16, int64_t M, int64_t K, int64_t ldx, void *q_e4m3,
                        int64_t ldq, float *sA, cudaStream_t stream)
{
    if (M < 0 || K < 0 || K % 128 != 0)
        return FP8BS_ERR_SHAPE;
    if (M == 0 || K == 0)
        return FP8BS_OK;
    if (!x_bf16 || !q_e4m3 || !sA)
        return FP8BS_ERR_NULL;
    if (ldx < K || ldq < K)
        return FP8BS_ERR_SHAPE;
    if (!aligned16(x_bf16) || !aligned16(q_e4m3) || !aligned4(sA) || (ldx * 2) % 16 != 0 ||
        ldq % 16 != 0)
        return FP8BS_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    CUtensorMap tmX;
    if (!encode_bf16_units_sw128(&tmX, x_bf16, (uint64_t)K, (uint64_t)M, (uint64_t)ldx))
        return FP8BS_ERR_ARG;
    const int64_t units = ((M + 127) / 128) * (K / 128);
    const int grid = (int)std::min<int64_t>(units, 3 * (int64_t)dev->num_sms);
    return launch_pdl(quant_act_1x128_kernel, dim3(grid), dim3(QUANT_THREADS), (size_t)quant_smem_bytes(), stream, 1,
                      tmX, M, (int64_t)(K / 128), static_cast<uint8_t *>(q_e4m3), ldq, sA, units,
                      wait_limit_single());
}

int fp8_quant_w_128x128(const void *w_bf16, int64_t R, int64_t C, int64_t ldw, void *q_e4m3,
                        int64_t ldq, float *sW, cudaStream_t stream)
{
    if (R < 0 || C < 0 || C % 128 != 0)
        return FP8BS_ERR_SHAPE;
    if (R == 0 || C == 0)
        return FP8BS_OK;
    if (!w_bf16 || !q_e4m3 || !sW)
        return FP8BS_ERR_NULL;
    if (ldw < C || ldq < C)
        return FP8BS_ERR_SHAPE;
    if (!aligned16(w_bf16) || !aligned16(q_e4m3) || !aligned4(sW) || (ldw * 2) % 16 != 0 ||
        ldq % 16 != 0)
        return FP8BS_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    const int64_t RB = (R + 127) / 128, CB = C / 128;
    CUtensorMap tmW;
    if (!encode_bf16_units(&tmW, w_bf16, (uint64_t)C, (uint64_t)R, (uint64_t)ldw))
        return FP8BS_ERR_ARG;
    const int64_t units = RB * CB;
    const int grid = (int)std::min<int64_t>(units, 3 * (int64_t)dev->num_sms);
    return launch_pdl(quant_w_128x128_kernel, dim3(grid), dim3(QUANT_THREADS), (size_t)quant_smem_bytes(), stream, 1,
                      tmW, R, CB, static_cast<uint8_t *>(q_e4m3), ldq, sW, units, wait_limit_single());
}

// Argument checks shared by the activation and weight quantisers: 0 when the
// operand is valid and non-empty, 1 when it is empty, else a status.
static int check_quant_operand(const void *x, int64_t rows, int64_t cols, int64_t ldx, const void *q, int64_t ldq,
                               const float *s)
{
    if (rows < 0 || cols < 0 || cols % 128 != 0)
        return FP8BS_ERR_SHAPE;
    if (rows == 0 || cols == 0)
        return 1;
    if (!x || !q || !s)
        return FP8BS_ERR_NULL;
    if (ldx < cols || ldq < cols)
        return FP8BS_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q) || !aligned4(s) || (ldx * 2) % 16 != 0 || ldq % 16 != 0)
        return FP8BS_ERR_ALIGN;
    return 0;
}

int fp8_quant_act_w(const void *x_bf16, int64_t M, int64_t K, int64_t ldx, void *qa_e4m3, int64_t ldqa, float *sA,
                    const void *w_bf16, int64_t R, int64_t C, int64_t ldw, void *qw_e4m3, int64_t ldqw, float *sW,
                    cudaStream_t stream)
{
    const int ca = check_quant_operand(x_bf16, M, K, ldx, qa_e4m3, ldqa, sA);
    if (ca < 0)
        return ca;
    const int cw = check_quant_operand(w_bf16, R, C, ldw, qw_e4m3, ldqw, sW);
    if (cw < 0)
        return cw;
    if (ca == 1 && cw == 1)
        return FP8BS_OK;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    CUtensorMap tmX, tmW;
    QuantPairArgs a = {};
    if (ca == 0) {
        if (!encode_bf16_units_sw128(&tmX, x_bf16, (uint64_t)K, (uint64_t)M, (uint64_t)ldx))
            return FP8BS_ERR_ARG;
        a.M = M;
        a.KB = K / 128;
        a.qa = static_cast<uint8_t *>(qa_e4m3);
        a.ldqa = ldqa;
        a.sA = sA;
        a.units_a = ((M + 127) / 128) * a.KB;
    }
    if (cw == 0) {
        if (!encode_bf16_units(&tmW, w_bf16, (uint64_t)C, (uint64_t)R, (uint64_t)ldw))
            return FP8BS_ERR_ARG;
        a.R = R;
        a.CB = C / 128;
        a.qw = static_cast<uint8_t *>(qw_e4m3);
        a.ldqw = ldqw;
        a.sW = sW;
    }
    if (ca != 0)
        tmX = tmW;                                // never read: no activation units
    if (cw != 0)
        tmW = tmX;                                // never read: no weight units
    a.units = a.units_a + (cw == 0 ? ((R + 127) / 128) * a.CB : 0);
    a.wait_ns = wait_limit_single();
    const int grid = (int)std::min<int64_t>(a.units, 3 * (int64_t)dev->num_sms);
    return launch_pdl(quant_act_w_kernel, dim3(grid), dim3(QUANT_THREADS), (size_t)quant_smem_bytes(), stream, 1, tmX,
                      tmW, a);
}

int fp8_gemm_blockscaled(const void *qA, const float *sA, const void *qB, const float *sB,
                         int64_t M, int64_t N, int64_t K, int b_major, void *C, int c_dtype,
                         int64_t ldc, cudaStream_t stream)
{
    if (b_major != FP8BS_B_KMAJOR && b_major != FP8BS_B_MNMAJOR)
        return FP8BS_ERR_ARG;
    if (int st = check_gemm_common(qA, sA, qB, sB, M, N, K, C, c_dtype, ldc))
        return st;
    if (M == 0 || N == 0)
        return FP8BS_OK;
    if (b_major == FP8BS_B_MNMAJOR && N % 128 != 0)
        return FP8BS_ERR_SHAPE;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    if (K == 0)
        return zero_output(C, c_dtype, ldc, M, N, stream);
    return launch_dense(dev, qA, sA, qB, sB, M, N, K, b_major, C, c_dtype, ldc, nullptr, stream);
}

int fp8_gemm_blockscaled_e4m3_out(const void *qA, const float *sA, const void *qB, const float *sB,
                                  int64_t M, int64_t N, int64_t K, int b_major, void *qC, int64_t ldqc,
                                  float *sC, cudaStream_t stream)
{
    if (b_major != FP8BS_B_KMAJOR && b_major != FP8BS_B_MNMAJOR)
        return FP8BS_ERR_ARG;
    if (M < 0 || N < 0 || K < 0 || K % 128 != 0 || N % 128 != 0)
        return FP8BS_ERR_SHAPE;
    if (M == 0 || N == 0)
        return FP8BS_OK;
    if (!qC || !sC || (K > 0 && (!qA || !sA || !qB || !sB)))
        return FP8BS_ERR_NULL;
    if (ldqc < N)
        return FP8BS_ERR_SHAPE;
    if (!aligned16(qC) || ldqc % 16 != 0 || !aligned4(sC) ||
        (K > 0 && (!aligned16(qA) || !aligned16(qB) || !aligned4(sA) || !aligned4(sB))))
        return FP8BS_ERR_ALIGN;
    if (M > INT32_MAX || N > INT32_MAX - 2 * BN || K > INT32_MAX)
        return FP8BS_ERR_SHAPE;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    if (K == 0) {
        // C == 0: every tile is all zero, so its codes are +0 and its scale 0
        if (cudaMemset2DAsync(qC, (size_t)ldqc, 0, (size_t)N, (size_t)M, stream) != cudaSuccess ||
            cudaMemsetAsync(sC, 0, (size_t)(N / 128) * (size_t)M * sizeof(float), stream) != cudaSuccess)
            return FP8BS_ERR_LAUNCH;
        return FP8BS_OK;
    }
    return launch_dense(dev, qA, sA, qB, sB, M, N, K, b_major, qC, FP8BS_OUT_BF16, ldqc, sC, stream);
}

int fp8_quant_act_1x128_gather(const void *x_bf16, int64_t T, int64_t K, int64_t ldx, const int32_t *rows,
                               int64_t M, void *q_e4m3, int64_t ldq, float *sA, cudaStream_t stream)
{
    if (T < 0 || M < 0 || K < 0 || K % 128 != 0)
        return FP8BS_ERR_SHAPE;
    if (M == 0 || K == 0)
        return FP8BS_OK;
    if (!x_bf16 || !rows || !q_e4m3 || !sA)
        return FP8BS_ERR_NULL;
    if (ldx < K || ldq < K)
        return FP8BS_ERR_SHAPE;
    if (!aligned16(x_bf16) || !aligned16(q_e4m3) || !aligned4(sA) || !aligned4(rows) || (ldx * 2) % 16 != 0 ||
        ldq % 16 != 0)
        return FP8BS_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    const int64_t KB = K / 128;
    const int64_t tasks = M * ((KB + GATHER_TILES - 1) / GATHER_TILES);
    const int64_t blocks = std::min<int64_t>((tasks * 32 + GATHER_THREADS - 1) / GATHER_THREADS,
                                             8 * (int64_t)dev->num_sms);
    quant_act_gather_kernel<false><<<(unsigned)blocks, GATHER_THREADS, 0, stream>>>(
        static_cast<const uint16_t *>(x_bf16), T, ldx, rows, M, KB, static_cast<uint8_t *>(q_e4m3), ldq, sA);
    return launch_status();
}

int fp8_quant_act_1x128_scatter(const void *x_bf16, int64_t T, int64_t K, int64_t ldx, const int32_t *dest, int topk,
                                int64_t M, void *q_e4m3, int64_t ldq, float *sA, cudaStream_t stream)
{
    if (T < 0 || M < 0 || K < 0 || K % 128 != 0)
        return FP8BS_ERR_SHAPE;
    if (topk < 1 || topk > SCATTER_MAX_TOPK)
        return FP8BS_ERR_ARG;
    if (T == 0 || K == 0)
        return FP8BS_OK;
    if (!x_bf16 || !dest || !q_e4m3 || !sA)
        return FP8BS_ERR_NULL;
    if (ldx < K || ldq < K)
        return FP8BS_ERR_SHAPE;
    if (!aligned16(x_bf16) || !aligned16(q_e4m3) || !aligned4(sA) || !aligned4(dest) || (ldx * 2) % 16 != 0 ||
        ldq % 16 != 0)
        return FP8BS_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    const int64_t KB = K / 128;
    const int64_t tasks = T * ((KB + GATHER_TILES - 1) / GATHER_TILES);
    const int64_t blocks = std::min<int64_t>((tasks * 32 + GATHER_THREADS - 1) / GATHER_THREADS,
                                             8 * (int64_t)dev->num_sms);
    return launch_pdl(quant_act_scatter_kernel<false>, dim3((unsigned)blocks), dim3(GATHER_THREADS), (size_t)0, stream, 1,
                      static_cast<const uint16_t *>(x_bf16), T, ldx, dest, topk, M, KB, static_cast<uint8_t *>(q_e4m3),
                      ldq, sA);
}

int fp8_ep_dispatch_pack(const void *x_bf16, int64_t T, int64_t K, int64_t ldx, const int32_t *rows, int64_t M,
                         void *packed, int64_t ld_packed, cudaStream_t stream)
{
    if (T < 0 || M < 0 || K < 0 || K % 128 != 0)
        return FP8BS_ERR_SHAPE;
    if (M == 0 || K == 0)
        return FP8BS_OK;
    if (!x_bf16 || !rows || !packed)
        return FP8BS_ERR_NULL;
    const int64_t KB = K / 128;
    if (ldx < K || ld_packed < K + 4 * KB)
        return FP8BS_ERR_SHAPE;
    if (!aligned16(x_bf16) || !aligned16(packed) || !aligned4(rows) || (ldx * 2) % 16 != 0 || ld_packed % 16 != 0)
        return FP8BS_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    const int64_t tasks = M * ((KB + GATHER_TILES - 1) / GATHER_TILES);
    const int64_t blocks = std::min<int64_t>((tasks * 32 + GATHER_THREADS - 1) / GATHER_THREADS,
                                             8 * (int64_t)dev->num_sms);
    quant_act_gather_kernel<true><<<(unsigned)blocks, GATHER_THREADS, 0, stream>>>(
        static_cast<const uint16_t *>(x_bf16), T, ldx, rows, M, KB, static_cast<uint8_t *>(packed), ld_packed,
        nullptr);
    return launch_status();
}

int fp8_ep_dispatch_pack_scatter(const void *x_bf16, int64_t T, int64_t K, int64_t ldx, const int32_t *dest, int topk,
                                 int64_t M, void *packed, int64_t ld_packed, cudaStream_t stream)
{
    if (T < 0 || M < 0 || K < 0 || K % 128 != 0)
        return FP8BS_ERR_SHAPE;
    if (topk < 1 || topk > SCATTER_MAX_TOPK)
        return FP8BS_ERR_ARG;
    if (T == 0 || K == 0)
        return FP8BS_OK;
    if (!x_bf16 || !dest || !packed)
        return FP8BS_ERR_NULL;
    const int64_t KB = K / 128;
    if (ldx < K || ld_packed < K + 4 * KB)
        return FP8BS_ERR_SHAPE;
    if (!aligned16(x_bf16) || !aligned16(packed) || !aligned4(dest) || (ldx * 2) % 16 != 0 || ld_packed % 16 != 0)
        return FP8BS_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    const int64_t tasks = T * ((KB + GATHER_TILES - 1) / GATHER_TILES);
    const int64_t blocks = std::min<int64_t>((tasks * 32 + GATHER_THREADS - 1) / GATHER_THREADS,
                                             8 * (int64_t)dev->num_sms);
    return launch_pdl(quant_act_scatter_kernel<true>, dim3((unsigned)blocks), dim3(GATHER_THREADS), (size_t)0, stream, 1,
                      static_cast<const uint16_t *>(x_bf16), T, ldx, dest, topk, M, KB, static_cast<uint8_t *>(packed),
                      ld_packed, static_cast<float *>(nullptr));
}

int fp8_ep_unpack(const void *packed, int64_t n_src, int64_t ld_packed, int64_t K, const int32_t *perm, int64_t M,
                  void *q_e4m3, int64_t ldq, float *sA, cudaStream_t stream)
{
    if (n_src < 0 || M < 0 || K < 0 || K % 128 != 0)
        return FP8BS_ERR_SHAPE;
    if (M == 0 || K == 0)
        return FP8BS_OK;
    if (!packed || !perm || !q_e4m3 || !sA)
        return FP8BS_ERR_NULL;
    const int64_t KB = K / 128;
    if (ld_packed < K + 4 * KB || ldq < K)
        return FP8BS_ERR_SHAPE;
    if (!aligned16(packed) || !aligned16(q_e4m3) || !aligned4(sA) || !aligned4(perm) || ld_packed % 16 != 0 ||
        ldq % 16 != 0)
        return FP8BS_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    const int64_t blocks = std::min<int64_t>((M + UNPACK_ROWS - 1) / UNPACK_ROWS, 4 * (int64_t)dev->num_sms);
    ep_unpack_kernel<<<(unsigned)blocks, UNPACK_THREADS, 0, stream>>>(
        static_cast<const uint8_t *>(packed), ld_packed, n_src, KB, perm, M, static_cast<uint8_t *>(q_e4m3), ldq, sA);
    return launch_status();
}

int fp8bs_gather_rows(const void *src, int64_t n_src, int64_t ld_src, const int32_t *rows, int64_t M,
                      int64_t row_bytes, void *dst, int64_t ld_dst, cudaStream_t stream)
{
    if (n_src < 0 || M < 0 || row_bytes < 0 || row_bytes % 16 != 0)
        return FP8BS_ERR_SHAPE;
    if (M == 0 || row_bytes == 0)
        return FP8BS_OK;
    if (!src || !rows || !dst)
        return FP8BS_ERR_NULL;
    if (ld_src < row_bytes || ld_dst < row_bytes)
        return FP8BS_ERR_SHAPE;
    if (!aligned16(src) || !aligned16(dst) || !aligned4(rows) || ld_src % 16 != 0 || ld_dst % 16 != 0)
        return FP8BS_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    const int64_t blocks = std::min<int64_t>((M * 32 + 255) / 256, 8 * (int64_t)dev->num_sms);
    gather_rows_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const uint8_t *>(src), n_src, ld_src, rows,
                                                             M, row_bytes / 16, static_cast<uint8_t *>(dst), ld_dst);
    return launch_status();
}

int fp8_quant_tokens_1x128(const void *x_bf16, int64_t T, int64_t F, int64_t ldx, void *qT, int64_t ldq,
                           float *s, cudaStream_t stream)
{
    if (T < 0 || F < 0 || T % 128 != 0)
        return FP8BS_ERR_SHAPE;
    if (T == 0 || F == 0)
        return FP8BS_OK;
    if (!x_bf16 || !qT || !s)
        return FP8BS_ERR_NULL;
    if (ldx < F || ldq < T)
        return FP8BS_ERR_SHAPE;
    if (!aligned16(x_bf16) || !aligned16(qT) || !aligned4(s) || (ldx * 2) % 16 != 0 || ldq % 16 != 0)
        return FP8BS_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    CUtensorMap tmX;
    if (!encode_bf16_units(&tmX, x_bf16, (uint64_t)F, (uint64_t)T, (uint64_t)ldx))
        return FP8BS_ERR_ARG;
    const int64_t FB = (F + 127) / 128;
    const int64_t units = (T / 128) * FB;
    const int grid = (int)std::min<int64_t>(units, 3 * (int64_t)dev->num_sms);
    return launch_pdl(quant_tokens_1x128_kernel, dim3(grid), dim3(QUANT_THREADS), (size_t)quant_smem_bytes(), stream, 1,
                      tmX, T, F, FB, static_cast<uint8_t *>(qT), ldq, s, units, wait_limit_single());
}

int fp8_gemm_wgrad(const void *qA, const float *sA, const void *qB, const float *sB, int64_t M, int64_t N,
                   int64_t K, void *C, int c_dtype, int64_t ldc, cudaStream_t stream)
{
    if (int st = check_gemm_common(qA, sA, qB, sB, M, N, K, C, c_dtype, ldc))
        return st;
    if (M == 0 || N == 0)
        return FP8BS_OK;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    if (K == 0)
        return zero_output(C, c_dtype, ldc, M, N, stream);
    return launch_dense(dev, qA, sA, qB, sB, M, N, K, FP8BS_B_KMAJOR, C, c_dtype, ldc, nullptr, stream, true);
}

int fp8_grouped_gemm_blockscaled(const void *qA, const float *sA, const void *qB,
                                 const float *sB, const int32_t *seg_offsets, int E,
                                 int64_t M_total, int64_t N, int64_t K, void *C, int c_dtype,
                                 int64_t ldc, cudaStream_t stream)
{
    if (E < 1 || E > MAX_EXPERTS)
        return FP8BS_ERR_ARG;
    if (int st = check_gemm_common(qA, sA, qB, sB, M_total, N, K, C, c_dtype, ldc))
        return st;
    if (M_total == 0 || N == 0)
        return FP8BS_OK;
    if (!seg_offsets)
        return FP8BS_ERR_NULL;
    if (!aligned4(seg_offsets))
        return FP8BS_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    if (K == 0)
        return zero_output(C, c_dtype, ldc, M_total, N, stream);

    CUtensorMap tmA, tmB;
    if (!encode_2d_u8(&tmA, qA, (uint64_t)K, (uint64_t)M_total, (uint64_t)K, BK, BM))
        return FP8BS_ERR_ARG;
    if (!encode_3d_u8(&tmB, qB, (uint64_t)K, (uint64_t)N, (uint64_t)E, BK, BN))
        return FP8BS_ERR_ARG;

    GemmArgs g{};
    g.M = M_total;
    g.N = N;
    g.K = K;
    g.ldc = ldc;
    g.sA = sA;
    g.sB = sB;
    g.C = C;
    g.offsets = seg_offsets;
    g.E = E;
    g.c_fp32 = c_dtype == FP8BS_OUT_FP32;
    g.wait_ns = wait_limit_single();
    CUtensorMap tmC = tmA;                        // unused unless the BF16 TMA epilogue runs
    g.c_tma = !g.c_fp32 && c_vector_ok(C, c_dtype, ldc) &&
              encode_c_bf16(&tmC, C, (uint64_t)N, (uint64_t)M_total, (uint64_t)ldc);
    g.num_m_blk = 0;
    g.num_n_blk = (int)((N + BN - 1) / BN);
    g.KB = (int)(K / BK);
    g.NB128 = (int)((N + 127) / 128);
    g.num_tiles = 0;
    return launch_pdl(fp8_gemm_kernel<true, false, false, 3>, dim3(dev->num_sms), dim3(GEMM_THREADS),
                      (size_t)gemm_smem_bytes<true, 3>(), stream, 1, tmA, tmB, tmC, g);
}

int fp8_quant_per_tensor_workspace_size(int64_t R, int64_t C, int64_t *bytes)
{
    if (!bytes)
        return FP8BS_ERR_NULL;
    if (R < 0 || C < 0 || C % 128 != 0)
        return FP8BS_ERR_SHAPE;
    *bytes = 4 * (((R + 127) / 128) * (C / 128) + 1);
    return FP8BS_OK;
}

int fp8_quant_per_tensor(const void *x_bf16, int64_t R, int64_t C, int64_t ldx, void *q_e4m3, int64_t ldq,
                         float *scale, void *workspace, int64_t workspace_bytes, cudaStream_t stream)
{
    const int st = check_quant_operand(x_bf16, R, C, ldx, q_e4m3, ldq, scale);
    if (st < 0)
        return st;
    if (st == 1)
        return FP8BS_OK;
    if (!workspace)
        return FP8BS_ERR_NULL;
    if (!aligned4(workspace))
        return FP8BS_ERR_ALIGN;
    const int64_t CB = C / 128, U = ((R + 127) / 128) * CB;
    if (workspace_bytes < 4 * (U + 1))
        return FP8BS_ERR_ARG;
    DeviceInfo *dev = nullptr;
    if (int s = current_device(&dev))
        return s;
    CUtensorMap tmX;
    if (!encode_bf16_units(&tmX, x_bf16, (uint64_t)C, (uint64_t)R, (uint64_t)ldx))
        return FP8BS_ERR_ARG;
    uint32_t *ws = static_cast<uint32_t *>(workspace);
    const int grid = (int)std::min<int64_t>(U, 3 * (int64_t)dev->num_sms);
    amax_units_kernel<<<grid, QUANT_THREADS, quant_smem_bytes(), stream>>>(tmX, CB, ws, U, wait_limit_single());
    amax_reduce_kernel<<<1, REDUCE_THREADS, 0, stream>>>(ws, U, scale);
    quant_fixed_kernel<false><<<grid, QUANT_THREADS, quant_smem_bytes(), stream>>>(
        tmX, R, CB, static_cast<uint8_t *>(q_e4m3), ldq, reinterpret_cast<const float *>(ws + U), scale, nullptr, U,
        wait_limit_single());
    return launch_status();
}

int fp8_quant_per_tensor_delayed(const void *x_bf16, int64_t R, int64_t C, int64_t ldx, const float *amax_in,
                                 void *q_e4m3, int64_t ldq, float *scale, float *amax_out, cudaStream_t stream)
{
    const int st = check_quant_operand(x_bf16, R, C, ldx, q_e4m3, ldq, scale);
    if (st < 0)
        return st;
    if (st == 1)
        return FP8BS_OK;
    if (!amax_in || !amax_out)
        return FP8BS_ERR_NULL;
    if (!aligned4(amax_in) || !aligned4(amax_out))
        return FP8BS_ERR_ALIGN;
    if (static_cast<const void *>(amax_in) == static_cast<const void *>(amax_out))
        return FP8BS_ERR_ARG;
    DeviceInfo *dev = nullptr;
    if (int s = current_device(&dev))
        return s;
    CUtensorMap tmX;
    if (!encode_bf16_units(&tmX, x_bf16, (uint64_t)C, (uint64_t)R, (uint64_t)ldx))
        return FP8BS_ERR_ARG;
    const int64_t CB = C / 128, U = ((R + 127) / 128) * CB;
    if (cudaMemsetAsync(amax_out, 0, sizeof(float), stream) != cudaSuccess)
        return FP8BS_ERR_LAUNCH;
    const int grid = (int)std::min<int64_t>(U, 3 * (int64_t)dev->num_sms);
    quant_fixed_kernel<true><<<grid, QUANT_THREADS, quant_smem_bytes(), stream>>>(
        tmX, R, CB, static_cast<uint8_t *>(q_e4m3), ldq, amax_in, scale, reinterpret_cast<uint32_t *>(amax_out), U,
        wait_limit_single());
    return launch_status();
}

int fp8_gemm_per_tensor(const void *qA, const float *sA, const void *qB, const float *sB, int64_t M, int64_t N,
                        int64_t K, int b_major, void *C, int c_dtype, int64_t ldc, cudaStream_t stream)
{
    if (b_major != FP8BS_B_KMAJOR && b_major != FP8BS_B_MNMAJOR)
        return FP8BS_ERR_ARG;
    if (int st = check_gemm_common(qA, sA, qB, sB, M, N, K, C, c_dtype, ldc))
        return st;
    if (M == 0 || N == 0)
        return FP8BS_OK;
    if (b_major == FP8BS_B_MNMAJOR && N % 16 != 0)
        return FP8BS_ERR_SHAPE;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    if (K == 0)
        return zero_output(C, c_dtype, ldc, M, N, stream);
    return launch_dense(dev, qA, sA, qB, sB, M, N, K, b_major, C, c_dtype, ldc, nullptr, stream, false, true);
}

int fp8bs_selftest_wait_timeout(int64_t limit_us, cudaStream_t stream)
{
    if (limit_us < 1 || limit_us > 1000000)
        return FP8BS_ERR_ARG;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    selftest_wait_kernel<<<1, 32, 0, stream>>>((uint64_t)limit_us * 1000u);
    return launch_status();
}

int fp8bs_last_error(cudaStream_t stream)
{
    if (cudaStreamSynchronize(stream) != cudaSuccess)
        return FP8BS_ERR_LAUNCH;
    if (cudaGetLastError() != cudaSuccess)
        return FP8BS_ERR_LAUNCH;
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_error_word, sizeof word) != cudaSuccess)
        return FP8BS_ERR_LAUNCH;
    if (word == 0)
        return FP8BS_OK;
    // Report one condition per call, the time-out first; clear only its bit,
    // so that a second condition is reported by the next call.
    const unsigned int bit = (word & 1u) ? 1u : (word & 2u) ? 2u : word;
    clear_error_bits_kernel<<<1, 1, 0, stream>>>(bit);
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(stream) != cudaSuccess)
        return FP8BS_ERR_LAUNCH;
    return bit == 1u ? FP8BS_ERR_TIMEOUT : FP8BS_ERR_INDEX;
}

int fp8bs_selftest_encode_e4m3(uint32_t first_bits, int64_t n, uint8_t *q, cudaStream_t stream)
{
    if (n < 0 || n > ((int64_t)1 << 32) - (int64_t)first_bits)
        return FP8BS_ERR_ARG;
    if (n == 0)
        return FP8BS_OK;
    if (!q)
        return FP8BS_ERR_NULL;
    DeviceInfo *dev = nullptr;
    if (int st = current_device(&dev))
        return st;
    const int64_t pairs = (n + 1) / 2;
    const int64_t blocks = std::min<int64_t>((pairs + 255) / 256, 16 * (int64_t)dev->num_sms);
    selftest_encode_kernel<<<(unsigned)blocks, 256, 0, stream>>>(first_bits, n, q);
    return launch_status();
}

int fp8bs_selftest_set_wait_limit(int64_t limit_ns)
{
    if (limit_ns < 0 || limit_ns > (int64_t)WAIT_LIMIT_NS)
        return FP8BS_ERR_ARG;
    g_test_wait_ns.store((uint64_t)limit_ns, std::memory_order_relaxed);
    return FP8BS_OK;
}

} // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free per-tensor quantisation.
//
// The scratch that fp8_quant_per_tensor takes from its caller (one word per
// 128x128 unit plus one) lives here instead, in a fixed array that every GPU
// holds from the moment it loads this library until the process exits.  In
// host code the name g_noalloc_scratch is only a host-side stand-in for the
// array, not a device address: it is never passed to a kernel.  The device
// address is looked up once per device, with that device current, by
// cudaGetSymbolAddress (on the first call of fp8_quant_per_tensor_noalloc on
// that device), and that address is what the kernels receive.
//
// Every call on a device uses the same array and leaves its contents behind.
// Nothing in it has to start at zero: the unit pass writes every word the
// reduction reads, and the reduction writes the word the encoding pass reads.
// Two calls whose kernels overlap on the GPU (on different streams) race on
// the array.
static __device__ __align__(256) uint32_t g_noalloc_scratch[FP8BS_NOALLOC_MAX_UNITS + 1];

namespace {
std::mutex g_noalloc_mutex;
uint32_t *g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device `dev`.
int noalloc_scratch(int dev, uint32_t **out)
{
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return FP8BS_ERR_DEVICE;
        }
        g_noalloc_ptr[dev] = static_cast<uint32_t *>(ptr);
    }
    *out = g_noalloc_ptr[dev];
    return FP8BS_OK;
}
} // namespace

extern "C" int fp8_quant_per_tensor_noalloc(const void *x_bf16, int64_t R, int64_t C, int64_t ldx, void *q_e4m3,
                                            int64_t ldq, float *scale, cudaStream_t stream)
{
    const int st = check_quant_operand(x_bf16, R, C, ldx, q_e4m3, ldq, scale);
    if (st < 0)
        return st;
    if (st == 1)
        return FP8BS_OK;
    const int64_t CB = C / 128, U = ((R + 127) / 128) * CB;
    if (U > FP8BS_NOALLOC_MAX_UNITS)
        return FP8BS_ERR_SCRATCH;
    DeviceInfo *dev = nullptr;
    if (int s = current_device(&dev))
        return s;
    int ordinal = 0;
    if (cudaGetDevice(&ordinal) != cudaSuccess)
        return FP8BS_ERR_DEVICE;
    uint32_t *ws = nullptr;
    if (int s = noalloc_scratch(ordinal, &ws))
        return s;
    CUtensorMap tmX;
    if (!encode_bf16_units(&tmX, x_bf16, (uint64_t)C, (uint64_t)R, (uint64_t)ldx))
        return FP8BS_ERR_ARG;
    const int grid = (int)std::min<int64_t>(U, 3 * (int64_t)dev->num_sms);
    amax_units_kernel<<<grid, QUANT_THREADS, quant_smem_bytes(), stream>>>(tmX, CB, ws, U, wait_limit_single());
    amax_reduce_kernel<<<1, REDUCE_THREADS, 0, stream>>>(ws, U, scale);
    quant_fixed_kernel<false><<<grid, QUANT_THREADS, quant_smem_bytes(), stream>>>(
        tmX, R, CB, static_cast<uint8_t *>(q_e4m3), ldq, reinterpret_cast<const float *>(ws + U), scale, nullptr, U,
        wait_limit_single());
    return launch_status();
}
