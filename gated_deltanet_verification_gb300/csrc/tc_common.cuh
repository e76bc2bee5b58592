// Helpers shared by the tensor-core kernels (TMA, tensor maps, launch set-up).
#pragma once

#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"
#include "sm100.cuh"

namespace bole {
namespace tc {

using namespace sm100;

constexpr int kD = 128;                            // d_k = d_v of the tensor-core kernels
constexpr uint64_t kWaitNs = 200ull * 1000 * 1000; // 200 ms bound on any device wait

// The dynamic shared-memory base rounded up to 1024 bytes.  The offset comes
// from the 32-bit shared address and is added to the __shared__ array
// itself, so the compiler keeps every derived pointer in the shared window
// (shared-memory instructions, not generic ones).
__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return p + ((1024u - (smem_addr(p) & 1023u)) & 1023u);
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int x, int y,
                                             int z)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(src)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(src)), "r"(x), "r"(y)
                 : "memory");
}

// Prefetch one tensor tile into L2 (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap *map, int x, int y, int z)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap *map, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float (&f)[8])
{
    const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const float2 x = __bfloat1622float2(p[t]);
        f[2 * t] = x.x;
        f[2 * t + 1] = x.y;
    }
}

// x rounded to the nearest tf32 (10 explicit mantissa bits; ties away from
// zero) by integer arithmetic on its IEEE-754 bits, so that a tf32 operand
// holds exactly this value whatever rounding the tensor core applies.
// Finite inputs below the largest float.
__device__ __forceinline__ float tf32_round(float x)
{
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u);
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// ---- host side ----

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// S viewed as a 2-D fp32 matrix [B*H*128 rows][128 cols], boxes of 32 x 128.
inline cudaError_t make_state_map(CUtensorMap *map, const float *S, int units)
{
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)units * kD};
    cuuint64_t strides[1] = {(cuuint64_t)kD * sizeof(float)};
    cuuint32_t box[2] = {32, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(S), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The states of `layers` GDN layers, layer l at S + l * layer_stride floats, as
// a 3-D fp32 tensor [layers][B*H*128 rows][128 cols], boxes of 32 x 128 x 1.
// One layer needs no stride (any valid value serves).
inline cudaError_t make_layered_state_map(CUtensorMap *map, const float *S, int units, int layers,
                                          int64_t layer_stride)
{
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const uint64_t slice = (uint64_t)units * kD * kD * sizeof(float);
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)units * kD, (cuuint64_t)layers};
    cuuint64_t strides[2] = {(cuuint64_t)kD * sizeof(float),
                             layers > 1 ? (cuuint64_t)layer_stride * sizeof(float) : slice};
    cuuint32_t box[3] = {32, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(S), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Kernel attributes are per device and per function: set them on the first
// launch of each kernel on each device only (they do not change), so later
// calls -- and stream capture -- meet no attribute call.  Keyed by the
// kernel's address.
inline cudaError_t configure_once(const void *fn, int smem, bool carveout)
{
    static std::mutex mu;
    constexpr int kMaxKernels = 64;
    static const void *fns[kMaxKernels] = {};
    static uint64_t done[kMaxKernels] = {}; // bit = device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    std::lock_guard<std::mutex> lock(mu);
    int slot = -1;
    for (int i = 0; i < kMaxKernels; ++i) {
        if (fns[i] == fn) { slot = i; break; }
        if (fns[i] == nullptr) { fns[i] = fn; slot = i; break; }
    }
    if (slot >= 0 && bit && (done[slot] & bit)) return cudaSuccess;
    if (carveout) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess && slot >= 0) done[slot] |= bit;
    return e;
}

// Launch configuration; with `overlap` the kernel may start while the previous
// kernel on the stream drains (programmatic dependent launch).
inline cudaLaunchConfig_t launch_config(dim3 grid, dim3 block, int smem, cudaStream_t s, bool overlap,
                                 cudaLaunchAttribute (&attr)[1])
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    return cfg;
}

// q, k or v [N][H][128] as a 3-D tensor: bf16 in boxes of 64 elements x 1
// head x `rows` nodes, or (f32) fp32 in boxes of 32 elements x 1 x `rows` --
// 128-byte box rows either way.
inline cudaError_t make_node_map(CUtensorMap *map, const void *x, int N, int H, int rows,
                                 bool f32 = false)
{
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)N};
    cuuint64_t strides[2] = {(cuuint64_t)kD * es, (cuuint64_t)H * kD * es};
    cuuint32_t box[3] = {f32 ? 32u : 64u, 1, (cuuint32_t)rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                    const_cast<void *>(x), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

} // namespace tc
} // namespace bole
