// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bole.h"

namespace bole {

constexpr int kMaxTree = BOLE_MAX_TREE_NODES;

// First fault wins: {code, request, node, detail}.  Out of line (cold path).
static __device__ __noinline__ void report(int32_t *st, int code, int b, int i, int aux)
{
    if (atomicCAS(st, 0, code) == 0) {
        st[1] = b;
        st[2] = i;
        st[3] = aux;
    }
}

__device__ __forceinline__ bool faulted(const int32_t *st)
{
    return *(const volatile int32_t *)st != 0;
}

// Programmatic dependent launch: let the next kernel on the stream start
// (it still waits for this one before reading what this one writes), and
// wait for the previous kernel's completion and memory.  Both are no-ops for
// launches without a programmatic dependency.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x)
{
    return __bfloat162float(x);
}

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x)
{
    return __float2bfloat16_rn(x);
}

// ---- launchers (one per kernel family; each returns the launch error) ----

cudaError_t launch_selftest_wait(int32_t *st, uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_pack(const int32_t *offsets, const int32_t *parent, int B, int N, int max_depth,
                        int32_t *depth, uint32_t *anc, int32_t *req_depth, int32_t *st,
                        cudaStream_t s);

struct VerifyArgs {
    const float *S_pre;
    const void *q, *k, *v;
    bole_dtype dtype;
    const float *gamma, *beta;
    const int32_t *offsets, *parent, *depth;
    const uint32_t *anc;
    const int32_t *req_depth;
    int B, H, dk, dv, N, max_T, max_depth;
    void *O;
    float *U, *logP;
    void *ws;
    size_t ws_bytes;
    int32_t *st;
    bool vk; // state stored [B, H, dv, dk] (BOLE_FLAG_STATE_VK)
    bool inline_topo; // depth / anc / req_depth formed by the kernel from parent
};

// One commit launch over `layers` GDN layers: layer l's S, k, U and logP start
// l strides (in elements) after the pointers below.
struct CommitArgs {
    float *S;
    const void *k;
    bole_dtype dtype;
    const float *U, *logP;
    const int32_t *offsets, *parent, *accepted;
    int B, H, dk, dv, N;
    int32_t *st;
    int layers;
    int64_t s_ls, k_ls, u_ls, lp_ls;
    bool vk; // state stored [B, H, dv, dk] (BOLE_FLAG_STATE_VK)
};

// Stage 1: tree-parallel convolution and gates.
struct ConvGatesArgs {
    const void *x, *conv_state;
    const float *conv_w, *conv_b, *a, *b, *gate_scale, *gate_bias;
    bole_dtype dtype;
    const int32_t *offsets, *parent;
    int B, H, dk, dv, N, W, max_T;
    void *q, *k, *v;
    float *gamma, *beta;
    int32_t *st;
};
cudaError_t launch_conv_gates(const ConvGatesArgs &a, cudaStream_t s);
cudaError_t launch_conv_commit(void *conv_state, const void *x, bole_dtype dtype,
                               const int32_t *offsets, const int32_t *parent,
                               const int32_t *accepted, int B, int C, int W, int N, int32_t *st,
                               cudaStream_t s);

// Device-side selection and forest build.
size_t select_workspace_bytes(int B);
cudaError_t launch_select(const float *p, const int32_t *cand_offsets, const int32_t *cand_parent,
                          const int32_t *caps, int B, int M, int budget, int32_t *offsets,
                          int32_t *parent, int32_t *src, float *rho, void *ws, int32_t *st,
                          cudaStream_t s);

size_t simt_workspace_bytes(int B, int H, int max_T);
cudaError_t launch_simt_verify(const VerifyArgs &a, cudaStream_t s);
bool simt_noalloc_fits(int B, int H, int max_T);
cudaError_t launch_simt_verify_noalloc(const VerifyArgs &a, cudaStream_t s);
cudaError_t launch_simt_commit(const CommitArgs &a, cudaStream_t s);

bool tc_vtile_supported(const VerifyArgs &a);
bool tc_vtile_preferred(const VerifyArgs &a);
cudaError_t launch_tc_vtile_verify(const VerifyArgs &a, cudaStream_t s, bool overlap);
bool tc_verify_supported(const VerifyArgs &a);
size_t tc_workspace_bytes(int B, int H, int max_T);
cudaError_t launch_tc_verify(const VerifyArgs &a, cudaStream_t s, bool overlap);
// The previous round's commit inputs for the deferred commit (bole_commit_verify).
struct PrevArgs {
    const void *k;
    const float *U, *logP;
    const int32_t *offsets, *parent, *accepted;
    int N;
};
bool tc_commit_verify_supported(const VerifyArgs &a);
cudaError_t launch_tc_commit_verify(const VerifyArgs &a, const PrevArgs &p, cudaStream_t s);
bool tc_big_supported(const VerifyArgs &a);
size_t tc_big_workspace_bytes(int B, int H);
cudaError_t launch_tc_big_verify(const VerifyArgs &a, cudaStream_t s);
bool tc_commit_supported(const CommitArgs &a);
cudaError_t launch_tc_commit(const CommitArgs &a, cudaStream_t s, bool overlap);

} // namespace bole
