// C ABI: host-side validation, kernel choice and launches.  No entry point
// allocates memory or keeps state between calls.
#include <stdint.h>

#include "common.cuh"

using namespace bole;

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_dim(int d) { return d >= 16 && d <= 128 && d % 16 == 0; }

bool valid_dtype(bole_dtype t) { return t == BOLE_F32 || t == BOLE_BF16; }

// The CUDA error behind the calling thread's last BOLE_ERR_CUDA.
thread_local int g_last_cuda_error = 0;

bole_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess) return BOLE_OK;
    g_last_cuda_error = (int)e;
    return BOLE_ERR_CUDA;
}

// Verification kernels: the value-tiled tensor-core kernel (trees of up to
// 32 nodes, depth <= 15, two CTAs per head; bf16 where the batch's heads
// would leave the one-CTA kernel short of a wave, fp32 always), the
// single-CTA tensor-core kernel (bf16, trees of up to 64 nodes, depth <=
// 15), the large-tree tensor-core kernel for larger or deeper bf16 trees (up
// to 128 nodes), else the FP32 CUDA-core kernels.
enum class VerifyPath { VTile, Fused, Big, Simt };

VerifyPath verify_path(const VerifyArgs &a, unsigned flags)
{
    if (flags & BOLE_FLAG_FORCE_SIMT) return VerifyPath::Simt;
    if (!(flags & BOLE_FLAG_ONE_TILE_PER_HEAD) && tc_vtile_supported(a) &&
        ((flags & BOLE_FLAG_VALUE_TILES) || a.dtype == BOLE_F32 || tc_vtile_preferred(a)))
        return VerifyPath::VTile;
    if (tc_verify_supported(a)) return VerifyPath::Fused;
    if (tc_big_supported(a)) return VerifyPath::Big;
    return VerifyPath::Simt;
}

size_t verify_workspace(const VerifyArgs &a, unsigned flags)
{
    switch (verify_path(a, flags)) {
    case VerifyPath::VTile: return 0; // every factor stays on chip
    case VerifyPath::Fused: return tc_workspace_bytes(a.B, a.H, a.max_T);
    case VerifyPath::Big: return 0; // [M; W] stays on chip
    default: return simt_workspace_bytes(a.B, a.H, a.max_T);
    }
}

} // namespace

extern "C" {

const char *bole_status_string(int status)
{
    switch (status) {
    case BOLE_OK: return "ok";
    case BOLE_ERR_INVALID_ARG: return "invalid argument";
    case BOLE_ERR_UNSUPPORTED: return "unsupported configuration";
    case BOLE_ERR_BAD_TOPOLOGY: return "bad tree topology";
    case BOLE_ERR_DEPTH: return "tree deeper than max_depth";
    case BOLE_ERR_WORKSPACE: return "workspace missing or too small";
    case BOLE_ERR_CUDA: return "CUDA runtime error";
    case BOLE_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
    }
}

int bole_version(void) { return 100; }

int bole_last_cuda_error(void) { return g_last_cuda_error; }

const char *bole_last_cuda_error_string(void)
{
    return g_last_cuda_error ? cudaGetErrorString((cudaError_t)g_last_cuda_error) : "no error";
}

bole_status bole_selftest_wait(int32_t *dev_status, uint64_t limit_ns, bole_stream_t stream)
{
    if (!dev_status || !aligned(dev_status, 16) || limit_ns > BOLE_SELFTEST_MAX_WAIT_NS)
        return BOLE_ERR_INVALID_ARG;
    return from_cuda(
        launch_selftest_wait(dev_status, limit_ns, reinterpret_cast<cudaStream_t>(stream)));
}

size_t bole_workspace_size(int B, int H, int dk, int dv, int max_T, int max_depth,
                           bole_dtype qkv_dtype, unsigned flags)
{
    if (B < 0 || H < 1 || !valid_dim(dk) || !valid_dim(dv) || max_T < 1 ||
        max_T > BOLE_MAX_TREE_NODES || max_depth < 0 || max_depth > BOLE_MAX_TREE_NODES - 1 ||
        !valid_dtype(qkv_dtype))
        return 0;
    VerifyArgs a = {};
    a.dtype = qkv_dtype;
    a.vk = (flags & BOLE_FLAG_STATE_VK) != 0;
    a.B = B; a.H = H; a.dk = dk; a.dv = dv; a.max_T = max_T; a.max_depth = max_depth;
    return verify_workspace(a, flags);
}

bole_status bole_pack_forest(const int32_t *offsets, const int32_t *parent, int B, int N,
                             int max_depth, int32_t *depth, uint32_t *anc, int32_t *req_depth,
                             int32_t *dev_status, bole_stream_t stream)
{
    if (B < 0 || N < 0 || max_depth < 0 || max_depth > BOLE_MAX_TREE_NODES - 1)
        return BOLE_ERR_INVALID_ARG;
    if (!offsets || !dev_status || (B > 0 && !req_depth)) return BOLE_ERR_INVALID_ARG;
    if (N > 0 && (!parent || !depth || !anc)) return BOLE_ERR_INVALID_ARG;
    if ((size_t)N > (size_t)B * BOLE_MAX_TREE_NODES) return BOLE_ERR_INVALID_ARG;
    if (!aligned(anc, 16) || !aligned(offsets, 4) || !aligned(parent, 4) || !aligned(depth, 4) ||
        !aligned(req_depth, 4) || !aligned(dev_status, 16))
        return BOLE_ERR_INVALID_ARG;
    return from_cuda(launch_pack(offsets, parent, B, N, max_depth, depth, anc, req_depth,
                                 dev_status, reinterpret_cast<cudaStream_t>(stream)));
}

bole_status bole_tree_verify(const float *S_pre, const void *q, const void *k, const void *v,
                             bole_dtype qkv_dtype, const float *gamma, const float *beta,
                             const int32_t *offsets, const int32_t *parent, const int32_t *depth,
                             const uint32_t *anc, const int32_t *req_depth, int B, int H, int dk,
                             int dv, int N, int max_T, int max_depth, void *O, float *U,
                             float *logP, void *workspace, size_t workspace_bytes,
                             int32_t *dev_status, unsigned flags, bole_stream_t stream)
{
    if (B < 0 || N < 0 || H < 1 || !valid_dim(dk) || !valid_dim(dv) || !valid_dtype(qkv_dtype))
        return BOLE_ERR_INVALID_ARG;
    if (max_T < 1 || max_T > BOLE_MAX_TREE_NODES || max_depth < 0 ||
        max_depth > BOLE_MAX_TREE_NODES - 1)
        return BOLE_ERR_INVALID_ARG;
    if ((size_t)N > (size_t)B * max_T) return BOLE_ERR_INVALID_ARG;
    // with the topology formed in the kernel, depth / anc / req_depth are unused
    const bool inl = (flags & BOLE_FLAG_INLINE_TOPOLOGY) != 0;
    if (!offsets || !dev_status || (B > 0 && (!S_pre || (!inl && !req_depth))))
        return BOLE_ERR_INVALID_ARG;
    if (N > 0 && (!q || !k || !v || !gamma || !beta || !parent || (!inl && (!depth || !anc)) ||
                  !O || !U || !logP))
        return BOLE_ERR_INVALID_ARG;
    const void *p16[] = {S_pre, q, k, v, O, U, anc, dev_status};
    for (const void *p : p16)
        if (!aligned(p, 16)) return BOLE_ERR_INVALID_ARG;
    const void *p4[] = {gamma, beta, offsets, parent, depth, req_depth, logP};
    for (const void *p : p4)
        if (!aligned(p, 4)) return BOLE_ERR_INVALID_ARG;

    VerifyArgs a;
    a.S_pre = S_pre; a.q = q; a.k = k; a.v = v; a.dtype = qkv_dtype;
    a.gamma = gamma; a.beta = beta;
    a.offsets = offsets; a.parent = parent; a.depth = depth; a.anc = anc; a.req_depth = req_depth;
    a.B = B; a.H = H; a.dk = dk; a.dv = dv; a.N = N; a.max_T = max_T; a.max_depth = max_depth;
    a.O = O; a.U = U; a.logP = logP; a.ws = workspace; a.ws_bytes = workspace ? workspace_bytes : 0;
    a.st = dev_status;
    a.vk = (flags & BOLE_FLAG_STATE_VK) != 0;
    a.inline_topo = inl;

    const VerifyPath path = verify_path(a, flags);
    if (inl && path != VerifyPath::VTile && path != VerifyPath::Fused)
        return BOLE_ERR_UNSUPPORTED; // these kernels read the masks bole_pack_forest builds
    const size_t need = verify_workspace(a, flags);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16)))
        return BOLE_ERR_WORKSPACE;
    if (B == 0 || N == 0) return BOLE_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (path) {
    case VerifyPath::VTile:
        return from_cuda(launch_tc_vtile_verify(a, s, (flags & BOLE_FLAG_OVERLAP_LAUNCH) != 0));
    case VerifyPath::Fused:
        return from_cuda(launch_tc_verify(a, s, (flags & BOLE_FLAG_OVERLAP_LAUNCH) != 0));
    case VerifyPath::Big: return from_cuda(launch_tc_big_verify(a, s));
    default: return from_cuda(launch_simt_verify(a, s));
    }
}

bole_status bole_tree_verify_noalloc(const float *S_pre, const void *q, const void *k,
                                     const void *v, bole_dtype qkv_dtype, const float *gamma,
                                     const float *beta, const int32_t *offsets,
                                     const int32_t *parent, const int32_t *depth,
                                     const uint32_t *anc, const int32_t *req_depth, int B, int H,
                                     int dk, int dv, int N, int max_T, int max_depth, void *O,
                                     float *U, float *logP, int32_t *dev_status,
                                     bole_stream_t stream)
{
    if (B < 0 || N < 0 || H < 1 || !valid_dim(dk) || !valid_dim(dv) || !valid_dtype(qkv_dtype))
        return BOLE_ERR_INVALID_ARG;
    if (max_T < 1 || max_T > BOLE_MAX_TREE_NODES || max_depth < 0 ||
        max_depth > BOLE_MAX_TREE_NODES - 1)
        return BOLE_ERR_INVALID_ARG;
    if ((size_t)N > (size_t)B * max_T) return BOLE_ERR_INVALID_ARG;
    if (!offsets || !dev_status || (B > 0 && (!S_pre || !req_depth))) return BOLE_ERR_INVALID_ARG;
    if (N > 0 && (!q || !k || !v || !gamma || !beta || !parent || !depth || !anc || !O || !U ||
                  !logP))
        return BOLE_ERR_INVALID_ARG;
    const void *p16[] = {S_pre, q, k, v, O, U, anc, dev_status};
    for (const void *p : p16)
        if (!aligned(p, 16)) return BOLE_ERR_INVALID_ARG;
    const void *p4[] = {gamma, beta, offsets, parent, depth, req_depth, logP};
    for (const void *p : p4)
        if (!aligned(p, 4)) return BOLE_ERR_INVALID_ARG;
    if (!simt_noalloc_fits(B, H, max_T)) return BOLE_ERR_UNSUPPORTED;
    if (B == 0 || N == 0) return BOLE_OK;

    VerifyArgs a;
    a.S_pre = S_pre; a.q = q; a.k = k; a.v = v; a.dtype = qkv_dtype;
    a.gamma = gamma; a.beta = beta;
    a.offsets = offsets; a.parent = parent; a.depth = depth; a.anc = anc; a.req_depth = req_depth;
    a.B = B; a.H = H; a.dk = dk; a.dv = dv; a.N = N; a.max_T = max_T; a.max_depth = max_depth;
    a.O = O; a.U = U; a.logP = logP; a.ws = nullptr; a.ws_bytes = 0; a.st = dev_status;
    a.vk = false;
    a.inline_topo = false;
    return from_cuda(launch_simt_verify_noalloc(a, reinterpret_cast<cudaStream_t>(stream)));
}

bole_status bole_commit_layers(float *S, int64_t s_layer_stride, const void *k,
                               int64_t k_layer_stride, bole_dtype k_dtype, const float *U,
                               int64_t u_layer_stride, const float *logP, int64_t lp_layer_stride,
                               const int32_t *offsets, const int32_t *parent,
                               const int32_t *accepted, int n_layers, int B, int H, int dk, int dv,
                               int N, int32_t *dev_status, unsigned flags, bole_stream_t stream)
{
    if (B < 0 || N < 0 || H < 1 || !valid_dim(dk) || !valid_dim(dv) || !valid_dtype(k_dtype))
        return BOLE_ERR_INVALID_ARG;
    if (n_layers < 0 || n_layers > 65535) return BOLE_ERR_INVALID_ARG;
    if ((size_t)N > (size_t)B * BOLE_MAX_TREE_NODES) return BOLE_ERR_INVALID_ARG;
    if (!offsets || !dev_status || (B > 0 && n_layers > 0 && (!S || !accepted)))
        return BOLE_ERR_INVALID_ARG;
    if (N > 0 && n_layers > 0 && (!k || !U || !logP || !parent)) return BOLE_ERR_INVALID_ARG;
    const void *p16[] = {S, k, U, dev_status};
    for (const void *p : p16)
        if (!aligned(p, 16)) return BOLE_ERR_INVALID_ARG;
    const void *p4[] = {logP, offsets, parent, accepted};
    for (const void *p : p4)
        if (!aligned(p, 4)) return BOLE_ERR_INVALID_ARG;
    // Layer strides: none negative; state slices disjoint (each layer writes
    // its own in place); every slice as aligned as the first.
    const int64_t ksize = k_dtype == BOLE_BF16 ? 2 : 4;
    if (s_layer_stride < 0 || k_layer_stride < 0 || u_layer_stride < 0 || lp_layer_stride < 0)
        return BOLE_ERR_INVALID_ARG;
    if (n_layers > 1 && s_layer_stride < (int64_t)B * H * dk * dv) return BOLE_ERR_INVALID_ARG;
    if ((s_layer_stride * 4) % 16 != 0 || (k_layer_stride * ksize) % 16 != 0 ||
        (u_layer_stride * 4) % 16 != 0)
        return BOLE_ERR_INVALID_ARG;
    if (B == 0 || N == 0 || n_layers == 0) return BOLE_OK;

    CommitArgs a;
    a.S = S; a.k = k; a.dtype = k_dtype; a.U = U; a.logP = logP;
    a.offsets = offsets; a.parent = parent; a.accepted = accepted;
    a.B = B; a.H = H; a.dk = dk; a.dv = dv; a.N = N; a.st = dev_status;
    a.layers = n_layers;
    a.s_ls = s_layer_stride; a.k_ls = k_layer_stride; a.u_ls = u_layer_stride;
    a.lp_ls = lp_layer_stride;
    a.vk = (flags & BOLE_FLAG_STATE_VK) != 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool tc = !(flags & BOLE_FLAG_FORCE_SIMT) && tc_commit_supported(a);
    return from_cuda(tc ? launch_tc_commit(a, s, (flags & BOLE_FLAG_OVERLAP_LAUNCH) != 0)
                        : launch_simt_commit(a, s));
}

bole_status bole_commit(float *S, const void *k, bole_dtype k_dtype, const float *U,
                        const float *logP, const int32_t *offsets, const int32_t *parent,
                        const int32_t *accepted, int B, int H, int dk, int dv, int N,
                        int32_t *dev_status, unsigned flags, bole_stream_t stream)
{
    return bole_commit_layers(S, 0, k, 0, k_dtype, U, 0, logP, 0, offsets, parent, accepted, 1, B,
                              H, dk, dv, N, dev_status, flags, stream);
}

bole_status bole_commit_verify(float *S, const void *k_prev, const float *U_prev,
                               const float *logP_prev, const int32_t *offsets_prev,
                               const int32_t *parent_prev, const int32_t *accepted_prev,
                               int N_prev, const void *q, const void *k, const void *v,
                               bole_dtype qkv_dtype, const float *gamma, const float *beta,
                               const int32_t *offsets, const int32_t *parent, int B, int H,
                               int dk, int dv, int N, int max_T, int max_depth, void *O, float *U,
                               float *logP, int32_t *dev_status, unsigned flags,
                               bole_stream_t stream)
{
    if (B < 0 || N < 0 || N_prev < 0 || H < 1 || !valid_dim(dk) || !valid_dim(dv) ||
        !valid_dtype(qkv_dtype))
        return BOLE_ERR_INVALID_ARG;
    if (max_T < 1 || max_T > BOLE_MAX_TREE_NODES || max_depth < 0 ||
        max_depth > BOLE_MAX_TREE_NODES - 1)
        return BOLE_ERR_INVALID_ARG;
    if ((size_t)N > (size_t)B * max_T || (size_t)N_prev > (size_t)B * BOLE_MAX_TREE_NODES)
        return BOLE_ERR_INVALID_ARG;
    if (flags & ~(unsigned)BOLE_FLAG_OVERLAP_LAUNCH) return BOLE_ERR_INVALID_ARG;
    if (!offsets || !offsets_prev || !accepted_prev || !dev_status || (B > 0 && !S))
        return BOLE_ERR_INVALID_ARG;
    if (N > 0 && (!q || !k || !v || !gamma || !beta || !parent || !O || !U || !logP))
        return BOLE_ERR_INVALID_ARG;
    if (N_prev > 0 && (!k_prev || !U_prev || !logP_prev || !parent_prev))
        return BOLE_ERR_INVALID_ARG;
    // this round's outputs must not overwrite the previous round's factors
    if (N > 0 && N_prev > 0 && (U == U_prev || logP == logP_prev)) return BOLE_ERR_INVALID_ARG;
    const void *p16[] = {S, q, k, v, O, U, k_prev, U_prev, dev_status};
    for (const void *p : p16)
        if (!aligned(p, 16)) return BOLE_ERR_INVALID_ARG;
    const void *p4[] = {gamma, beta, offsets, parent, logP, logP_prev, offsets_prev, parent_prev,
                        accepted_prev};
    for (const void *p : p4)
        if (!aligned(p, 4)) return BOLE_ERR_INVALID_ARG;

    VerifyArgs a = {};
    a.S_pre = S; a.q = q; a.k = k; a.v = v; a.dtype = qkv_dtype;
    a.gamma = gamma; a.beta = beta; a.offsets = offsets; a.parent = parent;
    a.B = B; a.H = H; a.dk = dk; a.dv = dv; a.N = N; a.max_T = max_T; a.max_depth = max_depth;
    a.O = O; a.U = U; a.logP = logP; a.st = dev_status;
    a.vk = false;
    a.inline_topo = true;
    if (!tc_commit_verify_supported(a)) return BOLE_ERR_UNSUPPORTED;
    if (B == 0 || (N == 0 && N_prev == 0)) return BOLE_OK;
    PrevArgs pr;
    pr.k = k_prev; pr.U = U_prev; pr.logP = logP_prev;
    pr.offsets = offsets_prev; pr.parent = parent_prev; pr.accepted = accepted_prev;
    pr.N = N_prev;
    return from_cuda(launch_tc_commit_verify(a, pr, reinterpret_cast<cudaStream_t>(stream)));
}

size_t bole_select_workspace_size(int B)
{
    if (B < 0 || B > BOLE_SELECT_MAX_REQUESTS) return 0;
    return select_workspace_bytes(B);
}

bole_status bole_select_forest(const float *p, const int32_t *cand_offsets,
                               const int32_t *cand_parent, const int32_t *caps, int B, int M,
                               int budget, int32_t *offsets, int32_t *parent, int32_t *src,
                               float *rho, void *workspace, size_t workspace_bytes,
                               int32_t *dev_status, unsigned flags, bole_stream_t stream)
{
    (void)flags;
    if (B < 0 || B > BOLE_SELECT_MAX_REQUESTS || M < 0 || budget < 0)
        return BOLE_ERR_INVALID_ARG;
    if (!cand_offsets || !offsets || !dev_status) return BOLE_ERR_INVALID_ARG;
    if (M > 0 && (!p || !cand_parent)) return BOLE_ERR_INVALID_ARG;
    if (budget > 0 && (!parent || !src)) return BOLE_ERR_INVALID_ARG;
    const void *p4[] = {p, cand_offsets, cand_parent, caps, offsets, parent, src, rho};
    for (const void *q : p4)
        if (!aligned(q, 4)) return BOLE_ERR_INVALID_ARG;
    if (!aligned(dev_status, 16)) return BOLE_ERR_INVALID_ARG;
    const size_t need = select_workspace_bytes(B);
    if (B > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16)))
        return BOLE_ERR_WORKSPACE;
    return from_cuda(launch_select(p, cand_offsets, cand_parent, caps, B, M, budget, offsets,
                                   parent, src, rho, workspace, dev_status,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

bole_status bole_conv_gates(const void *x, const void *conv_state, const float *conv_w,
                            const float *conv_b, const float *a, const float *b,
                            const float *gate_scale, const float *gate_bias, bole_dtype x_dtype,
                            const int32_t *offsets, const int32_t *parent, int B, int H, int dk,
                            int dv, int N, int max_T, int W, void *q, void *k, void *v,
                            float *gamma, float *beta, int32_t *dev_status, unsigned flags,
                            bole_stream_t stream)
{
    (void)flags;
    if (B < 0 || N < 0 || H < 1 || !valid_dim(dk) || !valid_dim(dv) || !valid_dtype(x_dtype))
        return BOLE_ERR_INVALID_ARG;
    if (W < 1 || W > BOLE_MAX_CONV_WIDTH) return BOLE_ERR_INVALID_ARG;
    if (max_T < 1 || max_T > BOLE_MAX_TREE_NODES) return BOLE_ERR_INVALID_ARG;
    if ((size_t)N > (size_t)B * max_T) return BOLE_ERR_INVALID_ARG;
    if (!offsets || !dev_status) return BOLE_ERR_INVALID_ARG;
    if (N > 0 && (!x || !conv_w || !a || !b || !parent || !q || !k || !v || !gamma || !beta ||
                  (W > 1 && !conv_state)))
        return BOLE_ERR_INVALID_ARG;
    const void *p16[] = {x, conv_state, conv_w, q, k, v, dev_status};
    for (const void *p : p16)
        if (!aligned(p, 16)) return BOLE_ERR_INVALID_ARG;
    const void *p4[] = {conv_b, a, b, gate_scale, gate_bias, offsets, parent, gamma, beta};
    for (const void *p : p4)
        if (!aligned(p, 4)) return BOLE_ERR_INVALID_ARG;
    if (B == 0 || N == 0) return BOLE_OK;
    ConvGatesArgs g;
    g.x = x; g.conv_state = conv_state; g.conv_w = conv_w; g.conv_b = conv_b; g.a = a; g.b = b;
    g.gate_scale = gate_scale; g.gate_bias = gate_bias; g.dtype = x_dtype;
    g.offsets = offsets; g.parent = parent;
    g.B = B; g.H = H; g.dk = dk; g.dv = dv; g.N = N; g.W = W; g.max_T = max_T;
    g.q = q; g.k = k; g.v = v; g.gamma = gamma; g.beta = beta; g.st = dev_status;
    return from_cuda(launch_conv_gates(g, reinterpret_cast<cudaStream_t>(stream)));
}

bole_status bole_conv_commit(void *conv_state, const void *x, bole_dtype x_dtype,
                             const int32_t *offsets, const int32_t *parent,
                             const int32_t *accepted, int B, int C, int W, int N,
                             int32_t *dev_status, unsigned flags, bole_stream_t stream)
{
    (void)flags;
    if (B < 0 || B > 65535 || N < 0 || C < 1 || C % 16 != 0 || W < 1 ||
        W > BOLE_MAX_CONV_WIDTH || !valid_dtype(x_dtype))
        return BOLE_ERR_INVALID_ARG;
    if ((size_t)N > (size_t)B * BOLE_MAX_TREE_NODES) return BOLE_ERR_INVALID_ARG;
    if (!offsets || !dev_status || (B > 0 && W > 1 && (!conv_state || !accepted)))
        return BOLE_ERR_INVALID_ARG;
    if (N > 0 && W > 1 && (!x || !parent)) return BOLE_ERR_INVALID_ARG;
    const void *p16[] = {conv_state, x, dev_status};
    for (const void *p : p16)
        if (!aligned(p, 16)) return BOLE_ERR_INVALID_ARG;
    const void *p4[] = {offsets, parent, accepted};
    for (const void *p : p4)
        if (!aligned(p, 4)) return BOLE_ERR_INVALID_ARG;
    if (B == 0 || N == 0 || W == 1) return BOLE_OK;
    return from_cuda(launch_conv_commit(conv_state, x, x_dtype, offsets, parent, accepted, B, C,
                                        W, N, dev_status,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

} // extern "C"
