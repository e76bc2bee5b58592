// FP32 CUDA-core path of the verification and the commit.
//
// It follows the pages' own kernel organisation ("Bole", Section IV-B/IV-C):
// a per-(request, head) producer builds the tree factors G and C into a
// short-lived workspace, and value-tiled CTAs each take b_v = 32 columns of
// S_pre and V, form R, run the d-step Neumann recurrence of Eq. (8) on chip
// and read out O = B0 + C U (Eq. (7)).  Every product is an FP32 FMA, so the
// path meets float32 accuracy; it serves float32 inputs and any shape the
// tensor-core kernels do not cover.
#include <mutex>

#include "common.cuh"

namespace bole {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTileV = 32; // b_v: value columns per solve CTA (one per lane)

__device__ __forceinline__ bool is_anc(const uint32_t *m, int j)
{
    return (m[j >> 5] >> (j & 31)) & 1u;
}

// Cumulative decay along parent links, L_i = log P_i = sum of log gamma over
// the ancestors-or-self of i (Lemma 1), by pointer jumping: after round s
// every node has summed its 2^s nearest path entries.  T <= 128 nodes.
__device__ void cumulative_log_decay(const float *__restrict__ gamma, const int32_t *__restrict__ parent,
                                     int o, int T, int H, int h, float *Ls, int *up)
{
    for (int i = threadIdx.x; i < T; i += blockDim.x) {
        Ls[i] = logf(gamma[(size_t)(o + i) * H + h]);
        up[i] = parent[o + i];
    }
    __syncthreads();
    for (int round = 0; round < 8; ++round) {
        float nl = 0.f;
        int nu = -1;
        const bool mine = threadIdx.x < T;
        bool active = false;
        if (mine) {
            const int a = up[threadIdx.x];
            active = a >= 0;
            nl = Ls[threadIdx.x] + (active ? Ls[a] : 0.f);
            nu = active ? up[a] : -1;
        }
        if (!__syncthreads_or(active)) break;
        if (mine) {
            Ls[threadIdx.x] = nl;
            up[threadIdx.x] = nu;
        }
        __syncthreads();
    }
}

// Producer: one CTA per (request, head).  Writes logP and the dense masked
// factors (Lemma 2 and the read-out of Lemma 1):
//   G_ij = beta_i exp(L_i - L_j) k_i.k_j   for j a strict ancestor of i
//   C_ij = exp(L_i - L_j) q_i.k_j          for j an ancestor of i or i itself
// Row-major [max_T][max_T] per unit in the workspace; other entries are 0.
// The exponent L_i - L_j <= 0 for an ancestor, and the factor is selected,
// never multiplied by a 0/1 mask, so an underflowed decay cannot give 0 * inf.
template <typename T>
__global__ void __launch_bounds__(kThreads) simt_factor_kernel(
    const T *__restrict__ q, const T *__restrict__ k, const float *__restrict__ gamma,
    const float *__restrict__ beta, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ parent, const uint32_t *__restrict__ anc, int H, int dk, int N,
    int max_T, float *__restrict__ logP, float *__restrict__ wsG, float *__restrict__ wsC,
    int32_t *st)
{
    __shared__ float Ls[kMaxTree];
    __shared__ int up[kMaxTree];
    const int unit = blockIdx.x;
    const int b = unit / H, h = unit % H;
    const bool prior_fault = faulted(st);
    const int o = offsets[b], Tn = offsets[b + 1] - o;
    if (__syncthreads_or(prior_fault)) return; // taken by the whole CTA
    if (Tn <= 0) return;
    if (Tn > max_T || o < 0 || o + Tn > N) {
        if (threadIdx.x == 0) report(st, BOLE_ERR_BAD_TOPOLOGY, b, -1, Tn);
        return;
    }
    cumulative_log_decay(gamma, parent, o, Tn, H, h, Ls, up);
    for (int i = threadIdx.x; i < Tn; i += blockDim.x) logP[(size_t)(o + i) * H + h] = Ls[i];

    float *G = wsG + (size_t)unit * max_T * max_T;
    float *C = wsC + (size_t)unit * max_T * max_T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = warp; i < max_T; i += kWarps) {
        uint32_t m[4] = {0u, 0u, 0u, 0u};
        float bi = 0.f, Li = 0.f;
        if (i < Tn) {
            const uint4 mm = *reinterpret_cast<const uint4 *>(anc + (size_t)(o + i) * 4);
            m[0] = mm.x; m[1] = mm.y; m[2] = mm.z; m[3] = mm.w;
            bi = beta[(size_t)(o + i) * H + h];
            Li = Ls[i];
        }
        const T *qi = q + ((size_t)(o + min(i, Tn - 1)) * H + h) * dk;
        const T *ki = k + ((size_t)(o + min(i, Tn - 1)) * H + h) * dk;
        for (int j = lane; j < max_T; j += 32) {
            float g = 0.f, c = 0.f;
            if (i < Tn && j <= i && is_anc(m, j)) {
                const T *kj = k + ((size_t)(o + j) * H + h) * dk;
                float qk = 0.f, kk = 0.f;
                for (int r = 0; r < dk; ++r) {
                    const float kjr = to_f32(kj[r]);
                    qk = fmaf(to_f32(qi[r]), kjr, qk);
                    kk = fmaf(to_f32(ki[r]), kjr, kk);
                }
                const float ratio = expf(Li - Ls[j]);
                c = ratio * qk;
                if (j != i) g = bi * ratio * kk;
            }
            G[(size_t)i * max_T + j] = g;
            C[(size_t)i * max_T + j] = c;
        }
    }
}

// Value-tiled solve: one CTA per (request, head, value tile of 32 columns).
// Lane = value column; warps stride over nodes.
//   B0 = D_P (Q S_pre^(r)),  R = D_beta (V^(r) - D_P (K S_pre^(r)))   (Eq. (7))
//   Z <- -G Z, U += Z for d steps (Eq. (8)), then O = B0 + C U.
// VK: the state is stored transposed ([dv][dk] per head, the slot layout).
template <typename T, bool VK>
__global__ void __launch_bounds__(kThreads) simt_solve_kernel(
    const float *__restrict__ S_pre, const T *__restrict__ q, const T *__restrict__ k,
    const T *__restrict__ v, const float *__restrict__ beta, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ req_depth, int H, int dk, int dv, int N, int max_T,
    const float *__restrict__ logP, const float *__restrict__ wsG, const float *__restrict__ wsC,
    T *__restrict__ O, float *__restrict__ Uout, int32_t *st)
{
    extern __shared__ float smem[];
    const int unit = blockIdx.x;
    const int b = unit / H, h = unit % H;
    const int c0 = blockIdx.y * kTileV;
    const bool prior_fault = faulted(st);
    const int o = offsets[b], Tn = offsets[b + 1] - o;
    if (__syncthreads_or(prior_fault)) return; // taken by the whole CTA
    if (Tn <= 0 || Tn > max_T || o < 0 || o + Tn > N) return; // reported by the producer
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool col_ok = c0 + lane < dv;

    float *Gs = smem;                        // [Tn][Tn]
    float *Ss = Gs + Tn * Tn;                // [dk][32]
    float *B0 = Ss + dk * kTileV;            // [Tn][32]
    float *Za = B0 + Tn * kTileV;            // [Tn][32]
    float *Zb = Za + Tn * kTileV;            // [Tn][32]
    float *Us = Zb + Tn * kTileV;            // [Tn][32]
    float *Pv = Us + Tn * kTileV;            // [Tn]
    float *Bv = Pv + Tn;                     // [Tn]

    const float *G = wsG + (size_t)unit * max_T * max_T;
    const float *C = wsC + (size_t)unit * max_T * max_T;
    for (int e = threadIdx.x; e < Tn * Tn; e += blockDim.x)
        Gs[e] = G[(size_t)(e / Tn) * max_T + (e % Tn)];
    const float *S = S_pre + (size_t)unit * dk * dv;
    for (int e = threadIdx.x; e < dk * kTileV; e += blockDim.x) {
        // consecutive threads read consecutive addresses in either layout
        const int r = VK ? e % dk : e / kTileV, c = VK ? e / dk : e % kTileV;
        Ss[r * kTileV + c] = (c0 + c < dv)
                                 ? S[VK ? (size_t)(c0 + c) * dk + r : (size_t)r * dv + c0 + c]
                                 : 0.f;
    }
    for (int i = threadIdx.x; i < Tn; i += blockDim.x) {
        Pv[i] = expf(logP[(size_t)(o + i) * H + h]);
        Bv[i] = beta[(size_t)(o + i) * H + h];
    }
    __syncthreads();

    for (int i = warp; i < Tn; i += kWarps) {
        const T *qi = q + ((size_t)(o + i) * H + h) * dk;
        const T *ki = k + ((size_t)(o + i) * H + h) * dk;
        float qs = 0.f, ks = 0.f;
        for (int r = 0; r < dk; ++r) {
            const float s = Ss[r * kTileV + lane];
            qs = fmaf(to_f32(qi[r]), s, qs);
            ks = fmaf(to_f32(ki[r]), s, ks);
        }
        const float vi = col_ok ? to_f32(v[((size_t)(o + i) * H + h) * dv + c0 + lane]) : 0.f;
        const float R = Bv[i] * (vi - Pv[i] * ks);
        B0[i * kTileV + lane] = Pv[i] * qs;
        Za[i * kTileV + lane] = R;
        Us[i * kTileV + lane] = R;
    }
    __syncthreads();

    const int d = min(req_depth[b], Tn - 1);
    float *Z = Za, *Zn = Zb;
    for (int m = 0; m < d; ++m) {
        for (int i = warp; i < Tn; i += kWarps) {
            float acc = 0.f;
            for (int j = 0; j < i; ++j) acc = fmaf(Gs[i * Tn + j], Z[j * kTileV + lane], acc);
            Zn[i * kTileV + lane] = -acc;
        }
        __syncthreads();
        for (int i = warp; i < Tn; i += kWarps) Us[i * kTileV + lane] += Zn[i * kTileV + lane];
        float *t = Z; Z = Zn; Zn = t;
        __syncthreads();
    }

    for (int i = warp; i < Tn; i += kWarps) {
        float acc = B0[i * kTileV + lane];
        const float *Ci = C + (size_t)i * max_T;
        for (int j = 0; j <= i; ++j) acc = fmaf(Ci[j], Us[j * kTileV + lane], acc);
        if (col_ok) {
            const size_t off = ((size_t)(o + i) * H + h) * dv + c0 + lane;
            O[off] = from_f32<T>(acc);
            Uout[off] = Us[i * kTileV + lane];
        }
    }
}

// Commit (Eq. (10)): one CTA per (request, head, block of 32 state rows,
// layer).  S[r][c] <- P_a S[r][c] + sum_t exp(L_a - L_{j_t}) k_{j_t}[r] u_{j_t}[c],
// the sum running over the accepted path j_t (root child .. a).  Layer l's
// buffers start l strides after the base pointers; with VK the state is
// stored transposed (element (r, c) at c * dk + r).
constexpr int kCommitRows = 32;
constexpr int kPathChunk = 32;

template <typename T, bool VK>
__global__ void __launch_bounds__(kThreads) simt_commit_kernel(
    float *__restrict__ S, const T *__restrict__ k, const float *__restrict__ U,
    const float *__restrict__ logP, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ parent, const int32_t *__restrict__ accepted, int H, int dk,
    int dv, int N, int64_t s_ls, int64_t k_ls, int64_t u_ls, int64_t lp_ls, int32_t *st)
{
    __shared__ int path[kMaxTree];
    __shared__ float coef[kMaxTree];
    __shared__ int path_len;
    __shared__ float ks[kPathChunk][kCommitRows];
    __shared__ float us[kPathChunk][128];
    const int unit = blockIdx.x;
    const int b = unit / H, h = unit % H;
    const int r0 = blockIdx.y * kCommitRows;
    const int layer = blockIdx.z;
    S += layer * s_ls;
    k += layer * k_ls;
    U += layer * u_ls;
    logP += layer * lp_ls;
    const bool prior_fault = faulted(st);
    const int a = accepted[b];
    const int o = offsets[b], Tn = offsets[b + 1] - o;
    if (__syncthreads_or(prior_fault)) return; // taken by the whole CTA
    if (a < 0) return;
    if (a >= Tn || o < 0 || o + Tn > N || Tn > kMaxTree) {
        if (threadIdx.x == 0) report(st, BOLE_ERR_BAD_TOPOLOGY, b, a, Tn);
        return;
    }
    if (threadIdx.x == 0) {
        int L = 0, j = a;
        bool ok = true;
        while (j >= 0) {
            if (L >= kMaxTree) { ok = false; break; }
            path[L++] = j;
            const int p = parent[o + j];
            if (p < -1 || p >= j) { ok = false; break; }
            j = p;
        }
        if (!ok) {
            report(st, BOLE_ERR_BAD_TOPOLOGY, b, j, -1);
            L = -1;
        }
        path_len = L;
    }
    __syncthreads();
    const int L = path_len;
    if (L < 0) return;
    const float La = logP[(size_t)(o + a) * H + h];
    for (int t = threadIdx.x; t < L; t += blockDim.x)
        coef[t] = expf(La - logP[(size_t)(o + path[t]) * H + h]);
    const float Pa = expf(La);
    const int rows = min(kCommitRows, dk - r0);
    float *Su = S + (size_t)unit * dk * dv;
    constexpr int kPer = kCommitRows * 128 / kThreads; // 16 elements per thread
    // element idx of the tile: (row rr, column c), consecutive threads on
    // consecutive addresses in either layout
    auto elem = [&](int idx, int &rr, int &c) {
        rr = VK ? idx % kCommitRows : idx / dv;
        c = VK ? idx / kCommitRows : idx % dv;
        return rr < rows && c < dv;
    };
    auto at = [&](int rr, int c) -> size_t {
        return VK ? (size_t)c * dk + r0 + rr : (size_t)(r0 + rr) * dv + c;
    };
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
        int rr, c;
        acc[e] = elem(threadIdx.x + e * kThreads, rr, c) ? Pa * Su[at(rr, c)] : 0.f;
    }
    __syncthreads();
    for (int t0 = 0; t0 < L; t0 += kPathChunk) {
        const int n = min(kPathChunk, L - t0);
        for (int e = threadIdx.x; e < n * kCommitRows; e += blockDim.x) {
            const int t = e / kCommitRows, rr = e % kCommitRows;
            const int j = path[t0 + t];
            ks[t][rr] = (rr < rows)
                            ? coef[t0 + t] * to_f32(k[((size_t)(o + j) * H + h) * dk + r0 + rr])
                            : 0.f;
        }
        for (int e = threadIdx.x; e < n * dv; e += blockDim.x) {
            const int t = e / dv, c = e % dv;
            us[t][c] = U[((size_t)(o + path[t0 + t]) * H + h) * dv + c];
        }
        __syncthreads();
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            int rr, c;
            if (elem(threadIdx.x + e * kThreads, rr, c)) {
                float s = acc[e];
                for (int t = 0; t < n; ++t) s = fmaf(ks[t][rr], us[t][c], s);
                acc[e] = s;
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
        int rr, c;
        if (elem(threadIdx.x + e * kThreads, rr, c)) Su[at(rr, c)] = acc[e];
    }
}

size_t solve_smem_bytes(int Tn, int dk)
{
    return sizeof(float) * ((size_t)Tn * Tn + (size_t)dk * kTileV + 4 * (size_t)Tn * kTileV + 2 * Tn);
}

template <typename T, bool VK> cudaError_t verify_typed(const VerifyArgs &a, cudaStream_t s)
{
    const size_t unit_ws = (size_t)a.max_T * a.max_T;
    float *wsG = static_cast<float *>(a.ws);
    float *wsC = wsG + (size_t)a.B * a.H * unit_ws;
    const int units = a.B * a.H;
    simt_factor_kernel<T><<<units, kThreads, 0, s>>>(
        static_cast<const T *>(a.q), static_cast<const T *>(a.k), a.gamma, a.beta, a.offsets,
        a.parent, a.anc, a.H, a.dk, a.N, a.max_T, a.logP, wsG, wsC, a.st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = solve_smem_bytes(a.max_T, a.dk);
    e = cudaFuncSetAttribute(simt_solve_kernel<T, VK>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(units, (a.dv + kTileV - 1) / kTileV);
    simt_solve_kernel<T, VK><<<grid, kThreads, smem, s>>>(
        a.S_pre, static_cast<const T *>(a.q), static_cast<const T *>(a.k),
        static_cast<const T *>(a.v), a.beta, a.offsets, a.req_depth, a.H, a.dk, a.dv, a.N, a.max_T,
        a.logP, wsG, wsC, static_cast<T *>(a.O), a.U, a.st);
    return cudaGetLastError();
}

template <typename T, bool VK> cudaError_t commit_typed(const CommitArgs &a, cudaStream_t s)
{
    dim3 grid(a.B * a.H, (a.dk + kCommitRows - 1) / kCommitRows, a.layers);
    simt_commit_kernel<T, VK><<<grid, kThreads, 0, s>>>(
        a.S, static_cast<const T *>(a.k), a.U, a.logP, a.offsets, a.parent, a.accepted, a.H, a.dk,
        a.dv, a.N, a.s_ls, a.k_ls, a.u_ls, a.lp_ls, a.st);
    return cudaGetLastError();
}

} // namespace

size_t simt_workspace_bytes(int B, int H, int max_T)
{
    return 2 * sizeof(float) * (size_t)B * H * max_T * max_T;
}

cudaError_t launch_simt_verify(const VerifyArgs &a, cudaStream_t s)
{
    if (a.B * a.H == 0 || a.N == 0) return cudaSuccess;
    if (a.dtype == BOLE_BF16)
        return a.vk ? verify_typed<__nv_bfloat16, true>(a, s) : verify_typed<__nv_bfloat16, false>(a, s);
    return a.vk ? verify_typed<float, true>(a, s) : verify_typed<float, false>(a, s);
}

cudaError_t launch_simt_commit(const CommitArgs &a, cudaStream_t s)
{
    if (a.B * a.H == 0 || a.N == 0 || a.layers == 0) return cudaSuccess;
    if (a.dtype == BOLE_BF16)
        return a.vk ? commit_typed<__nv_bfloat16, true>(a, s) : commit_typed<__nv_bfloat16, false>(a, s);
    return a.vk ? commit_typed<float, true>(a, s) : commit_typed<float, false>(a, s);
}

// ---- verification without any allocation ----
// Some callers cannot allocate device memory when they verify: hosts that hand
// the library only tensors they already own and no allocator, and serving
// loops that forbid allocation on the hot path because an allocation can
// synchronise the device.  For them the G, C scratch of the CUDA-core path
// lives in this fixed, library-owned array (8 MiB, held by every GPU that
// loads the library until the process exits).  Every call shares it and it
// keeps the previous call's contents; the producer kernel rewrites every
// entry the solve kernel reads, so nothing has to start at zero.  Calls whose
// kernels overlap on the GPU race on the array.
static __device__ __align__(256) float g_noalloc_scratch[2 * (size_t)BOLE_NOALLOC_MAX_FACTOR_ELEMS];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices] = {};
} // namespace

// The array's device address on the current device, resolved once per device
// (host code cannot use the symbol itself: it names a host-side stand-in).
static cudaError_t noalloc_scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

bool simt_noalloc_fits(int B, int H, int max_T)
{
    return (size_t)B * H * max_T * max_T <= (size_t)BOLE_NOALLOC_MAX_FACTOR_ELEMS;
}

cudaError_t launch_simt_verify_noalloc(const VerifyArgs &a, cudaStream_t s)
{
    if (a.B * a.H == 0 || a.N == 0) return cudaSuccess;
    void *scratch = nullptr;
    cudaError_t e = noalloc_scratch_address(&scratch);
    if (e != cudaSuccess) return e;
    VerifyArgs b = a;
    b.ws = scratch;
    return launch_simt_verify(b, s);
}

} // namespace bole
