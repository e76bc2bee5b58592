// Tree-parallel stage 1 of a GDN layer: the short causal depthwise
// convolution along parent links, its bias, SiLU, the per-head L2
// normalisation of q and k, and the decay / write gates -- every node at once
// ("Bole", Section IV-C: the first of the three per-layer stages fuses the
// convolution, bias, SiLU and gate preparation along parent links).  Also the
// commit of the convolution state to the accepted path.
//
// A node's causal window is itself, its parent, grandparent, ... (nearest
// first) and, once the path reaches the committed root, the committed
// prefix's last W-1 tokens (the request's convolution state, row W-2 the most
// recent).  In token order this is the usual causal convolution
//     y_t[c] = bias[c] + sum_w conv_w[c][w] x_{t-W+1+w}[c].
//
// The stage is HBM-bound: each node's in-projection row is read once from
// DRAM into shared memory and its q, k, v rows are written once; the window
// products read shared memory.  No tensor-core work.
#include "common.cuh"
#include "sm100.cuh"
#include "tc_common.cuh"

namespace bole {
namespace {

using namespace sm100;

constexpr int kMaxConv = 8;          // widest supported convolution
constexpr int kS1Warps = 4;
constexpr int kS1Threads = 32 * kS1Warps;
constexpr int kMaxChan = 128;        // d_k, d_v <= 128

template <typename T> struct Vec4;
template <> struct Vec4<__nv_bfloat16> {
    using raw = uint2; // four elements, moved as they are
    __device__ static uint2 load_raw(const __nv_bfloat16 *p)
    {
        return __ldg(reinterpret_cast<const uint2 *>(p));
    }
    __device__ static void unpack(const uint2 &u, float (&f)[4])
    {
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&u.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&u.y);
        const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
        f[0] = fa.x; f[1] = fa.y; f[2] = fb.x; f[3] = fb.y;
    }
    __device__ static void store(__nv_bfloat16 *p, const float (&f)[4])
    {
        __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]);
        __nv_bfloat162 b = __floats2bfloat162_rn(f[2], f[3]);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&a);
        u.y = *reinterpret_cast<uint32_t *>(&b);
        *reinterpret_cast<uint2 *>(p) = u;
    }
};
template <> struct Vec4<float> {
    using raw = float4;
    __device__ static float4 load_raw(const float *p)
    {
        return __ldg(reinterpret_cast<const float4 *>(p));
    }
    __device__ static void unpack(const float4 &u, float (&f)[4])
    {
        f[0] = u.x; f[1] = u.y; f[2] = u.z; f[3] = u.w;
    }
    __device__ static void store(float *p, const float (&f)[4])
    {
        *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
    }
};

// Eight consecutive elements: one 16-byte access (bf16) or two (float32).
template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
    struct raw { uint4 u; };
    __device__ static raw load(const __nv_bfloat16 *p)
    {
        return raw{*reinterpret_cast<const uint4 *>(p)};
    }
    __device__ static void unpack(const raw &r, float (&f)[8])
    {
        const uint32_t w[4] = {r.u.x, r.u.y, r.u.z, r.u.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[t]));
            f[2 * t] = x.x;
            f[2 * t + 1] = x.y;
        }
    }
    __device__ static void store(__nv_bfloat16 *p, const float (&f)[8])
    {
        uint32_t w[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * t], f[2 * t + 1]);
            w[t] = *reinterpret_cast<uint32_t *>(&h);
        }
        *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct Vec8<float> {
    struct raw { float4 a, b; };
    __device__ static raw load(const float *p)
    {
        return raw{reinterpret_cast<const float4 *>(p)[0], reinterpret_cast<const float4 *>(p)[1]};
    }
    __device__ static void unpack(const raw &r, float (&f)[8])
    {
        f[0] = r.a.x; f[1] = r.a.y; f[2] = r.a.z; f[3] = r.a.w;
        f[4] = r.b.x; f[5] = r.b.y; f[6] = r.b.z; f[7] = r.b.w;
    }
    __device__ static void store(float *p, const float (&f)[8])
    {
        reinterpret_cast<float4 *>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4 *>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
};

// x * sigmoid(x); the quotient by the fast approximate division (2 ulp)
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.f + __expf(-x)); }

// x * sigmoid(x) = h + h tanh(h), h = x / 2, with the hardware tanh
// approximation (one multi-function op; relative error near 2^-11, below the
// bf16 rounding of the outputs it feeds)
__device__ __forceinline__ float silu_tanh(float x)
{
    const float h = 0.5f * x;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return fmaf(h, t, h);
}

// log(1 + e^x) without overflow: x + log1p(e^-x) for x > 0
__device__ __forceinline__ float softplus(float x)
{
    return x > 0.f ? x + log1pf(expf(-x)) : log1pf(expf(x));
}

// One CTA per (request, head, part), part 0 = q, 1 = k, 2 = v.  The CTA's
// channel slice of every row it needs -- the request's T node rows and the
// W-1 committed state rows -- arrives in shared memory by TMA tiles (node
// rows in boxes of 16, the state rows in one box, all on one mbarrier: a
// handful of copies per CTA rather than one per row), so each row leaves
// DRAM once and the window products read shared memory.  The
// set-up reads (parent links, taps, bias, gate pre-activations) are issued
// together, one item per thread (T, n <= 128 = the block).  Each warp pass
// takes two nodes, 16 lanes per node and eight channels per lane.  The v
// CTAs also form the gates.
//   window[i][d], d = 0..W-1: the shared-memory row of the token at distance
//   d before node i (d = 0 is i itself): row = node index < T, or Tpad + s
//   for state row s (Tpad = T rounded up to the 16-row box).
constexpr uint64_t kS1WaitNs = 200ull * 1000 * 1000;
constexpr int kRowBox = 16;          // node rows per TMA box
static_assert(kS1Threads >= kMaxTree && kS1Threads >= kMaxChan, "one set-up item per thread");

template <typename T, int MAXW>
__global__ void __launch_bounds__(kS1Threads)
conv_gates_kernel(const __grid_constant__ CUtensorMap tmXqk, const __grid_constant__ CUtensorMap tmXv,
                  const __grid_constant__ CUtensorMap tmCqk, const __grid_constant__ CUtensorMap tmCv,
                  const float *__restrict__ conv_w, const float *__restrict__ conv_b,
                  const float *__restrict__ ga, const float *__restrict__ gb,
                  const float *__restrict__ gate_scale, const float *__restrict__ gate_bias,
                  const int32_t *__restrict__ offsets, const int32_t *__restrict__ parent, int H,
                  int dk, int dv, int N, int W, int max_T, T *__restrict__ q, T *__restrict__ k,
                  T *__restrict__ v, float *__restrict__ gamma, float *__restrict__ beta,
                  int32_t *st)
{
    extern __shared__ __align__(16) uint8_t rows_raw[]; // [Tpad(max_T) + W - 1][n] elements
    __shared__ int32_t spar[kMaxTree];
    __shared__ int32_t window[kMaxTree][MAXW];
    __shared__ __align__(16) float wts[MAXW][kMaxChan]; // tap-major
    __shared__ __align__(16) float bias[kMaxChan];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int bad;

    const int unit = blockIdx.x, b = unit / H, h = unit % H, part = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = part < 2 ? dk : dv;
    const int cb = part == 0 ? h * dk : part == 1 ? (H + h) * dk : 2 * H * dk + h * dv;
    // One round trip for what needs nothing else: the status word, the
    // request's extent and this slice's taps and bias (thread = channel).
    // The exit on an earlier failure is taken by the whole CTA.
    const bool has_chan = tid < n;
    float wv[MAXW];
#pragma unroll
    for (int t = 0; t < MAXW; ++t)
        wv[t] = (has_chan && t < W) ? conv_w[(size_t)(cb + tid) * W + t] : 0.f;
    const float bv = (has_chan && conv_b) ? conv_b[cb + tid] : 0.f;
    const bool prior_fault = faulted(st);
    const int o = offsets[b], Tn = offsets[b + 1] - o;
    if (__syncthreads_or(prior_fault)) return;
    if (Tn <= 0) return;
    if (Tn > max_T || o < 0 || o + Tn > N) {
        if (tid == 0 && h == 0 && part == 0) report(st, BOLE_ERR_BAD_TOPOLOGY, b, -1, Tn);
        return;
    }
    // TMA destinations 128-byte aligned (the launch adds the slack)
    T *rows = reinterpret_cast<T *>((reinterpret_cast<uintptr_t>(rows_raw) + 127) & ~(uintptr_t)127);
    const int Tpad = (Tn + kRowBox - 1) / kRowBox * kRowBox;
    const uint32_t row_bytes = (uint32_t)n * sizeof(T);
    if (tid == 0) {
        bad = 0;
        mbar_init(&bar, 1);
        fence_mbar_init();
        const CUtensorMap *mx = part < 2 ? &tmXqk : &tmXv;
        mbar_arrive_expect_tx(&bar, (uint32_t)(Tpad + W - 1) * row_bytes);
        for (int r0 = 0; r0 < Tn; r0 += kRowBox) // rows past N arrive as zeros
            tma_load_2d(rows + (size_t)r0 * n, mx, &bar, cb, o + r0);
        if (W > 1)
            tma_load_2d(rows + (size_t)Tpad * n, part < 2 ? &tmCqk : &tmCv, &bar, cb, b * (W - 1));
    }
    // request reads, in flight together with the rows: thread tid = node tid
    const bool has_node = tid < Tn;
    const int par_t = has_node ? parent[o + tid] : 0;
    const bool gates = part == 2 && has_node;
    const size_t nh_t = (size_t)(o + tid) * H + h;
    const float av = gates ? ga[nh_t] : 0.f, bgv = gates ? gb[nh_t] : 0.f;
    const float gs = (gates && gate_scale) ? gate_scale[h] : 1.f;
    const float gbias = (gates && gate_bias) ? gate_bias[h] : 0.f;
    if (has_node) spar[tid] = par_t;
    if (has_chan) {
#pragma unroll
        for (int t = 0; t < MAXW; ++t)
            if (t < W) wts[t][tid] = wv[t];
        bias[tid] = bv;
    }
    if (gates) {
        gamma[nh_t] = expf(-gs * softplus(av + gbias));
        beta[nh_t] = 1.f / (1.f + expf(-bgv));
    }
    __syncthreads();
    // causal window of node tid along parent links (every link checked)
    if (has_node) {
        int j = tid, d = 0;
        for (; d < W && j >= 0; ++d) {
            window[tid][d] = j;
            const int pj = spar[j];
            if (pj >= j || pj < -1) {
                report(st, BOLE_ERR_BAD_TOPOLOGY, b, o + j, pj);
                bad = 1;
                break;
            }
            j = pj;
        }
        if (j < 0)
            for (int s = W - 2; d < W; ++d, --s) window[tid][d] = Tpad + s;
    }
    __syncthreads();
    const bool ok = mbar_wait(&bar, 0, kS1WaitNs); // the copies end even when unused
    if (bad) return;
    if (!ok) {
        if (tid == 0) report(st, BOLE_ERR_TIMEOUT, b, -1, 30);
        return;
    }

    T *out = part == 0 ? q : part == 1 ? k : v;
    const int sub = lane >> 4, sl = lane & 15; // node of this half-warp, lane within it
    const int c0 = 8 * sl;
    const bool act = c0 < n;
    // this lane's eight channels: taps and bias stay in registers for every node
    float wr[MAXW][8], br[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) br[e] = act ? bias[c0 + e] : 0.f;
#pragma unroll
    for (int d = 0; d < MAXW; ++d)
#pragma unroll
        for (int e = 0; e < 8; ++e) wr[d][e] = (act && d < W) ? wts[W - 1 - d][c0 + e] : 0.f;
    for (int i0 = 2 * warp; i0 < Tn; i0 += 2 * kS1Warps) {
        const int i = i0 + sub;
        const bool live = i < Tn && act;
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = 0.f;
        if (live) {
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = br[e];
#pragma unroll
            for (int d = 0; d < MAXW; ++d) {
                if (d >= W) break;
                float xv[8];
                Vec8<T>::unpack(Vec8<T>::load(rows + (size_t)window[i][d] * n + c0), xv);
                // channel pairs as packed fp32 FMAs (each lane rounded as fmaf)
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float2 acc = __ffma2_rn(make_float2(wr[d][e], wr[d][e + 1]),
                                                  make_float2(xv[e], xv[e + 1]),
                                                  make_float2(y[e], y[e + 1]));
                    y[e] = acc.x;
                    y[e + 1] = acc.y;
                }
            }
            // bf16 outputs: the one-op form; float32 outputs: the accurate one
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = sizeof(T) == 2 ? silu_tanh(y[e]) : silu(y[e]);
        }
        if (part < 2) { // q and k leave as unit vectors per head
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(y[e], y[e], ss);
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float r = rsqrtf(ss);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const float2 yr = __fmul2_rn(make_float2(y[e], y[e + 1]), make_float2(r, r));
                y[e] = yr.x;
                y[e + 1] = yr.y;
            }
        }
        if (live) Vec8<T>::store(out + ((size_t)(o + i) * H + h) * n + c0, y);
    }
}

// Convolution-state commit: four channels per thread of one request.  The new
// rows are the last W-1 tokens ending at the accepted node a: a (row W-2),
// its parent (row W-3), ... then the old rows shifted down.  Each thread reads
// its channels' old rows before writing any, so the update is in place
// (C is a multiple of 16).
constexpr int kCommitThreadsS1 = 256;
template <typename T>
__global__ void __launch_bounds__(kCommitThreadsS1)
conv_commit_kernel(T *__restrict__ conv_state, const T *__restrict__ x,
                   const int32_t *__restrict__ offsets, const int32_t *__restrict__ parent,
                   const int32_t *__restrict__ accepted, int C, int W, int N, int32_t *st)
{
    __shared__ int32_t toks[kMaxConv];
    __shared__ int32_t spar[kMaxTree];
    __shared__ int ok;
    const int b = blockIdx.y;
    const bool prior_fault = faulted(st); // one round trip with the request's reads
    const int a = accepted[b];
    const int o = offsets[b], Tn = offsets[b + 1] - o;
    if (__syncthreads_or(prior_fault)) return; // taken by the whole CTA
    if (a < 0) return;
    if (a >= Tn || o < 0 || o + Tn > N || Tn > kMaxTree) {
        if (threadIdx.x == 0 && blockIdx.x == 0) report(st, BOLE_ERR_BAD_TOPOLOGY, b, a, Tn);
        return;
    }
    for (int i = threadIdx.x; i <= a; i += blockDim.x) spar[i] = parent[o + i];
    __syncthreads();
    if (threadIdx.x == 0) {
        int j = a, d = 0, good = 1;
        for (; d < W - 1 && j >= 0; ++d) {
            toks[d] = j;
            const int pj = spar[j];
            if (pj >= j || pj < -1) {
                good = 0;
                if (blockIdx.x == 0) report(st, BOLE_ERR_BAD_TOPOLOGY, b, o + j, pj);
                break;
            }
            j = pj;
        }
        // the old row each remaining position takes: the most recent first
        for (int s = W - 2; d < W - 1; ++d, --s) toks[d] = -(s + 1);
        ok = good;
    }
    __syncthreads();
    if (!ok) return;
    const int c = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (c >= C) return;
    using V = typename Vec4<T>::raw;
    V *row0 = reinterpret_cast<V *>(conv_state + (size_t)b * (W - 1) * C + c);
    const size_t rs = (size_t)C / 4; // row stride in vectors
    V old[kMaxConv - 1], nv[kMaxConv - 1];
#pragma unroll
    for (int s = 0; s < kMaxConv - 1; ++s)
        if (s < W - 1) old[s] = row0[s * rs];
#pragma unroll
    for (int d = 0; d < kMaxConv - 1; ++d) {
        if (d >= W - 1) break;
        const int tok = toks[d];
        V val = old[0];
        if (tok >= 0) val = *reinterpret_cast<const V *>(x + (size_t)(o + tok) * C + c);
#pragma unroll
        for (int s = 1; s < kMaxConv - 1; ++s) // old row -(tok + 1), selected in registers
            if (tok == -(s + 1)) val = old[s];
        nv[d] = val;
    }
#pragma unroll
    for (int d = 0; d < kMaxConv - 1; ++d)
        if (d < W - 1) row0[(W - 2 - d) * rs] = nv[d];
}

size_t conv_rows_bytes(const ConvGatesArgs &a, size_t elem)
{
    const size_t tpad = (size_t)(a.max_T + kRowBox - 1) / kRowBox * kRowBox;
    return (tpad + a.W - 1) * (size_t)(a.dk > a.dv ? a.dk : a.dv) * elem + 128; // + alignment
}

// rows x C row-major (x: N rows, the convolution state: B (W-1) rows) as a
// 2-D tensor whose boxes are `cols` channels x `box_rows` rows
cudaError_t make_rows_map(CUtensorMap *map, const void *base, bole_dtype dt, int C, int rows,
                          int cols, int box_rows)
{
    auto fn = tc::encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const size_t es = dt == BOLE_BF16 ? 2 : 4;
    cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)C * es};
    cuuint32_t box[2] = {(cuuint32_t)cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dt == BOLE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                    2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <typename T, int MAXW> cudaError_t conv_gates_typed(const ConvGatesArgs &a, cudaStream_t s)
{
    const size_t smem = conv_rows_bytes(a, sizeof(T));
    const int C = a.H * (2 * a.dk + a.dv);
    CUtensorMap xqk, xv, cqk, cv;
    cudaError_t e = make_rows_map(&xqk, a.x, a.dtype, C, a.N, a.dk, kRowBox);
    if (e == cudaSuccess) e = make_rows_map(&xv, a.x, a.dtype, C, a.N, a.dv, kRowBox);
    if (e == cudaSuccess && a.W > 1) {
        e = make_rows_map(&cqk, a.conv_state, a.dtype, C, a.B * (a.W - 1), a.dk, a.W - 1);
        if (e == cudaSuccess)
            e = make_rows_map(&cv, a.conv_state, a.dtype, C, a.B * (a.W - 1), a.dv, a.W - 1);
    } else {
        cqk = xqk; // unused: no state rows
        cv = xv;
    }
    if (e != cudaSuccess) return e;
    auto kernel = conv_gates_kernel<T, MAXW>;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<dim3(a.B * a.H, 3), kS1Threads, smem, s>>>(
        xqk, xv, cqk, cv, a.conv_w, a.conv_b,
        a.a, a.b, a.gate_scale, a.gate_bias, a.offsets, a.parent, a.H, a.dk, a.dv, a.N, a.W,
        a.max_T, static_cast<T *>(a.q), static_cast<T *>(a.k), static_cast<T *>(a.v), a.gamma,
        a.beta, a.st);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_conv_gates(const ConvGatesArgs &a, cudaStream_t s)
{
    if (a.B * a.H == 0 || a.N == 0) return cudaSuccess;
    if (a.dtype == BOLE_BF16)
        return a.W <= 4 ? conv_gates_typed<__nv_bfloat16, 4>(a, s)
                        : conv_gates_typed<__nv_bfloat16, 8>(a, s);
    return a.W <= 4 ? conv_gates_typed<float, 4>(a, s) : conv_gates_typed<float, 8>(a, s);
}

cudaError_t launch_conv_commit(void *conv_state, const void *x, bole_dtype dtype,
                               const int32_t *offsets, const int32_t *parent,
                               const int32_t *accepted, int B, int C, int W, int N, int32_t *st,
                               cudaStream_t s)
{
    if (B == 0 || N == 0 || W <= 1) return cudaSuccess;
    dim3 grid((C / 4 + kCommitThreadsS1 - 1) / kCommitThreadsS1, B);
    if (dtype == BOLE_BF16)
        conv_commit_kernel<__nv_bfloat16><<<grid, kCommitThreadsS1, 0, s>>>(
            static_cast<__nv_bfloat16 *>(conv_state), static_cast<const __nv_bfloat16 *>(x),
            offsets, parent, accepted, C, W, N, st);
    else
        conv_commit_kernel<float><<<grid, kCommitThreadsS1, 0, s>>>(static_cast<float *>(conv_state),
                                                       static_cast<const float *>(x), offsets,
                                                       parent, accepted, C, W, N, st);
    return cudaGetLastError();
}

} // namespace bole
