// Round-level topology step: validate the packed forest and derive each
// node's depth and ancestor-or-self bit mask ("Bole", Section IV-C, and the
// flat-ragged packed forest of the review's Section 3).  Integer only.
#include "common.cuh"

namespace bole {
namespace {

// One warp per request.  The request's parent array (at most 128 entries) is
// staged in shared memory with coalesced loads, validated, and then every lane
// walks its nodes' parent links there (at most 128 steps, guaranteed to end
// because every parent index was checked to be smaller); depth = bits - 1.
constexpr int kPackWarps = 4;

__global__ void __launch_bounds__(32 * kPackWarps) pack_kernel(
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ parent, int B, int N,
    int max_depth, int32_t *__restrict__ depth, uint32_t *__restrict__ anc,
    int32_t *__restrict__ req_depth, int32_t *st)
{
    __shared__ int sp[kPackWarps][kMaxTree];
    pdl_launch_dependents(); // a verification launched to overlap may start its state reads
    const int wib = threadIdx.x >> 5;
    const int b = (int)blockIdx.x * kPackWarps + wib;
    const int lane = threadIdx.x & 31;
    if (b >= B) return;
    const int o = offsets[b], e = offsets[b + 1];
    const int T = e - o;
    const bool bad_off = o < 0 || e > N || T < 0 || T > kMaxTree || (b == 0 && o != 0) ||
                         (b == B - 1 && e != N);
    if (bad_off) {
        if (lane == 0) {
            req_depth[b] = 0;
            report(st, BOLE_ERR_BAD_TOPOLOGY, b, -1, T);
        }
        return;
    }
    int *par = sp[wib];
    int bad_i = -1;
    for (int i = lane; i < T; i += 32) {
        const int p = parent[o + i];
        par[i] = p;
        if ((p < -1 || p >= i) && bad_i < 0) bad_i = i;
    }
    const unsigned badm = __ballot_sync(0xffffffffu, bad_i >= 0);
    if (badm) {
        const int src = __ffs(badm) - 1;
        const int bi = __shfl_sync(0xffffffffu, bad_i, src);
        if (lane == 0) {
            req_depth[b] = 0;
            report(st, BOLE_ERR_BAD_TOPOLOGY, b, bi, par[bi]);
        }
        return;
    }
    __syncwarp();
    int dmax = 0;
    for (int i = lane; i < T; i += 32) {
        uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
        for (int j = i; j >= 0; j = par[j]) {
            const uint32_t bit = 1u << (j & 31);
            if (j < 32) w0 |= bit;
            else if (j < 64) w1 |= bit;
            else if (j < 96) w2 |= bit;
            else w3 |= bit;
        }
        const int d = __popc(w0) + __popc(w1) + __popc(w2) + __popc(w3) - 1;
        depth[o + i] = d;
        *reinterpret_cast<uint4 *>(anc + (size_t)(o + i) * 4) = make_uint4(w0, w1, w2, w3);
        dmax = max(dmax, d);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) dmax = max(dmax, __shfl_xor_sync(0xffffffffu, dmax, s));
    if (lane == 0) {
        req_depth[b] = dmax;
        if (dmax > max_depth) report(st, BOLE_ERR_DEPTH, b, -1, dmax);
    }
}

} // namespace

cudaError_t launch_pack(const int32_t *offsets, const int32_t *parent, int B, int N, int max_depth,
                        int32_t *depth, uint32_t *anc, int32_t *req_depth, int32_t *st,
                        cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(st, 0, sizeof(int32_t) * BOLE_STATUS_WORDS, s);
    if (e != cudaSuccess) return e;
    if (B <= 0) return cudaSuccess;
    const int blocks = (B + kPackWarps - 1) / kPackWarps;
    pack_kernel<<<blocks, 32 * kPackWarps, 0, s>>>(offsets, parent, B, N, max_depth, depth, anc,
                                                   req_depth, st);
    return cudaGetLastError();
}

} // namespace bole
