// Round-level topology step: validate the packed forest and derive each
// node's depth and ancestor-or-self bit mask ("Bole", Section IV-C, and the
// flat-ragged packed forest of the review's Section 3).  Integer only.
#include "common.cuh"
#include "sm100.cuh"

namespace bole {
namespace {

// One warp per request.  The request's parent array (at most 128 entries) is
// staged in shared memory with coalesced loads and validated; then the
// ancestor-or-self masks are built by pointer jumping: node i starts with
// {i} and a jump to its parent, and each round ORs in the mask held at its
// jump target and doubles the jump (jump <- jump of the jump), so after
// ceil(log2 128) = 7 rounds every mask holds the whole path to the root (a
// path of length l is covered after ceil(log2 l) rounds).  Rounds alternate
// between two copies of the masks and jumps so a lane never reads a value
// another lane is writing.  depth = bits - 1.
// A batch of at most 32 requests runs as one CTA (one warp per request) that
// also clears the status block before any warp can report, so no separate
// reset is needed; larger batches run CTAs of four warps after a reset copy.
constexpr int kPackWarps = 4;
constexpr int kPackOneCTA = 32;
constexpr int kPackWarpSmem = 2 * kMaxTree * (16 + 4); // masks and jumps, two copies

template <bool ONE_CTA>
__global__ void __launch_bounds__(32 * (ONE_CTA ? kPackOneCTA : kPackWarps)) pack_kernel(
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ parent, int B, int N,
    int max_depth, int32_t *__restrict__ depth, uint32_t *__restrict__ anc,
    int32_t *__restrict__ req_depth, int32_t *st)
{
    extern __shared__ __align__(16) uint8_t pack_smem[];
    pdl_launch_dependents(); // a verification launched to overlap may start its state reads
    const int warps = (int)blockDim.x >> 5;
    const int wib = threadIdx.x >> 5;
    const int b = (int)blockIdx.x * warps + wib;
    const int lane = threadIdx.x & 31;
    if (ONE_CTA) { // the status block is clear before anyone can report
        if (threadIdx.x < BOLE_STATUS_WORDS) st[threadIdx.x] = 0;
        __syncthreads();
    }
    // this warp's two copies of the masks and jumps
    uint4 (*smask)[kMaxTree] = reinterpret_cast<uint4 (*)[kMaxTree]>(pack_smem + wib * kPackWarpSmem);
    int (*sjump)[kMaxTree] =
        reinterpret_cast<int (*)[kMaxTree]>(pack_smem + wib * kPackWarpSmem + 2 * kMaxTree * 16);
    if (b >= B) return;
    const int o = offsets[b], e = offsets[b + 1];
    const int T = e - o;
    const bool bad_off = o < 0 || e > N || T < 0 || T > kMaxTree || (b == 0 && o != 0);
    if (bad_off) {
        if (lane == 0) {
            req_depth[b] = 0;
            report(st, BOLE_ERR_BAD_TOPOLOGY, b, -1, T);
        }
        return;
    }
    int bad_i = -1, bad_p = 0;
    for (int i = lane; i < T; i += 32) {
        const int p = parent[o + i];
        if ((p < -1 || p >= i) && bad_i < 0) {
            bad_i = i;
            bad_p = p;
        }
        const uint32_t bit = 1u << (i & 31), w = (uint32_t)(i >> 5);
        smask[0][i] = make_uint4(w == 0 ? bit : 0u, w == 1 ? bit : 0u, w == 2 ? bit : 0u,
                                      w == 3 ? bit : 0u);
        sjump[0][i] = p;
    }
    const unsigned badm = __ballot_sync(0xffffffffu, bad_i >= 0);
    if (badm) {
        const int src = __ffs(badm) - 1;
        const int bi = __shfl_sync(0xffffffffu, bad_i, src);
        const int bp = __shfl_sync(0xffffffffu, bad_p, src);
        if (lane == 0) {
            req_depth[b] = 0;
            report(st, BOLE_ERR_BAD_TOPOLOGY, b, bi, bp);
        }
        return;
    }
    __syncwarp();
    // every link points backwards, so jumps stay in [-1, i) and the rounds
    // only ever read indices below the one they write
    int cur = 0;
    for (int round = 0; (1 << round) < T; ++round) {
        for (int i = lane; i < T; i += 32) {
            uint4 mk = smask[cur][i];
            int j = sjump[cur][i];
            if (j >= 0) {
                const uint4 mj = smask[cur][j];
                mk.x |= mj.x; mk.y |= mj.y; mk.z |= mj.z; mk.w |= mj.w;
                j = sjump[cur][j];
            }
            smask[cur ^ 1][i] = mk;
            sjump[cur ^ 1][i] = j;
        }
        __syncwarp();
        cur ^= 1;
    }
    int dmax = 0;
    for (int i = lane; i < T; i += 32) {
        const uint4 mk = smask[cur][i];
        const int d = __popc(mk.x) + __popc(mk.y) + __popc(mk.z) + __popc(mk.w) - 1;
        depth[o + i] = d;
        *reinterpret_cast<uint4 *>(anc + (size_t)(o + i) * 4) = mk;
        dmax = max(dmax, d);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) dmax = max(dmax, __shfl_xor_sync(0xffffffffu, dmax, s));
    if (lane == 0) {
        req_depth[b] = dmax;
        if (dmax > max_depth) report(st, BOLE_ERR_DEPTH, b, -1, dmax);
    }
}

// Self-test of the bounded device wait every kernel uses: one thread waits on
// an mbarrier that nothing arrives on, with the caller's limit; the wait gives
// up and the timeout is reported with the time actually waited (microseconds).
__global__ void selftest_wait_kernel(int32_t *st, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    sm100::mbar_init(&bar, 1);
    sm100::fence_mbar_init();
    const uint64_t t0 = sm100::global_ns();
    const bool arrived = sm100::mbar_wait(&bar, 0, limit_ns);
    const uint64_t us = (sm100::global_ns() - t0) / 1000;
    if (!arrived) report(st, BOLE_ERR_TIMEOUT, -1, -1, (int)(us < 0x7fffffffu ? us : 0x7fffffffu));
}

} // namespace

cudaError_t launch_selftest_wait(int32_t *st, uint64_t limit_ns, cudaStream_t s)
{
    selftest_wait_kernel<<<1, 32, 0, s>>>(st, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_pack(const int32_t *offsets, const int32_t *parent, int B, int N, int max_depth,
                        int32_t *depth, uint32_t *anc, int32_t *req_depth, int32_t *st,
                        cudaStream_t s)
{
    if (B >= 1 && B <= kPackOneCTA) { // one CTA clears the status block itself
        const size_t smem = (size_t)B * kPackWarpSmem;
        static bool configured[64] = {};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64 || !configured[dev]) {
            e = cudaFuncSetAttribute(pack_kernel<true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kPackOneCTA * kPackWarpSmem);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) configured[dev] = true;
        }
        pack_kernel<true><<<1, 32 * B, smem, s>>>(offsets, parent, B, N, max_depth, depth, anc,
                                                  req_depth, st);
        return cudaGetLastError();
    }
    cudaError_t e = cudaMemsetAsync(st, 0, sizeof(int32_t) * BOLE_STATUS_WORDS, s);
    if (e != cudaSuccess) return e;
    if (B <= 0) return cudaSuccess;
    const int blocks = (B + kPackWarps - 1) / kPackWarps;
    pack_kernel<false><<<blocks, 32 * kPackWarps, kPackWarps * kPackWarpSmem, s>>>(
        offsets, parent, B, N, max_depth, depth, anc, req_depth, st);
    return cudaGetLastError();
}

} // namespace bole
