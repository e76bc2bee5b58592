// Device-side proposal selection and forest build: the runtime rule of the
// hardware-aware budget ("Bole", Section IV: every drafted candidate scores
// the product of the drafter's edge probabilities along its path, and the
// round's budget is filled with the globally highest-scoring candidates;
// since a child never outscores its parent, each request's selection is
// ancestor-closed), followed by the flat ragged forest build -- the
// "selection -> forest build" steps the pages keep on the GPU.
//
// Three small kernels, all integer decisions taken on float32 scores
// accumulated root-down, rho(v) = rho(parent) * p(v):
//   1. select_local_kernel (one CTA per request): parent-link depths by
//      pointer jumping, the scores level by level, every candidate's 64-bit
//      order key, a bitonic sort, and the request's best min(cap, 128, M_b)
//      keys into a per-request list.
//   2. select_global_kernel (one CTA per request, 8 threads per list entry):
//      each request's best key is reserved (in global order while the
//      budget lasts); every other listed key is selected when fewer than
//      the remaining budget of the other lists' keys precede it -- its
//      global rank, counted by binary search in every request's sorted list
//      (an eighth of the lists per thread).  The selected keys of a request
//      are a prefix of its list.
//   3. build_forest_kernel (one CTA per request): the request's offset (sum
//      of the earlier counts), its selected candidates in candidate order
//      (parent before child), and their request-local parent links.
// Order key, ascending = better: [63:32] = ~bits(rho) (rho >= 0, so larger
// rho first), [31:22] depth, [21:10] request, [9:0] candidate index -- the
// global order (rho, depth, request, index) in one 64-bit comparison.
#include "common.cuh"

namespace bole {
namespace {

constexpr int kMaxCand = BOLE_MAX_CANDIDATES; // candidates per request
constexpr int kListLen = kMaxTree;            // a request's tree holds at most 128 nodes
constexpr int kSelThreads = 512;
constexpr int kGlobThreads = kListLen;        // build: one thread per list entry
constexpr int kRankSplit = 8;                 // rank: list entry x eighth of the lists
constexpr int kRankThreads = kListLen * kRankSplit;
constexpr int kChunkLists = 40;               // lists staged per pass (40 KB)

__device__ __forceinline__ uint64_t order_key(float rho, int depth, int b, int i)
{
    return ((uint64_t)(0xFFFFFFFFu - __float_as_uint(rho)) << 32) |
           ((uint64_t)depth << 22) | ((uint64_t)b << 10) | (uint64_t)i;
}

__global__ void __launch_bounds__(kSelThreads)
select_local_kernel(const float *__restrict__ p, const int32_t *__restrict__ cand_offsets,
                    const int32_t *__restrict__ cand_parent, const int32_t *__restrict__ caps,
                    int M_total, float *__restrict__ rho_out, uint64_t *__restrict__ lists,
                    int32_t *__restrict__ lens, int32_t *st)
{
    __shared__ float sp[kMaxCand], srho[kMaxCand];
    __shared__ int32_t spar[kMaxCand];
    __shared__ int32_t sdep[2][kMaxCand], sanc[2][kMaxCand];
    __shared__ uint64_t keys[kMaxCand];
    __shared__ int maxd, bad;
    const int b = blockIdx.x, tid = threadIdx.x;
    const int o = cand_offsets[b], M = cand_offsets[b + 1] - o;
    if (tid == 0) {
        maxd = 0;
        bad = (M < 0 || M > kMaxCand || o < 0 || o + M > M_total) ? 1 : 0;
        if (bad) report(st, BOLE_ERR_BAD_TOPOLOGY, b, -1, M);
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) lens[b] = 0;
        return;
    }
    for (int i = tid; i < M; i += kSelThreads) {
        const int pi = cand_parent[o + i];
        sp[i] = p[o + i];
        spar[i] = pi;
        if (pi < -1 || pi >= i) {
            report(st, BOLE_ERR_BAD_TOPOLOGY, b, o + i, pi);
            bad = 1;
        }
        sdep[0][i] = pi >= 0 ? 1 : 0;
        sanc[0][i] = pi;
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) lens[b] = 0;
        return;
    }
    // depth = strict ancestors, by pointer jumping (ceil(log2 M) rounds)
    int cur = 0;
    for (int len = 1; len < M; len <<= 1) {
        for (int i = tid; i < M; i += kSelThreads) {
            const int a = sanc[cur][i];
            sdep[cur ^ 1][i] = sdep[cur][i] + (a >= 0 ? sdep[cur][a] : 0);
            sanc[cur ^ 1][i] = a >= 0 ? sanc[cur][a] : -1;
        }
        cur ^= 1;
        __syncthreads();
    }
    for (int i = tid; i < M; i += kSelThreads) atomicMax(&maxd, sdep[cur][i]);
    __syncthreads();
    // scores level by level: rho(v) = rho(parent) * p(v), root-down as defined
    const int D = maxd;
    for (int l = 0; l <= D; ++l) {
        for (int i = tid; i < M; i += kSelThreads)
            if (sdep[cur][i] == l) srho[i] = spar[i] < 0 ? sp[i] : srho[spar[i]] * sp[i];
        __syncthreads();
    }
    int n2 = 1;
    while (n2 < M) n2 <<= 1;
    for (int i = tid; i < n2; i += kSelThreads)
        keys[i] = i < M ? order_key(srho[i], sdep[cur][i], b, i) : ~0ull;
    if (rho_out)
        for (int i = tid; i < M; i += kSelThreads) rho_out[o + i] = srho[i];
    __syncthreads();
    // bitonic sort, ascending
    for (int k = 2; k <= n2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < n2; i += kSelThreads) {
                const int l = i ^ j;
                if (l > i) {
                    const uint64_t a = keys[i], c = keys[l];
                    const bool up = (i & k) == 0;
                    if ((a > c) == up) {
                        keys[i] = c;
                        keys[l] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    int cap = caps ? caps[b] : kListLen;
    cap = min(max(cap, 0), min(kListLen, M));
    for (int j = tid; j < cap; j += kSelThreads) lists[(size_t)b * kListLen + j] = keys[j];
    if (tid == 0) lens[b] = cap;
}

// lower_bound of x in s[0, n): the number of entries < x
__device__ __forceinline__ int count_less(const uint64_t *s, int n, uint64_t x)
{
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s[mid] < x) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ int block_sum(int v, int *red)
{
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    int s = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
    return s;
}

// Thread (q, j): list entry j of this request against the staged lists r with
// r % kRankSplit == q; the partial counts are summed in shared memory.
__global__ void __launch_bounds__(kRankThreads)
select_global_kernel(const uint64_t *__restrict__ lists, const int32_t *__restrict__ lens, int B,
                     int budget, int32_t *__restrict__ counts)
{
    __shared__ uint64_t stage[kChunkLists][kListLen];
    __shared__ int32_t slen[kChunkLists];
    __shared__ int32_t part[kRankSplit][kListLen];
    __shared__ int red[kRankThreads / 32];
    const int b = blockIdx.x, tid = threadIdx.x;
    const int q = tid / kListLen, j = tid % kListLen;
    const int len = lens[b];
    const uint64_t first = len > 0 ? lists[(size_t)b * kListLen] : ~0ull;
    const bool has_x = j >= 1 && j < len; // a non-reserved entry of this list
    const uint64_t x = has_x ? lists[(size_t)b * kListLen + j] : 0ull;
    // requests with a list, and how many of their best keys precede this one's
    int nonempty = 0, ahead = 0;
    for (int r = tid; r < B; r += kRankThreads) {
        if (lens[r] > 0) {
            ++nonempty;
            ahead += lists[(size_t)r * kListLen] < first;
        }
    }
    nonempty = block_sum(nonempty, red);
    ahead = block_sum(ahead, red);
    const bool reserved = len > 0 && ahead < budget;
    const int rest = budget - min(budget, nonempty);
    // global rank of x among every list's non-reserved entries (1..len-1)
    int rank = 0;
    for (int c0 = 0; c0 < B; c0 += kChunkLists) {
        const int nl = min(kChunkLists, B - c0);
        __syncthreads();
        if (tid < nl) slen[tid] = lens[c0 + tid];
        for (int e = tid; e < nl * kListLen; e += kRankThreads)
            stage[e / kListLen][e % kListLen] = lists[(size_t)c0 * kListLen + e];
        __syncthreads();
        if (has_x)
            for (int r = q; r < nl; r += kRankSplit)
                if (slen[r] > 1) rank += count_less(&stage[r][1], slen[r] - 1, x);
    }
    part[q][j] = rank;
    __syncthreads();
    int mine = 0;
    if (q == 0 && has_x) {
        int tot = 0;
#pragma unroll
        for (int k = 0; k < kRankSplit; ++k) tot += part[k][j];
        mine = tot < rest ? 1 : 0;
    }
    const int n = block_sum(mine, red);
    if (tid == 0) counts[b] = (reserved ? 1 : 0) + n;
}

__global__ void __launch_bounds__(kGlobThreads)
build_forest_kernel(const uint64_t *__restrict__ lists, const int32_t *__restrict__ counts,
                    const int32_t *__restrict__ cand_offsets,
                    const int32_t *__restrict__ cand_parent, int B, int32_t *__restrict__ offsets,
                    int32_t *__restrict__ parent, int32_t *__restrict__ src, int32_t *st)
{
    __shared__ int32_t idx[kListLen];
    __shared__ int16_t pos[kMaxCand];
    __shared__ int red[kGlobThreads / 32];
    const int b = blockIdx.x, tid = threadIdx.x;
    int before = 0;
    for (int r = tid; r < b; r += kGlobThreads) before += counts[r];
    const int off = block_sum(before, red);
    const int c = counts[b];
    if (tid == 0) {
        if (b == 0) offsets[0] = 0;
        offsets[b + 1] = off + c;
    }
    if (c == 0) return;
    const int o = cand_offsets[b], M = cand_offsets[b + 1] - o;
    // the selected candidates (a prefix of the sorted list), in candidate order
    idx[tid] = tid < c ? (int)(lists[(size_t)b * kListLen + tid] & 1023u) : 0x7FFFFFFF;
    for (int i = tid; i < M; i += kGlobThreads) pos[i] = -1;
    __syncthreads();
    for (int k = 2; k <= kListLen; k <<= 1)
        for (int jj = k >> 1; jj > 0; jj >>= 1) {
            const int l = tid ^ jj;
            if (l > tid) {
                const int a = idx[tid], e = idx[l];
                if ((a > e) == ((tid & k) == 0)) {
                    idx[tid] = e;
                    idx[l] = a;
                }
            }
            __syncthreads();
        }
    if (tid < c) pos[idx[tid]] = (int16_t)tid;
    __syncthreads();
    if (tid < c) {
        const int ci = idx[tid];
        const int cp = cand_parent[o + ci];
        int lp = -1;
        if (cp >= 0) {
            lp = pos[cp];
            if (lp < 0) { // a child outscored its parent: p outside [0, 1]
                report(st, BOLE_ERR_BAD_TOPOLOGY, b, o + ci, cp);
                lp = -1;
            }
        }
        parent[off + tid] = lp;
        src[off + tid] = o + ci;
    }
}

} // namespace

size_t select_workspace_bytes(int B)
{
    return (size_t)B * kListLen * sizeof(uint64_t) + 2 * (size_t)B * sizeof(int32_t);
}

cudaError_t launch_select(const float *p, const int32_t *cand_offsets, const int32_t *cand_parent,
                          const int32_t *caps, int B, int M, int budget, int32_t *offsets,
                          int32_t *parent, int32_t *src, float *rho, void *ws, int32_t *st,
                          cudaStream_t s)
{
    uint64_t *lists = static_cast<uint64_t *>(ws);
    int32_t *lens = reinterpret_cast<int32_t *>(lists + (size_t)B * kListLen);
    int32_t *counts = lens + B;
    cudaError_t e = cudaMemsetAsync(st, 0, BOLE_STATUS_WORDS * sizeof(int32_t), s);
    if (e != cudaSuccess) return e;
    if (B == 0) return cudaMemsetAsync(offsets, 0, sizeof(int32_t), s); // the empty forest
    select_local_kernel<<<B, kSelThreads, 0, s>>>(p, cand_offsets, cand_parent, caps, M, rho,
                                                  lists, lens, st);
    select_global_kernel<<<B, kRankThreads, 0, s>>>(lists, lens, B, budget, counts);
    build_forest_kernel<<<B, kGlobThreads, 0, s>>>(lists, counts, cand_offsets, cand_parent, B,
                                                   offsets, parent, src, st);
    return cudaGetLastError();
}

} // namespace bole
