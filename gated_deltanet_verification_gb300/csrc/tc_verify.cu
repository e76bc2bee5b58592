// Tensor-core (TMA + tcgen05) verification and commit for bf16 q/k/v with
// d_k = d_v = 128 -- the Qwen3.5-shaped GDN head of the pages' evaluation.
//
// Verification, one CTA per (request, head), two CTAs per SM, trees of up to
// 64 nodes and depth <= 15:
//   1. TMA streams the head's S_pre (128 x 128 fp32, 128B-swizzled, four
//      32-column boxes) into shared memory while the CTA stages [Q;K] of the
//      tree as one 128 x 128 bf16 operand (rows 0..63 = q, 64..127 = k).
//   2. S_pre is split exactly into bf16 S_hi + S_lo (S - S_hi rounds to bf16
//      with ~2^-18 relative residue), and tcgen05 computes in tensor memory the
//      Gram [Q;K] K^T and the state products [Q;K] (S_hi + S_lo), all with bf16
//      products (exact) and fp32 accumulation.
//   3. From the Gram the CTA forms the ancestor-masked factors
//      G_ij = beta_i (P_i/P_j) k_i.k_j and C_ij = (P_i/P_j) q_i.k_j (Lemma 2,
//      Lemma 1), stored compactly by ancestor depth, and runs the d-step
//      Neumann recurrence Z <- -G Z, W += Z (Eq. (8)) on the identity, which
//      yields W = (I+G)^{-1} (Lemma 3); M = C W follows.  All on chip.
//   4. Epilogue of the state products: B0 = D_P Q S_pre stays in tensor
//      memory, R = D_beta (V - D_P K S_pre) goes to shared memory (as R^T).
//   5. One more tcgen05 product (tf32) [M; W] R accumulates M R onto B0
//      (giving O) and writes W R (= U) in the other 64 rows.
// Deviation from the pages' kernel: the Neumann recurrence runs on the
// T x T identity instead of on each value tile's R.  The tree factor W does
// not depend on the value columns, so the d dependent steps stay small and
// off the state-streaming path, and propagation + read-out become one dense
// tensor-core product per head.  The result is the same polynomial, Eq. (6).
//
// Commit, one CTA per (request, head) with an accepted node: TMA loads S,
// one tcgen05 product (D_a K_a)^T U_a over the accepted path (K chunks of 32
// path nodes), the epilogue adds P_a S and TMA stores S in place (Eq. (10)).
#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"
#include "sm100.cuh"

namespace bole {
namespace {

using namespace sm100;

constexpr int kT = 64;        // padded tree extent
constexpr int kD = 128;       // d_k = d_v
constexpr int kSlots = 16;    // depth slots in the compact factors: depth <= 15
constexpr int kLd = 17;       // padded row stride of the compact factors (bank spread)
constexpr uint64_t kWaitNs = 200ull * 1000 * 1000; // 200 ms bound on any device wait

// ---- per-head pair records: the factor kernel's output, the solve kernel's input ----
// For head (b, h) the records start at ((offsets[b] * H) + h * T_b) * kSlots and hold,
// for every pair (node i, ancestor slot t <= depth(i)) with j the ancestor of i at
// depth t: M_ij = (C W)_ij and W_ij.  At most T_b * kSlots records per head, so the
// workspace is bounded by N * H * kSlots records (plus one count per head).
struct PairRec {
    float m, w;
    int i, j;
};
static_assert(sizeof(PairRec) == 16, "16-byte records");

// =====================================================================
// factor kernel: the per-(request, head) producer of the tree factors
// =====================================================================
// One CTA per (request, head), three CTAs per SM (58 KB shared memory, 64
// tensor-memory columns).  It forms the cumulative decay, the Gram [Q;K] K^T
// on tcgen05 (bf16 products, exact, fp32 accumulation), the ancestor-masked
//   C_ij = exp(L_i - L_j) q_i.k_j        (j an ancestor of i or i itself)
//   G_ij = beta_i exp(L_i - L_j) k_i.k_j (j a strict ancestor of i)
// compactly by ancestor depth, runs the d-step Neumann recurrence
// Z <- -G Z, W += Z on the identity (Eq. (8)), which gives W = (I+G)^{-1}
// (Lemma 3), and writes M = C W and W as pair records.
constexpr int kFThreads = 256;
constexpr int kMaxPairs = kT * kSlots;
constexpr int F_A1 = 0;                         // [Q;K] bf16 K-major, then the staged Gram
constexpr int F_FAC = 32768;                    // G, C, Za, Zb, W: [64][17] f32 each
constexpr int F_FAC_BYTES = kT * kLd * 4;
constexpr int F_ANCAT = F_FAC + 5 * F_FAC_BYTES; // [64][16] u8
constexpr int F_PAIRS = F_ANCAT + kT * kSlots;   // u16 (i << 8 | t)
constexpr int F_L = F_PAIRS + kMaxPairs * 2;
constexpr int F_BETA = F_L + kT * 4;
constexpr int F_DEPTH = F_BETA + kT * 4;
constexpr int F_BAR = F_DEPTH + kT * 4;         // mbarriers: A1, Gram
constexpr int F_MISC = F_BAR + 16;              // TMEM slot, pair count
constexpr int FACTOR_SMEM = F_MISC + 16 + 1024;
static_assert(FACTOR_SMEM <= 75 * 1024, "three factor CTAs per SM");

constexpr uint32_t IDESC_GRAM = idesc_bf16(128, 64, false, false);  // [Q;K] K^T

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__global__ void __launch_bounds__(kFThreads, 3)
tc_factor_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const float *__restrict__ gamma, const float *__restrict__ beta,
                 const int32_t *__restrict__ offsets, const int32_t *__restrict__ depth_g,
                 const uint32_t *__restrict__ anc_g, const int32_t *__restrict__ req_depth, int H,
                 int N, float *__restrict__ logP, PairRec *__restrict__ recs,
                 int32_t *__restrict__ counts, int32_t *st)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *sA1 = sm + F_A1;
    float *gram = reinterpret_cast<float *>(sm + F_A1); // [128][64], column XOR row % 32
    float *Gc = reinterpret_cast<float *>(sm + F_FAC);
    float *Cc = Gc + kT * kLd;
    float *Za = Cc + kT * kLd;
    float *Zb = Za + kT * kLd;
    float *Wc = Zb + kT * kLd;
    uint8_t *ancat = sm + F_ANCAT;
    uint16_t *pairs = reinterpret_cast<uint16_t *>(sm + F_PAIRS);
    float *Ls = reinterpret_cast<float *>(sm + F_L);
    float *Bs = reinterpret_cast<float *>(sm + F_BETA);
    int *Ds = reinterpret_cast<int *>(sm + F_DEPTH);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + F_BAR); // A1, Gram
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + F_MISC);
    int *npair = reinterpret_cast<int *>(sm + F_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x;
    const int b = unit / H, h = unit % H;
    if (faulted(st)) return;
    const int o = offsets[b], T = offsets[b + 1] - o;
    if (T <= 0) return;
    const int d = req_depth[b];
    if (T > kT || o < 0 || o + T > N || d < 0 || d >= kSlots || d >= T) {
        if (tid == 0)
            report(st, T > kT || o < 0 || o + T > N ? BOLE_ERR_BAD_TOPOLOGY : BOLE_ERR_DEPTH, b,
                   -1, T > kT ? T : d);
        return;
    }

    if (tid == 32) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, 64);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool ok = true;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[0], 32768);
#pragma unroll
        for (int ka = 0; ka < 2; ++ka) {
            tma_load_3d(sA1 + ka * 16384, &tmQ, &bar[0], 64 * ka, h, o);
            tma_load_3d(sA1 + ka * 16384 + 8192, &tmK, &bar[0], 64 * ka, h, o);
        }
    }

    // ---- topology, cumulative decay and the (node, ancestor slot) pair list ----
    // Warps 0 and 1 own rows 0..63 (row = tid) and also read the partner row
    // tid ^ 32, so each warp sees every row's gate and depth through shuffles:
    // L_i = sum of log gamma over the ancestors-or-self of i (the prefix along
    // parent links, Lemma 1), the ancestor-by-depth table, and the offsets of
    // each row's pairs by a 64-row scan, without a barrier.
    if (tid < kT) {
        const int i = tid, ip = i ^ 32;
        int di = -1, dp = -1;
        uint64_t mi = 0;
        float bi = 0.f, lgi = 0.f, lgp = 0.f;
        if (i < T) {
            const size_t nh = (size_t)(o + i) * H + h;
            di = depth_g[o + i];
            const uint2 m2 = *reinterpret_cast<const uint2 *>(anc_g + (size_t)(o + i) * 4);
            mi = ((uint64_t)m2.y << 32) | m2.x;
            bi = beta[nh];
            lgi = logf(gamma[nh]);
        }
        if (ip < T) {
            dp = depth_g[o + ip];
            lgp = logf(gamma[(size_t)(o + ip) * H + h]);
        }
        const float lg_lo = (i < 32) ? lgi : lgp; // log gamma of row `lane`
        const float lg_hi = (i < 32) ? lgp : lgi; // log gamma of row `lane` + 32
        const int cnt = di + 1;
        int maxcnt = cnt;
#pragma unroll
        for (int sft = 16; sft > 0; sft >>= 1)
            maxcnt = max(maxcnt, __shfl_xor_sync(0xffffffffu, maxcnt, sft));
        float L = 0.f;
        uint64_t mm = mi;
        for (int t = 0; t < maxcnt; ++t) {
            const int j = mm ? __ffsll((long long)mm) - 1 : 0;
            const float vlo = __shfl_sync(0xffffffffu, lg_lo, j & 31);
            const float vhi = __shfl_sync(0xffffffffu, lg_hi, j & 31);
            if (mm) {
                L += (j < 32) ? vlo : vhi;
                ancat[i * kSlots + t] = (uint8_t)j;
                mm &= mm - 1;
            }
        }
        int c_lo = (i < 32) ? cnt : dp + 1, c_hi = (i < 32) ? dp + 1 : cnt;
#pragma unroll
        for (int sft = 1; sft < 32; sft <<= 1) {
            const int ylo = __shfl_up_sync(0xffffffffu, c_lo, sft);
            const int yhi = __shfl_up_sync(0xffffffffu, c_hi, sft);
            if (lane >= sft) {
                c_lo += ylo;
                c_hi += yhi;
            }
        }
        const int tot_lo = __shfl_sync(0xffffffffu, c_lo, 31);
        const int tot_hi = __shfl_sync(0xffffffffu, c_hi, 31);
        const int start = ((i < 32) ? c_lo : tot_lo + c_hi) - cnt;
        for (int t = 0; t < cnt; ++t) {
            pairs[start + t] = (uint16_t)((i << 8) | t);
            const float id = (t == di) ? 1.f : 0.f; // Z^(0) = W = identity
            Za[i * kLd + t] = id;
            Wc[i * kLd + t] = id;
        }
        Ds[i] = di;
        Bs[i] = bi;
        Ls[i] = L;
        if (i < T) logP[(size_t)(o + i) * H + h] = L;
        if (i == 0) *npair = tot_lo + tot_hi;
    }

    // ---- Gram [Q;K] K^T on the tensor core, staged back into the [Q;K] buffer ----
    if (tid == 0) {
        ok &= mbar_wait(&bar[0], 0, kWaitNs);
        tc_fence_after();
        const uint32_t a1 = smem_addr(sA1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16_ss(tmem, sdesc_sw128(a1 + off, 16, 1024),
                        sdesc_sw128(a1 + off + 8192, 16, 1024), IDESC_GRAM, kk > 0);
        }
        mma_commit(&bar[1]);
    }
    ok &= mbar_wait(&bar[1], 0, kWaitNs);
    tc_fence_after();
    {
        const int rowgrp = warp & 3, half = warp >> 2;
        const int m = rowgrp * 32 + lane; // row 0..63 q_i.k_j, 64..127 k_i.k_j
        float g[32];
        tmem_ld32(tmem + ((uint32_t)(rowgrp * 32) << 16) + half * 32, g);
#pragma unroll
        for (int t = 0; t < 32; ++t) gram[m * 64 + ((half * 32 + t) ^ (m & 31))] = g[t];
    }
    tc_fence_before();
    __syncthreads();
    const int P = *npair;

    // ---- compact C and G, one thread per (node, ancestor slot) pair ----
    for (int p = tid; p < P; p += kFThreads) {
        const int pr = pairs[p];
        const int i = pr >> 8, t = pr & 255;
        const int j = ancat[i * kSlots + t];
        const float ratio = __expf(Ls[i] - Ls[j]);
        Cc[i * kLd + t] = ratio * gram[i * 64 + (j ^ (i & 31))];
        if (t < Ds[i]) Gc[i * kLd + t] = Bs[i] * ratio * gram[(64 + i) * 64 + (j ^ (i & 31))];
    }
    __syncthreads();

    // ---- W = sum_{m<=d} (-G)^m by Z <- -G Z, W += Z (Eq. (8) on the identity) ----
    // Pair (i, t): row i's coefficient on its ancestor at depth t.  Z^(m) can be
    // nonzero only where depth(i) - t >= m; one thread per pair.
    {
        float *Zc = Za, *Zn = Zb;
        for (int step = 0; step < d; ++step) {
            for (int p = tid; p < P; p += kFThreads) {
                const int pr = pairs[p];
                const int i = pr >> 8, t = pr & 255;
                const int di = Ds[i];
                if (t + step >= di) continue;
                const float *gi = Gc + i * kLd;
                const uint8_t *ai = ancat + i * kSlots;
                float v0 = 0.f, v1 = 0.f;
                int s2 = t + step;
                for (; s2 + 1 < di; s2 += 2) {
                    v0 = fmaf(gi[s2], Zc[ai[s2] * kLd + t], v0);
                    v1 = fmaf(gi[s2 + 1], Zc[ai[s2 + 1] * kLd + t], v1);
                }
                if (s2 < di) v0 = fmaf(gi[s2], Zc[ai[s2] * kLd + t], v0);
                const float val = -(v0 + v1);
                Zn[i * kLd + t] = val;
                Wc[i * kLd + t] += val;
            }
            __syncthreads();
            float *tmp = Zc; Zc = Zn; Zn = tmp;
        }
    }

    // ---- M = C W and W as pair records ----
    PairRec *out = recs + ((size_t)o * H + (size_t)h * T) * kSlots;
    for (int p = tid; p < P; p += kFThreads) {
        const int pr = pairs[p];
        const int i = pr >> 8, t = pr & 255;
        const int di = Ds[i];
        const float *ci = Cc + i * kLd;
        const uint8_t *ai = ancat + i * kSlots;
        float mval = 0.f;
        for (int s2 = t; s2 <= di; ++s2) mval = fmaf(ci[s2], Wc[ai[s2] * kLd + t], mval);
        PairRec r;
        r.m = mval;
        r.w = Wc[i * kLd + t];
        r.i = i;
        r.j = ai[t];
        out[p] = r;
    }
    if (tid == 0) {
        counts[unit] = P;
        if (!ok) report(st, BOLE_ERR_TIMEOUT, b, -1, 0);
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

// =====================================================================
// solve kernel: value tile = the whole head (b_v = d_v = 128)
// =====================================================================
// Shared-memory plan (bytes from a 1024-aligned base), two CTAs per SM:
//   S buffer (64 KB): four 16 KB boxes [128 rows x 128 B] of fp32 S_pre; the
//     in-place split turns boxes (0,1) into (S_hi, S_lo) of columns 0..63 and
//     boxes (2,3) into those of columns 64..127 (bf16, 128B-swizzled,
//     N-contiguous); after the state products it holds [M;W] (first 32 KB,
//     tf32 K-major) and R^T (second 32 KB, tf32 K-major).
//   A1 (32 KB): [Q;K] bf16 K-major (rows 0..63 q, 64..127 k).
//   V (16 KB): the head's value rows, two 128B-swizzled boxes [64 rows x 64
//     bf16], loaded by TMA beside the state so the epilogue reads them from
//     shared memory (row-per-thread global loads cost several microseconds).
// Tensor memory (256 columns, 128 lanes = operand rows): columns 0..127 hold
// [Q S_pre; K S_pre], columns 128..255 the propagation [M R; W R].  The
// epilogues only read it, so no tensor-memory store sits between the state
// products and the second MMA.
constexpr int OFF_SBUF = 0;
constexpr int SBUF_BYTES = 65536;
constexpr int OFF_A1 = SBUF_BYTES;
constexpr int OFF_V = OFF_A1 + 32768;
constexpr int OFF_BAR = OFF_V + 16384;        // mbarriers
constexpr int OFF_MISC = OFF_BAR + 8 * 8;     // TMEM slot
constexpr int SOLVE_END = OFF_MISC + 16;
// Two CTAs per SM leave 113 KB each (228 KB less 1 KB reserved per CTA); the
// plan fills 112 KB and keeps 256 B of slack for the 1024 B alignment of the
// dynamic base, which is aligned when the kernel has no static shared memory
// (checked in the kernel).  A request at the 113 KB edge would drop to one CTA
// per SM as soon as anything else claimed shared memory.
constexpr int SOLVE_SMEM = SOLVE_END + 256;
static_assert(2 * (SOLVE_SMEM + 1024) <= 228 * 1024, "two solve CTAs per SM");
static_assert(3 * SOLVE_SMEM > 228 * 1024, "at most two solve CTAs (2 x 256 TMEM columns) per SM");

constexpr int kComputeThreads = 256;          // warps 0..7: split, epilogues, scatter
constexpr int kThreads = kComputeThreads + 32; // warp 8: TMA and tcgen05 issue

constexpr uint32_t IDESC_STATE = idesc_bf16(128, 128, false, true); // [Q;K] S, S N-contiguous
constexpr uint32_t IDESC_TF32 = idesc_tf32(128, 128, false, false); // both K-major

// mbarrier slots
constexpr int BAR_S = 0, BAR_A1 = 1, BAR_STATE = 2, BAR_MMA2 = 3, BAR_CONV = 4, BAR_OPS = 5,
              BAR_V = 6;


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


__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Barrier among the compute warps only (the issue warp keeps running).
__device__ __forceinline__ void compute_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kComputeThreads) : "memory");
}

// One CTA per (request, head): state products on tcgen05, R, and the
// propagation + read-out product [M; W] R.  Warp 8 streams operands and
// issues the tensor-core products; warps 0..7 do everything else.  All waits
// are bounded.
__global__ void __launch_bounds__(kThreads, 2)
tc_solve_kernel(const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmQ,
                const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const float *__restrict__ beta, const int32_t *__restrict__ offsets,
                const int32_t *__restrict__ req_depth, const float *__restrict__ logP,
                const PairRec *__restrict__ recs, const int32_t *__restrict__ counts, int H, int N,
                __nv_bfloat16 *__restrict__ O, float *__restrict__ Uout, int32_t *st)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *sbuf = sm + OFF_SBUF;
    uint8_t *sA1 = sm + OFF_A1;
    uint8_t *sV = sm + OFF_V;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x;
    const int b = unit / H, h = unit % H;

    // Uniform early exits, before any barrier or tensor-memory allocation
    // (the factor kernel reported any fault of this head).
    if (faulted(st)) return;
    const int o = offsets[b], T = offsets[b + 1] - o;
    if (T <= 0) return;
    const int d = req_depth[b];
    if (T > kT || o < 0 || o + T > N || d < 0 || d >= kSlots || d >= T) return;
    if (sm + SOLVE_END > smem_raw + SOLVE_SMEM) { // dynamic base too far from 1024 B
        if (tid == 0) report(st, BOLE_ERR_CUDA, b, -1, -1);
        return;
    }

    if (tid == 32) {
        for (int i = BAR_S; i <= BAR_MMA2; ++i) mbar_init(&bar[i], 1);
        mbar_init(&bar[BAR_V], 1);
        mbar_init(&bar[BAR_CONV], kComputeThreads);
        mbar_init(&bar[BAR_OPS], kComputeThreads);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == kComputeThreads / 32) {
        // =========================== issue warp ===========================
        const uint32_t a1 = smem_addr(sA1), s0 = smem_addr(sbuf);
        bool ok = true;
        if (lane == 0) {
            mbar_arrive_expect_tx(&bar[BAR_S], SBUF_BYTES);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tma_load_2d(sbuf + c * 16384, &tmS, &bar[BAR_S], 32 * c, unit * kD);
            mbar_arrive_expect_tx(&bar[BAR_A1], 32768);
#pragma unroll
            for (int ka = 0; ka < 2; ++ka) {
                tma_load_3d(sA1 + ka * 16384, &tmQ, &bar[BAR_A1], 64 * ka, h, o);
                tma_load_3d(sA1 + ka * 16384 + 8192, &tmK, &bar[BAR_A1], 64 * ka, h, o);
            }
            mbar_arrive_expect_tx(&bar[BAR_V], 16384);
            tma_load_3d(sV, &tmV, &bar[BAR_V], 0, h, o);
            tma_load_3d(sV + 8192, &tmV, &bar[BAR_V], 64, h, o);
        }
        // state products [Q;K] (S_hi + S_lo) once the split is in place
        ok &= mbar_wait(&bar[BAR_A1], 0, kWaitNs);
        ok &= mbar_wait(&bar[BAR_CONV], 0, kWaitNs);
        tc_fence_after();
        if (lane == 0) {
            const uint32_t slo = s0 + 16384;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad = sdesc_sw128(a1 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                mma_bf16_ss(tmem, ad, sdesc_sw128(s0 + kk * 2048, 32768, 1024), IDESC_STATE, kk > 0);
                mma_bf16_ss(tmem, ad, sdesc_sw128(slo + kk * 2048, 32768, 1024), IDESC_STATE, 1);
            }
            mma_commit(&bar[BAR_STATE]);
        }
        __syncwarp();
        // propagation + read-out: [M; W] R accumulated onto [B0; 0]
        ok &= mbar_wait(&bar[BAR_OPS], 0, kWaitNs);
        tc_fence_after();
        if (lane == 0) {
            const uint32_t b2 = s0 + 32768;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_tf32_ss(tmem + 128, sdesc_sw128(s0 + off, 16, 1024),
                            sdesc_sw128(b2 + off, 16, 1024), IDESC_TF32, kk > 0);
            }
            mma_commit(&bar[BAR_MMA2]);
        }
        __syncwarp();
        if (!ok && lane == 0) report(st, BOLE_ERR_TIMEOUT, b, -1, 0);
    } else {
        // ========================== compute warps =========================
        const int rowgrp = warp & 3, half = warp >> 2;
        const int m = rowgrp * 32 + lane;    // TMEM lane = operand row
        const uint32_t lane_base = (uint32_t)(rowgrp * 32) << 16;
        bool ok = true;
        // this thread's operand row: P_i for both halves, beta_i for the K half
        const int i = m & 63;
        const float p = (i < T) ? expf(logP[(size_t)(o + i) * H + h]) : 0.f;
        const float bt = (m >= 64 && i < T) ? beta[(size_t)(o + i) * H + h] : 0.f;
        // this thread's pair records (at most kMaxPairs / 256 = 4), fetched early
        const int P = counts[unit];
        const PairRec *rin = recs + ((size_t)o * H + (size_t)h * T) * kSlots;
        PairRec rec[kMaxPairs / kComputeThreads];
#pragma unroll
        for (int u = 0; u < kMaxPairs / kComputeThreads; ++u) {
            const int p = tid + u * kComputeThreads;
            if (p < P) rec[u] = rin[p];
        }

        // ---- S_pre = S_hi + S_lo in place (bf16, N-contiguous, 64-column atoms) ----
        ok &= mbar_wait(&bar[BAR_S], 0, kWaitNs);
        {
            const int r = tid & 127, p = tid >> 7; // row r, columns 64p .. 64p+63
            uint8_t *box0 = sbuf + (2 * p) * 16384, *box1 = box0 + 16384;
            float x[64];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 a0 = *reinterpret_cast<const float4 *>(box0 + sw128_chunk(r, c));
                const float4 a1v = *reinterpret_cast<const float4 *>(box1 + sw128_chunk(r, c));
                x[4 * c + 0] = a0.x; x[4 * c + 1] = a0.y; x[4 * c + 2] = a0.z; x[4 * c + 3] = a0.w;
                x[32 + 4 * c + 0] = a1v.x; x[32 + 4 * c + 1] = a1v.y;
                x[32 + 4 * c + 2] = a1v.z; x[32 + 4 * c + 3] = a1v.w;
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float x0 = x[8 * c + 2 * t], x1 = x[8 * c + 2 * t + 1];
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
                    const float2 hf = __bfloat1622float2(h2);
                    const __nv_bfloat162 l2 = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
                    hw[t] = *reinterpret_cast<const uint32_t *>(&h2);
                    lw[t] = *reinterpret_cast<const uint32_t *>(&l2);
                }
                *reinterpret_cast<uint4 *>(box0 + sw128_chunk(r, c)) =
                    make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4 *>(box1 + sw128_chunk(r, c)) =
                    make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bar[BAR_CONV]);

        // ---- state epilogue: rows 0..63 zero the [M; W] operand; rows 64..127
        //      write R^T = (beta (v - P K S_pre))^T.  No tensor-memory stores:
        //      Q S_pre stays in columns 0..127 and is scaled by P at the output ----
        ok &= mbar_wait(&bar[BAR_STATE], 0, kWaitNs);
        tc_fence_after();
        if (m < 64) {
            float4 *a2z = reinterpret_cast<float4 *>(sbuf);
            const int zt = (half * 64 + m); // 0..127
#pragma unroll
            for (int e = 0; e < 16; ++e) a2z[zt + e * 128] = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            uint8_t *sB2 = sbuf + 32768;
            uint8_t *dst = sB2 + (i >> 5) * 16384;
            const uint8_t *vrow = sV + half * 8192 + i * 128; // 64 columns of row i
            ok &= mbar_wait(&bar[BAR_V], 0, kWaitNs);
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
                const int col0 = half * 64 + cc * 32;
                float x[32];
                tmem_ld32(tmem + lane_base + col0, x);
#pragma unroll
                for (int uu = 0; uu < 4; ++uu) {
                    float f[8];
                    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(
                                      vrow + (((cc * 4 + uu) ^ (i & 7)) << 4)), f);
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const int c = 8 * uu + t;
                        const float r = (i < T) ? bt * (f[t] - p * x[c]) : 0.f;
                        *reinterpret_cast<float *>(dst + sw128_offset(col0 + c, i & 31)) = r;
                    }
                }
            }
        }
        compute_sync(); // operand zeroed
        // ---- [M; W] from the factor kernel's pair records ----
#pragma unroll
        for (int u = 0; u < kMaxPairs / kComputeThreads; ++u) {
            if (tid + u * kComputeThreads < P) {
                const PairRec r = rec[u];
                uint8_t *col = sbuf + (r.j >> 5) * 16384;
                *reinterpret_cast<float *>(col + sw128_offset(r.i, r.j & 31)) = r.m;
                *reinterpret_cast<float *>(col + sw128_offset(64 + r.i, r.j & 31)) = r.w;
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bar[BAR_OPS]);

        // ---- outputs: O = P (Q S_pre) + M R (bf16), U = W R (fp32) ----
        ok &= mbar_wait(&bar[BAR_MMA2], 0, kWaitNs);
        tc_fence_after();
        {
            const bool store = ok && i < T;
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
                const int col0 = half * 64 + cc * 32;
                float x[32];
                tmem_ld32(tmem + 128 + lane_base + col0, x);
                if (m < 64) {
                    float y[32];
                    tmem_ld32(tmem + lane_base + col0, y);
#pragma unroll
                    for (int t = 0; t < 32; ++t) x[t] = fmaf(p, y[t], x[t]);
                }
                if (!store) continue;
                const size_t row = ((size_t)(o + i) * H + h) * kD + col0;
                if (m < 64) {
                    uint4 *dst = reinterpret_cast<uint4 *>(O + row);
#pragma unroll
                    for (int uu = 0; uu < 4; ++uu) {
                        __nv_bfloat162 p2[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t)
                            p2[t] = __floats2bfloat162_rn(x[8 * uu + 2 * t], x[8 * uu + 2 * t + 1]);
                        dst[uu] = *reinterpret_cast<uint4 *>(p2);
                    }
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(Uout + row);
#pragma unroll
                    for (int uu = 0; uu < 8; ++uu)
                        dst[uu] = make_float4(x[4 * uu], x[4 * uu + 1], x[4 * uu + 2], x[4 * uu + 3]);
                }
            }
        }
        if (!ok && tid == 0) report(st, BOLE_ERR_TIMEOUT, b, -1, 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---- commit ----
// One CTA per (request, head, 64-column half of the state): value tiling as in
// the pages' kernel, so four CTAs fit on an SM and overlap their TMA load,
// tensor-core product and TMA store.
constexpr int kCommitThreads = 128;
constexpr int kChunk = 16;                    // path nodes per MMA K chunk
constexpr int kHalf = 64;                     // state columns per CTA
constexpr int CO_S = 0;                       // S half: 2 boxes x [128 rows x 128 B] = 32 KB
constexpr int CO_A = 32768;                   // (D_a K_a)^T chunk: 128 rows x 16 tf32 (64 B rows)
constexpr int CO_B = CO_A + 8192;             // U_a^T chunk: 64 rows x 16 tf32
constexpr int CO_PATH = CO_B + 4096;          // int[128]
constexpr int CO_COEF = CO_PATH + 512;        // float[128]
constexpr int CO_BAR = CO_COEF + 512;         // 2 mbarriers
constexpr int CO_TSLOT = CO_BAR + 16;
constexpr int CO_MISC = CO_TSLOT + 4;         // path length, flag
constexpr int CO_PAR = CO_MISC + 16;          // int[128]: the request's parent links
constexpr int COMMIT_SMEM = CO_PAR + 512 + 1024;

constexpr uint32_t IDESC_COMMIT = idesc_tf32(128, kHalf, false, false);

// 64-byte-swizzled K-major operand with 64-byte rows (16 tf32): the 16-byte
// chunk index (0..3) is XORed with (row / 2) % 4.
__device__ __forceinline__ uint32_t sw64_offset(int row, int col_f32)
{
    return (uint32_t)row * 64u + ((((uint32_t)col_f32 >> 2) ^ (((uint32_t)row >> 1) & 3u)) << 4) +
           (((uint32_t)col_f32 & 3u) << 2);
}

// 64B-swizzle variant of the shared-memory descriptor (layout code 4).
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (4ull << 61);
}

__global__ void __launch_bounds__(kCommitThreads)
tc_commit_kernel(const __grid_constant__ CUtensorMap tmS, const __nv_bfloat16 *__restrict__ k,
                 const float *__restrict__ U, const float *__restrict__ logP,
                 const int32_t *__restrict__ offsets, const int32_t *__restrict__ parent,
                 const int32_t *__restrict__ accepted, int H, int N, int32_t *st)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *sS = sm + CO_S;
    uint8_t *sA = sm + CO_A;
    uint8_t *sB = sm + CO_B;
    int *path = reinterpret_cast<int *>(sm + CO_PATH);
    float *coef = reinterpret_cast<float *>(sm + CO_COEF);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + CO_BAR); // tma, mma
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + CO_TSLOT);
    int *plen = reinterpret_cast<int *>(sm + CO_MISC);
    int *flag = plen + 1;
    int *spar = reinterpret_cast<int *>(sm + CO_PAR);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int unit = blockIdx.x, hv = blockIdx.y; // head unit, value half
    const int b = unit / H, h = unit % H;
    if (faulted(st)) return;
    const int a = accepted[b];
    if (a < 0) return;
    const int o = offsets[b], T = offsets[b + 1] - o;
    if (a >= T || o < 0 || o + T > N || T > kMaxTree) {
        if (tid == 0 && hv == 0) report(st, BOLE_ERR_BAD_TOPOLOGY, b, a, T);
        return;
    }
    if (warp == 0) {
        tmem_alloc(tslot, 64);
        tmem_relinquish();
    }
    if (tid == 32) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        *flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (tid == 0) {
        prefetch_tensormap(&tmS);
        mbar_arrive_expect_tx(&bar[0], 2 * 16384);
        tma_load_2d(sS, &tmS, &bar[0], kHalf * hv, unit * kD);
        tma_load_2d(sS + 16384, &tmS, &bar[0], kHalf * hv + 32, unit * kD);
    }
    // stage the request's parent links (coalesced), then walk the accepted path
    for (int i = tid; i < T; i += kCommitThreads) spar[i] = parent[o + i];
    __syncthreads();
    if (tid == 0) {
        int L = 0, j = a;
        bool ok = true;
        while (j >= 0) {
            if (L >= kMaxTree) { ok = false; break; }
            path[L++] = j;
            const int p = spar[j];
            if (p < -1 || p >= j) { ok = false; break; }
            j = p;
        }
        if (!ok) {
            if (hv == 0) report(st, BOLE_ERR_BAD_TOPOLOGY, b, j, -1);
            *flag = 1;
        }
        *plen = L;
    }
    __syncthreads();
    const int L = *plen;
    const float La = logP[(size_t)(o + a) * H + h];
    for (int t = tid; t < L; t += kCommitThreads)
        coef[t] = expf(La - logP[(size_t)(o + path[t]) * H + h]);
    __syncthreads();

    const uint32_t sa = smem_addr(sA), sb = smem_addr(sB);
    const int nchunks = (*(volatile int *)flag != 0) ? 0 : (L + kChunk - 1) / kChunk;
    for (int ch = 0; ch < nchunks; ++ch) {
        // A[r][t] = coef_t k_{j_t}[r] (row r = tid), K-major, 64-byte rows
        {
            const int r = tid;
            float av[kChunk];
#pragma unroll
            for (int tt = 0; tt < kChunk; ++tt) {
                const int t = ch * kChunk + tt;
                av[tt] = (t < L) ? coef[t] * __bfloat162float(k[((size_t)(o + path[t]) * H + h) * kD + r])
                                 : 0.f;
            }
#pragma unroll
            for (int c4 = 0; c4 < kChunk / 4; ++c4)
                *reinterpret_cast<float4 *>(sA + sw64_offset(r, 4 * c4)) =
                    make_float4(av[4 * c4], av[4 * c4 + 1], av[4 * c4 + 2], av[4 * c4 + 3]);
        }
        // B^T[c][t] = u_{j_t}[64 hv + c] (row c < 64), K-major, 64-byte rows
        if (tid < kHalf) {
            const int c = tid;
#pragma unroll
            for (int t4 = 0; t4 < kChunk / 4; ++t4) {
                float uv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = ch * kChunk + 4 * t4 + e;
                    uv[e] = (t < L) ? U[((size_t)(o + path[t]) * H + h) * kD + kHalf * hv + c] : 0.f;
                }
                *reinterpret_cast<float4 *>(sB + sw64_offset(c, 4 * t4)) =
                    make_float4(uv[0], uv[1], uv[2], uv[3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kChunk / 8; ++kk)
                mma_tf32_ss(tmem, sdesc_sw64(sa + kk * 32, 512), sdesc_sw64(sb + kk * 32, 512),
                            IDESC_COMMIT, (ch > 0 || kk > 0));
            mma_commit(&bar[1]);
        }
        if (!mbar_wait(&bar[1], ch & 1, kWaitNs)) {
            report(st, BOLE_ERR_TIMEOUT, b, -1, 7);
            *flag = 1;
        }
        tc_fence_after();
        __syncthreads();
    }

    // epilogue: S <- P_a S + D, in shared memory, then TMA store in place
    if (!mbar_wait(&bar[0], 0, kWaitNs)) {
        report(st, BOLE_ERR_TIMEOUT, b, -1, 8);
        *flag = 1;
    }
    const bool ok = *(volatile int *)flag == 0;
    if (ok && nchunks > 0) {
        const float Pa = expf(La);
        const int r = tid;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
        for (int cb = 0; cb < 2; ++cb) {
            float x[32];
            tmem_ld32(tmem + lane_base + cb * 32, x);
            uint8_t *tile = sS + cb * 16384;
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                float4 *p = reinterpret_cast<float4 *>(tile + sw128_offset(r, 4 * c4));
                float4 s4 = *p;
                s4.x = fmaf(Pa, s4.x, x[4 * c4 + 0]);
                s4.y = fmaf(Pa, s4.y, x[4 * c4 + 1]);
                s4.z = fmaf(Pa, s4.z, x[4 * c4 + 2]);
                s4.w = fmaf(Pa, s4.w, x[4 * c4 + 3]);
                *p = s4;
            }
        }
        fence_proxy_async_smem();
    }
    __syncthreads();
    if (tid == 0 && ok && nchunks > 0) {
        tma_store_2d(&tmS, sS, kHalf * hv, unit * kD);
        tma_store_2d(&tmS, sS + 16384, kHalf * hv + 32, unit * kD);
        bulk_commit_group();
        bulk_wait_group_read0();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

// ---- host side ----

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
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
cudaError_t make_state_map(CUtensorMap *map, const float *S, int units)
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

} // namespace

bool tc_verify_supported(const VerifyArgs &a)
{
    return a.dtype == BOLE_BF16 && a.dk == kD && a.dv == kD && a.max_T <= kT &&
           a.max_depth < kSlots;
}

size_t tc_workspace_bytes(int B, int H, int max_T)
{
    const size_t recs = (size_t)B * max_T * H * kSlots * sizeof(PairRec);
    return recs + (size_t)B * H * sizeof(int32_t);
}

// q or k [N][H][128] bf16 as a 3-D tensor, boxes of 64 elements x 1 head x 64 nodes.
cudaError_t make_node_map(CUtensorMap *map, const void *x, int N, int H)
{
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)N};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kT};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(x), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_tc_verify(const VerifyArgs &a, cudaStream_t s)
{
    const int units = a.B * a.H;
    if (units == 0 || a.N == 0) return cudaSuccess;
    CUtensorMap mS, mQ, mK, mV;
    cudaError_t e = make_state_map(&mS, a.S_pre, units);
    if (e == cudaSuccess) e = make_node_map(&mQ, a.q, a.N, a.H);
    if (e == cudaSuccess) e = make_node_map(&mK, a.k, a.N, a.H);
    if (e == cudaSuccess) e = make_node_map(&mV, a.v, a.N, a.H);
    if (e != cudaSuccess) return e;
    PairRec *recs = static_cast<PairRec *>(a.ws);
    int32_t *counts = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(a.ws) +
                                                  (size_t)a.B * a.max_T * a.H * kSlots * sizeof(PairRec));
    e = cudaFuncSetAttribute(tc_factor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             FACTOR_SMEM);
    if (e != cudaSuccess) return e;
    tc_factor_kernel<<<units, kFThreads, FACTOR_SMEM, s>>>(
        mQ, mK, a.gamma, a.beta, a.offsets, a.depth, a.anc, a.req_depth, a.H, a.N, a.logP, recs,
        counts, a.st);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(tc_solve_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(tc_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SOLVE_SMEM);
    if (e != cudaSuccess) return e;
    tc_solve_kernel<<<units, kThreads, SOLVE_SMEM, s>>>(
        mS, mQ, mK, mV, a.beta, a.offsets, a.req_depth,
        a.logP, recs, counts, a.H, a.N, static_cast<__nv_bfloat16 *>(a.O), a.U, a.st);
    return cudaGetLastError();
}

bool tc_commit_supported(const CommitArgs &a)
{
    return a.dtype == BOLE_BF16 && a.dk == kD && a.dv == kD;
}

cudaError_t launch_tc_commit(const CommitArgs &a, cudaStream_t s)
{
    const int units = a.B * a.H;
    if (units == 0 || a.N == 0) return cudaSuccess;
    CUtensorMap map;
    cudaError_t e = make_state_map(&map, a.S, units);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(tc_commit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             COMMIT_SMEM);
    if (e != cudaSuccess) return e;
    tc_commit_kernel<<<dim3(units, kD / kHalf), kCommitThreads, COMMIT_SMEM, s>>>(
        map, static_cast<const __nv_bfloat16 *>(a.k), a.U, a.logP, a.offsets, a.parent,
        a.accepted, a.H, a.N, a.st);
    return cudaGetLastError();
}

} // namespace bole
