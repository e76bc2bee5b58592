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

// ---- verification shared-memory plan (bytes from a 1024-aligned base) ----
// One head per CTA, two CTAs per SM: while one CTA waits on memory or on the
// tensor core, the other computes.
//   S buffer (64 KB): four 16 KB boxes [128 rows x 128 B] of fp32 S_pre; the
//     in-place split turns boxes (0,1) into (S_hi, S_lo) of columns 0..63 and
//     boxes (2,3) into those of columns 64..127 (bf16, 128B-swizzled,
//     N-contiguous); after the state products it holds [M;W] (first 32 KB,
//     tf32 K-major) and R^T (second 32 KB, tf32 K-major).
//   A1 (32 KB): [Q;K] bf16 K-major; once the state products are done it
//     holds the compact factors G, C, the Neumann iterates and W.
constexpr int OFF_SBUF = 0;
constexpr int SBUF_BYTES = 65536;
constexpr int OFF_A1 = SBUF_BYTES;
constexpr int FAC_BYTES = kT * kLd * 4;       // one compact factor [64][17] f32
constexpr int OFF_G = OFF_A1;                 // compact G (slot = ancestor depth)
constexpr int OFF_C = OFF_G + FAC_BYTES;      // compact C
constexpr int OFF_ZA = OFF_C + FAC_BYTES;     // Neumann iterates
constexpr int OFF_ZB = OFF_ZA + FAC_BYTES;
constexpr int OFF_W = OFF_ZB + FAC_BYTES;     // W = sum of iterates
static_assert(OFF_W + FAC_BYTES <= OFF_A1 + 32768, "factors fit in the [Q;K] buffer");
constexpr int OFF_ANCAT = OFF_A1 + 32768;     // [64][16] u8: ancestor at depth s
constexpr int OFF_PAIRS = OFF_ANCAT + kT * kSlots; // u16 (i << 8 | t), t <= depth(i)
constexpr int OFF_LG = OFF_PAIRS + kT * kSlots * 2; // log gamma
constexpr int OFF_L = OFF_LG + kT * 4;        // log P
constexpr int OFF_P = OFF_L + kT * 4;
constexpr int OFF_BETA = OFF_P + kT * 4;
constexpr int OFF_DEPTH = OFF_BETA + kT * 4;
constexpr int OFF_SCAN = OFF_DEPTH + kT * 4;  // per-row inclusive pair counts
constexpr int OFF_MASK = OFF_SCAN + kT * 4;   // u64 ancestor-or-self masks
constexpr int OFF_BAR = OFF_MASK + kT * 8;    // mbarriers
constexpr int OFF_MISC = OFF_BAR + 16 * 8;    // TMEM slot, flag, pair count
constexpr int VERIFY_SMEM = OFF_MISC + 32 + 1024; // + alignment slack
static_assert(VERIFY_SMEM <= 113 * 1024, "two verification CTAs per SM");

constexpr int kComputeThreads = 256;          // warps 0..7: factors, splits, epilogues
constexpr int kThreads = kComputeThreads + 32; // warp 8: TMA and tcgen05 issue

constexpr uint32_t IDESC_GRAM = idesc_bf16(128, 64, false, false);  // [Q;K] K^T
constexpr uint32_t IDESC_STATE = idesc_bf16(128, 128, false, true); // [Q;K] S, S N-contiguous
constexpr uint32_t IDESC_TF32 = idesc_tf32(128, 128, false, false); // both K-major

// mbarrier slots
constexpr int BAR_S = 0, BAR_A1 = 1, BAR_GRAM = 2, BAR_STATE = 3, BAR_MMA2 = 4, BAR_CONV = 5,
              BAR_OPS = 6;

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
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

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z)
                 : "memory");
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

// Verification kernel: one CTA per (request, head), trees of up to 64 nodes
// and depth <= 15.  Warp 8 streams operands and issues the tensor-core
// products; warps 0..7 do everything else.  All waits are bounded.
__global__ void __launch_bounds__(kThreads, 2)
tc_verify_kernel(const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmQ,
                 const __grid_constant__ CUtensorMap tmK, const __nv_bfloat16 *__restrict__ v,
                 const float *__restrict__ gamma, const float *__restrict__ beta,
                 const int32_t *__restrict__ offsets, const int32_t *__restrict__ depth_g,
                 const uint32_t *__restrict__ anc_g, const int32_t *__restrict__ req_depth, int H,
                 int N, __nv_bfloat16 *__restrict__ O, float *__restrict__ Uout,
                 float *__restrict__ logP, int32_t *st)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *sbuf = sm + OFF_SBUF;
    uint8_t *sA1 = sm + OFF_A1;
    float *Gc = reinterpret_cast<float *>(sm + OFF_G);
    float *Cc = reinterpret_cast<float *>(sm + OFF_C);
    float *Za = reinterpret_cast<float *>(sm + OFF_ZA);
    float *Zb = reinterpret_cast<float *>(sm + OFF_ZB);
    float *Wc = reinterpret_cast<float *>(sm + OFF_W);
    uint8_t *ancat = sm + OFF_ANCAT;
    uint16_t *pairs = reinterpret_cast<uint16_t *>(sm + OFF_PAIRS);
    float *Lg = reinterpret_cast<float *>(sm + OFF_LG);
    float *Ls = reinterpret_cast<float *>(sm + OFF_L);
    float *Ps = reinterpret_cast<float *>(sm + OFF_P);
    float *Bs = reinterpret_cast<float *>(sm + OFF_BETA);
    int *Ds = reinterpret_cast<int *>(sm + OFF_DEPTH);
    int *scan = reinterpret_cast<int *>(sm + OFF_SCAN);
    uint64_t *msk = reinterpret_cast<uint64_t *>(sm + OFF_MASK);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
    int *flag = reinterpret_cast<int *>(sm + OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x;
    const int b = unit / H, h = unit % H;

    // Uniform early exits, before any barrier or tensor-memory allocation.
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

    if (warp == 0) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int i = BAR_S; i <= BAR_MMA2; ++i) mbar_init(&bar[i], 1);
        mbar_init(&bar[BAR_CONV], kComputeThreads);
        mbar_init(&bar[BAR_OPS], kComputeThreads);
        *flag = 0;
        fence_mbar_init();
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
            mbar_arrive_expect_tx(&bar[BAR_A1], 32768);
#pragma unroll
            for (int ka = 0; ka < 2; ++ka) {
                tma_load_3d(sA1 + ka * 16384, &tmQ, &bar[BAR_A1], 64 * ka, h, o);
                tma_load_3d(sA1 + ka * 16384 + 8192, &tmK, &bar[BAR_A1], 64 * ka, h, o);
            }
            mbar_arrive_expect_tx(&bar[BAR_S], SBUF_BYTES);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tma_load_2d(sbuf + c * 16384, &tmS, &bar[BAR_S], 32 * c, unit * kD);
        }
        // Gram [Q;K] K^T
        ok &= mbar_wait(&bar[BAR_A1], 0, kWaitNs);
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_bf16_ss(tmem + 128, sdesc_sw128(a1 + off, 16, 1024),
                            sdesc_sw128(a1 + off + 8192, 16, 1024), IDESC_GRAM, kk > 0);
            }
            mma_commit(&bar[BAR_GRAM]);
        }
        __syncwarp();
        // state products [Q;K] (S_hi + S_lo) once the split is in place
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
                mma_tf32_ss(tmem, sdesc_sw128(s0 + off, 16, 1024), sdesc_sw128(b2 + off, 16, 1024),
                            IDESC_TF32, 1);
            }
            mma_commit(&bar[BAR_MMA2]);
        }
        __syncwarp();
        if (!ok && lane == 0) {
            report(st, BOLE_ERR_TIMEOUT, b, -1, 0);
            *flag = 1;
        }
    } else {
        // ========================== compute warps =========================
        const int rowgrp = warp & 3, half = warp >> 2;
        const int m = rowgrp * 32 + lane;    // TMEM lane = operand row
        const uint32_t lane_base = (uint32_t)(rowgrp * 32) << 16;
        bool ok = true;

        // ---- topology and gates ----
        if (tid < kT) {
            const int i = tid;
            if (i < T) {
                const size_t nh = (size_t)(o + i) * H + h;
                Ds[i] = depth_g[o + i];
                const uint2 m2 = *reinterpret_cast<const uint2 *>(anc_g + (size_t)(o + i) * 4);
                msk[i] = ((uint64_t)m2.y << 32) | m2.x;
                Bs[i] = beta[nh];
                Lg[i] = logf(gamma[nh]);
            } else {
                Ds[i] = -1;
                msk[i] = 0;
                Bs[i] = 0.f;
                Lg[i] = 0.f;
            }
        }
        compute_sync();
        // ---- cumulative decay L_i = sum of log gamma over the ancestors-or-self
        //      (the prefix along parent links, Lemma 1) and the ancestor-by-depth
        //      table; per-row pair counts scanned within each warp ----
        if (tid < kT) {
            const int i = tid;
            float L = 0.f;
            if (i < T) {
                uint64_t mm = msk[i];
                int t = 0;
                while (mm) {
                    const int j = __ffsll((long long)mm) - 1;
                    ancat[i * kSlots + t++] = (uint8_t)j;
                    L += Lg[j];
                    mm &= mm - 1;
                }
                logP[(size_t)(o + i) * H + h] = L;
            }
            Ls[i] = L;
            Ps[i] = (i < T) ? expf(L) : 0.f;
            int incl = Ds[i] + 1;
#pragma unroll
            for (int sft = 1; sft < 32; sft <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, sft);
                if (lane >= sft) incl += y;
            }
            scan[i] = incl;
        }
        compute_sync();
        // pair list (node i, ancestor slot t), t <= depth(i)
        if (tid < kT) {
            const int i = tid;
            const int incl = scan[i] + ((i >= 32) ? scan[31] : 0);
            const int di = Ds[i];
            const int start = incl - (di + 1);
            for (int t = 0; t <= di; ++t) pairs[start + t] = (uint16_t)((i << 8) | t);
        }
        const int P = scan[31] + scan[63];
        compute_sync();

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

        // ---- Gram epilogue: compact G and C (Lemma 2 / Lemma 1 read-out), written
        //      into the [Q;K] buffer once the state products have consumed it ----
        ok &= mbar_wait(&bar[BAR_GRAM], 0, kWaitNs);
        ok &= mbar_wait(&bar[BAR_STATE], 0, kWaitNs);
        tc_fence_after();
        {
            // stage the Gram rows in the S buffer (free once the state products are
            // done): [128 rows][64 + 1] f32, rows 0..63 q_i.k_j, rows 64..127 k_i.k_j
            float *gram = reinterpret_cast<float *>(sbuf);
            float g[32];
            tmem_ld32(tmem + lane_base + 128 + half * 32, g);
#pragma unroll
            for (int t = 0; t < 32; ++t) gram[m * 65 + half * 32 + t] = g[t];
        }
        compute_sync();
        // one thread per (row, ancestor): C for rows 0..63, G (strict ancestors) for 64..127
        {
            const int r = tid >> 1, part = tid & 1; // two threads per operand row
            const int i = r & 63;
            if (i < T) {
                const bool isG = r >= 64;
                uint64_t bits = msk[i];
                if (isG) bits &= ~(1ull << i);
                const float *grow = reinterpret_cast<const float *>(sbuf) + r * 65;
                float *dst = (isG ? Gc : Cc) + i * kLd;
                const float Li = Ls[i], scale = isG ? Bs[i] : 1.f;
                int n = 0;
#pragma unroll 1
                while (bits) {
                    const int j = __ffsll((long long)bits) - 1;
                    bits &= bits - 1;
                    if ((n++ & 1) == part) dst[Ds[j]] = scale * __expf(Li - Ls[j]) * grow[j];
                }
            }
        }
        // Neumann start Z^(0) = W = identity (the self entry sits at slot depth(i))
        for (int p = tid; p < P; p += kComputeThreads) {
            const int pr = pairs[p];
            const int i = pr >> 8, t = pr & 255;
            const float id = (t == Ds[i]) ? 1.f : 0.f;
            Za[i * kLd + t] = id;
            Wc[i * kLd + t] = id;
        }
        compute_sync();

        // ---- W = sum_{m<=d} (-G)^m by Z <- -G Z, W += Z (Eq. (8) on the identity) ----
        // Pair (i, t): row i's coefficient on its ancestor at depth t.  Z^(m)
        // can be nonzero only where depth(i) - t >= m; one thread per pair.
        {
            float *Zc = Za, *Zn = Zb;
            for (int step = 0; step < d; ++step) {
                for (int p = tid; p < P; p += kComputeThreads) {
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
                compute_sync();
                float *tmp = Zc; Zc = Zn; Zn = tmp;
            }
        }

        // ---- state epilogue: B0 = P Q S_pre in place; R^T = (beta (v - P K S_pre))^T;
        //      [M; W] operand zeroed ----
        {
            float4 *a2z = reinterpret_cast<float4 *>(sbuf);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                a2z[tid + e * kComputeThreads] = make_float4(0.f, 0.f, 0.f, 0.f);
            uint8_t *sB2 = sbuf + 32768;
            const int i = m & 63;
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
                const int col0 = half * 64 + cc * 32;
                float x[32];
                tmem_ld32(tmem + lane_base + col0, x);
                if (m < 64) {
                    const float p = Ps[i];
#pragma unroll
                    for (int t = 0; t < 32; ++t) x[t] *= p;
                    tmem_st32(tmem + lane_base + col0, x);
                } else {
                    const float p = Ps[i], bt = Bs[i];
                    uint8_t *dst = sB2 + (i >> 5) * 16384;
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        v + ((size_t)(o + (i < T ? i : 0)) * H + h) * kD + col0);
#pragma unroll
                    for (int uu = 0; uu < 4; ++uu) {
                        float f[8];
                        bf16x8_to_f32(src[uu], f);
#pragma unroll
                        for (int t = 0; t < 8; ++t) {
                            const int c = 8 * uu + t;
                            const float r = (i < T) ? bt * (f[t] - p * x[c]) : 0.f;
                            *reinterpret_cast<float *>(dst + sw128_offset(col0 + c, i & 31)) = r;
                        }
                    }
#pragma unroll
                    for (int t = 0; t < 32; ++t) x[t] = 0.f;
                    tmem_st32(tmem + lane_base + col0, x);
                }
            }
        }
        compute_sync(); // operand zeroed; W final
        // ---- scatter M = C W (rows 0..63) and W (rows 64..127) into [M; W] ----
        for (int p = tid; p < P; p += kComputeThreads) {
            const int pr = pairs[p];
            const int i = pr >> 8, t = pr & 255;
            const int di = Ds[i];
            const float *ci = Cc + i * kLd;
            const uint8_t *ai = ancat + i * kSlots;
            float mval = 0.f;
            for (int s2 = t; s2 <= di; ++s2) mval = fmaf(ci[s2], Wc[ai[s2] * kLd + t], mval);
            const int j = ai[t];
            uint8_t *col = sbuf + (j >> 5) * 16384;
            *reinterpret_cast<float *>(col + sw128_offset(i, j & 31)) = mval;
            *reinterpret_cast<float *>(col + sw128_offset(64 + i, j & 31)) = Wc[i * kLd + t];
        }
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar[BAR_OPS]);

        // ---- outputs: rows 0..63 O (bf16), rows 64..127 U (fp32) ----
        ok &= mbar_wait(&bar[BAR_MMA2], 0, kWaitNs);
        tc_fence_after();
        {
            const int i = m & 63;
            const bool store = ok && i < T;
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
                const int col0 = half * 64 + cc * 32;
                float x[32];
                tmem_ld32(tmem + lane_base + col0, x);
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
constexpr int COMMIT_SMEM = CO_MISC + 16 + 1024;

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
    CUtensorMap mS, mQ, mK;
    cudaError_t e = make_state_map(&mS, a.S_pre, units);
    if (e == cudaSuccess) e = make_node_map(&mQ, a.q, a.N, a.H);
    if (e == cudaSuccess) e = make_node_map(&mK, a.k, a.N, a.H);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(tc_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             VERIFY_SMEM);
    if (e != cudaSuccess) return e;
    tc_verify_kernel<<<units, kThreads, VERIFY_SMEM, s>>>(
        mS, mQ, mK, static_cast<const __nv_bfloat16 *>(a.v), a.gamma, a.beta, a.offsets, a.depth,
        a.anc, a.req_depth, a.H, a.N, static_cast<__nv_bfloat16 *>(a.O), a.U, a.logP, a.st);
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
