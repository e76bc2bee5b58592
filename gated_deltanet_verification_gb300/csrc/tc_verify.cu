// Tensor-core (TMA + tcgen05) verification and commit for bf16 q/k/v with
// d_k = d_v = 128 -- the Qwen3.5-shaped GDN head of the pages' evaluation.
//
// Verification, one CTA per (request, head), trees of up to 64 nodes:
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
constexpr int kSlots = 32;    // depth slots in the compact factors: depth <= 31
constexpr int kLd = 33;       // padded row stride of the compact factors (bank spread)
constexpr int kThreads = 256;
constexpr uint64_t kWaitNs = 200ull * 1000 * 1000; // 200 ms bound on any device wait

// ---- verification shared-memory plan (bytes from a 1024-aligned base) ----
constexpr int OFF_ST = 0;                     // S_pre fp32 staging: 4 x [128 rows x 128 B]
constexpr int OFF_A2 = OFF_ST;                // [M;W] tf32, K-major, 2 K-atoms (after the split)
constexpr int OFF_B2 = OFF_ST + 32768;        // R^T tf32, K-major, 2 K-atoms
constexpr int OFF_SHI = OFF_ST + 65536;       // S_hi bf16, MN-major, 2 N-atoms x 16 KB
constexpr int OFF_SLO = OFF_SHI + 32768;      // S_lo bf16
constexpr int OFF_A1 = OFF_SLO + 32768;       // [Q;K] bf16, K-major, 2 K-atoms x 16 KB
constexpr int OFF_G = OFF_A1 + 32768;         // compact G  [64][33] f32
constexpr int OFF_C = OFF_G + kT * kLd * 4;   // compact C
constexpr int OFF_ZA = OFF_C + kT * kLd * 4;  // Neumann iterates
constexpr int OFF_ZB = OFF_ZA + kT * kLd * 4;
constexpr int OFF_W = OFF_ZB + kT * kLd * 4;  // W = sum of iterates
constexpr int OFF_ANCAT = OFF_W + kT * kLd * 4; // [64][32] u8: ancestor at depth s
constexpr int OFF_L = OFF_ANCAT + kT * kSlots;
constexpr int OFF_P = OFF_L + kT * 4;
constexpr int OFF_BETA = OFF_P + kT * 4;
constexpr int OFF_DEPTH = OFF_BETA + kT * 4;
constexpr int OFF_UP = OFF_DEPTH + kT * 4;
constexpr int OFF_MASK = OFF_UP + kT * 4;     // u64 ancestor-or-self masks
constexpr int OFF_BAR = OFF_MASK + kT * 8;    // 4 mbarriers
constexpr int OFF_TSLOT = OFF_BAR + 4 * 8;
constexpr int OFF_FLAG = OFF_TSLOT + 4;
constexpr int VERIFY_SMEM = OFF_FLAG + 16 + 1024; // + alignment slack
static_assert(VERIFY_SMEM <= 227 * 1024, "verification shared memory");

constexpr uint32_t IDESC_GRAM = idesc_bf16(128, 64, false, false);  // [Q;K] K^T
constexpr uint32_t IDESC_STATE = idesc_bf16(128, 128, false, true); // [Q;K] S, S N-contiguous
constexpr uint32_t IDESC_TF32 = idesc_tf32(128, 128, false, false); // both K-major

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

__global__ void __launch_bounds__(kThreads, 1)
tc_verify_kernel(const __grid_constant__ CUtensorMap tmS, const __nv_bfloat16 *__restrict__ q,
                 const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                 const float *__restrict__ gamma, const float *__restrict__ beta,
                 const int32_t *__restrict__ offsets, const int32_t *__restrict__ parent,
                 const int32_t *__restrict__ depth_g, const uint32_t *__restrict__ anc_g,
                 const int32_t *__restrict__ req_depth, int H, int N,
                 __nv_bfloat16 *__restrict__ O, float *__restrict__ Uout,
                 float *__restrict__ logP, int32_t *st)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    float *sSt = reinterpret_cast<float *>(sm + OFF_ST);
    uint8_t *sHi = sm + OFF_SHI;
    uint8_t *sLo = sm + OFF_SLO;
    uint8_t *sA1 = sm + OFF_A1;
    uint8_t *sA2 = sm + OFF_A2;
    uint8_t *sB2 = sm + OFF_B2;
    float *Gc = reinterpret_cast<float *>(sm + OFF_G);
    float *Cc = reinterpret_cast<float *>(sm + OFF_C);
    float *Za = reinterpret_cast<float *>(sm + OFF_ZA);
    float *Zb = reinterpret_cast<float *>(sm + OFF_ZB);
    float *Wc = reinterpret_cast<float *>(sm + OFF_W);
    uint8_t *ancat = sm + OFF_ANCAT;
    float *Ls = reinterpret_cast<float *>(sm + OFF_L);
    float *Ps = reinterpret_cast<float *>(sm + OFF_P);
    float *Bs = reinterpret_cast<float *>(sm + OFF_BETA);
    int *Ds = reinterpret_cast<int *>(sm + OFF_DEPTH);
    int *up = reinterpret_cast<int *>(sm + OFF_UP);
    uint64_t *msk = reinterpret_cast<uint64_t *>(sm + OFF_MASK);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + OFF_BAR); // tma, gram, state, mma2
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_TSLOT);
    int *flag = reinterpret_cast<int *>(sm + OFF_FLAG);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x;
    const int b = unit / H, h = unit % H;

    // Uniform early exits, before any barrier or tensor-memory allocation.
    if (faulted(st)) return;
    const int o = offsets[b], T = offsets[b + 1] - o;
    if (T <= 0) return;
    if (T > kT || o < 0 || o + T > N) {
        if (tid == 0) report(st, BOLE_ERR_BAD_TOPOLOGY, b, -1, T);
        return;
    }
    const int d = req_depth[b];
    if (d < 0 || d >= kSlots || d >= T) {
        if (tid == 0) report(st, BOLE_ERR_DEPTH, b, -1, d);
        return;
    }

    // ---- set-up: tensor memory, barriers, the S_pre stream ----
    if (warp == 0) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
        *flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (tid == 0) {
        prefetch_tensormap(&tmS);
        mbar_arrive_expect_tx(&bar[0], 4 * 32 * 128 * 4);
#pragma unroll
        for (int c = 0; c < 4; ++c) tma_load_2d(sSt + c * 4096, &tmS, &bar[0], 32 * c, unit * kD);
    }

    // ---- topology and gates ----
    if (tid < kT) {
        const int i = tid;
        if (i < T) {
            const size_t nh = (size_t)(o + i) * H + h;
            Ds[i] = depth_g[o + i];
            const uint2 m2 = *reinterpret_cast<const uint2 *>(anc_g + (size_t)(o + i) * 4);
            msk[i] = ((uint64_t)m2.y << 32) | m2.x;
            Bs[i] = beta[nh];
            Ls[i] = logf(gamma[nh]);
            up[i] = parent[o + i];
        } else {
            Ds[i] = 0;
            msk[i] = 0;
            Bs[i] = 0.f;
            Ls[i] = 0.f;
            up[i] = -1;
        }
    }
    // [Q;K] -> bf16 K-major operand (two 64-element K-atoms; zeros beyond the tree)
    for (int item = tid; item < 128 * 16; item += kThreads) {
        const int m = item >> 4, g = item & 15;
        const int node = m & 63;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (node < T)
            val = *reinterpret_cast<const uint4 *>(((m < 64) ? q : k) +
                                                   ((size_t)(o + node) * H + h) * kD + g * 8);
        *reinterpret_cast<uint4 *>(sA1 + (g >> 3) * 16384 + sw128_chunk(m, g & 7)) = val;
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ---- MMA 1a: Gram [Q;K] K^T (one elected thread) ----
    const uint32_t a1 = smem_addr(sA1);
    if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16_ss(tmem + 128, sdesc_sw128(a1 + off, 16, 1024),
                        sdesc_sw128(a1 + off + 8192, 16, 1024), IDESC_GRAM, kk > 0);
        }
        mma_commit(&bar[1]);
    }

    // cumulative decay by pointer jumping along parent links (Lemma 1)
    for (int round = 0; round < 6; ++round) {
        float nl = 0.f;
        int nu = -1;
        bool active = false;
        if (tid < T) {
            const int a = up[tid];
            active = a >= 0;
            nl = Ls[tid] + (active ? Ls[a] : 0.f);
            nu = active ? up[a] : -1;
        }
        if (!__syncthreads_or(active)) break;
        if (tid < T) {
            Ls[tid] = nl;
            up[tid] = nu;
        }
        __syncthreads();
    }
    if (tid < kT) {
        const int i = tid;
        Ps[i] = (i < T) ? expf(Ls[i]) : 0.f;
        if (i < T) {
            logP[(size_t)(o + i) * H + h] = Ls[i];
            int t = 0;
            uint64_t mm = msk[i];
            while (mm) {
                const int j = __ffsll((long long)mm) - 1;
                ancat[i * kSlots + t++] = (uint8_t)j;
                mm &= mm - 1;
            }
        }
    }
    // Neumann start: Z^(0) = W = identity (the self entry sits at slot depth(i))
    for (int e = tid; e < kT * kSlots; e += kThreads) {
        const int i = e >> 5, t = e & 31;
        const float val = (i < T && t == Ds[i]) ? 1.f : 0.f;
        Za[i * kLd + t] = val;
        Wc[i * kLd + t] = val;
    }

    // ---- S_pre = S_hi + S_lo, both bf16, MN-major (64-column atoms) ----
    if (!mbar_wait(&bar[0], 0, kWaitNs)) {
        report(st, BOLE_ERR_TIMEOUT, b, -1, 1);
        *flag = 1;
    }
    for (int item = tid; item < 128 * 16; item += kThreads) {
        const int r = item >> 4, c8 = item & 15; // row r, columns 8*c8 .. 8*c8+7
        const uint8_t *box = reinterpret_cast<const uint8_t *>(sSt) + (c8 >> 2) * 16384;
        const float4 x0 = *reinterpret_cast<const float4 *>(box + sw128_chunk(r, (c8 & 3) * 2));
        const float4 x1 = *reinterpret_cast<const float4 *>(box + sw128_chunk(r, (c8 & 3) * 2 + 1));
        const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        __nv_bfloat162 hi2[4], lo2[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const __nv_bfloat16 h0 = __float2bfloat16_rn(xs[2 * t]);
            const __nv_bfloat16 h1 = __float2bfloat16_rn(xs[2 * t + 1]);
            hi2[t] = __halves2bfloat162(h0, h1);
            lo2[t] = __floats2bfloat162_rn(xs[2 * t] - __bfloat162float(h0),
                                           xs[2 * t + 1] - __bfloat162float(h1));
        }
        const uint32_t off = (c8 >> 3) * 16384 + sw128_chunk(r, c8 & 7);
        *reinterpret_cast<uint4 *>(sHi + off) = *reinterpret_cast<const uint4 *>(hi2);
        *reinterpret_cast<uint4 *>(sLo + off) = *reinterpret_cast<const uint4 *>(lo2);
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ---- MMA 1b: state products [Q;K] (S_hi + S_lo) ----
    if (tid == 0) {
        tc_fence_after();
        const uint32_t shi = smem_addr(sHi), slo = smem_addr(sLo);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad = sdesc_sw128(a1 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
            mma_bf16_ss(tmem, ad, sdesc_sw128(shi + kk * 2048, 16384, 1024), IDESC_STATE, kk > 0);
            mma_bf16_ss(tmem, ad, sdesc_sw128(slo + kk * 2048, 16384, 1024), IDESC_STATE, 1);
        }
        mma_commit(&bar[2]);
    }

    // ---- Gram epilogue: compact G and C (Lemma 2 / Lemma 1 read-out) ----
    const int rowgrp = warp & 3, half = warp >> 2;
    const int m = rowgrp * 32 + lane;
    const uint32_t lane_base = (uint32_t)(rowgrp * 32) << 16;
    if (!mbar_wait(&bar[1], 0, kWaitNs)) {
        report(st, BOLE_ERR_TIMEOUT, b, -1, 2);
        *flag = 1;
    }
    tc_fence_after();
    {
        float g[32];
        tmem_ld32(tmem + lane_base + 128 + half * 32, g);
        const int i = m & 63;
        if (i < T) {
            const uint64_t mi = msk[i];
            const float Li = Ls[i], bi = Bs[i];
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                const int j = half * 32 + t;
                if (j < T && ((mi >> j) & 1ull)) {
                    const float ratio = expf(Li - Ls[j]);
                    if (m < 64) Cc[i * kLd + Ds[j]] = ratio * g[t];
                    else if (j != i) Gc[i * kLd + Ds[j]] = bi * ratio * g[t];
                }
            }
        }
    }
    __syncthreads();

    // ---- W = sum_{m<=d} (-G)^m by Z <- -G Z, W += Z (Eq. (8) on the identity) ----
    {
        float *Zc = Za, *Zn = Zb;
        for (int step = 0; step < d; ++step) {
            for (int e = tid; e < kT * kSlots; e += kThreads) {
                const int i = e & 63, t = e >> 6;
                float val = 0.f;
                if (i < T) {
                    const int di = Ds[i];
                    for (int s = t + step; s < di; ++s)
                        val = fmaf(-Gc[i * kLd + s], Zc[ancat[i * kSlots + s] * kLd + t], val);
                }
                Zn[i * kLd + t] = val;
                Wc[i * kLd + t] += val;
            }
            __syncthreads();
            float *tmp = Zc; Zc = Zn; Zn = tmp;
        }
    }

    // ---- state epilogue: B0 = P Q S_pre in place; R^T = (beta (v - P K S_pre))^T ----
    if (!mbar_wait(&bar[2], 0, kWaitNs)) {
        report(st, BOLE_ERR_TIMEOUT, b, -1, 3);
        *flag = 1;
    }
    tc_fence_after();
    {
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
                float vv[32];
                if (i < T) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        v + ((size_t)(o + i) * H + h) * kD + col0);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        float f[8];
                        bf16x8_to_f32(src[u], f);
#pragma unroll
                        for (int t = 0; t < 8; ++t) vv[u * 8 + t] = f[t];
                    }
                }
                // R^T: row = value column c, K index = node i (tf32, K-major)
                uint8_t *dst = sB2 + (i >> 5) * 16384;
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const float r = (i < T) ? bt * (vv[t] - p * x[t]) : 0.f;
                    *reinterpret_cast<float *>(dst + sw128_offset(col0 + t, i & 31)) = r;
                    x[t] = 0.f;
                }
                tmem_st32(tmem + lane_base + col0, x);
            }
        }
        tmem_wait_st();
    }
    // [M; W] -> tf32 K-major operand: rows 0..63 M = C W, rows 64..127 W
    for (int item = tid; item < 128 * 16; item += kThreads) {
        const int r = item >> 4, ch = item & 15;
        const int i = r & 63;
        float vals[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int j = ch * 4 + jj;
            float val = 0.f;
            if (i < T && j < T && ((msk[i] >> j) & 1ull)) {
                const int dj = Ds[j];
                if (r >= 64) {
                    val = Wc[i * kLd + dj];
                } else {
                    const int di = Ds[i];
                    for (int s = dj; s <= di; ++s)
                        val = fmaf(Cc[i * kLd + s], Wc[ancat[i * kSlots + s] * kLd + dj], val);
                }
            }
            vals[jj] = val;
        }
        *reinterpret_cast<float4 *>(sA2 + (ch >> 3) * 16384 + sw128_offset(r, (ch & 7) * 4)) =
            make_float4(vals[0], vals[1], vals[2], vals[3]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA 2 (tf32): [M; W] R accumulated onto [B0; 0] ----
    if (tid == 0) {
        tc_fence_after();
        const uint32_t a2 = smem_addr(sA2), b2 = smem_addr(sB2);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_tf32_ss(tmem, sdesc_sw128(a2 + off, 16, 1024), sdesc_sw128(b2 + off, 16, 1024),
                        IDESC_TF32, 1);
        }
        mma_commit(&bar[3]);
    }
    if (!mbar_wait(&bar[3], 0, kWaitNs)) {
        report(st, BOLE_ERR_TIMEOUT, b, -1, 4);
        *flag = 1;
    }
    tc_fence_after();

    // ---- outputs: rows 0..63 O (bf16), rows 64..127 U (fp32) ----
    {
        const int i = m & 63;
        const bool store = i < T && *(volatile int *)flag == 0;
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
                for (int u = 0; u < 4; ++u) {
                    __nv_bfloat162 p2[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        p2[t] = __floats2bfloat162_rn(x[8 * u + 2 * t], x[8 * u + 2 * t + 1]);
                    dst[u] = *reinterpret_cast<uint4 *>(p2);
                }
            } else {
                float4 *dst = reinterpret_cast<float4 *>(Uout + row);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    dst[u] = make_float4(x[4 * u], x[4 * u + 1], x[4 * u + 2], x[4 * u + 3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---- commit ----
constexpr int kCommitThreads = 128;
constexpr int kChunk = 32; // path nodes per MMA K chunk
constexpr int CO_S = 0;                       // S tile, 64 KB
constexpr int CO_A = 65536;                   // (D_a K_a)^T chunk: 128 rows x 32 tf32, 16 KB
constexpr int CO_B = CO_A + 16384;            // U_a^T chunk: 128 rows x 32 tf32, 16 KB
constexpr int CO_PATH = CO_B + 16384;         // int[128]
constexpr int CO_COEF = CO_PATH + 512;        // float[128]
constexpr int CO_BAR = CO_COEF + 512;         // 2 mbarriers
constexpr int CO_TSLOT = CO_BAR + 16;
constexpr int CO_MISC = CO_TSLOT + 4;         // path length, flag
constexpr int COMMIT_SMEM = CO_MISC + 16 + 1024;

__global__ void __launch_bounds__(kCommitThreads)
tc_commit_kernel(const __grid_constant__ CUtensorMap tmS, const __nv_bfloat16 *__restrict__ k,
                 const float *__restrict__ U, const float *__restrict__ logP,
                 const int32_t *__restrict__ offsets, const int32_t *__restrict__ parent,
                 const int32_t *__restrict__ accepted, int H, int N, int32_t *st)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    float *sS = reinterpret_cast<float *>(sm + CO_S);
    uint8_t *sA = sm + CO_A;
    uint8_t *sB = sm + CO_B;
    int *path = reinterpret_cast<int *>(sm + CO_PATH);
    float *coef = reinterpret_cast<float *>(sm + CO_COEF);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + CO_BAR); // tma, mma
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + CO_TSLOT);
    int *plen = reinterpret_cast<int *>(sm + CO_MISC);
    int *flag = plen + 1;

    const int tid = threadIdx.x, warp = tid >> 5;
    const int unit = blockIdx.x;
    const int b = unit / H, h = unit % H;
    if (faulted(st)) return;
    const int a = accepted[b];
    if (a < 0) return;
    const int o = offsets[b], T = offsets[b + 1] - o;
    if (a >= T || o < 0 || o + T > N || T > kMaxTree) {
        if (tid == 0) report(st, BOLE_ERR_BAD_TOPOLOGY, b, a, T);
        return;
    }
    if (warp == 0) {
        tmem_alloc(tslot, 128);
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
        mbar_arrive_expect_tx(&bar[0], 4 * 128 * 128);
#pragma unroll
        for (int c = 0; c < 4; ++c) tma_load_2d(sS + c * 4096, &tmS, &bar[0], 32 * c, unit * kD);
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
        // A[r][t] = coef_t k_{j_t}[r]  (row r = tid), K-major, one 128-byte atom
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
                *reinterpret_cast<float4 *>(sA + sw128_offset(r, 4 * c4)) =
                    make_float4(av[4 * c4], av[4 * c4 + 1], av[4 * c4 + 2], av[4 * c4 + 3]);
        }
        // B^T[c][t] = u_{j_t}[c] (row c = tid), K-major, one 128-byte atom
        {
            const int c = tid;
#pragma unroll
            for (int t4 = 0; t4 < kChunk / 4; ++t4) {
                float uv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = ch * kChunk + 4 * t4 + e;
                    uv[e] = (t < L) ? U[((size_t)(o + path[t]) * H + h) * kD + c] : 0.f;
                }
                *reinterpret_cast<float4 *>(sB + sw128_offset(c, 4 * t4)) =
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
                mma_tf32_ss(tmem, sdesc_sw128(sa + kk * 32, 16, 1024),
                            sdesc_sw128(sb + kk * 32, 16, 1024), IDESC_TF32, (ch > 0 || kk > 0));
            mma_commit(&bar[1]);
        }
        if (!mbar_wait(&bar[1], ch & 1, kWaitNs)) {
            report(st, BOLE_ERR_TIMEOUT, b, -1, 5);
            *flag = 1;
        }
        tc_fence_after();
        __syncthreads();
    }

    // epilogue: S <- P_a S + D, in shared memory, then TMA store in place
    if (!mbar_wait(&bar[0], 0, kWaitNs)) {
        report(st, BOLE_ERR_TIMEOUT, b, -1, 6);
        *flag = 1;
    }
    const bool ok = *(volatile int *)flag == 0;
    if (ok && nchunks > 0) {
        const float Pa = expf(La);
        const int r = tid;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
            float x[32];
            tmem_ld32(tmem + lane_base + cb * 32, x);
            uint8_t *tile = reinterpret_cast<uint8_t *>(sS + cb * 4096);
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
#pragma unroll
        for (int c = 0; c < 4; ++c) tma_store_2d(&tmS, sS + c * 4096, 32 * c, unit * kD);
        bulk_commit_group();
        bulk_wait_group_read0();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
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

cudaError_t launch_tc_verify(const VerifyArgs &a, cudaStream_t s)
{
    const int units = a.B * a.H;
    if (units == 0 || a.N == 0) return cudaSuccess;
    CUtensorMap map;
    cudaError_t e = make_state_map(&map, a.S_pre, units);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(tc_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             VERIFY_SMEM);
    if (e != cudaSuccess) return e;
    tc_verify_kernel<<<units, kThreads, VERIFY_SMEM, s>>>(
        map, static_cast<const __nv_bfloat16 *>(a.q), static_cast<const __nv_bfloat16 *>(a.k),
        static_cast<const __nv_bfloat16 *>(a.v), a.gamma, a.beta, a.offsets, a.parent, a.depth,
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
    tc_commit_kernel<<<units, kCommitThreads, COMMIT_SMEM, s>>>(
        map, static_cast<const __nv_bfloat16 *>(a.k), a.U, a.logP, a.offsets, a.parent,
        a.accepted, a.H, a.N, a.st);
    return cudaGetLastError();
}

} // namespace bole
