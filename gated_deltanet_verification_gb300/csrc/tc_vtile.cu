// Value-tiled tensor-core verification for small trees: d_k = d_v = 128,
// trees of up to 32 nodes, depth <= 15 (the batched Qwen3.5-shaped workloads
// of the pages' evaluation), bf16 or fp32 q/k/v.
//
// The pages' kernel splits d_v into N_v = d_v / b_v value tiles and gives each
// (request, head, tile) its own CTA, so a request yields H * N_v
// independently schedulable CTAs ("Bole", Section IV-B, value-tiled kernel).
// Here b_v = 64, N_v = 2: each CTA streams its 128 x 64 tile of S_pre by TMA,
// forms the tree factors of its head on chip (both tiles of a head repeat
// that small T x T work instead of exchanging it), and writes its 64 columns
// of O and U.  bf16 inputs: 66 KB of shared memory and 128 tensor-memory
// columns, three CTAs per SM; the library runs this form for batches whose
// heads would leave the one-CTA-per-head kernel short of a wave (a single
// request's heads, say): there the extra CTAs add parallelism, while on
// larger batches the one-CTA kernel keeps more state bytes in flight per SM.
// fp32 inputs: 111 KB, two CTAs per SM, the tensor-core path for every fp32
// batch it covers.
//
// Per CTA (T <= 32 nodes of one head, value columns c0 .. c0 + 63):
//   1. TMA: [Q;K] of the tree (q rows 0..31, k rows 32..63 of each K-atom)
//      and (bf16) the value rows of the tile; once the per-node reads have
//      returned, the two 32-column boxes of the S_pre tile.  fp32 value rows
//      go straight to the registers of the threads that form R^T.
//   2. Warp 0: cumulative decay L_i along the ancestor-or-self mask (Lemma 1),
//      the decay ratios exp(L_i - L_j) of each node's ancestors.
//   3. tcgen05 Gram [Q;K] K^T (bf16 products, fp32 accumulation); warps 0, 5
//      stage its rows in shared memory; warp 0 gathers the compact
//        C_ij = exp(L_i - L_j) q_i.k_j          (j an ancestor of i, or i)
//        G_ij = beta_i exp(L_i - L_j) k_i.k_j   (j a strict ancestor of i)
//      by ancestor depth; rows of W = (I+G)^{-1} (warp 0) and M = C W
//      (warp 5) by backward substitution along each node's ancestor path --
//      the finite Neumann sum of Eq. (6), term for term.
//   4. Warps 1..4 split the S_pre tile in place as soon as it lands; tcgen05
//      [Q;K] S_pre with exact bf16 products and fp32 accumulation gives
//      Q S_pre and K S_pre of the tile (Eq. (7)).
//   5. Warps 1, 5: R^T = (beta (v - P K S_pre))^T of the tile; warps 0, 5
//      write [M; W] -- both into the tile buffer the products released.
//   6. tcgen05 tf32 [M; W] R (K = the tree's nodes) into the Gram's
//      tensor-memory columns; warps 0, 4 write O = P Q S_pre + M R, warps
//      1, 5 U = W R (fp32).
//
// Precision.  bf16 inputs: S_pre = S_hi + S_lo in bf16 (a relative residue
// of about 2^-17 per element), q and k exact, [M; W] and R in tf32.  fp32
// inputs (the 1e-5 bound): every fp32 operand x of the Gram and the state
// products is written as x1 + x2 + x3 in bf16 (x1 = bf16(x), x2 = bf16(x -
// x1), x3 = bf16(x - x1 - x2): 24 significant bits, x itself for normal
// floats), and the product keeps the six terms of order up to 2^-16,
//   sum_{i + j <= 4} x_i y_j   (i, j >= 1),
// dropping terms of order 2^-24; [M; W] and R^T are written as hi + lo in
// tf32 (rounded to nearest here, so the hardware's reading of an operand
// is exact) and the propagation keeps hi hi + hi lo + lo hi (dropped term
// ~2^-22).  Accumulation is fp32 throughout.
//
// [Q;K] is stored without padding (64 rows per K-atom); the M = 128 products
// read the 8 KB behind each atom as rows 64..127, whose results land in
// tensor-memory lanes 64..127 that nothing reads.  The same holds for [M; W].
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm100.cuh"
#include "tc_common.cuh"

namespace bole {
namespace {

using namespace sm100;
using namespace tc;

constexpr int kVT = 32;     // tree nodes per CTA
constexpr int kVB = 64;     // b_v: value columns per CTA
constexpr int kVSlots = 16; // depth slots of the compact factors: depth <= 15
constexpr int kVLd = 17;    // padded row stride of the compact factors

// ---- shared-memory plan (bytes from a 1024-aligned base) ----
//   S: the state tile lands as two fp32 boxes [128 rows x 32 columns]
//     (32 KB) and is split in place into bf16 copies, N-contiguous [128 d_k
//     rows x 64 columns], 16 KB each: S_hi, S_lo (bf16 inputs) or S_1, S_2,
//     S_3 (fp32 inputs, 48 KB).  After the state products: [M; W] (rows
//     0..63, tf32 K-major, 128 B per row) and R^T (64 value rows x 32 nodes,
//     tf32 K-major): bf16 inputs [M; W] at 0, R^T at 16 KB; fp32 inputs
//     [M; W] hi at 0, lo at 16 KB, R^T hi at 32 KB, lo at 40 KB.  After the
//     propagation: the staged O and U rows.
//   QK: K-atoms [64 rows x 128 B] of [Q;K] (q rows 0..31, k rows 32..63):
//     bf16 inputs two atoms (16 KB) loaded as they are; fp32 inputs four fp32
//     atoms (32 KB) loaded, then rewritten as three bf16 copies of two atoms
//     each (48 KB, copy c atom a at (2 c + a) x 8 KB).  The M = 128 products
//     read 8 KB past each atom.
//   V (bf16 inputs, 4 KB): the tile's value rows [32 nodes x 64 bf16],
//     128B-swizzled.
//   G (8 KB): the staged Gram rows [64 x 32 fp32] (q.k rows 0..31, k.k rows
//     32..63), 16-byte chunks XOR-swizzled by row.
//   X: compact C, G [32][17], ancestor table [32][16] u8, L, depth, log gamma.
constexpr int VT_FAC = kVT * kVLd * 4;
template <bool F32> struct VtPlan {
    static constexpr int S = 0;
    static constexpr int QK = S + (F32 ? 3 : 2) * 16384;
    static constexpr int QK_ATOMS = F32 ? 6 : 2; // 8 KB K-atoms after the split
    static constexpr int V = QK + QK_ATOMS * 8192;
    static constexpr int G = V + (F32 ? 0 : 4096);
    static constexpr int X = G + 8192;
    static constexpr int GC = X;
    static constexpr int CC = GC + VT_FAC;
    static constexpr int ANCAT = CC + VT_FAC;
    static constexpr int L = ANCAT + kVT * kVSlots;
    static constexpr int DEPTH = L + kVT * 4;
    static constexpr int LG = DEPTH + kVT * 4;
    static constexpr int BAR = LG + kVT * 4;
    static constexpr int MISC = BAR + 16 * 8; // TMEM slot, status copy, wait-failure flag,
                                              // first bad node, request depth
    static constexpr int END = MISC + 24;
    static constexpr int SMEM = END + 1024;   // slack for the 1024-byte alignment of the base
    static constexpr int PER_SM = F32 ? 2 : 3;
    static_assert(ANCAT % 16 == 0 && BAR % 8 == 0, "aligned scratch");
    static_assert(QK + (QK_ATOMS - 1) * 8192 + 16384 <= X,
                  "the products' reads past [Q;K] stay inside the CTA's buffers");
    static_assert(PER_SM * (SMEM + 1024) <= 228 * 1024, "CTAs per SM");
};

constexpr int kVTCompute = 192;               // warps 0..5
constexpr int kVTThreads = kVTCompute + 32;   // warp 6: TMA and tcgen05 issue
constexpr uint32_t TM_COLS = 128;             // tensor-memory columns per CTA
constexpr uint32_t TM_GP = 64;                // Gram, then the propagation [M R; W R]

constexpr uint32_t IDESC_VGRAM = idesc_bf16(128, 32, false, false);  // [Q;K] K^T
constexpr uint32_t IDESC_VSTATE = idesc_bf16(128, kVB, false, true); // [Q;K] S, S N-contiguous
constexpr uint32_t IDESC_VPROP = idesc_tf32(128, kVB, false, false); // [M; W] R

// The six (x copy, y copy) pairs of the fp32 products, smallest first.
__device__ constexpr int kSplitA[6] = {2, 1, 0, 1, 0, 0};
__device__ constexpr int kSplitB[6] = {0, 1, 2, 0, 1, 0};

// mbarrier slots
constexpr int VB_S = 0, VB_QK = 1, VB_V = 2, VB_GRAM = 3, VB_STATE = 4, VB_PROP = 5,
              VB_TOPO = 6, VB_STAGED = 7, VB_CG = 8, VB_CONV = 9, VB_OPS = 10, VB_DRAIN = 11,
              VB_QKS = 12; // fp32: [Q;K] split into its bf16 copies

// x -> x1 + x2 + x3 (bf16 each) for eight consecutive floats, packed as
// three 16-byte chunks.
__device__ __forceinline__ void split3_bf16x8(const float *x, uint4 &c1, uint4 &c2, uint4 &c3)
{
    uint32_t w1[4], w2[4], w3[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const float x0 = x[2 * t], x1 = x[2 * t + 1];
        const __nv_bfloat162 b1 = __floats2bfloat162_rn(x0, x1);
        const float2 f1 = __bfloat1622float2(b1);
        const float r0 = x0 - f1.x, r1 = x1 - f1.y; // exact
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(r0, r1);
        const float2 f2 = __bfloat1622float2(b2);
        const __nv_bfloat162 b3 = __floats2bfloat162_rn(r0 - f2.x, r1 - f2.y);
        w1[t] = *reinterpret_cast<const uint32_t *>(&b1);
        w2[t] = *reinterpret_cast<const uint32_t *>(&b2);
        w3[t] = *reinterpret_cast<const uint32_t *>(&b3);
    }
    c1 = make_uint4(w1[0], w1[1], w1[2], w1[3]);
    c2 = make_uint4(w2[0], w2[1], w2[2], w2[3]);
    c3 = make_uint4(w3[0], w3[1], w3[2], w3[3]);
}

template <bool F32>
__global__ void __launch_bounds__(kVTThreads, VtPlan<F32>::PER_SM)
tc_vtile_kernel(const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmQ,
                const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const float *__restrict__ gamma, const float *__restrict__ beta,
                const int32_t *__restrict__ offsets, const uint32_t *__restrict__ anc,
                const int32_t *__restrict__ req_depth, int H, int N,
                void *__restrict__ Oout, float *__restrict__ Uout,
                float *__restrict__ logP, int32_t *st, int pf_stride, int early_alloc,
                const int32_t *__restrict__ parent, int max_depth, int inline_topo,
                const float *__restrict__ vf32)
{
    using P = VtPlan<F32>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *sS = sm + P::S, *sQK = sm + P::QK, *sV = sm + P::V, *sG = sm + P::G;
    float *Gc = reinterpret_cast<float *>(sm + P::GC);
    float *Cc = reinterpret_cast<float *>(sm + P::CC);
    uint8_t *ancat = sm + P::ANCAT;
    float *Ls = reinterpret_cast<float *>(sm + P::L);
    int *Ds = reinterpret_cast<int *>(sm + P::DEPTH);
    float *LGs = reinterpret_cast<float *>(sm + P::LG);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + P::BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + P::MISC);
    int *sfault = reinterpret_cast<int *>(sm + P::MISC + 4);
    volatile int *sfail = reinterpret_cast<volatile int *>(sm + P::MISC + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x >> 1, vh = blockIdx.x & 1; // (request, head), value tile
    const int b = unit / H, h = unit % H;
    const int c0 = vh * kVB; // first value column of the tile

    if (sm + P::END > smem_raw + P::SMEM) { // dynamic base too far from 1024 B
        if (tid == 0) report(st, BOLE_ERR_CUDA, b, -1, -5);
        return;
    }
    // A launch of its own allocates tensor memory first (the SM starts the
    // next CTA once this one has given up its allocation permit); a launch
    // overlapping the previous kernel allocates after its prologue.
    if (early_alloc && warp == 0) {
        tmem_alloc(tslot, TM_COLS);
        tmem_relinquish();
    }
    pdl_launch_dependents();
    const int o = offsets[b], T = offsets[b + 1] - o;
    const bool in_range = T > 0 && T <= kVT && o >= 0 && o + T <= N;
    const bool issuer = tid == kVTCompute;
    if (issuer) {
        for (int k = VB_S; k <= VB_PROP; ++k) mbar_init(&bar[k], 1);
        mbar_init(&bar[VB_TOPO], 32);
        mbar_init(&bar[VB_STAGED], 64);
        mbar_init(&bar[VB_CG], 32);
        mbar_init(&bar[VB_CONV], 128);
        mbar_init(&bar[VB_OPS], kVTCompute);
        mbar_init(&bar[VB_DRAIN], 1);
        mbar_init(&bar[VB_QKS], 128);
        fence_mbar_init();
        if (in_range) {
            if constexpr (F32) {
                // q rows 0..31 and k rows 32..63 of the four fp32 K-atoms
                mbar_arrive_expect_tx(&bar[VB_QK], 32768);
#pragma unroll
                for (int ka = 0; ka < 4; ++ka) {
                    tma_load_3d(sQK + ka * 8192, &tmQ, &bar[VB_QK], 32 * ka, h, o);
                    tma_load_3d(sQK + ka * 8192 + 4096, &tmK, &bar[VB_QK], 32 * ka, h, o);
                }
            } else {
                // q rows 0..31 and k rows 32..63 of both K-atoms; the tile's value rows
                mbar_arrive_expect_tx(&bar[VB_QK], 16384);
#pragma unroll
                for (int ka = 0; ka < 2; ++ka) {
                    tma_load_3d(sQK + ka * 8192, &tmQ, &bar[VB_QK], 64 * ka, h, o);
                    tma_load_3d(sQK + ka * 8192 + 4096, &tmK, &bar[VB_QK], 64 * ka, h, o);
                }
                mbar_arrive_expect_tx(&bar[VB_V], 4096);
                tma_load_3d(sV, &tmV, &bar[VB_V], c0, h, o);
            }
        }
    }
    // per-thread tree inputs: warp 0 (node = lane) the gates of its row, warps
    // 1 and 5 (node = lane, the K-side rows) beta for R^T
    const int i = lane;
    float bt = 0.f, g_i = 1.f;
    int my_par = -1; // warp 0, topology formed here: the parent of node i
    // fp32 inputs: warps 1 and 5 hold the 32 value columns of node i they
    // turn into R^T (columns c0 + 32 (warp / 5) ...), read now so the loads
    // complete long before R^T is formed
    float vreg[F32 ? 32 : 1];
    if constexpr (F32) {
#pragma unroll
        for (int c = 0; c < 32; ++c) vreg[c] = 0.f;
    }
    if (in_range && i < T && (warp == 0 || warp == 1 || warp == 5)) {
        bt = beta[(size_t)(o + i) * H + h];
        if (warp == 0) g_i = gamma[(size_t)(o + i) * H + h];
        if (warp == 0 && inline_topo) my_par = parent[o + i];
        if constexpr (F32) {
            if (warp != 0) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    vf32 + ((size_t)(o + i) * H + h) * kD + c0 + (warp == 5 ? 32 : 0));
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float4 t4 = src[u];
                    vreg[4 * u] = t4.x; vreg[4 * u + 1] = t4.y;
                    vreg[4 * u + 2] = t4.z; vreg[4 * u + 3] = t4.w;
                }
            }
        }
    }
    // What the previous call wrote (the status word pack reset, the request's
    // depth, each node's ancestor-or-self mask) is read after the wait.
    pdl_wait();
    if (tid == 0) {
        *sfault = *(const volatile int32_t *)st; // one read: a uniform exit
        *sfail = 0;
    }
    int *stopo = reinterpret_cast<int *>(sm + P::MISC + 12); // first bad node, depth
    const int d_read = inline_topo ? 0 : req_depth[b];
    int my_depth = -1;
    uint32_t my_mask = 0;
    int wdepth = 0; // warp 0, topology formed here: the request's depth
    if (!inline_topo) {
        if (warp == 0 && in_range && i < T) {
            my_mask = anc[(size_t)(o + i) * 4]; // a tree of <= 32 nodes: the first word
            my_depth = __popc(my_mask) - 1;
        }
    } else if (warp == 0) {
        // The round's topology step in the kernel (Section IV-C): pointer
        // jumping over the lanes, so after log2(32) = 5 rounds each mask holds
        // the node's whole path; a link that does not point backwards is a
        // fault (reported below) and is not followed.
        const bool live = in_range && i < T;
        const bool badp = live && (my_par < -1 || my_par >= i);
        uint32_t mk = live ? (1u << i) : 0u;
        int jp = (live && !badp) ? my_par : -1;
#pragma unroll
        for (int r = 0; r < 5; ++r) {
            const int src = jp >= 0 ? jp : i;
            const uint32_t m2 = __shfl_sync(0xffffffffu, mk, src);
            const int j2 = __shfl_sync(0xffffffffu, jp, src);
            if (jp >= 0) {
                mk |= m2;
                jp = j2;
            }
        }
        const unsigned badm = __ballot_sync(0xffffffffu, badp);
        if (live) {
            my_mask = mk;
            my_depth = __popc(mk) - 1;
        }
        wdepth = __reduce_max_sync(0xffffffffu, live ? my_depth : 0);
        if (lane == 0) stopo[0] = badm ? __ffs(badm) - 1 : kVT;
        if (lane == 0) stopo[1] = wdepth;
    }
    if (my_depth >= kVSlots) my_depth = -1; // the request is refused below
    if (warp == 0) LGs[i] = logf(g_i); // consumes gamma before the barrier
    if (!early_alloc && warp == 0) {
        tmem_alloc(tslot, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int fault = *sfault;
    const int d = inline_topo ? stopo[1] : d_read;
    const int bad_node = inline_topo && in_range ? stopo[0] : kVT;
    const bool bad = !in_range || d < 0 || d >= kVSlots || d >= T || bad_node < kVT ||
                     (inline_topo && d > max_depth);
    if (issuer && fault == 0 && T > 0 && !bad) {
        // The state tile is requested once the small reads have returned:
        // requested at entry it queued them behind every CTA's state burst
        // (28.1 -> 26.3 us on the batched forest).
        mbar_arrive_expect_tx(&bar[VB_S], 32768);
        tma_load_2d(sS, &tmS, &bar[VB_S], c0, unit * kD);
        tma_load_2d(sS + 16384, &tmS, &bar[VB_S], c0 + 32, unit * kD);
    }
    if (fault != 0 || T <= 0 || bad) {
        if (fault == 0 && h == 0 && vh == 0 && (T > 0 || (inline_topo && T < 0))) {
            if (bad_node < kVT) { // the first node whose link does not point backwards
                if (tid == bad_node) report(st, BOLE_ERR_BAD_TOPOLOGY, b, bad_node, my_par);
            } else if (bad && tid == 0) {
                report(st, T > kVT || T < 0 || o < 0 || o + T > N ? BOLE_ERR_BAD_TOPOLOGY
                                                                   : BOLE_ERR_DEPTH,
                       b, -1, T > kVT || T < 0 ? T : d);
            }
        }
        if (issuer) { // the copies in flight end before the CTA retires
            if (in_range) {
                mbar_wait(&bar[VB_QK], 0, kWaitNs);
                if (!F32) mbar_wait(&bar[VB_V], 0, kWaitNs);
            }
        }
        if (warp == 0) tmem_dealloc(tmem, TM_COLS);
        return;
    }
    const int quad = warp & 3; // the tensor-memory lanes this warp reaches
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    auto waitb = [&](int k) -> bool {
        const bool r = mbar_wait(&bar[k], 0, kWaitNs);
        if (!r) *sfail = 1;
        return r;
    };
    // staged Gram row r (0..63): 32 fp32, chunks XOR-swizzled by r & 7
    auto staged = [&](int r) -> float * { return reinterpret_cast<float *>(sG + r * 128); };

    if (warp == kVTCompute / 32) {
        // =========================== issue warp ===========================
        bool ok = true;
        if (lane == 0) {
            const uint32_t qk = smem_addr(sQK), s0 = smem_addr(sS);
            do { // every step ends the issue once a wait anywhere in the CTA gave up
                ok &= waitb(F32 ? VB_QKS : VB_QK);
                if (!ok || *sfail) break;
                tc_fence_after();
                if constexpr (F32) {
                    // Gram from the bf16 copies: the six pairs, 16 d_k per step
#pragma unroll
                    for (int t = 0; t < 6; ++t)
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
                            mma_bf16_ss(tmem + TM_GP,
                                        sdesc_sw128(qk + kSplitA[t] * 16384 + off, 16, 1024),
                                        sdesc_sw128(qk + kSplitB[t] * 16384 + off + 4096, 16, 1024),
                                        IDESC_VGRAM, t > 0 || kk > 0);
                        }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) { // Gram [Q;K] K^T, 16 d_k per step
                        const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
                        mma_bf16_ss(tmem + TM_GP, sdesc_sw128(qk + off, 16, 1024),
                                    sdesc_sw128(qk + off + 4096, 16, 1024), IDESC_VGRAM, kk > 0);
                    }
                }
                mma_commit(&bar[VB_GRAM]);
                ok &= waitb(VB_CONV);
                if (!ok || *sfail) break;
                tc_fence_after();
                if constexpr (F32) {
                    // [Q;K] S_pre from the bf16 copies of both: the six pairs
#pragma unroll
                    for (int t = 0; t < 6; ++t)
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
                            mma_bf16_ss(tmem, sdesc_sw128(qk + kSplitA[t] * 16384 + off, 16, 1024),
                                        sdesc_sw128(s0 + kSplitB[t] * 16384 + kk * 2048, 16384,
                                                    1024),
                                        IDESC_VSTATE, t > 0 || kk > 0);
                        }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) { // [Q;K] (S_hi + S_lo), 16 d_k rows per step
                        const uint64_t ad =
                            sdesc_sw128(qk + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024);
                        mma_bf16_ss(tmem, ad, sdesc_sw128(s0 + kk * 2048, 16384, 1024),
                                    IDESC_VSTATE, kk > 0);
                        mma_bf16_ss(tmem, ad, sdesc_sw128(s0 + 16384 + kk * 2048, 16384, 1024),
                                    IDESC_VSTATE, 1);
                    }
                }
                mma_commit(&bar[VB_STATE]);
                // the state tile of the CTA one wave later goes to L2 now that
                // this CTA's own tile has landed
                const int nx = (int)blockIdx.x + pf_stride;
                if (pf_stride > 0 && nx < (int)gridDim.x) {
                    tma_prefetch_l2_2d(&tmS, (nx & 1) * kVB, (nx >> 1) * kD);
                    tma_prefetch_l2_2d(&tmS, (nx & 1) * kVB + 32, (nx >> 1) * kD);
                }
                ok &= waitb(VB_OPS);
                if (!ok || *sfail) break;
                tc_fence_after();
                if constexpr (F32) {
                    // [M; W] R as lo hi + hi lo + hi hi, over the tree's nodes
#pragma unroll
                    for (int t = 0; t < 3; ++t) {
                        const uint32_t a = s0 + (t == 0 ? 16384 : 0);
                        const uint32_t bb = s0 + (t == 1 ? 40960 : 32768);
                        for (int kk = 0; kk < (T + 7) / 8; ++kk)
                            mma_tf32_ss(tmem + TM_GP, sdesc_sw128(a + kk * 32, 16, 1024),
                                        sdesc_sw128(bb + kk * 32, 16, 1024), IDESC_VPROP,
                                        t > 0 || kk > 0);
                    }
                } else {
                    for (int kk = 0; kk < (T + 7) / 8; ++kk) // [M; W] R over the tree's nodes
                        mma_tf32_ss(tmem + TM_GP, sdesc_sw128(s0 + kk * 32, 16, 1024),
                                    sdesc_sw128(s0 + 16384 + kk * 32, 16, 1024), IDESC_VPROP,
                                    kk > 0);
                }
                mma_commit(&bar[VB_PROP]);
            } while (0);
        }
        __syncwarp();
        if (!ok) report(st, BOLE_ERR_TIMEOUT, b, -1, 30);
    } else {
        // ========================== compute warps =========================
        bool ok = true;
        float ratio[kVSlots];          // warp 0: exp(L_i - L_j), j the ancestor at depth t
        uint32_t aw[4] = {0, 0, 0, 0}; // warp 0: ancestor-by-depth table, packed bytes
        if (warp == 0) {
            // Topology and cumulative decay (node i = lane): the ancestors come
            // out of the mask in depth order (parents precede children), so the
            // partial sums of log gamma are their L_j (Lemma 1).
            __syncwarp();
            int jt[kVSlots];
            uint32_t mm = my_depth >= 0 ? my_mask : 0u;
#pragma unroll
            for (int t = 0; t < kVSlots; ++t) {
                jt[t] = mm ? __ffs(mm) - 1 : 0;
                mm &= mm - 1;
            }
            float lgv[kVSlots];
#pragma unroll
            for (int t = 0; t < kVSlots; ++t) lgv[t] = LGs[jt[t]];
            float L = 0.f;
#pragma unroll
            for (int t = 0; t < kVSlots; ++t) {
                if (t <= my_depth) {
                    L += lgv[t];
                    aw[t >> 2] |= (uint32_t)jt[t] << (8 * (t & 3));
                }
                ratio[t] = L;
            }
#pragma unroll
            for (int t = 0; t < kVSlots; ++t)
                ratio[t] = F32 ? expf(L - ratio[t]) : __expf(L - ratio[t]);
            *reinterpret_cast<uint4 *>(ancat + i * kVSlots) = make_uint4(aw[0], aw[1], aw[2], aw[3]);
            Ls[i] = L;
            Ds[i] = my_depth;
            if (vh == 0 && i < T) logP[(size_t)(o + i) * H + h] = L;
            mbar_arrive(&bar[VB_TOPO]);
        }
        if constexpr (F32) {
            if (warp >= 1 && warp <= 4) {
                // [Q;K] -> three bf16 copies: thread (row r, d_k half hf)
                // reads its 64 floats from fp32 atoms 2 hf, 2 hf + 1 and
                // writes 64 bf16 of row r into atom hf of each copy.  Row r's
                // outputs overwrite only row r's inputs, and both halves of a
                // row sit in one warp (adjacent lanes), so a warp-level sync
                // orders the reads before the writes.
                const int t = tid - 32, r = t >> 1, hf = t & 1;
                ok &= waitb(VB_QK);
                float x[64];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 a0 = *reinterpret_cast<const float4 *>(
                        sQK + (2 * hf) * 8192 + sw128_chunk(r, c));
                    const float4 a1 = *reinterpret_cast<const float4 *>(
                        sQK + (2 * hf + 1) * 8192 + sw128_chunk(r, c));
                    x[4 * c + 0] = a0.x; x[4 * c + 1] = a0.y; x[4 * c + 2] = a0.z;
                    x[4 * c + 3] = a0.w;
                    x[32 + 4 * c + 0] = a1.x; x[32 + 4 * c + 1] = a1.y;
                    x[32 + 4 * c + 2] = a1.z; x[32 + 4 * c + 3] = a1.w;
                }
                __syncwarp();
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 c1, c2, c3;
                    split3_bf16x8(x + 8 * c, c1, c2, c3);
                    *reinterpret_cast<uint4 *>(sQK + hf * 8192 + sw128_chunk(r, c)) = c1;
                    *reinterpret_cast<uint4 *>(sQK + (2 + hf) * 8192 + sw128_chunk(r, c)) = c2;
                    *reinterpret_cast<uint4 *>(sQK + (4 + hf) * 8192 + sw128_chunk(r, c)) = c3;
                }
                fence_proxy_async_smem();
                mbar_arrive(&bar[VB_QKS]);
            }
        }
        if (warp == 0 || warp == 5) {
            // stage the Gram rows: q.k (warp 0, lanes 0..31), k.k (warp 5,
            // lanes 32..63 -- warp 1, which reaches the same lanes, is
            // splitting the state tile meanwhile)
            ok &= waitb(VB_GRAM);
            tc_fence_after();
            __syncwarp();
            const int r = (warp == 0 ? 0 : 32) + lane;
            float4 *srow = reinterpret_cast<float4 *>(staged(r));
            float x[32];
            tmem_ld32(tmem + TM_GP + lane_base, x);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
                srow[c4 ^ (r & 7)] = make_float4(x[4 * c4], x[4 * c4 + 1], x[4 * c4 + 2],
                                                 x[4 * c4 + 3]);
            mbar_arrive(&bar[VB_STAGED]);
        }
        if (warp == 0) {
            // compact C and G of row i, gathered in depth order
            ok &= waitb(VB_STAGED);
            const float *qk = staged(i), *kk = staged(32 + i);
            float *crow = Cc + i * kVLd, *grow = Gc + i * kVLd;
            float qv[kVSlots], kv[kVSlots];
#pragma unroll
            for (int t = 0; t < kVSlots; ++t) {
                const int j = (aw[t >> 2] >> (8 * (t & 3))) & 0xff;
                const int sw = (((j >> 2) ^ (i & 7)) << 2) | (j & 3);
                qv[t] = qk[sw];
                kv[t] = kk[sw];
            }
#pragma unroll
            for (int t = 0; t < kVSlots; ++t) {
                if (t <= my_depth) {
                    crow[t] = ratio[t] * qv[t];
                    if (t < my_depth) grow[t] = bt * ratio[t] * kv[t];
                }
            }
            mbar_arrive(&bar[VB_CG]);
        }
        if (warp >= 1 && warp <= 4) {
            // S_pre tile split in place (row r): both boxes' row r (columns
            // 0..31, 32..63) become 64 bf16 of each copy, N-contiguous and
            // 128B-swizzled -- S_hi in the first box and S_lo in the second
            // (bf16 inputs), or S_1, S_2 there and S_3 after them (fp32)
            const int r = tid - 32;
            ok &= waitb(VB_S);
            uint8_t *box0 = sS, *box1 = sS + 16384;
            float x[64];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 a0 = *reinterpret_cast<const float4 *>(box0 + sw128_chunk(r, c));
                const float4 a1 = *reinterpret_cast<const float4 *>(box1 + sw128_chunk(r, c));
                x[4 * c + 0] = a0.x; x[4 * c + 1] = a0.y; x[4 * c + 2] = a0.z; x[4 * c + 3] = a0.w;
                x[32 + 4 * c + 0] = a1.x; x[32 + 4 * c + 1] = a1.y;
                x[32 + 4 * c + 2] = a1.z; x[32 + 4 * c + 3] = a1.w;
            }
            if constexpr (F32) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 c1, c2, c3;
                    split3_bf16x8(x + 8 * c, c1, c2, c3);
                    *reinterpret_cast<uint4 *>(box0 + sw128_chunk(r, c)) = c1;
                    *reinterpret_cast<uint4 *>(box1 + sw128_chunk(r, c)) = c2;
                    *reinterpret_cast<uint4 *>(sS + 32768 + sw128_chunk(r, c)) = c3;
                }
            } else {
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
            mbar_arrive(&bar[VB_CONV]);
        }
        ok &= waitb(VB_TOPO);
        const float p = (i < T) ? expf(Ls[i]) : 0.f; // P_i of node i = lane

        if (warp == 0 || warp == 5) {
            // Rows of W (warp 0: y) and M (warp 5: z) of node n = lane by
            // backward substitution along its ancestor path a_0 .. a_d = n:
            //   y_t = [t = d] - sum_{u > t} y_u G(a_u, a_t),
            //   z_t = C(n, a_t) - sum_{u > t} z_u G(a_u, a_t),
            // the finite Neumann sum of Eq. (6) restricted to the path (Lemma 3).
            // Formed while the state products run; written into the [M; W]
            // operand once they have released the tile buffer.
            const int n = lane;
            const bool wrow = warp == 0;
            ok &= waitb(VB_CG);
            float vals[kVSlots];
            uint32_t aw4[4] = {0, 0, 0, 0};
            int di = -1;
            if (n < T) {
                di = Ds[n];
                const uint4 a4 = *reinterpret_cast<const uint4 *>(ancat + n * kVSlots);
                aw4[0] = a4.x; aw4[1] = a4.y; aw4[2] = a4.z; aw4[3] = a4.w;
                const float *ci = Cc + n * kVLd;
                float cv[kVSlots], acc[kVSlots], gcur[kVSlots];
#pragma unroll
                for (int t = 0; t < kVSlots; ++t) {
                    cv[t] = wrow ? 0.f : ci[t];
                    acc[t] = 0.f;
                }
                {
                    const float *gr = Gc + n * kVLd;
#pragma unroll
                    for (int t = 0; t < kVSlots - 1; ++t) gcur[t] = gr[t];
                }
#pragma unroll
                for (int u = kVSlots - 1; u >= 0; --u) {
                    vals[u] = 0.f;
                    if (u <= di) {
                        float gnext[kVSlots];
                        if (u >= 1) { // G row of the ancestor at depth u - 1, one step ahead
                            const int an = (aw4[(u - 1) >> 2] >> (8 * ((u - 1) & 3))) & 0xff;
                            const float *gr = Gc + an * kVLd;
#pragma unroll
                            for (int t = 0; t < u - 1; ++t) gnext[t] = gr[t];
                        }
                        const float val = wrow ? ((u == di) ? 1.f : -acc[u]) : cv[u] - acc[u];
                        vals[u] = val;
#pragma unroll
                        for (int t = 0; t < u; ++t) acc[t] = fmaf(val, gcur[t], acc[t]);
#pragma unroll
                        for (int t = 0; t < u - 1; ++t) gcur[t] = gnext[t];
                    }
                }
            } else {
#pragma unroll
                for (int u = 0; u < kVSlots; ++u) vals[u] = 0.f;
            }
            ok &= waitb(VB_STATE);
            const int orow = wrow ? 32 + n : n; // [M; W]: M rows 0..31, W rows 32..63
#pragma unroll
            for (int c = 0; c < 8; ++c) { // K extent <= 32 nodes: one 128-byte row
                *reinterpret_cast<float4 *>(sS + sw128_chunk(orow, c)) =
                    make_float4(0.f, 0.f, 0.f, 0.f);
                if (F32) // the tf32 low part
                    *reinterpret_cast<float4 *>(sS + 16384 + sw128_chunk(orow, c)) =
                        make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kVSlots; ++u) {
                if (u <= di) {
                    const int au = (aw4[u >> 2] >> (8 * (u & 3))) & 0xff;
                    if constexpr (F32) {
                        const float hi = tf32_round(vals[u]);
                        *reinterpret_cast<float *>(sS + sw128_offset(orow, au)) = hi;
                        *reinterpret_cast<float *>(sS + 16384 + sw128_offset(orow, au)) =
                            tf32_round(vals[u] - hi);
                    } else {
                        *reinterpret_cast<float *>(sS + sw128_offset(orow, au)) = vals[u];
                    }
                }
            }
        }
        if (warp == 1 || warp == 5) {
            // R^T of the tile's columns 32 (warp / 5) .. + 31 for node i = lane:
            // K S_pre from tensor-memory lanes 32..63, the value row from V.
            ok &= waitb(VB_STATE);
            if (!F32) ok &= waitb(VB_V);
            tc_fence_after();
            __syncwarp();
            const int col0 = warp == 5 ? 32 : 0;
            float x[32];
            tmem_ld32(tmem + lane_base + col0, x);
            if constexpr (F32) {
                // R^T as tf32 hi (32 KB) + lo (40 KB); the value row from registers
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float r = (i < T) ? bt * (vreg[c] - p * x[c]) : 0.f;
                    const float hi = tf32_round(r);
                    *reinterpret_cast<float *>(sS + 32768 + sw128_offset(col0 + c, i)) = hi;
                    *reinterpret_cast<float *>(sS + 40960 + sw128_offset(col0 + c, i)) =
                        tf32_round(r - hi);
                }
            } else {
                uint8_t *dst = sS + 16384;
                const uint8_t *vrow = sV + i * 128;
                uint4 vv[4]; // read ahead of the scattered stores below, which could alias
#pragma unroll
                for (int uu = 0; uu < 4; ++uu)
                    vv[uu] = *reinterpret_cast<const uint4 *>(
                        vrow + ((((col0 >> 3) + uu) ^ (i & 7)) << 4));
#pragma unroll
                for (int uu = 0; uu < 4; ++uu) {
                    float f[8];
                    bf16x8_to_f32(vv[uu], f);
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const int c = 8 * uu + t;
                        const float r = (i < T) ? bt * (f[t] - p * x[c]) : 0.f;
                        *reinterpret_cast<float *>(dst + sw128_offset(col0 + c, i)) = r;
                    }
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bar[VB_OPS]);

        // ---- outputs: O = P (Q S_pre) + M R (warps 0, 4), U = W R (warps 1, 5) ----
        // Each thread puts its 32 columns of row i into the tile buffer the
        // propagation has released (rows padded by 16 B); then the compute
        // warps store the tile's rows segment by segment (row-per-thread
        // global stores touch 32 cache lines per instruction).
        constexpr int kOR = kVB * (F32 ? 4 : 2) + 16, kUR = kVB * 4 + 16; // staged row strides
        uint8_t *stO = sS, *stU = sS + kVT * kOR;
        if (quad < 2) {
            ok &= waitb(VB_PROP);
            tc_fence_after();
            __syncwarp();
            const int col0 = warp >= 4 ? 32 : 0;
            float x[32];
            if (quad == 0) {
                float y[32];
                tmem_ld32_async(tmem + TM_GP + lane_base + col0, x);
                tmem_ld32_async(tmem + lane_base + col0, y);
                tmem_wait_ld32(x);
                tmem_wait_ld32(y);
#pragma unroll
                for (int t = 0; t < 32; ++t) x[t] = fmaf(p, y[t], x[t]);
                if constexpr (F32) {
                    float4 *dsto = reinterpret_cast<float4 *>(stO + i * kOR + col0 * 4);
#pragma unroll
                    for (int uu = 0; uu < 8; ++uu)
                        dsto[uu] =
                            make_float4(x[4 * uu], x[4 * uu + 1], x[4 * uu + 2], x[4 * uu + 3]);
                } else {
                    uint4 *dsto = reinterpret_cast<uint4 *>(stO + i * kOR + col0 * 2);
#pragma unroll
                    for (int uu = 0; uu < 4; ++uu) {
                        __nv_bfloat162 p2[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t)
                            p2[t] = __floats2bfloat162_rn(x[8 * uu + 2 * t], x[8 * uu + 2 * t + 1]);
                        dsto[uu] = *reinterpret_cast<uint4 *>(p2);
                    }
                }
            } else {
                tmem_ld32(tmem + TM_GP + lane_base + col0, x);
                float4 *dstu = reinterpret_cast<float4 *>(stU + i * kUR + col0 * 4);
#pragma unroll
                for (int uu = 0; uu < 8; ++uu)
                    dstu[uu] = make_float4(x[4 * uu], x[4 * uu + 1], x[4 * uu + 2], x[4 * uu + 3]);
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kVTCompute) : "memory");
        if (ok && !*sfail) {
            if constexpr (F32) {
                float *O = static_cast<float *>(Oout);
                for (int c = tid; c < T * 16; c += kVTCompute) { // O: 16 chunks of 16 B per row
                    const int r = c >> 4, q = c & 15;
                    *reinterpret_cast<uint4 *>(O + ((size_t)(o + r) * H + h) * kD + c0 + q * 4) =
                        *reinterpret_cast<const uint4 *>(stO + r * kOR + q * 16);
                }
            } else {
                __nv_bfloat16 *O = static_cast<__nv_bfloat16 *>(Oout);
                for (int c = tid; c < T * 8; c += kVTCompute) { // O: 8 chunks of 16 B per row
                    const int r = c >> 3, q = c & 7;
                    *reinterpret_cast<uint4 *>(O + ((size_t)(o + r) * H + h) * kD + c0 + q * 8) =
                        *reinterpret_cast<const uint4 *>(stO + r * kOR + q * 16);
                }
            }
            for (int c = tid; c < T * 16; c += kVTCompute) { // U: 16 chunks per row
                const int r = c >> 4, q = c & 15;
                *reinterpret_cast<float4 *>(Uout + ((size_t)(o + r) * H + h) * kD + c0 + q * 4) =
                    *reinterpret_cast<const float4 *>(stU + r * kUR + q * 16);
            }
        }
        if (!ok) report(st, BOLE_ERR_TIMEOUT, b, -1, 31);
    }
    tc_fence_before();
    __syncthreads();
    if (*sfail) { // read after the barrier: the same value in every thread
        // after a timeout the products and copies this CTA issued end
        // (bounded) before its tensor and shared memory go to another CTA
        if (issuer) {
            mma_commit(&bar[VB_DRAIN]);
            mbar_wait(&bar[VB_DRAIN], 0, kWaitNs);
            mbar_wait(&bar[VB_QK], 0, kWaitNs);
            if (!F32) mbar_wait(&bar[VB_V], 0, kWaitNs);
            mbar_wait(&bar[VB_S], 0, kWaitNs);
        }
        __syncthreads();
    }
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

} // namespace

// CTAs of a launch resident at once (per_sm per SM), 0 if unknown
static int vtile_resident_ctas(int per_sm)
{
    static int sms[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        sms[dev] = n;
    }
    return per_sm * sms[dev];
}

bool tc_vtile_supported(const VerifyArgs &a)
{
    return (a.dtype == BOLE_BF16 || a.dtype == BOLE_F32) && a.dk == kD && a.dv == kD &&
           a.max_T <= kVT && a.max_depth < kVSlots && !a.vk;
}

// Value tiles pay off while the heads of the batch leave the one-CTA
// kernel (two CTAs per SM) short of one wave: measured on the 16-head
// single request, 7.5 vs 7.8 us; on 512 heads, 28 vs 22 us (each CTA's
// latency chain is as long as the one-CTA kernel's, so halving its state
// bytes leaves fewer bytes in flight per SM).
bool tc_vtile_preferred(const VerifyArgs &a)
{
    const int slots = vtile_resident_ctas(2);
    return slots > 0 && a.B * a.H < slots;
}

template <bool F32>
static cudaError_t launch_vtile(const VerifyArgs &a, cudaStream_t s, bool overlap)
{
    using P = VtPlan<F32>;
    const int units = a.B * a.H;
    CUtensorMap mS, mQ, mK, mV;
    cudaError_t e = make_state_map(&mS, a.S_pre, units);
    if (e == cudaSuccess) e = make_node_map(&mQ, a.q, a.N, a.H, kVT, F32);
    if (e == cudaSuccess) e = make_node_map(&mK, a.k, a.N, a.H, kVT, F32);
    if (e == cudaSuccess) e = make_node_map(&mV, a.v, a.N, a.H, kVT, F32);
    if (e != cudaSuccess) return e;
    e = configure_once(reinterpret_cast<const void *>(tc_vtile_kernel<F32>), P::SMEM, true);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = launch_config(dim3(2 * units), dim3(kVTThreads), P::SMEM, s,
                                                 overlap, attr);
    return cudaLaunchKernelEx(&cfg, tc_vtile_kernel<F32>, mS, mQ, mK, mV, a.gamma, a.beta,
                              a.offsets, a.anc, a.req_depth, a.H, a.N, a.O, a.U, a.logP, a.st,
                              vtile_resident_ctas(P::PER_SM), overlap ? 0 : 1, a.parent,
                              a.max_depth, a.inline_topo ? 1 : 0,
                              static_cast<const float *>(F32 ? a.v : nullptr));
}

cudaError_t launch_tc_vtile_verify(const VerifyArgs &a, cudaStream_t s, bool overlap)
{
    if (a.B * a.H == 0 || a.N == 0) return cudaSuccess;
    return a.dtype == BOLE_F32 ? launch_vtile<true>(a, s, overlap)
                               : launch_vtile<false>(a, s, overlap);
}

} // namespace bole
