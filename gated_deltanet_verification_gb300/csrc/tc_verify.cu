// Tensor-core (TMA + tcgen05) verification and commit for bf16 q/k/v with
// d_k = d_v = 128 -- the Qwen3.5-shaped GDN head of the pages' evaluation.
//
// Verification, one CTA per (request, head), two CTAs per SM, trees of up to
// 64 nodes and depth <= 15.  Everything between the inputs and (O, U, logP)
// stays on chip:
//   1. TMA streams the head's S_pre (128 x 128 fp32, four 32-column
//      128B-swizzled boxes) and [Q;K] of the tree (one 128 x 128 bf16
//      operand, rows 0..63 q, 64..127 k).
//   2. While S_pre is in flight: the cumulative decay L_i = sum of log gamma
//      over the ancestors-or-self of i (Lemma 1), the Gram [Q;K] K^T on
//      tcgen05, the ancestor-masked factors
//        C_ij = exp(L_i - L_j) q_i.k_j          (j an ancestor of i or i)
//        G_ij = beta_i exp(L_i - L_j) k_i.k_j   (j a strict ancestor of i)
//      stored compactly by ancestor depth, and the rows of W = (I+G)^{-1}
//      and M = C W by backward substitution along each node's ancestor path
//      (below).  The value rows follow by TMA once the factor scratch is free.
//   3. S_pre is split exactly into bf16 S_hi + S_lo (S - S_hi rounds to bf16
//      with ~2^-18 relative residue); tcgen05 computes [Q;K] (S_hi + S_lo)
//      with bf16 products (exact) and fp32 accumulation.
//   4. Epilogue: R = D_beta (V - D_P K S_pre) goes to shared memory as R^T,
//      [M; W] is scattered into the other operand buffer.
//   5. One tcgen05 product (tf32) [M; W] R gives M R and W R = U; the output
//      adds D_P Q S_pre to M R (Eq. (6)), so O and U leave in one pass.
//
// Rows of W and M.  Restricted to the ancestor path a_0 (root), ..., a_d = i
// of node i, I + G is the (d+1) x (d+1) unit lower-triangular matrix
// L[u][t] = G(a_u, a_t) (u > t), and row i of the inverse only involves that
// path (Lemma 3: every chain of G from i ends at an ancestor).  So row i of W
// is the y with y^T L = e_d^T, and row i of M = C W is the z with
// z^T L = c^T, c_t = C(i, a_t): both by backward substitution from t = d,
//   y_t = [t = d] - sum_{u > t} y_u G(a_u, a_t),
//   z_t = c_t     - sum_{u > t} z_u G(a_u, a_t),
// which equals the d-step Neumann sum of Eq. (8) (nilpotent G, G^{d+1} = 0)
// term by term, with one thread per node and no barrier between steps.
//
// Deviations from the pages' kernel: the inverse is formed once on the
// T x T tree (not applied to each value tile's R by the recurrence), so the
// dependent steps stay off the state-streaming path and propagation +
// read-out become one dense tensor-core product per head.  The result is the
// same polynomial, Eq. (6).
//
// Commit, one CTA per (request, head, 64-column half) with an accepted node:
// TMA loads the half of S, one tcgen05 product (D_a K_a)^T U_a over the
// accepted path (K chunks of 16 path nodes), the epilogue adds P_a S and TMA
// stores S in place (Eq. (10)).
#include <cudaTypedefs.h>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "sm100.cuh"
#include "tc_common.cuh"

namespace bole {
namespace {

using namespace sm100;
using namespace tc;

constexpr int kT = 64;        // padded tree extent
constexpr int kSlots = 16;    // depth slots in the compact factors: depth <= 15
constexpr int kLd = 17;       // padded row stride of the compact factors (bank spread)

// ---- verification shared-memory plan (bytes from a 1024-aligned base) ----
//   S buffer (64 KB): four 16 KB boxes [128 rows x 128 B] of fp32 S_pre; the
//     in-place split turns boxes (0,1) into (S_hi, S_lo) of columns 0..63 and
//     boxes (2,3) into those of columns 64..127 (bf16, 128B-swizzled,
//     N-contiguous).  Once the first d_k half of the state products has
//     read rows 0..63 of every box, those rows (first 8 KB of each box) hold
//     the staged Gram; after the whole product the first 32 KB hold [M;W]
//     and the second 32 KB R^T, both tf32 K-major.
//   A1 (32 KB): [Q;K] bf16 K-major, operand of the Gram and the state
//     products; once the first d_k half is done, its first 16 KB take the
//     head's value rows by TMA (two 128B-swizzled boxes [64 rows x 64 bf16]),
//     read by the epilogue from shared memory.
//   X (11 KB): the factor scratch (compact C and G, ancestor table, decays,
//     depths, log gammas).
// Tensor memory (256 columns, lane = operand row): columns 0..127 hold
// [Q S_pre; K S_pre], columns 128..255 the propagation [M R; W R]; before the
// propagation, 128..191 hold the Gram.  The epilogues only read tensor memory.
//
// Trees of at most 32 nodes (the small variant) load q and k as 32-row boxes,
// so rows 32..63 and 96..127 of each [Q;K] K-atom are padding that the
// products read into tensor-memory lanes nobody reads.  Those 16 KB take the
// value rows (TMA at entry, rows 32..63 of both atoms) and the staged Gram
// (q.k rows 96..127 of atom 0, k.k rows 96..127 of atom 1, 128 B per row),
// so the factor chain -- Gram, gather, substitution -- no longer waits for
// the first d_k half of the state products and runs beside the S_pre
// stream; the rows of W and M are held in registers until the state
// products release the S buffer.
constexpr int kTSmall = 32;
constexpr int SM_V = 4096;                    // value rows: + 16384 for columns 64..127
constexpr int SM_GQK = 12288, SM_GKK = 28672; // staged q.k and k.k Gram rows
constexpr int OFF_SBUF = 0;
constexpr int SBUF_BYTES = 65536;
constexpr int OFF_A1 = SBUF_BYTES;
constexpr int OFF_X = OFF_A1 + 32768;         // factor scratch
constexpr int X_BYTES = 11264;
constexpr int OFF_BAR = OFF_X + X_BYTES;      // mbarriers
constexpr int OFF_MISC = OFF_BAR + 16 * 8;    // TMEM slot
constexpr int VERIFY_END = OFF_MISC + 16;
// factor scratch
constexpr int FAC_BYTES = kT * kLd * 4;       // one compact factor [64][17] f32
constexpr int X_G = OFF_X;                    // G (row i, ancestor slot t < depth(i))
constexpr int X_C = X_G + FAC_BYTES;          // C (row i, ancestor slot t <= depth(i))
constexpr int X_ANCAT = X_C + FAC_BYTES;      // [64][16] u8: ancestor of row i at depth t
constexpr int X_L = X_ANCAT + kT * kSlots;    // L_i
constexpr int X_DEPTH = X_L + kT * 4;
constexpr int X_LG = X_DEPTH + kT * 4;        // log gamma_i
// topology formed in the kernel (no pack before it): ancestor masks and jumps
constexpr int X_JMASK = X_LG + kT * 4;        // u64 [64]
constexpr int X_JUMP = X_JMASK + kT * 8;      // int [64]
static_assert(X_JUMP + kT * 4 <= OFF_X + X_BYTES, "factor scratch fits its region");
static_assert(X_JMASK % 8 == 0, "aligned masks");
constexpr int OFF_TOPO = OFF_BAR + 13 * 8;    // int [2]: first bad node, request depth
static_assert(X_ANCAT % 16 == 0, "vector-aligned ancestor rows");
// Deferred commit of the previous round (the FUSE kernels): its tree's parent
// links, the accepted path (node first) and two words (path length, failure)
// follow the mbarriers; the two operands of its product, (D_a K_a)^T and
// U_a^T as 128 x 8 tf32 K-major tiles (32B-swizzled), use the compact-factor
// scratch, which the gather writes only after that product has ended.
constexpr int kFzMaxPath = 16;                // two K chunks of eight path nodes
constexpr int OFF_FZ = VERIFY_END;            // int [128]
constexpr int FZ_PATH = OFF_FZ + kMaxTree * 4; // int [16]
constexpr int FZ_MISC = FZ_PATH + kFzMaxPath * 4; // int [2], then the mbarrier below
constexpr int FZ_DONE = FZ_MISC + 8;          // one phase: the whole commit product has ended
constexpr int FZ_DRAIN = FZ_MISC + 16;        // after a timeout: the product's issuer drains
constexpr int VERIFY_END_FZ = FZ_MISC + 24;
static_assert(FZ_DONE % 8 == 0, "aligned mbarrier");
constexpr int FZ_A = X_G, FZ_B = X_G + 4096;
static_assert(FZ_B + 4096 <= X_ANCAT && FZ_A % 256 == 0, "commit operands in the compact factors");
// Two CTAs per SM leave 113 KB each (228 KB less 1 KB reserved per CTA); the
// plan fills 112 KB and keeps 256 B of slack for the 1024 B alignment of the
// dynamic base, which is aligned when the kernel has no static shared memory
// (checked in the kernel).  A request at the 113 KB edge would drop to one CTA
// per SM as soon as anything else claimed shared memory.
constexpr int VERIFY_SMEM = VERIFY_END_FZ + 256;
static_assert(2 * (VERIFY_SMEM + 1024) <= 228 * 1024, "two verification CTAs per SM");
static_assert(3 * VERIFY_SMEM > 228 * 1024,
              "at most two verification CTAs (2 x 256 TMEM columns) per SM");

constexpr int kORow = kD * 2 + 16, kURow = kD * 4 + 16; // staged output rows, padded
static_assert(kT * kORow <= 32768 && kT * kURow <= SBUF_BYTES, "staged outputs fit");
constexpr int kComputeThreads = 256;          // warps 0..7: factors, split, epilogues
constexpr int kThreads = kComputeThreads + 32; // warp 8: TMA and tcgen05 issue

constexpr uint32_t IDESC_GRAM = idesc_bf16(128, 64, false, false);  // [Q;K] K^T
constexpr uint32_t IDESC_GRAM_S = idesc_bf16(128, 32, false, false); // small trees
constexpr uint32_t IDESC_STATE = idesc_bf16(128, 128, false, true); // [Q;K] S, S N-contiguous
constexpr uint32_t IDESC_STATE_VK = idesc_bf16(128, 128, false, false); // S stored [dv][dk]
constexpr uint32_t IDESC_TF32 = idesc_tf32(128, 128, false, false); // both K-major
constexpr uint32_t TM_GRAM = 128, TM_PROP = 128;                  // tensor-memory columns

// mbarrier slots
constexpr int BAR_S = 0, BAR_A1 = 1, BAR_GRAM = 2, BAR_V = 3, BAR_STATE_A = 4, BAR_STATE = 5,
              BAR_MMA2 = 6, BAR_TOPO = 7, BAR_STAGED = 8, BAR_CG = 9, BAR_CONV = 10, BAR_OPS = 11,
              BAR_DRAIN = 12;
constexpr int BAR_FZ = 15; // deferred commit: a chunk's product done (slot 13 holds the
                           // topology words)

// The previous round's commit inputs for the deferred commit (FUSE): what
// bole_commit would read, for the same B requests and H heads.
struct PrevRound {
    const __nv_bfloat16 *k;              // [N][H][128], the keys its verification read
    const float *U, *logP;               // its outputs, [N][H][128] and [N][H]
    const int32_t *offsets, *parent, *accepted;
    int N;
};

// Verification kernel: one CTA per (request, head).  Warp 8 streams operands
// and issues the tensor-core products.  Warps 0..7 share the rest:
//   warps 0, 1  topology, decay ratios, staging the q.k Gram rows, gathering
//               the compact C and G, the rows of W;
//   warps 2, 3  staging the k.k Gram rows, then R^T for columns 0..63;
//   warps 4..7  splitting S_pre as soon as it lands; then warps 4, 5 the
//               rows of M, warps 6, 7 R^T for columns 64..127.
// The state products run in two halves of d_k: the first half releases the
// [Q;K] columns that the value rows then overwrite and the S_pre rows where
// the Gram is staged, so neither waits for the whole product.  All waits are
// bounded.
// VK: the state is stored transposed, [dv][dk] per head (the serving
// runtime's slot layout).  The same TMA boxes and the same split then give
// K-major operand rows (row = value column, 64 d_k entries per 128 B), the
// first d_k half of the product reads the boxes (0, 1) whole, and the Gram
// is staged in those 32 KB instead.
// SMALL (trees of at most 32 nodes): the Gram and the value rows live in the
// [Q;K] padding; warps 0 and 2 stage the Gram, warp 0 gathers and forms the
// rows of W, warp 1 those of M (both before the state products end); warps
// 2 and 6 form R^T; only the lanes of rows 0..31 and 64..95 carry outputs.
// FUSE (deferred commit): before verifying, the CTA applies the previous
// round's commit (Eq. (10)) to the state tile it has just loaded and stores
// the committed state in place, so one state read serves both.  Warps 4..7
// request the previous accepted node and parent links in the prologue, walk
// the path after it and stage the path operands; one of their threads runs
// the product (D_a K_a)^T U_a into tensor-memory columns 0..127 (free until
// the state products); they add P_a S_r to it row by row, store each
// 64-column half by TMA and split the committed values.  In the 64-node
// layout C and G are then gathered from the Gram in tensor memory (the
// staging would wait for the state side).
template <bool VK, bool SMALL, bool FUSE>
__global__ void __launch_bounds__(kThreads, 2)
tc_verify_kernel(const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmQ,
                 const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const float *__restrict__ gamma, const float *__restrict__ beta,
                 const int32_t *__restrict__ offsets, const uint32_t *__restrict__ anc,
                 const int32_t *__restrict__ req_depth, int H, int N,
                 __nv_bfloat16 *__restrict__ O, float *__restrict__ Uout,
                 float *__restrict__ logP, int32_t *st, int pf_stride, int early_alloc,
                 const int32_t *__restrict__ parent, int max_depth, int inline_topo,
                 const PrevRound prev)
{
    static_assert(!(FUSE && VK), "the deferred commit supports the default state layout");
    constexpr bool kColGather = FUSE && !SMALL; // C and G gathered from tensor memory
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *sbuf = sm + OFF_SBUF;
    uint8_t *sA1 = sm + OFF_A1;
    uint8_t *sV = sm + OFF_A1; // value rows over the first d_k half of [Q;K]
    float *Gc = reinterpret_cast<float *>(sm + X_G);
    float *Cc = reinterpret_cast<float *>(sm + X_C);
    uint8_t *ancat = sm + X_ANCAT;
    float *Ls = reinterpret_cast<float *>(sm + X_L);
    int *Ds = reinterpret_cast<int *>(sm + X_DEPTH);
    float *LGs = reinterpret_cast<float *>(sm + X_LG);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x;
    const int b = unit / H, h = unit % H;

    if (sm + VERIFY_END_FZ > smem_raw + VERIFY_SMEM) { // dynamic base too far from 1024 B
        if (tid == 0) report(st, BOLE_ERR_CUDA, b, -1, -1);
        return;
    }
    // Tensor memory: the SM starts the next CTA of a kernel that allocates
    // tensor memory only once the resident one has given up its allocation
    // permit.  A launch of its own allocates first, so the second CTA of each
    // SM is not held back by the prologue; a launch overlapping the previous
    // kernel allocates after the prologue (measured faster there: the CTAs
    // that wait for the previous kernel then do not all start at once).
    if (early_alloc && warp == 0) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    // An overlapped commit may start its state reads; the deferred-commit form
    // writes the state, so nothing after it starts before it has ended.
    if (!FUSE) pdl_launch_dependents();
    // Caller inputs first (a launch that overlaps pack reads only these before
    // it waits): the request's extent, then the small, latency-critical reads
    // -- [Q;K] and the per-thread gamma, beta -- before the 64 KB state tile,
    // which every CTA requests at once.
    const int o = offsets[b], T = offsets[b + 1] - o;
    constexpr int kTmax = SMALL ? kTSmall : kT;
    const bool in_range = T > 0 && T <= kTmax && o >= 0 && o + T <= N;
    const bool issuer = tid == kComputeThreads;
    if (issuer) {
        for (int i = BAR_S; i <= BAR_MMA2; ++i) mbar_init(&bar[i], 1);
        mbar_init(&bar[BAR_TOPO], kT);
        mbar_init(&bar[BAR_STAGED], SMALL ? 64 : 128);
        mbar_init(&bar[BAR_CG], kColGather ? 128 : kT); // C and G gathered apart
        mbar_init(&bar[BAR_CONV], 128);
        mbar_init(&bar[BAR_OPS], kComputeThreads);
        mbar_init(&bar[BAR_DRAIN], 1);
        if (FUSE) {
            mbar_init(&bar[BAR_FZ], 1);
            mbar_init(reinterpret_cast<uint64_t *>(sm + FZ_DONE), 1);
            mbar_init(reinterpret_cast<uint64_t *>(sm + FZ_DRAIN), 1);
        }
        fence_mbar_init();
        if (in_range) {
            // q rows 0.., k rows 64.. of each K-atom (boxes of kTmax rows)
            mbar_arrive_expect_tx(&bar[BAR_A1], SMALL ? 16384 : 32768);
#pragma unroll
            for (int ka = 0; ka < 2; ++ka) {
                tma_load_3d(sA1 + ka * 16384, &tmQ, &bar[BAR_A1], 64 * ka, h, o);
                tma_load_3d(sA1 + ka * 16384 + 8192, &tmK, &bar[BAR_A1], 64 * ka, h, o);
            }
        }
    }
    const int rowgrp = warp & 3, half = warp >> 2;
    const int m = rowgrp * 32 + lane; // TMEM lane = operand row
    const int i = m & 63;             // this thread's node
    const bool topo = tid < kT;       // warps 0, 1: row i = tid
    float bt = 0.f;                   // beta_i (topology rows and the K-side rows)
    float g_i = 1.f;
    int my_par = -1;                  // topology rows, topology formed here: parent of i
    if (warp < 8 && in_range && i < T) {
        if (topo || m >= 64) bt = beta[(size_t)(o + i) * H + h];
        if (topo) g_i = gamma[(size_t)(o + i) * H + h];
        if (topo && inline_topo) my_par = parent[o + i];
    }
    if (issuer) {
        if (!FUSE) { // (the deferred-commit form requests it after the prologue)
            mbar_arrive_expect_tx(&bar[BAR_S], SBUF_BYTES);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tma_load_2d(sbuf + c * 16384, &tmS, &bar[BAR_S], 32 * c, unit * kD);
        }
        if (SMALL && in_range) { // value rows into the padding of the q boxes
            mbar_arrive_expect_tx(&bar[BAR_V], 8192);
            tma_load_3d(sA1 + SM_V, &tmV, &bar[BAR_V], 0, h, o);
            tma_load_3d(sA1 + SM_V + 16384, &tmV, &bar[BAR_V], 64, h, o);
        }
        if (!SMALL && in_range) {
            // 64-node layout: the value rows can only be loaded once the first
            // d_k half of the state products has released their buffer, and
            // R^T waits for them; requested into L2 now, that load is an L2 hit
            // (first wave of config 3: R^T found them 5.7 K cycles late)
            tma_prefetch_l2_3d(&tmV, 0, h, o);
            tma_prefetch_l2_3d(&tmV, 64, h, o);
        }
    }
    // What the previous call wrote (the status word pack reset, the
    // per-request depth, each node's ancestor-or-self mask) is read after the
    // wait; the reads above are already in flight, so without an overlapped
    // launch they all arrive in one round trip.
    pdl_wait();
    int *sfault = reinterpret_cast<int *>(sm + OFF_MISC + 4);
    // Set by any thread whose bounded wait gave up; the issuing thread then
    // issues no further copy or product.
    volatile int *sfail = reinterpret_cast<volatile int *>(sm + OFF_MISC + 8);
    if (tid == 0) {
        *sfault = *(const volatile int32_t *)st; // one read: a uniform exit
        *sfail = 0;
    }
    int *stopo = reinterpret_cast<int *>(sm + OFF_TOPO);
    const int d_read = inline_topo ? 0 : req_depth[b];
    int my_depth = -1;
    uint64_t my_mask = 0;
    if (!inline_topo) {
        // Depth and ancestor-or-self mask of each node as pack built them
        // (rows below 64: the first two words of the 128-bit mask).  A tree
        // pack found malformed or too deep has set the status or a depth the
        // check below refuses, so such a launch ends before any output; every
        // bit indexes a row below 64 whatever the input.
        if (topo && in_range && i < T) {
            const uint2 mk = *reinterpret_cast<const uint2 *>(anc + (size_t)(o + i) * 4);
            my_mask = ((uint64_t)mk.y << 32) | mk.x;
            my_depth = __popcll(my_mask) - 1;
        }
    } else if (topo) {
        // The round's topology step in the kernel (Section IV-C): each node
        // starts with itself and a jump to its parent, and every round ORs in
        // the mask at its jump target and doubles the jump, so after
        // log2(64) = 6 rounds the mask holds the whole path to the root.
        // A link that does not point backwards is a fault (reported below)
        // and is not followed, so every jump indexes an earlier node.
        uint64_t *smk = reinterpret_cast<uint64_t *>(sm + X_JMASK);
        int *sjp = reinterpret_cast<int *>(sm + X_JUMP);
        const bool live = in_range && i < T;
        const bool badp = live && (my_par < -1 || my_par >= i);
        uint64_t mk = live ? (1ull << i) : 0ull;
        int jp = (live && !badp) ? my_par : -1;
        if (tid == 0) {
            stopo[0] = kT;
            stopo[1] = 0;
        }
        smk[i] = mk;
        sjp[i] = jp;
        asm volatile("bar.sync 3, 64;" ::: "memory");
        if (badp) atomicMin(&stopo[0], i);
#pragma unroll 1
        for (int r = 0; r < 6; ++r) {
            uint64_t m2 = 0;
            int j2 = -1;
            if (jp >= 0) {
                m2 = smk[jp];
                j2 = sjp[jp];
            }
            asm volatile("bar.sync 3, 64;" ::: "memory");
            if (jp >= 0) {
                mk |= m2;
                jp = j2;
            }
            smk[i] = mk;
            sjp[i] = jp;
            asm volatile("bar.sync 3, 64;" ::: "memory");
        }
        if (live) {
            my_mask = mk;
            my_depth = __popcll(mk) - 1;
            atomicMax(&stopo[1], my_depth);
        }
    }
    // FUSE, warps 4..7 (row r): the previous round's accepted node, tree
    // extent and parent link r, requested in the prologue (the walk along them
    // runs after the prologue, so it never holds up the CTA's topology step).
    int fz_o = 0, fz_ap = -1, fz_Tp = 0, fz_par = -1;
    bool fz_go = false;
    if (FUSE && warp >= 4 && warp < 8) {
        const int r = tid - 128;
        fz_ap = prev.accepted[b];
        fz_o = prev.offsets[b];
        fz_Tp = prev.offsets[b + 1] - fz_o;
        const bool ext_ok = fz_Tp > 0 && fz_Tp <= kMaxTree && fz_o >= 0 && fz_o + fz_Tp <= prev.N;
        fz_go = fz_ap >= 0 && fz_ap < fz_Tp && ext_ok;
        if (fz_go && r < fz_Tp) fz_par = prev.parent[fz_o + r];
    }
    // FUSE, warps 4..7 (row r): log P of the accepted node and, for the first
    // eight path nodes, log P_t, k_t[r] and u_t[r].
    float fz_La = 0.f, fz_lp[8], fz_kv[8], fz_uv[8];
    if (my_depth >= kSlots) my_depth = -1; // no work for this row (the request is refused)
    if (!early_alloc && warp == 0) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (FUSE && issuer) {
        // The deferred-commit form requests the state tile only now, once the
        // small prologue reads (this round's and the previous round's) have
        // returned: the tile waits for the commit product anyway, and requested
        // at entry it queued those reads behind every CTA's state burst.  Every
        // CTA requests it (the commit of an empty or refused tree needs it, and
        // the exit path waits for it).
        mbar_arrive_expect_tx(&bar[BAR_S], SBUF_BYTES);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            tma_load_2d(sbuf + c * 16384, &tmS, &bar[BAR_S], 32 * c, unit * kD);
    }
    const int fault = *sfault;
    const int d = inline_topo ? stopo[1] : d_read;
    const int bad_node = inline_topo && in_range ? stopo[0] : kT;
    const bool bad = !in_range || d < 0 || d >= kSlots || d >= T || bad_node < kT ||
                     (inline_topo && d > max_depth);
    const uint32_t lane_base = (uint32_t)(rowgrp * 32) << 16;
    // Bounded wait on phase 0 of barrier `i`; a timeout is recorded CTA-wide.
    auto waitb = [&](int i) -> bool {
        const bool r = mbar_wait(&bar[i], 0, kWaitNs);
        if (!r) *sfail = 1;
        return r;
    };
    // ---- deferred commit (FUSE) ----
    // Issuing thread: one kind::tf32 product per chunk, (D_a K_a)^T U_a into
    // tensor-memory columns 0..127 (lane = row of the state).
    uint64_t *fz_done = reinterpret_cast<uint64_t *>(sm + FZ_DONE);
    uint64_t *fz_drain = reinterpret_cast<uint64_t *>(sm + FZ_DRAIN);
    // Split warps (row r): the previous tree's parent links staged, the
    // accepted path walked by one thread with bole_commit's checks (a fault is
    // reported and nothing is committed), then the first chunk's path rows
    // read.  Returns the path length (0: nothing to commit, and fz_done is
    // completed at once for the gather that waits on it).
    auto fz_walk = [&](int r) -> int {
        int *fpar = reinterpret_cast<int *>(sm + OFF_FZ);
        int *fpath = reinterpret_cast<int *>(sm + FZ_PATH);
        int *fmisc = reinterpret_cast<int *>(sm + FZ_MISC);
        if (fz_go && r < fz_Tp) fpar[r] = fz_par;
        asm volatile("bar.sync 4, 128;" ::: "memory");
        if (r == 0) {
            int L = 0, fail = 0, at = fz_ap, aux = fz_Tp;
            if (fz_go) {
                int j = fz_ap;
                while (j >= 0) {
                    if (L >= kFzMaxPath) { // a longer path than this kernel commits
                        fail = BOLE_ERR_DEPTH;
                        aux = kFzMaxPath;
                        break;
                    }
                    fpath[L++] = j;
                    const int p = fpar[j];
                    if (p < -1 || p >= j) {
                        fail = BOLE_ERR_BAD_TOPOLOGY;
                        at = j;
                        aux = -1;
                        break;
                    }
                    j = p;
                }
            } else if (fz_ap >= 0) {
                fail = BOLE_ERR_BAD_TOPOLOGY;
            }
            if (fail != 0) {
                if (h == 0) report(st, fail, b, at, aux);
                L = 0;
            }
            fmisc[0] = L;
            if (L == 0) mbar_arrive(fz_done);
        }
        asm volatile("bar.sync 4, 128;" ::: "memory");
        const int L = fmisc[0];
        if (L > 0) {
            fz_La = prev.logP[(size_t)(fz_o + fpath[0]) * H + h];
#pragma unroll
            for (int tt = 0; tt < 8; ++tt) {
                const bool on = tt < L;
                const size_t nh = (size_t)(fz_o + (on ? fpath[tt] : 0)) * H + h;
                fz_lp[tt] = on ? prev.logP[nh] : 0.f;
                fz_kv[tt] = on ? __bfloat162float(prev.k[nh * kD + r]) : 0.f;
                fz_uv[tt] = on ? prev.U[nh * kD + r] : 0.f;
            }
        }
        return L;
    };
    // Split warps (row r): the operands of each chunk of eight path nodes,
    // A[r][t] = (P_a / P_t) k_t[r] and B^T[r][t] = u_t[r] (node first, as
    // bole_commit forms them), and one kind::tf32 product per chunk,
    // (D_a K_a)^T U_a into tensor-memory columns 0..127 (lane = row of the
    // state), issued by thread r = 0 -- not the issuing warp, whose next
    // product (the Gram) waits for [Q;K]; then the wait for the whole
    // product.  Returns P_a.
    auto fz_stage = [&](int r, int fz_len) -> float {
        const int fz_nch = (fz_len + 7) >> 3;
        const int *fpath = reinterpret_cast<const int *>(sm + FZ_PATH);
        const float La = fz_La;
        uint8_t *fa = sm + FZ_A, *fb = sm + FZ_B;
        const uint32_t fa_s = smem_addr(fa), fb_s = smem_addr(fb);
#pragma unroll 1
        for (int ch = 0; ch < fz_nch; ++ch) {
            float lp[8], kv[8], uv[8];
            if (ch == 0) { // read in the prologue
#pragma unroll
                for (int tt = 0; tt < 8; ++tt) {
                    lp[tt] = fz_lp[tt];
                    kv[tt] = fz_kv[tt];
                    uv[tt] = fz_uv[tt];
                }
            } else {
                // the previous chunk's product has read the operand buffers
                if (!mbar_wait(&bar[BAR_FZ], (uint32_t)(ch - 1) & 1u, kWaitNs)) {
                    *sfail = 1;
                    break;
                }
#pragma unroll
                for (int tt = 0; tt < 8; ++tt) {
                    const int t = 8 * ch + tt;
                    const bool on = t < fz_len;
                    const size_t nh = (size_t)(fz_o + (on ? fpath[t] : 0)) * H + h;
                    lp[tt] = on ? prev.logP[nh] : 0.f;
                    kv[tt] = on ? __bfloat162float(prev.k[nh * kD + r]) : 0.f;
                    uv[tt] = on ? prev.U[nh * kD + r] : 0.f;
                }
            }
            float av[8];
#pragma unroll
            for (int tt = 0; tt < 8; ++tt)
                av[tt] = 8 * ch + tt < fz_len ? expf(La - lp[tt]) * kv[tt] : 0.f;
            *reinterpret_cast<float4 *>(fa + sw32_chunk(r, 0)) = make_float4(av[0], av[1], av[2], av[3]);
            *reinterpret_cast<float4 *>(fa + sw32_chunk(r, 1)) = make_float4(av[4], av[5], av[6], av[7]);
            *reinterpret_cast<float4 *>(fb + sw32_chunk(r, 0)) = make_float4(uv[0], uv[1], uv[2], uv[3]);
            *reinterpret_cast<float4 *>(fb + sw32_chunk(r, 1)) = make_float4(uv[4], uv[5], uv[6], uv[7]);
            fence_proxy_async_smem();
            asm volatile("bar.sync 4, 128;" ::: "memory");
            if (r == 0 && !*sfail) {
                tc_fence_after();
                mma_tf32_ss(tmem, sdesc_sw32(fa_s, 256), sdesc_sw32(fb_s, 256), IDESC_TF32,
                            ch > 0 ? 1u : 0u);
                mma_commit(&bar[BAR_FZ]);
                // a barrier with a single phase for the end of the whole product
                // (waiters may come before or after any chunk)
                if (ch == fz_nch - 1) mma_commit(fz_done);
            }
        }
        if (!mbar_wait(fz_done, 0, kWaitNs)) *sfail = 1;
        tc_fence_after();
        return expf(La);
    };
    // After a timeout, the products thread r = 0 issued end (bounded) before
    // the CTA frees its tensor memory.
    auto fz_drain_products = [&](int fz_len) {
        if (FUSE && tid == 128 && fz_len > 0) {
            mma_commit(fz_drain);
            mbar_wait(fz_drain, 0, kWaitNs);
        }
    };
    // Split warps: every row r of the state tile becomes P_a S + D (D in
    // tensor memory), in place in shared memory, one 64-column half at a time;
    // one thread stores each half by TMA (in place in global memory) as soon
    // as it is written, one bulk group per half.
    auto fz_commit_tile = [&](int r, float Pa) {
#pragma unroll 1
        for (int pc = 0; pc < 2; ++pc) {
            float d0[32], d1[32]; // both tensor-memory loads in flight at once
            tmem_ld32_async(tmem + lane_base + 64 * pc, d0);
            tmem_ld32_async(tmem + lane_base + 64 * pc + 32, d1);
            tmem_wait_ld32(d0);
            tmem_wait_ld32(d1);
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                uint8_t *box = sbuf + (2 * pc + hb) * 16384;
                const float *dv = hb ? d1 : d0;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float4 *p4 = reinterpret_cast<float4 *>(box + sw128_chunk(r, c));
                    float4 v = *p4;
                    v.x = fmaf(Pa, v.x, dv[4 * c + 0]);
                    v.y = fmaf(Pa, v.y, dv[4 * c + 1]);
                    v.z = fmaf(Pa, v.z, dv[4 * c + 2]);
                    v.w = fmaf(Pa, v.w, dv[4 * c + 3]);
                    *p4 = v;
                }
            }
            fence_proxy_async_smem();
            asm volatile("bar.sync 4, 128;" ::: "memory");
            if (r == 0 && !*sfail) { // no store of a product that timed out
                tma_store_2d(&tmS, sbuf + (2 * pc) * 16384, 64 * pc, unit * kD);
                tma_store_2d(&tmS, sbuf + (2 * pc + 1) * 16384, 64 * pc + 32, unit * kD);
                bulk_commit_group();
            }
        }
    };
    // Split warps: before half pc is overwritten, its store has read it.
    auto fz_wait_half = [&](int r, int pc) {
        if (r == 0) {
            if (pc == 0) bulk_wait_group_read1();
            else bulk_wait_group_read0();
        }
        asm volatile("bar.sync 4, 128;" ::: "memory");
    };
    if (fault != 0 || T <= 0 || bad) {
        if (fault == 0 && h == 0 && (T > 0 || (inline_topo && T < 0))) {
            if (bad_node < kT) { // the first node whose link does not point backwards
                if (tid == bad_node) report(st, BOLE_ERR_BAD_TOPOLOGY, b, bad_node, my_par);
            } else if (bad && tid == 0) {
                report(st, T > kTmax || T < 0 || o < 0 || o + T > N ? BOLE_ERR_BAD_TOPOLOGY
                                                                     : BOLE_ERR_DEPTH,
                       b, -1, T > kTmax || T < 0 ? T : d);
            }
        }
        // FUSE: the previous round's commit still applies when this round's
        // tree is empty or refused (the commit's own inputs being valid).
        int fzL = 0;
        if (FUSE && fault == 0 && warp >= 4 && warp < 8) {
            const int r = tid - 128;
            fzL = fz_walk(r);
            if (fzL > 0) {
                const float Pa = fz_stage(r, fzL);
                waitb(BAR_S); // every thread goes on (the update holds named barriers);
                              // after a timeout nothing is stored
                fz_commit_tile(r, Pa);
                fz_wait_half(r, 1);
            }
        }
        if (issuer) { // drain the copies in flight before the CTA retires
            if (in_range) mbar_wait(&bar[BAR_A1], 0, kWaitNs);
            if (SMALL && in_range) mbar_wait(&bar[BAR_V], 0, kWaitNs);
            mbar_wait(&bar[BAR_S], 0, kWaitNs);
        }
        if (FUSE) { // a product in flight after a timeout ends before the tensor memory goes
            tc_fence_before();
            __syncthreads();
            if (*sfail) fz_drain_products(fzL);
            __syncthreads();
            tc_fence_after();
        }
        if (warp == 0) tmem_dealloc(tmem, 256);
        return;
    }
    bool v_issued = SMALL; // the value rows' copy (issued at entry for small trees)
    int fzL = 0;           // FUSE, split warps: the previous accepted path's length

    if (warp == kComputeThreads / 32) {
        // =========================== issue warp ===========================
        bool ok = true;
        if (lane == 0) {
            const uint32_t a1 = smem_addr(sA1), s0 = smem_addr(sbuf);
            do { // every step ends the issue once a wait anywhere in the CTA gave up
            // Gram [Q;K] K^T
            ok &= waitb(BAR_A1);
            if (!ok || *sfail) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_bf16_ss(tmem + TM_GRAM, sdesc_sw128(a1 + off, 16, 1024),
                            sdesc_sw128(a1 + off + 8192, 16, 1024),
                            SMALL ? IDESC_GRAM_S : IDESC_GRAM, kk > 0);
            }
            mma_commit(&bar[BAR_GRAM]);
            // state products [Q;K] (S_hi + S_lo) once the split is in place,
            // in two halves of d_k (rows 0..63 of S_pre, then 64..127)
            ok &= waitb(BAR_CONV);
            if (!ok || *sfail) break;
            tc_fence_after();
            const uint32_t slo = s0 + 16384;
            constexpr uint32_t idesc_s = VK ? IDESC_STATE_VK : IDESC_STATE;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad = sdesc_sw128(a1 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                // 16 d_k rows of S: N-contiguous atoms 32 KB apart, or (VK) a
                // 32 B step along the K-major rows of box pair kk / 4
                const uint32_t boff = VK ? (kk >> 2) * 32768 + (kk & 3) * 32 : kk * 2048;
                const uint32_t lbo = VK ? 16 : 32768;
                mma_bf16_ss(tmem, ad, sdesc_sw128(s0 + boff, lbo, 1024), idesc_s, kk > 0);
                mma_bf16_ss(tmem, ad, sdesc_sw128(slo + boff, lbo, 1024), idesc_s, 1);
                if (kk == 3) mma_commit(&bar[BAR_STATE_A]);
            }
            mma_commit(&bar[BAR_STATE]);
            // The state tile of the CTA one wave ahead (pf_stride = resident
            // CTAs of the launch) goes to L2 now that this CTA's own tile has
            // landed, so the next wave finds it there.
            if (pf_stride > 0 && unit + pf_stride < (int)gridDim.x) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    tma_prefetch_l2_2d(&tmS, 32 * c, (unit + pf_stride) * kD);
            }
            // value rows over the [Q;K] columns the first half has released
            // (small trees: loaded at entry)
            if (!SMALL) {
                ok &= waitb(BAR_STATE_A);
                if (!ok || *sfail) break;
                v_issued = true;
                mbar_arrive_expect_tx(&bar[BAR_V], 16384);
                tma_load_3d(sV, &tmV, &bar[BAR_V], 0, h, o);
                tma_load_3d(sV + 8192, &tmV, &bar[BAR_V], 64, h, o);
            }
            // propagation + read-out: [M; W] R into its own 128 columns
            // (the K extent is the tree: ceil(T / 8) steps of 8 nodes)
            ok &= waitb(BAR_OPS);
            if (!ok || *sfail) break;
            tc_fence_after();
            const uint32_t b2 = s0 + 32768;
            for (int kk = 0; kk < (T + 7) / 8; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_tf32_ss(tmem + TM_PROP, sdesc_sw128(s0 + off, 16, 1024),
                            sdesc_sw128(b2 + off, 16, 1024), IDESC_TF32, kk > 0);
            }
            mma_commit(&bar[BAR_MMA2]);
            } while (0);
        }
        __syncwarp();
        if (!ok) report(st, BOLE_ERR_TIMEOUT, b, -1, 0);
    } else {
        // ========================== compute warps =========================
        bool ok = true;
        // Gram row m is staged in the S_pre rows the first d_k half released:
        // rows 32p..32p+31 in the first 8 KB of box p (VK: the first 32 KB,
        // boxes 0 and 1), 256 B per row, 16-byte chunks XOR-swizzled by row.
        // Small trees: rows 0..31 and 64..95 in the [Q;K] padding, 128 B per
        // row (32 columns), chunks XOR-swizzled by row & 7.
        auto staged_row = [&](int row) -> float * {
            if (SMALL)
                return reinterpret_cast<float *>(
                    sA1 + (row < 64 ? SM_GQK + row * 128 : SM_GKK + (row - 64) * 128));
            return reinterpret_cast<float *>(
                sbuf + (VK ? row * 256 : (row >> 5) * 16384 + (row & 31) * 256));
        };
        float ratio[kSlots]; // topology rows: exp(L_i - L_j), j the ancestor at depth t
        uint32_t aw[4] = {0, 0, 0, 0}; // topology rows: ancestor-by-depth table, packed bytes
        if (topo) {
            // Topology and cumulative decay (row = tid).  L_i is the sum of log
            // gamma over the ancestors-or-self of i (the prefix along parent
            // links, Lemma 1).  The ancestors come out of the mask in depth
            // order (parents precede children), so the partial sums are their
            // L_j.  All log gammas are read in one batch after a barrier of
            // the two topology warps.
            const uint64_t mi = my_depth >= 0 ? my_mask : 0ull;
            LGs[i] = logf(g_i);
            asm volatile("bar.sync 2, 64;" ::: "memory");
            int jt[kSlots];
            uint64_t mm = mi;
#pragma unroll
            for (int t = 0; t < kSlots; ++t) {
                jt[t] = mm ? __ffsll((long long)mm) - 1 : 0;
                mm &= mm - 1;
            }
            float lgv[kSlots];
#pragma unroll
            for (int t = 0; t < kSlots; ++t) lgv[t] = LGs[jt[t]];
            float L = 0.f;
#pragma unroll
            for (int t = 0; t < kSlots; ++t) {
                if (t <= my_depth) {
                    L += lgv[t];
                    aw[t >> 2] |= (uint32_t)jt[t] << (8 * (t & 3));
                }
                ratio[t] = L; // L_j of the ancestor at depth t
            }
#pragma unroll
            for (int t = 0; t < kSlots; ++t) ratio[t] = __expf(L - ratio[t]);
            *reinterpret_cast<uint4 *>(ancat + i * kSlots) = make_uint4(aw[0], aw[1], aw[2], aw[3]);
            Ls[i] = L;
            Ds[i] = my_depth;
            if (kColGather) reinterpret_cast<uint64_t *>(sm + X_JMASK)[i] = mi; // for the G gather
            if (i < T) logP[(size_t)(o + i) * H + h] = L;
            mbar_arrive(&bar[BAR_TOPO]);
        }
        if (kColGather && warp < 4) {
            // Deferred commit, 64-node layout: the compact C (warps 0-1, Gram rows
            // q_i . k_j) and G (warps 2-3, rows k_i . k_j) of node i straight from
            // the Gram in tensor memory, with no staging -- which would wait for
            // the state rows the first d_k half of the products frees, and in this
            // form the state side (the commit first) is the long one.  Each thread
            // holds its row and, column by column, writes exp(L_i - L_j) times the
            // entry of every ancestor(-or-self) j into slot depth(j).  (Slower than
            // the staging where the state side is short: the plain kernel stages.)
            ok &= waitb(BAR_GRAM);
            ok &= waitb(BAR_TOPO);
            if (FUSE && // the commit operands live where C and G go
                !mbar_wait(fz_done, 0, kWaitNs)) {
                *sfail = 1;
                ok = false;
            }
            tc_fence_after();
            __syncwarp();
            const int node = m & 63;
            const bool gsel = m >= 64; // G: strict ancestors, times beta_i
            const uint64_t mask =
                node < T ? reinterpret_cast<const uint64_t *>(sm + X_JMASK)[node] : 0ull;
            const float Li = Ls[node];
            const float sc = gsel ? bt : 1.f;
            float *row = (gsel ? Gc : Cc) + node * kLd;
#pragma unroll 1
            for (int hc = 0; hc < 2; ++hc) {
                const uint32_t mw = (uint32_t)(mask >> (32 * hc));
                // columns that are an ancestor of some row of the warp (warp-uniform:
                // the others are skipped, and a half no row needs is not loaded)
                const uint32_t any = __reduce_or_sync(0xffffffffu, mw);
                if (any == 0u) continue;
                float x[32];
                tmem_ld32(tmem + TM_GRAM + 32 * hc + lane_base, x);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    if ((any >> c) & 1u) {
                        const int j = 32 * hc + c;
                        const bool anc = ((mw >> c) & 1u) && !(gsel && j == node);
                        if (anc) row[Ds[j]] = sc * __expf(Li - Ls[j]) * x[c];
                    }
                }
            }
            mbar_arrive(&bar[BAR_CG]);
        }
        if (SMALL ? (warp == 0 || warp == 2) : (!kColGather && warp < 4)) {
            // Stage the Gram rows (q.k for rows 0..63, k.k for 64..127; small
            // trees: rows 0..31 and 64..95, columns 0..31, with no wait for
            // the state products).
            ok &= waitb(BAR_GRAM);
            if (!SMALL) ok &= waitb(BAR_STATE_A);
            tc_fence_after();
            __syncwarp();
            float4 *srow = reinterpret_cast<float4 *>(staged_row(m));
#pragma unroll 1
            for (int hc = 0; hc < (SMALL ? 1 : 2); ++hc) {
                float x[32];
                tmem_ld32(tmem + TM_GRAM + 32 * hc + lane_base, x);
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4)
                    srow[(8 * hc + c4) ^ (m & (SMALL ? 7 : 15))] =
                        make_float4(x[4 * c4], x[4 * c4 + 1], x[4 * c4 + 2], x[4 * c4 + 3]);
            }
            mbar_arrive(&bar[BAR_STAGED]);
        }
        if (!kColGather && topo) {
            // Compact C and G of row i, gathered in depth order (small trees:
            // warp 0 only, the rows of warp 1 are past the tree).
            ok &= waitb(BAR_STAGED);
            if (FUSE && // the commit operands live where C and G go
                !mbar_wait(fz_done, 0, kWaitNs)) {
                *sfail = 1;
                ok = false;
            }
            const float *qk = staged_row(i), *kk = staged_row(64 + i);
            float *crow = Cc + i * kLd, *grow = Gc + i * kLd;
            float qv[kSlots], kv[kSlots]; // every load first, then the products
#pragma unroll
            for (int t = 0; t < kSlots; ++t) {
                const int j = (aw[t >> 2] >> (8 * (t & 3))) & 0xff;
                const int sw = (((j >> 2) ^ (i & (SMALL ? 7 : 15))) << 2) | (j & 3);
                qv[t] = (!SMALL || warp == 0) ? qk[sw] : 0.f;
                kv[t] = (!SMALL || warp == 0) ? kk[sw] : 0.f;
            }
#pragma unroll
            for (int t = 0; t < kSlots; ++t) {
                if (t <= my_depth) {
                    crow[t] = ratio[t] * qv[t];
                    if (t < my_depth) grow[t] = bt * ratio[t] * kv[t];
                }
            }
            mbar_arrive(&bar[BAR_CG]);
        } else if (warp >= 4) {
            // --------- split warps: S_pre = S_hi + S_lo in place (row r) ---------
            // bf16, N-contiguous, 64-column atoms: boxes (0,1) <- columns 0..63,
            // boxes (2,3) <- columns 64..127.
            const int r = tid - 128;
            // FUSE: first the previous round's commit of the tile (P_a S + D, each
            // half stored by TMA as soon as it is written), then the split of the
            // committed values, each half once its store has read it.
            fzL = FUSE ? fz_walk(r) : 0;
            const bool fzc = fzL > 0;
            float Pa = 1.f; // P_a of the previous accepted node
            if (fzc) Pa = fz_stage(r, fzL);
            ok &= waitb(BAR_S);
            if (fzc) fz_commit_tile(r, Pa); // the previous round's commit, stored
#pragma unroll 1
            for (int pc = 0; pc < 2; ++pc) {
                uint8_t *box0 = sbuf + (2 * pc) * 16384, *box1 = box0 + 16384;
                if (fzc) fz_wait_half(r, pc); // the committed half's store has read it
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
            if (FUSE) tc_fence_before(); // the commit product's tensor-memory reads
            mbar_arrive(&bar[BAR_CONV]);
        }
        ok &= waitb(BAR_TOPO);
        const float p = (i < T) ? expf(Ls[i]) : 0.f; // P_i

        if (SMALL && warp < 2) {
            // Rows of W (warp 0: y) and M (warp 1: z) of node n = lane by the
            // same backward substitution, formed while the state products
            // run and written into the [M; W] operand once they are done.
            const int n = lane;
            const bool wrow = warp == 0;
            ok &= waitb(BAR_CG);
            float vals[kSlots];
            uint32_t aw4[4] = {0, 0, 0, 0};
            int di = -1;
            if (n < T) {
                di = Ds[n];
                const uint4 a4 = *reinterpret_cast<const uint4 *>(ancat + n * kSlots);
                aw4[0] = a4.x; aw4[1] = a4.y; aw4[2] = a4.z; aw4[3] = a4.w;
                const float *ci = Cc + n * kLd;
                float cv[kSlots], acc[kSlots], gcur[kSlots];
#pragma unroll
                for (int t = 0; t < kSlots; ++t) {
                    cv[t] = wrow ? 0.f : ci[t];
                    acc[t] = 0.f;
                }
                {
                    const float *gr = Gc + n * kLd;
#pragma unroll
                    for (int t = 0; t < kSlots - 1; ++t) gcur[t] = gr[t];
                }
#pragma unroll
                for (int u = kSlots - 1; u >= 0; --u) {
                    vals[u] = 0.f;
                    if (u <= di) {
                        float gnext[kSlots];
                        if (u >= 1) {
                            const int an = (aw4[(u - 1) >> 2] >> (8 * ((u - 1) & 3))) & 0xff;
                            const float *gr = Gc + an * kLd;
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
            }
            ok &= waitb(BAR_STATE);
            const int orow = wrow ? 64 + n : n;
#pragma unroll
            for (int c = 0; c < 8; ++c) // K extent <= 32 nodes: the first K-atom
                *reinterpret_cast<float4 *>(sbuf + sw128_chunk(orow, c)) =
                    make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < kSlots; ++u) {
                if (u <= di) {
                    const int au = (aw4[u >> 2] >> (8 * (u & 3))) & 0xff;
                    *reinterpret_cast<float *>(sbuf + sw128_offset(orow, au)) = vals[u];
                }
            }
        } else if (SMALL && rowgrp == 2) {
            // R^T of nodes 0..31 (warp 2: columns 0..63, warp 6: 64..127),
            // value rows from the [Q;K] padding.
            ok &= waitb(BAR_STATE);
            ok &= waitb(BAR_V);
            tc_fence_after();
            __syncwarp();
            uint8_t *dst = sbuf + 32768;
            const uint8_t *vrow = sA1 + SM_V + half * 16384 + i * 128;
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
                const int col0 = half * 64 + cc * 32;
                float x[32];
                tmem_ld32(tmem + lane_base + col0, x);
                uint4 vv[4]; // read ahead of the scattered stores below, which could alias
#pragma unroll
                for (int uu = 0; uu < 4; ++uu)
                    vv[uu] = *reinterpret_cast<const uint4 *>(vrow +
                                                              (((cc * 4 + uu) ^ (i & 7)) << 4));
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
        } else if (SMALL) {
            // lanes of the padding rows: nothing to form
        } else if (m < 64 && (topo || warp >= 4)) {
            // Rows of W (warps 0, 1: y) and of M (warps 4, 5: z) by backward
            // substitution along the ancestor path, written straight into the
            // [M; W] operand (row i of M, row 64 + i of W, column = ancestor)
            // once the gathers and the state products have released it.  Each
            // thread zeroes its own row first (program order keeps the values).
            ok &= waitb(BAR_CG);
            ok &= waitb(BAR_STATE);
            const bool wrow = topo;
            const int orow = wrow ? 64 + i : i;
#pragma unroll
            for (int c = 0; c < 16; ++c) // 2 K-atoms x 8 chunks of 16 B
                *reinterpret_cast<float4 *>(sbuf + (c >> 3) * 16384 + sw128_chunk(orow, c & 7)) =
                    make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < T) {
                const int di = Ds[i];
                const uint4 a4 = *reinterpret_cast<const uint4 *>(ancat + i * kSlots);
                const uint32_t aw4[4] = {a4.x, a4.y, a4.z, a4.w};
                const float *ci = Cc + i * kLd;
                float cv[kSlots];
#pragma unroll
                for (int t = 0; t < kSlots; ++t) cv[t] = wrow ? 0.f : ci[t];
                float acc[kSlots]; // sum_{u > t} (y or z)_u G(a_u, a_t)
#pragma unroll
                for (int t = 0; t < kSlots; ++t) acc[t] = 0.f;
                // G row of the ancestor at depth u, read one step ahead
                float gcur[kSlots];
                {
                    const float *gr = Gc + i * kLd;
#pragma unroll
                    for (int t = 0; t < kSlots - 1; ++t) gcur[t] = gr[t];
                }
#pragma unroll
                for (int u = kSlots - 1; u >= 0; --u) {
                    if (u <= di) {
                        float gnext[kSlots];
                        if (u >= 1) {
                            const int an = (aw4[(u - 1) >> 2] >> (8 * ((u - 1) & 3))) & 0xff;
                            const float *gr = Gc + an * kLd;
#pragma unroll
                            for (int t = 0; t < u - 1; ++t) gnext[t] = gr[t];
                        }
                        const float val = wrow ? ((u == di) ? 1.f : -acc[u]) : cv[u] - acc[u];
                        const int au = (aw4[u >> 2] >> (8 * (u & 3))) & 0xff;
                        *reinterpret_cast<float *>(sbuf + (au >> 5) * 16384 +
                                                   sw128_offset(orow, au & 31)) = val;
#pragma unroll
                        for (int t = 0; t < u; ++t) acc[t] = fmaf(val, gcur[t], acc[t]);
#pragma unroll
                        for (int t = 0; t < u - 1; ++t) gcur[t] = gnext[t];
                    }
                }
            }
        } else if (m >= 64) {
            // R^T = (beta (v - P K S_pre))^T for columns 64 half .. +63 of the
            // rows 64..127 (warps 2, 3, 6, 7), once the staged Gram in this
            // buffer has been gathered.
            ok &= waitb(BAR_STATE);
            ok &= waitb(BAR_CG);
            ok &= waitb(BAR_V);
            tc_fence_after();
            __syncwarp();
            uint8_t *dst = sbuf + 32768 + (i >> 5) * 16384;
            const uint8_t *vrow = sV + half * 8192 + i * 128; // 64 columns of row i
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
                const int col0 = half * 64 + cc * 32;
                float x[32];
                tmem_ld32(tmem + lane_base + col0, x);
                uint4 vv[4]; // read ahead of the scattered stores below, which could alias
#pragma unroll
                for (int uu = 0; uu < 4; ++uu)
                    vv[uu] = *reinterpret_cast<const uint4 *>(vrow +
                                                              (((cc * 4 + uu) ^ (i & 7)) << 4));
#pragma unroll
                for (int uu = 0; uu < 4; ++uu) {
                    float f[8];
                    bf16x8_to_f32(vv[uu], f);
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const int c = 8 * uu + t;
                        const float r = (i < T) ? bt * (f[t] - p * x[c]) : 0.f;
                        *reinterpret_cast<float *>(dst + sw128_offset(col0 + c, i & 31)) = r;
                    }
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bar[BAR_OPS]);

        // ---- outputs: O = P (Q S_pre) + M R (bf16), U = W R (fp32) ----
        ok &= waitb(BAR_MMA2);
        tc_fence_after();
        __syncwarp();
        // Each thread puts its 64 columns of row i of O (bf16, rows 0..63) or
        // U (fp32, rows 64..127) into shared memory the propagation has
        // released (O rows in the [Q;K] buffer, U rows in the state buffer,
        // padded by 16 B so the row-per-thread writes are conflict-free);
        // then the compute warps store the rows with 16 lanes per 256-byte
        // row segment -- row-per-thread global stores touched 32 cache lines
        // per instruction.
        if (!SMALL || !(rowgrp & 1)) { // small trees: no output in the padding lanes
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
                const int col0 = half * 64 + cc * 32;
                float x[32];
                if (m < 64) { // both loads in flight at once
                    float y[32];
                    tmem_ld32_async(tmem + TM_PROP + lane_base + col0, x);
                    tmem_ld32_async(tmem + lane_base + col0, y);
                    tmem_wait_ld32(x);
                    tmem_wait_ld32(y);
#pragma unroll
                    for (int t = 0; t < 32; ++t) x[t] = fmaf(p, y[t], x[t]);
                    uint4 *dsto = reinterpret_cast<uint4 *>(sA1 + i * kORow + col0 * 2);
#pragma unroll
                    for (int uu = 0; uu < 4; ++uu) {
                        __nv_bfloat162 p2[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t)
                            p2[t] = __floats2bfloat162_rn(x[8 * uu + 2 * t], x[8 * uu + 2 * t + 1]);
                        dsto[uu] = *reinterpret_cast<uint4 *>(p2);
                    }
                } else {
                    tmem_ld32(tmem + TM_PROP + lane_base + col0, x);
                    float4 *dstu = reinterpret_cast<float4 *>(sbuf + i * kURow + col0 * 4);
#pragma unroll
                    for (int uu = 0; uu < 8; ++uu)
                        dstu[uu] = make_float4(x[4 * uu], x[4 * uu + 1], x[4 * uu + 2], x[4 * uu + 3]);
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kComputeThreads) : "memory");
        if (ok && !*sfail) {
            // O: T rows of 16 chunks of 16 B; U: T rows of 32 chunks
            for (int c = tid; c < T * 16; c += kComputeThreads) {
                const int r = c >> 4, q = c & 15;
                *reinterpret_cast<uint4 *>(O + ((size_t)(o + r) * H + h) * kD + q * 8) =
                    *reinterpret_cast<const uint4 *>(sA1 + r * kORow + q * 16);
            }
            for (int c = tid; c < T * 32; c += kComputeThreads) {
                const int r = c >> 5, q = c & 31;
                *reinterpret_cast<float4 *>(Uout + ((size_t)(o + r) * H + h) * kD + q * 4) =
                    *reinterpret_cast<const float4 *>(sbuf + r * kURow + q * 16);
            }
        }
        if (!ok) report(st, BOLE_ERR_TIMEOUT, b, -1, 1);
    }
    tc_fence_before();
    __syncthreads();
    if (*sfail) { // read after the barrier: the same value in every thread
        // After a timeout the products and copies this CTA issued must end
        // before its tensor memory and shared memory go to another CTA: wait
        // (bounded) for every one of them.
        if (issuer) {
            mma_commit(&bar[BAR_DRAIN]);
            mbar_wait(&bar[BAR_DRAIN], 0, kWaitNs);
            mbar_wait(&bar[BAR_A1], 0, kWaitNs);
            mbar_wait(&bar[BAR_S], 0, kWaitNs);
            if (v_issued) mbar_wait(&bar[BAR_V], 0, kWaitNs);
        }
        fz_drain_products(fzL); // FUSE: the commit products of the split warps
        __syncthreads();
    }
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---- commit ----
// One CTA per (request, head, 64-column half of the state, layer): value
// tiling as in the pages' kernel.  The half is staged one 32-column box at a
// time through a 16 KB buffer (both boxes are prefetched into L2 ahead of
// use, so the second load is an L2 hit), which lets seven CTAs share an SM and a
// batch of 1024 tiles run in one wave.  (Narrower tiles fit more CTAs but
// repeat the path operand's gather and measured slower.)  One launch covers
// every layer of a unified cross-layer commit: layer l's state, keys, deltas
// and decays start l strides after the base pointers.
// The stored tile is always 128 rows x 64 columns.  [dk][dv] state: rows are
// d_k (operand A = (D_a K_a)^T, 128 x path), columns a d_v half (operand B^T =
// U_a^T of that half).  VK ([dv][dk], the slot layout): rows are d_v (A =
// U_a^T), columns a d_k half (B^T = (D_a K_a)^T of that half) -- the same
// product, transposed.
// Precision: bf16 keys are exact in tf32 and U_a is rounded to tf32.  fp32
// keys (the 1e-5 bound): both operands are written as tf32 hi + lo (rounded
// to nearest here, so the hardware reads them exactly) and each chunk keeps
// lo hi + hi lo + hi hi (the dropped lo lo term is ~2^-22 relative).
constexpr int kCommitThreads = 128;
constexpr int kChunk = 16;                    // path nodes per MMA K chunk
constexpr int kBatch = 8;                     // path nodes whose operands are read at once
constexpr int kTile = 64;                     // state columns per CTA
template <bool F32> struct CoPlan {
    static constexpr int S = 0;               // one box of the half: [128 rows x 128 B] = 16 KB
    static constexpr int A = 16384;           // (D_a K_a)^T chunk: 128 rows x 16 tf32 (64 B rows)
    static constexpr int B = A + 8192;        // U_a^T chunk: 64 rows x 16 tf32
    static constexpr int AL = B + 4096;       // fp32: the tf32 low parts of A and B
    static constexpr int BL = AL + 8192;
    static constexpr int PATH = F32 ? BL + 4096 : AL; // int[128]
    static constexpr int BAR = PATH + 512;    // 5 mbarriers: box, product, drain, 2 row buffers
    static constexpr int TSLOT = BAR + 40;
    static constexpr int MISC = TSLOT + 4;    // path length, flag, status copy
    static constexpr int PAR = MISC + 16;     // int[128]: the request's parent links
    static constexpr int COEF = PAR + 512;    // float[128]: exp(L_a - L_j) along a long path
    static constexpr int SMEM = COEF + 512 + 1024;
    static constexpr int CTAS = F32 ? 5 : 7;  // per SM (x 64 tensor memory columns)
    static_assert(CTAS * (SMEM + 1024) <= 228 * 1024, "commit CTAs per SM");
    static_assert((CTAS + 1) * (SMEM + 1024) > 228 * 1024,
                  "never more (the tensor memory columns would still fit; keep the margin)");
};

constexpr uint32_t IDESC_COMMIT = idesc_tf32(128, kTile, false, false);

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

// A long accepted path (default layout, bf16 keys), by warp 0: chunk cc's
// rows into half cc % 2 of the state buffer -- 16 key rows (256 B), then 16
// U half-rows of this CTA's columns (256 B) -- one bulk copy per lane,
// completing on bar[3 + cc % 2].
template <typename KT>
__device__ __forceinline__ void stage_path_rows(uint8_t *sS, uint64_t *bar, const int *path,
                                                const KT *k, const float *U, int cc, int L, int o,
                                                int H, int h, int hv)
{
    const int lane = threadIdx.x & 31, buf = cc & 1;
    const int tn = min(kChunk, L - cc * kChunk);
    uint8_t *dst = sS + buf * 8192;
    if (lane == 0) mbar_arrive_expect_tx(&bar[3 + buf], (uint32_t)tn * 512u);
    __syncwarp();
    const int t = lane & 15;
    if (t < tn) {
        const size_t nh = (size_t)(o + path[cc * kChunk + t]) * H + h;
        if (lane < 16) bulk_load(dst + t * 256, k + nh * kD, 256, &bar[3 + buf]);
        else bulk_load(dst + 4096 + t * 256, U + nh * kD + kTile * hv, 256, &bar[3 + buf]);
    }
}

template <bool VK, bool F32>
__global__ void __launch_bounds__(kCommitThreads, CoPlan<F32>::CTAS)
tc_commit_kernel(const __grid_constant__ CUtensorMap tmS, const void *__restrict__ kptr,
                 const float *__restrict__ U, const float *__restrict__ logP,
                 const int32_t *__restrict__ offsets, const int32_t *__restrict__ parent,
                 const int32_t *__restrict__ accepted, int H, int N, int64_t k_ls, int64_t u_ls,
                 int64_t lp_ls, int32_t *st)
{
    using P = CoPlan<F32>;
    using KT = typename std::conditional<F32, float, __nv_bfloat16>::type;
    const KT *k = static_cast<const KT *>(kptr);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *sS = sm + P::S;
    uint8_t *sA = sm + P::A;
    uint8_t *sB = sm + P::B;
    uint8_t *sAL = sm + P::AL, *sBL = sm + P::BL; // fp32 only
    int *path = reinterpret_cast<int *>(sm + P::PATH);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + P::BAR); // tma, mma, drain
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + P::TSLOT);
    int *plen = reinterpret_cast<int *>(sm + P::MISC);
    int *flag = plen + 1;
    int *spar = reinterpret_cast<int *>(sm + P::PAR);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int unit = blockIdx.x, hv = blockIdx.y; // head unit, column half
    const int layer = blockIdx.z;
    const int b = unit / H, h = unit % H;
    k += layer * k_ls;
    U += layer * u_ls;
    logP += layer * lp_ls;
    // The first box of the half goes to L2 now, the second once the path
    // reads are in flight (prefetching both at entry queued those small,
    // dependent reads behind every CTA's state traffic); the first box is
    // requested into shared memory beside the first batch of path reads.
    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
        prefetch_tensormap(&tmS);
        tma_prefetch_l2_3d(&tmS, kTile * hv, unit * kD, layer);
    }
    // Tensor memory at entry: the SM starts the next CTA of the kernel once
    // this one has given up its allocation permit, so all seven CTAs of an SM
    // start together and, in a launch overlapping the verification, begin
    // their state prefetch during its last wave (config 2 step 35.2 -> 33.5 us;
    // allocating after the first round trip staggered them by one each).
    if (warp == 0) {
        tmem_alloc(tslot, 64);
        tmem_relinquish();
    }
    // The request's extent and its parent links are caller inputs that no
    // call of the round writes: read before the wait, so that a launch
    // overlapping the verification has them during its last wave.  What the
    // verification (or the sampler) wrote -- U, log P, the accepted node, the
    // status -- is read after it; the status word and the accepted node come
    // in one round trip (uniform early exit: the status is read by one thread).
    static_assert(kCommitThreads >= kMaxTree, "one parent link per thread");
    const int o = offsets[b], T = offsets[b + 1] - o;
    const bool ext_ok = T > 0 && T <= kMaxTree && o >= 0 && o + T <= N;
    const int my_par = (ext_ok && tid < T) ? parent[o + tid] : -1;
    pdl_wait();
    int *sfault = plen + 2;
    if (tid == 0) *sfault = *(const volatile int32_t *)st;
    const int a = accepted[b];
    const bool bad = a >= 0 && (a >= T || !ext_ok);
    const bool work = a >= 0 && !bad;
    // stage the parent links, then walk the accepted path
    if (work && tid < T) spar[tid] = my_par;
    int *staged = plen + 3; // last chunk whose path rows were requested (long path)
    if (tid == 32) *flag = 0;
    if (tid == 33) *staged = -1;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int fault = *sfault;
    if (fault != 0 || !work) {
        if (bad && fault == 0 && tid == 0 && hv == 0 && layer == 0)
            report(st, BOLE_ERR_BAD_TOPOLOGY, b, a, T);
        if (warp == 0) tmem_dealloc(tmem, 64); // unused
        return;
    }
    // The accepted path, node first: one thread walks the parent links (and
    // reports a bad one).  In a tree of more than 32 nodes the walk stops
    // after one chunk of nodes; a longer path is then read off a's
    // ancestor-or-self mask, formed for every node at once by pointer jumping
    // (log2 of the depth rounds, in the operand buffer, unused yet) --
    // ancestors have smaller indices, so by index the mask lists the path
    // root first.
    if (tid == 0) {
        int L = 0, j = a;
        bool ok = true;
        while (j >= 0) {
            if (L >= kMaxTree) { ok = false; break; }
            if (L == kChunk && T > 32) { L = -1; break; } // the long walk below
            path[L++] = j;
            const int p = spar[j];
            if (p < -1 || p >= j) { ok = false; break; }
            j = p;
        }
        if (!ok) {
            if (hv == 0 && layer == 0) report(st, BOLE_ERR_BAD_TOPOLOGY, b, j, -1);
            *flag = 1;
        }
        *plen = L;
    }
    __syncthreads();
    if (*plen < 0) {
        uint32_t *smk = reinterpret_cast<uint32_t *>(sA);         // [128][4]
        int *sjp = reinterpret_cast<int *>(sA + 16 * kMaxTree);    // [128]
        uint4 mk = make_uint4(0u, 0u, 0u, 0u);
        int jp = -1;
        if (tid < T) {
            const uint32_t bit = 1u << (tid & 31);
            mk = make_uint4(tid < 32 ? bit : 0u, (tid >> 5) == 1 ? bit : 0u,
                            (tid >> 5) == 2 ? bit : 0u, (tid >> 5) == 3 ? bit : 0u);
            jp = spar[tid];
            if (jp >= tid) jp = -1; // a link that is not backwards ends the walk (checked below)
            *reinterpret_cast<uint4 *>(smk + 4 * tid) = mk;
            sjp[tid] = jp;
        }
#pragma unroll 1
        for (int r = 0; r < 7; ++r) { // 2^7 >= 128 nodes
            if (!__syncthreads_or(jp >= 0)) break;
            uint4 nm = make_uint4(0u, 0u, 0u, 0u);
            int j2 = -1;
            if (jp >= 0) {
                nm = *reinterpret_cast<const uint4 *>(smk + 4 * jp);
                j2 = sjp[jp];
            }
            __syncthreads();
            if (jp >= 0) {
                mk.x |= nm.x; mk.y |= nm.y; mk.z |= nm.z; mk.w |= nm.w;
                jp = j2;
            }
            if (tid < T) {
                *reinterpret_cast<uint4 *>(smk + 4 * tid) = mk;
                sjp[tid] = jp;
            }
        }
        __syncthreads();
        const uint4 ma = *reinterpret_cast<const uint4 *>(smk + 4 * a);
        const int La_len = __popc(ma.x) + __popc(ma.y) + __popc(ma.z) + __popc(ma.w);
        if (tid < T) {
            const int wd = tid >> 5;
            const uint32_t w = wd == 0 ? ma.x : wd == 1 ? ma.y : wd == 2 ? ma.z : ma.w;
            if ((w >> (tid & 31)) & 1u) { // on the path: position by the path nodes below it
                const int rank = __popc(w & ((1u << (tid & 31)) - 1u)) +
                                 (wd > 0 ? __popc(ma.x) : 0) + (wd > 1 ? __popc(ma.y) : 0) +
                                 (wd > 2 ? __popc(ma.z) : 0);
                path[La_len - 1 - rank] = tid;
                if (rank == 0 && spar[tid] != -1) { // the path ends in a bad link
                    if (hv == 0 && layer == 0) report(st, BOLE_ERR_BAD_TOPOLOGY, b, tid, -1);
                    *flag = 1;
                }
            }
        }
        if (tid == 0) *plen = La_len;
    }
    __syncthreads();
    const int L = *plen;
    // A path of more than one chunk (default layout, bf16 keys): its rows are
    // staged by bulk copies two chunks ahead instead of read per thread in
    // dependent batches.
    const bool longp = !VK && !F32 && L > kChunk &&
                       ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(U)) & 15) == 0;
    if (!longp && L > kBatch && *(volatile int *)flag == 0) {
        // A path longer than one batch: every node's key and delta rows go
        // to L2 now, so that the batches below, each a dependent round trip,
        // meet L2 instead of DRAM.  A side: the row of 128 (key, or VK: U),
        // B side: this CTA's 64-entry half (U, or VK: key).
        constexpr uint32_t kRowK = kD * sizeof(KT), kHalfK = kTile * sizeof(KT);
        for (int t = tid; t < L; t += kCommitThreads) {
            const size_t nh = (size_t)(o + path[t]) * H + h;
            if (VK) {
                bulk_prefetch_l2(U + nh * kD, kD * 4);
                bulk_prefetch_l2(k + nh * kD + kTile * hv, kHalfK);
            } else {
                bulk_prefetch_l2(k + nh * kD, kRowK);
                bulk_prefetch_l2(U + nh * kD + kTile * hv, kTile * 4);
            }
        }
    }
    const float La = logP[(size_t)(o + a) * H + h];

    const uint32_t sa = smem_addr(sA), sb = smem_addr(sB);
    int nload = 0; // state boxes requested on bar[0] (thread 0)
    const int nchunks = (*(volatile int *)flag != 0) ? 0 : (L + kChunk - 1) / kChunk;
    // Long path: the rows of chunks 0 and 1 are requested into the state
    // buffer (free until the epilogue), each later chunk's once the buffer
    // half it reuses has been read.
    float *scoef = reinterpret_cast<float *>(sm + P::COEF);
    if (longp && nchunks > 0) {
        if (warp == 0) {
            stage_path_rows(sS, bar, path, k, U, 0, L, o, H, h, hv);
            stage_path_rows(sS, bar, path, k, U, 1, L, o, H, h, hv); // L > 16: two chunks
            if (tid == 0) *staged = 1;
            if (tid == 0) tma_prefetch_l2_3d(&tmS, kTile * hv + 32, unit * kD, layer); // second box
        }
        // the key-side coefficients exp(L_a - L_j) of every path node at once
        if (tid < L) scoef[tid] = expf(La - logP[(size_t)(o + path[tid]) * H + h]);
        __syncthreads();
    }
    for (int ch = 0; ch < nchunks; ++ch) {
        const int tn = min(kChunk, L - ch * kChunk); // path nodes in this chunk
        if constexpr (!VK && !F32) {
            if (longp) {
                const int buf = ch & 1;
                if (!mbar_wait(&bar[3 + buf], (uint32_t)(ch >> 1) & 1u, kWaitNs)) {
                    report(st, BOLE_ERR_TIMEOUT, b, -1, 9);
                    *flag = 1;
                }
                const __nv_bfloat16 *krow = reinterpret_cast<const __nv_bfloat16 *>(sS + buf * 8192);
                const float *urow = reinterpret_cast<const float *>(sS + buf * 8192 + 4096);
                // A[r][t] = coef_t k_t[r] (row r = tid), B^T[c][t] = U_t[64 hv + c]
                // (row c = tid < 64); columns past the path are zeros
#pragma unroll
                for (int c4 = 0; c4 < kChunk / 4; ++c4) {
                    float av[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int t = 4 * c4 + e;
                        av[e] = t < tn ? scoef[ch * kChunk + t] * __bfloat162float(krow[t * kD + tid])
                                       : 0.f;
                    }
                    *reinterpret_cast<float4 *>(sA + sw64_offset(tid, 4 * c4)) =
                        make_float4(av[0], av[1], av[2], av[3]);
                    if (tid < kTile) {
                        float bv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int t = 4 * c4 + e;
                            bv[e] = t < tn ? urow[t * kTile + tid] : 0.f;
                        }
                        *reinterpret_cast<float4 *>(sB + sw64_offset(tid, 4 * c4)) =
                            make_float4(bv[0], bv[1], bv[2], bv[3]);
                    }
                }
            }
        }
#pragma unroll 1
        for (int t0 = 0; t0 < (longp ? 0 : kChunk); t0 += kBatch) {
            // Every path-dependent read of the batch at once: the decay of
            // each path node (each thread forms its own coefficients), entry
            // r = tid of the A-side row (key, or VK: U) and, for c = tid < 64,
            // entry 64 hv + c of the B-side row (U, or VK: key).  Columns past
            // the path are written as zeros.
            float lp[kBatch], av_[kBatch], bv_[kBatch];
#pragma unroll
            for (int tt = 0; tt < kBatch; ++tt) {
                const bool on = t0 + tt < tn;
                const size_t nh =
                    (size_t)(o + (on ? path[ch * kChunk + t0 + tt] : 0)) * H + h;
                lp[tt] = on ? logP[nh] : 0.f;
                if (VK) {
                    av_[tt] = on ? U[nh * kD + tid] : 0.f;
                    bv_[tt] = (on && tid < kTile) ? to_f32(k[nh * kD + kTile * hv + tid]) : 0.f;
                } else {
                    av_[tt] = on ? to_f32(k[nh * kD + tid]) : 0.f;
                    bv_[tt] = (on && tid < kTile) ? U[nh * kD + kTile * hv + tid] : 0.f;
                }
            }
            if (ch == 0 && t0 == 0 && tid == 0) {
                ++nload;
                mbar_arrive_expect_tx(&bar[0], 16384);
                tma_load_3d(sS, &tmS, &bar[0], kTile * hv, unit * kD, layer);
                tma_prefetch_l2_3d(&tmS, kTile * hv + 32, unit * kD, layer); // second box
            }
            // The key side carries the coefficients exp(L_a - L_j).
            float coef[kBatch];
#pragma unroll
            for (int tt = 0; tt < kBatch; ++tt)
                coef[tt] = (t0 + tt < tn) ? expf(La - lp[tt]) : 0.f;
            // A[r][t] (row r = tid), K-major, 64-byte rows
#pragma unroll
            for (int c4 = 0; c4 < kBatch / 4; ++c4) {
                float av[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tt = 4 * c4 + e;
                    av[e] = VK ? av_[tt] : coef[tt] * av_[tt];
                }
                if constexpr (F32) {
                    float hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        hi[e] = tf32_round(av[e]);
                        lo[e] = tf32_round(av[e] - hi[e]);
                    }
                    *reinterpret_cast<float4 *>(sA + sw64_offset(tid, t0 + 4 * c4)) =
                        make_float4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<float4 *>(sAL + sw64_offset(tid, t0 + 4 * c4)) =
                        make_float4(lo[0], lo[1], lo[2], lo[3]);
                } else {
                    *reinterpret_cast<float4 *>(sA + sw64_offset(tid, t0 + 4 * c4)) =
                        make_float4(av[0], av[1], av[2], av[3]);
                }
            }
            // B^T[c][t] (row c = tid < 64), K-major, 64-byte rows
            if (tid < kTile) {
#pragma unroll
                for (int t4 = 0; t4 < kBatch / 4; ++t4) {
                    float bv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int tt = 4 * t4 + e;
                        bv[e] = VK ? coef[tt] * bv_[tt] : bv_[tt];
                    }
                    if constexpr (F32) {
                        float hi[4], lo[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            hi[e] = tf32_round(bv[e]);
                            lo[e] = tf32_round(bv[e] - hi[e]);
                        }
                        *reinterpret_cast<float4 *>(sB + sw64_offset(tid, t0 + 4 * t4)) =
                            make_float4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<float4 *>(sBL + sw64_offset(tid, t0 + 4 * t4)) =
                            make_float4(lo[0], lo[1], lo[2], lo[3]);
                    } else {
                        *reinterpret_cast<float4 *>(sB + sw64_offset(tid, t0 + 4 * t4)) =
                            make_float4(bv[0], bv[1], bv[2], bv[3]);
                    }
                }
            }
            if (t0 + kBatch >= tn && t0 + kBatch < kChunk) { // the rest of the chunk is zero
#pragma unroll
                for (int c4 = kBatch / 4; c4 < kChunk / 4; ++c4) {
                    *reinterpret_cast<float4 *>(sA + sw64_offset(tid, 4 * c4)) =
                        make_float4(0.f, 0.f, 0.f, 0.f);
                    if (tid < kTile)
                        *reinterpret_cast<float4 *>(sB + sw64_offset(tid, 4 * c4)) =
                            make_float4(0.f, 0.f, 0.f, 0.f);
                    if (F32) {
                        *reinterpret_cast<float4 *>(sAL + sw64_offset(tid, 4 * c4)) =
                            make_float4(0.f, 0.f, 0.f, 0.f);
                        if (tid < kTile)
                            *reinterpret_cast<float4 *>(sBL + sw64_offset(tid, 4 * c4)) =
                                make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                break;
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            if constexpr (F32) {
                const uint32_t sal = smem_addr(sAL), sbl = smem_addr(sBL);
#pragma unroll
                for (int t = 0; t < 3; ++t) // lo hi, hi lo, hi hi
#pragma unroll
                    for (int kk = 0; kk < kChunk / 8; ++kk)
                        mma_tf32_ss(tmem, sdesc_sw64((t == 0 ? sal : sa) + kk * 32, 512),
                                    sdesc_sw64((t == 1 ? sbl : sb) + kk * 32, 512), IDESC_COMMIT,
                                    (ch > 0 || t > 0 || kk > 0));
            } else {
#pragma unroll
                for (int kk = 0; kk < kChunk / 8; ++kk)
                    mma_tf32_ss(tmem, sdesc_sw64(sa + kk * 32, 512),
                                sdesc_sw64(sb + kk * 32, 512), IDESC_COMMIT, (ch > 0 || kk > 0));
            }
            mma_commit(&bar[1]);
        }
        // Long path: every thread has read this chunk's staged rows, so its
        // buffer takes the rows of chunk ch + 2, or, after the last chunk, the
        // first state box (the whole buffer is free then).
        if (longp && warp == 0 &&
            __shfl_sync(0xffffffffu, (int)(*(volatile int *)flag == 0), 0) != 0) {
            if (ch + 2 < nchunks) {
                stage_path_rows(sS, bar, path, k, U, ch + 2, L, o, H, h, hv);
                if (tid == 0) *staged = ch + 2;
            } else if (ch == nchunks - 1 && tid == 0) {
                ++nload;
                mbar_arrive_expect_tx(&bar[0], 16384);
                tma_load_3d(sS, &tmS, &bar[0], kTile * hv, unit * kD, layer);
            }
        }
        if (!mbar_wait(&bar[1], ch & 1, kWaitNs)) {
            report(st, BOLE_ERR_TIMEOUT, b, -1, 7);
            *flag = 1;
        }
        tc_fence_after();
        __syncthreads();
        if (*(volatile int *)flag != 0) break; // no further product after a timeout
    }

    // epilogue, one 32-column box at a time: S <- P_a S + D in shared memory,
    // then TMA store in place; the second box is requested into the buffer
    // once the first one's store has read it (an L2 hit: prefetched at entry)
    bool ok = *(volatile int *)flag == 0;
    if (nchunks > 0) {
        const float Pa = expf(La);
        const int r = tid;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
        for (int cb = 0; cb < 2; ++cb) {
            if (cb == 1 && tid == 0) {
                bulk_wait_group_read0(); // the first box's store has read the buffer
                if (ok) {
                    ++nload;
                    mbar_arrive_expect_tx(&bar[0], 16384);
                    tma_load_3d(sS, &tmS, &bar[0], kTile * hv + 32, unit * kD, layer);
                }
            }
            if (cb == 1) {
                __syncthreads();
                if (!ok) break;
            }
            if (ok && !mbar_wait(&bar[0], (uint32_t)cb, kWaitNs)) {
                report(st, BOLE_ERR_TIMEOUT, b, -1, 8);
                *flag = 1;
            }
            if (*(volatile int *)flag == 0) {
                float x[32];
                tmem_ld32(tmem + lane_base + cb * 32, x);
#pragma unroll
                for (int q = 0; q < 2; ++q) { // the row in two halves (fewer live registers)
                    float4 s4[4];
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
                        s4[c4] = *reinterpret_cast<const float4 *>(sS + sw128_offset(r, 16 * q + 4 * c4));
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        float4 v = s4[c4];
                        const float *xq = x + 16 * q + 4 * c4;
                        v.x = fmaf(Pa, v.x, xq[0]);
                        v.y = fmaf(Pa, v.y, xq[1]);
                        v.z = fmaf(Pa, v.z, xq[2]);
                        v.w = fmaf(Pa, v.w, xq[3]);
                        *reinterpret_cast<float4 *>(sS + sw128_offset(r, 16 * q + 4 * c4)) = v;
                    }
                }
                fence_proxy_async_smem();
            }
            __syncthreads();
            ok = *(volatile int *)flag == 0;
            if (tid == 0 && ok) {
                tma_store_3d(&tmS, sS, kTile * hv + 32 * cb, unit * kD, layer);
                bulk_commit_group();
            }
        }
        if (tid == 0) bulk_wait_group_read0();
    }
    tc_fence_before();
    __syncthreads();
    if (*(volatile int *)flag != 0 && nchunks > 0) {
        // after a timeout: the products and the state copy this CTA issued
        // end (bounded) before its tensor and shared memory are released
        if (tid == 0) {
            mma_commit(&bar[2]);
            mbar_wait(&bar[2], 0, kWaitNs);
            if (nload > 0) mbar_wait(&bar[0], (uint32_t)(nload - 1) & 1u, kWaitNs);
            // the last requested chunk of each staging buffer
            const int last = *staged;
            for (int cc = last; cc >= 0 && cc >= last - 1; --cc)
                mbar_wait(&bar[3 + (cc & 1)], (uint32_t)(cc >> 1) & 1u, kWaitNs);
        }
        __syncthreads();
    }
    if (warp == 0) tmem_dealloc(tmem, 64);
}

// ---- host side ----

} // namespace

// CTAs of a launch resident at once (per_sm per SM), cached per device.
static int resident_ctas(int per_sm)
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

bool tc_verify_supported(const VerifyArgs &a)
{
    return a.dtype == BOLE_BF16 && a.dk == kD && a.dv == kD && a.max_T <= kT &&
           a.max_depth < kSlots;
}

size_t tc_workspace_bytes(int, int, int) { return 0; }

cudaError_t launch_tc_verify(const VerifyArgs &a, cudaStream_t s, bool overlap)
{
    const int units = a.B * a.H;
    if (units == 0 || a.N == 0) return cudaSuccess;
    // trees of at most 32 nodes take the small variant (q, k, v boxes of 32 rows)
    const bool small = a.max_T <= kTSmall;
    const int rows = small ? kTSmall : kT;
    CUtensorMap mS, mQ, mK, mV;
    cudaError_t e = make_state_map(&mS, a.S_pre, units);
    if (e == cudaSuccess) e = make_node_map(&mQ, a.q, a.N, a.H, rows);
    if (e == cudaSuccess) e = make_node_map(&mK, a.k, a.N, a.H, rows);
    if (e == cudaSuccess) e = make_node_map(&mV, a.v, a.N, a.H, rows);
    if (e != cudaSuccess) return e;
    auto kernel = small ? (a.vk ? tc_verify_kernel<true, true, false>
                                : tc_verify_kernel<false, true, false>)
                        : (a.vk ? tc_verify_kernel<true, false, false>
                                : tc_verify_kernel<false, false, false>);
    e = configure_once(reinterpret_cast<const void *>(kernel), VERIFY_SMEM, true);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = launch_config(dim3(units), dim3(kThreads), VERIFY_SMEM, s,
                                                 overlap, attr);
    return cudaLaunchKernelEx(&cfg, kernel, mS, mQ, mK, mV, a.gamma, a.beta, a.offsets, a.anc,
                              a.req_depth, a.H, a.N, static_cast<__nv_bfloat16 *>(a.O), a.U,
                              a.logP, a.st, resident_ctas(2), overlap ? 0 : 1, a.parent,
                              a.max_depth, a.inline_topo ? 1 : 0, PrevRound{});
}

bool tc_commit_verify_supported(const VerifyArgs &a)
{
    return tc_verify_supported(a) && !a.vk;
}

cudaError_t launch_tc_commit_verify(const VerifyArgs &a, const PrevArgs &p, cudaStream_t s)
{
    const int units = a.B * a.H;
    if (units == 0) return cudaSuccess;
    const bool small = a.max_T <= kTSmall;
    const int rows = small ? kTSmall : kT;
    CUtensorMap mS, mQ, mK, mV;
    // N may be 0 (every tree of this round empty: only the commit runs); the
    // node maps then describe an extent over the previous keys that no copy
    // reads (no tree, no q / k / v load).
    const int n_map = a.N > 0 ? a.N : rows;
    cudaError_t e = make_state_map(&mS, a.S_pre, units);
    if (e == cudaSuccess) e = make_node_map(&mQ, a.N > 0 ? a.q : p.k, n_map, a.H, rows);
    if (e == cudaSuccess) e = make_node_map(&mK, a.N > 0 ? a.k : p.k, n_map, a.H, rows);
    if (e == cudaSuccess) e = make_node_map(&mV, a.N > 0 ? a.v : p.k, n_map, a.H, rows);
    if (e != cudaSuccess) return e;
    auto kernel = small ? tc_verify_kernel<false, true, true> : tc_verify_kernel<false, false, true>;
    e = configure_once(reinterpret_cast<const void *>(kernel), VERIFY_SMEM, true);
    if (e != cudaSuccess) return e;
    const PrevRound prev{static_cast<const __nv_bfloat16 *>(p.k), p.U, p.logP, p.offsets,
                         p.parent, p.accepted, p.N};
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = launch_config(dim3(units), dim3(kThreads), VERIFY_SMEM, s,
                                                 false, attr);
    return cudaLaunchKernelEx(&cfg, kernel, mS, mQ, mK, mV, a.gamma, a.beta, a.offsets, a.anc,
                              a.req_depth, a.H, a.N, static_cast<__nv_bfloat16 *>(a.O), a.U,
                              a.logP, a.st, resident_ctas(2), 1, a.parent, a.max_depth, 1, prev);
}

bool tc_commit_supported(const CommitArgs &a)
{
    return (a.dtype == BOLE_BF16 || a.dtype == BOLE_F32) && a.dk == kD && a.dv == kD;
}

cudaError_t launch_tc_commit(const CommitArgs &a, cudaStream_t s, bool overlap)
{
    const int units = a.B * a.H;
    if (units == 0 || a.N == 0 || a.layers == 0) return cudaSuccess;
    CUtensorMap map;
    cudaError_t e = make_layered_state_map(&map, a.S, units, a.layers, a.s_ls);
    if (e != cudaSuccess) return e;
    const bool f32 = a.dtype == BOLE_F32;
    auto kernel = f32 ? (a.vk ? tc_commit_kernel<true, true> : tc_commit_kernel<false, true>)
                      : (a.vk ? tc_commit_kernel<true, false> : tc_commit_kernel<false, false>);
    const int smem = f32 ? CoPlan<true>::SMEM : CoPlan<false>::SMEM;
    e = configure_once(reinterpret_cast<const void *>(kernel), smem, false);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = launch_config(dim3(units, kD / kTile, a.layers),
                                                 dim3(kCommitThreads), smem, s, overlap, attr);
    return cudaLaunchKernelEx(&cfg, kernel, map, a.k, a.U, a.logP, a.offsets, a.parent,
                              a.accepted, a.H, a.N, a.k_ls, a.u_ls, a.lp_ls, a.st);
}

} // namespace bole
