/*
 * bole.h -- C ABI of the GB300 (sm_103a) library for closed-form tree
 * verification of Gated DeltaNet layers.
 *
 * The method is the one of "Bole: Efficient Tree Speculation for
 * Hybrid-Attention Language Models":
 *   - every proposal node i of a tree sees the committed prefix and its own
 *     proposal ancestors A(i), never a sibling branch (Section II-B);
 *   - its output is given in closed form from one immutable pre-tree state
 *     S_pre (Theorem 1, Eq. (2)):
 *         O = D_P Q S_pre + C (I+G)^{-1} D_beta (V - D_P K S_pre)
 *     with the cumulative decay P_i = prod of gamma over A(i) and i (Lemma 1,
 *     Eq. (4)), G_ij = beta_i (P_i/P_j) k_i.k_j for j in A(i) (Lemma 2,
 *     Eq. (5)), C_ij = (P_i/P_j) q_i.k_j for j in A(i) or j = i, and the
 *     inverse equal to the finite Neumann sum of (-G)^m, m <= d (Lemma 3,
 *     Eq. (6)).  The same finite polynomial is evaluated three ways: the
 *     CUDA-core kernels run the pages' recurrence Z <- -G Z, U += Z
 *     (Eq. (8)) on each value tile; the tensor-core kernel for trees of up
 *     to 64 nodes forms each row of (I+G)^{-1} by backward substitution
 *     along the node's ancestor path; the large-tree tensor-core kernel by
 *     log-depth doubling, (I - G) prod_k (I + G^(2^k)).  Only the rounding
 *     order differs;
 *   - the per-node factors (P, K, U) replace per-node state snapshots
 *     (Eq. (9)); after sampling, commit rebuilds the accepted node a's exact
 *     state S_new = P_a S_pre + (D_a K_a)^T U_a (Eq. (10)), in place.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library allocates no device memory.  Its global state is limited to
 *     set-up done once per device (kernel attributes, the tensor-map
 *     encoder's entry point) and one exception: the fixed scratch array of
 *     bole_tree_verify_noalloc, which every call of that entry point shares
 *     (see there).  All calls are asynchronous on `stream` (a cudaStream_t;
 *     NULL selects the legacy default stream); apart from
 *     bole_tree_verify_noalloc (see there), they may be captured in CUDA
 *     graphs.
 *   - Packed forest: B requests' trees are concatenated node-major.
 *     offsets[B+1] (int32, offsets[0] = 0, non-decreasing, offsets[B] <= N)
 *     delimits request b's nodes [offsets[b], offsets[b+1]); N is the
 *     length (capacity) of the node arrays and nodes past offsets[B] are
 *     ignored, so a forest built on the device needs no host round trip.  parent[N]
 *     (int32) holds request-LOCAL parent indices, -1 = the committed root,
 *     and parent[i] < i (parent before child).  At most 128 nodes per tree.
 *   - Depth of a node = number of strict proposal ancestors (a child of the
 *     committed root has depth 0).  `max_depth` is an upper bound; the
 *     kernels run exactly the per-request depth (extra Neumann steps would
 *     add exact zeros since G^(d+1) = 0).
 *   - Layouts (row-major, last index contiguous):
 *       S_pre / S     [B, H, dk, dv] float32 (one dk x dv state per head);
 *                     [B, H, dv, dk] with BOLE_FLAG_STATE_VK
 *       q, k          [N, H, dk]  bf16 or float32 (bole_dtype)
 *       v             [N, H, dv]  same dtype as q, k
 *       gamma, beta   [N, H] float32; gamma in (0, 1] (decay), beta = write gate
 *       O             [N, H, dv]  same dtype as q/k/v
 *       U             [N, H, dv]  float32 (the propagated deltas u_i)
 *       logP          [N, H]      float32, log of the cumulative decay P_i
 *   - Supported sizes: dk, dv multiples of 16 in [16, 128]; H >= 1;
 *     B >= 0 (B = 0 or N = 0 launches nothing); 16-byte aligned pointers.
 *   - Errors: arguments that the host can check (null pointers, sizes,
 *     alignment, workspace) make the call return an error code synchronously
 *     and launch nothing.  Faults in device data (topology, depth, sizes
 *     larger than declared) are written to `dev_status` (int32[4]:
 *     {code, request, node, detail}); the first fault wins, later kernels of
 *     the round see it and write no outputs.  No kernel traps or spins
 *     without bound; a bounded wait that expires records BOLE_ERR_TIMEOUT.
 *     BOLE_ERR_CUDA means a CUDA runtime call (launch, attribute) failed.
 */
#ifndef BOLE_H_
#define BOLE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *bole_stream_t; /* same type as cudaStream_t */

typedef enum bole_status {
    BOLE_OK = 0,
    BOLE_ERR_INVALID_ARG = 1,  /* null pointer, size out of range, misalignment */
    BOLE_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement */
    BOLE_ERR_BAD_TOPOLOGY = 3, /* parent[i] >= i or < -1, tree > 128 nodes, bad offsets */
    BOLE_ERR_DEPTH = 4,        /* a tree is deeper than max_depth */
    BOLE_ERR_WORKSPACE = 5,    /* workspace missing or smaller than bole_workspace_size */
    BOLE_ERR_CUDA = 6,         /* a CUDA runtime call failed */
    BOLE_ERR_TIMEOUT = 7       /* a bounded device-side wait expired */
} bole_status;

typedef enum bole_dtype { BOLE_F32 = 0, BOLE_BF16 = 1 } bole_dtype;

#define BOLE_MAX_TREE_NODES 128
#define BOLE_STATUS_WORDS 4

/* Flags for bole_tree_verify / bole_commit / bole_workspace_size. */
#define BOLE_FLAG_FORCE_SIMT 0x1u /* use the FP32 CUDA-core kernels even where the
                                     tcgen05 tensor-core kernels apply */
/* Overlap the launch with the kernel before it on the stream (programmatic
 * dependent launch; tensor-core kernels only).  The caller asserts that the
 * previous kernel on the stream is the round's bole_pack_forest (before
 * bole_tree_verify), a bole_tree_verify (before the next layer's
 * bole_tree_verify, or before bole_commit / bole_commit_layers), or any
 * kernel that does not let its dependents start early.  The kernel may then
 * begin while that one drains: before waiting for it, it reads only
 * caller-owned inputs that none of these calls writes (S_pre / S, q, k, v,
 * gamma, beta, offsets, parent); the status word and everything the previous call
 * produced are read after the wait.  Without the flag every launch starts
 * only after the previous kernel has ended. */
#define BOLE_FLAG_OVERLAP_LAUNCH 0x2u
/* State slots in the serving runtime's canonical layout (Section IV-D, the
 * state lifecycle of Fig. 6): S_pre / S stored [B, H, dv, dk] -- each head's
 * state transposed, d_k contiguous -- instead of [B, H, dk, dv].  Accepted by
 * bole_workspace_size, bole_tree_verify, bole_commit and bole_commit_layers;
 * every kernel reads and writes that layout directly (no transposed copy).
 * The results are the same numbers as with the default layout. */
#define BOLE_FLAG_STATE_VK 0x4u
/* Verification of bf16 trees of up to 32 nodes (depth <= 15, dk = dv = 128,
 * default state layout) has two tensor-core kernels: one CTA per (request,
 * head), or the value-tiled kernel -- two CTAs per head, 64 value columns
 * each (Section IV-B: H * N_v independently schedulable CTAs per request).
 * By default the value tiles serve batches whose B * H heads would not fill
 * one wave of the one-CTA kernel (two CTAs per SM), where the extra CTAs
 * add parallelism; larger batches run one CTA per head, which moves more
 * state bytes per resident CTA.  These flags force either kernel (same
 * results up to rounding order); they are ignored elsewhere.  fp32 trees in
 * the same envelope run the value-tiled kernel's fp32 form by default (no
 * one-CTA fp32 kernel exists: with BOLE_FLAG_ONE_TILE_PER_HEAD they run the
 * FP32 CUDA-core kernels). */
#define BOLE_FLAG_ONE_TILE_PER_HEAD 0x8u
#define BOLE_FLAG_VALUE_TILES 0x10u
/* bole_tree_verify only: the round's topology step runs inside the
 * verification (Section IV-C), so no bole_pack_forest precedes it.  Each CTA
 * derives its tree's ancestor-or-self masks and depths from `parent` and
 * validates the tree: a link that does not point backwards is reported as
 * BOLE_ERR_BAD_TOPOLOGY {code, request, node, parent}, a tree deeper than
 * max_depth as BOLE_ERR_DEPTH {code, request, -1, depth}, bad extents as
 * bole_pack_forest reports them; that request's outputs are left unwritten
 * (other requests' are written, and a later bole_commit of the round then
 * writes nothing).  depth, anc and req_depth are not read and may be NULL.
 * Nothing clears dev_status in this mode: zero it once, check it after the
 * round, and zero it again after handling a fault (until then every later
 * kernel sees the fault and writes nothing).  Supported where the
 * tensor-core kernels for trees of up to 64 nodes apply (bf16, dk = dv =
 * 128, max_T <= 64, max_depth <= 15, default state layout); elsewhere the
 * call returns BOLE_ERR_UNSUPPORTED with nothing launched. */
#define BOLE_FLAG_INLINE_TOPOLOGY 0x20u

/* Human-readable name of a status code (static storage, never NULL). */
const char *bole_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int bole_version(void);

/* The cudaError_t behind the calling host thread's most recent BOLE_ERR_CUDA
 * (0 if none yet), and its CUDA description (static storage, never NULL).
 * A launch can also return the sticky error of an earlier kernel that
 * faulted. */
int bole_last_cuda_error(void);
const char *bole_last_cuda_error_string(void);

/* Self-test of the bounded device waits.  Every device wait of the library
 * (an mbarrier wait for a copy or a tensor-core product) gives up after a
 * limit and reports BOLE_ERR_TIMEOUT in the status block instead of hanging;
 * this call launches one thread that waits on an mbarrier nothing arrives
 * on, with the given limit (at most BOLE_SELFTEST_MAX_WAIT_NS), so that the
 * timeout path can be exercised without a fault: afterwards dev_status holds
 * {BOLE_ERR_TIMEOUT, -1, -1, microseconds waited} (first error wins, as
 * everywhere) and the context stays usable.  dev_status: device, 16-byte
 * aligned, BOLE_STATUS_WORDS words, not cleared by this call. */
#define BOLE_SELFTEST_MAX_WAIT_NS 1000000000ull
bole_status bole_selftest_wait(int32_t *dev_status, uint64_t limit_ns, bole_stream_t stream);

/* Bytes of device workspace bole_tree_verify needs for these sizes (0 when
 * the chosen kernel keeps every intermediate on chip, as both tensor-core
 * kernels do).  max_T bounds every tree's node count (1..128) and max_depth
 * every tree's depth (0..127); pass the same values, dtype and flags as to
 * bole_tree_verify.  The workspace holds the short-lived tree factors of one
 * call -- the "verification scratch" of the pages' state lifecycle (Section
 * IV-D): dense G, C on the CUDA-core path -- and may be reused by the next
 * call once that call's kernels have finished. */
size_t bole_workspace_size(int B, int H, int dk, int dv, int max_T, int max_depth,
                           bole_dtype qkv_dtype, unsigned flags);

/* Round-level topology step (Section IV-C; forest packing, review Section 3).
 * Validates the packed forest and derives, per node, its depth and its
 * ancestor-or-self bit mask, and per request its depth.
 *   offsets [B+1], parent [N]   in: the packed forest (device)
 *   depth   [N]   int32         out: strict-ancestor count
 *   anc     [N,4] uint32        out: bit j of word j/32 set iff local node j is
 *                                    an ancestor of the node or the node itself
 *   req_depth [B] int32         out: max depth over the request (0 if empty)
 *   dev_status [4] int32        out: zeroed by this call, then the first fault:
 *                                    BOLE_ERR_BAD_TOPOLOGY or BOLE_ERR_DEPTH
 * Integer only; results are exact. */
bole_status bole_pack_forest(const int32_t *offsets, const int32_t *parent, int B, int N,
                             int max_depth, int32_t *depth, uint32_t *anc, int32_t *req_depth,
                             int32_t *dev_status, bole_stream_t stream);

/* Closed-form verification of every node of every tree (Theorem 1, Eq. (2);
 * state products as in Eq. (7); propagation by the finite Neumann sum of
 * Eq. (6), evaluated per kernel as described at the top of this file: the
 * recurrence of Eq. (8) on the CUDA-core path, backward substitution or
 * log-depth doubling on the tensor-core paths).  S_pre is read only
 * (immutable during verification, Section IV-D).  Inputs: S_pre, q, k, v, gamma, beta as laid out above; offsets and
 * parent of the packed forest; depth, anc, req_depth from bole_pack_forest.
 * (With BOLE_FLAG_INLINE_TOPOLOGY the verification forms depth, anc and
 * req_depth itself and they may be NULL; see the flag.)
 * max_T bounds the tree sizes (1..128), max_depth the depths (0..127).
 * Outputs: O (dtype of q/k/v), U (float32) and logP (float32) -- U, logP and
 * the caller's k buffer are the factors commit needs; keep them alive until
 * bole_commit.  workspace: device buffer of at least
 * bole_workspace_size(...) bytes (NULL allowed when that size is 0).
 * Kernel choice: bf16 inputs with dk = dv = 128, max_T <= 64 and
 * max_depth <= 15 run the single-CTA TMA + tcgen05 kernel (state products on
 * a bf16 hi/lo split of S_pre -- the low part is itself rounded to bf16, so
 * each state element keeps a relative residue of about 2^-17 -- with exact
 * bf16 products and fp32 accumulation, every factor on chip); fp32 inputs with
 * dk = dv = 128, max_T <= 32 and max_depth <= 15 run the value-tiled tcgen05
 * kernel (two CTAs per head) with every fp32 operand of the Gram and the state
 * products written as three bf16 parts (24 significant bits) and the six
 * products of order up to 2^-16 kept, the propagation as tf32 hi + lo (three
 * products), fp32 accumulation -- within the float32 bound; bf16 inputs with
 * dk = dv = 128 and larger or deeper trees (up to 128 nodes, any depth) run
 * one tcgen05 kernel per (request, head) that forms the
 * factors [M; W] by log-depth doubling and keeps them in tensor memory for the
 * state products and the propagation (no workspace; when the caller passes
 * one of at least B * H * 256 * 128 * 4 bytes anyway, [M; W] is also written
 * there, unit-major, 256 rows of 128 floats, for inspection); everything
 * else, or flags & BOLE_FLAG_FORCE_SIMT, runs the FP32 CUDA-core kernels
 * (producer of G, C into the workspace + value-tiled solve). */
bole_status bole_tree_verify(const float *S_pre, const void *q, const void *k, const void *v,
                             bole_dtype qkv_dtype, const float *gamma, const float *beta,
                             const int32_t *offsets, const int32_t *parent, const int32_t *depth,
                             const uint32_t *anc, const int32_t *req_depth, int B, int H, int dk,
                             int dv, int N, int max_T, int max_depth, void *O, float *U,
                             float *logP, void *workspace, size_t workspace_bytes,
                             int32_t *dev_status, unsigned flags, bole_stream_t stream);

/* Verification that allocates nothing -- the paper has no counterpart; this
 * entry point exists for callers that cannot allocate device memory when they
 * verify: hosts that give the library only tensors they already own and no
 * allocator, and serving loops that forbid allocation on the hot path because
 * an allocation can synchronise the device.  Same arguments, layouts, results
 * and device-status behaviour as bole_tree_verify with BOLE_FLAG_FORCE_SIMT
 * (the FP32 CUDA-core kernels), but the G, C scratch those kernels need lives
 * in a fixed 8 MiB array owned by the library (every GPU that loads the
 * library holds it until the process exits); no workspace is passed and
 * nothing is allocated.
 *   - Limit: B * H * max_T * max_T <= BOLE_NOALLOC_MAX_FACTOR_ELEMS; larger
 *     problems return BOLE_ERR_UNSUPPORTED with nothing launched (use
 *     bole_tree_verify with a caller-allocated workspace instead).
 *   - The first call on each device resolves the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.  A failure there returns BOLE_ERR_CUDA.
 *   - Every call shares the one array and it keeps the previous call's
 *     contents; calls whose kernels overlap on the GPU (different streams, or
 *     several host threads) race on it -- order them on one stream. */
#define BOLE_NOALLOC_MAX_FACTOR_ELEMS (1u << 20)
bole_status bole_tree_verify_noalloc(const float *S_pre, const void *q, const void *k,
                                     const void *v, bole_dtype qkv_dtype, const float *gamma,
                                     const float *beta, const int32_t *offsets,
                                     const int32_t *parent, const int32_t *depth,
                                     const uint32_t *anc, const int32_t *req_depth, int B, int H,
                                     int dk, int dv, int N, int max_T, int max_depth, void *O,
                                     float *U, float *logP, int32_t *dev_status,
                                     bole_stream_t stream);

/* Factorised commit (Eq. (10)): for every request b with accepted[b] = a >= 0
 * (request-local node index) and every head,
 *     S <- P_a S + sum over j on the path root..a of (P_a / P_j) k_j u_j^T
 * written in place over S ([B,H,dk,dv] float32, which held S_pre during the
 * verification that produced U and logP).  accepted[b] = -1 leaves request b's
 * state untouched.  k is the same buffer verification read; U and logP are its
 * outputs.  dk = dv = 128 uses the TMA + tcgen05 kernel (one tensor-core
 * product per 64-column half of each head's state over the accepted path, tf32
 * operands; fp32 k writes both operands as tf32 hi + lo and keeps three
 * products, for the float32 bound); otherwise, or with BOLE_FLAG_FORCE_SIMT,
 * the FP32 CUDA-core kernel.  Must be stream-ordered after
 * the verification.  Device faults go to dev_status and leave that request's
 * state as it was: accepted[b] >= tree size, {BOLE_ERR_BAD_TOPOLOGY, b,
 * accepted[b], tree size}; a parent link on the accepted path that does not
 * point to an earlier node of the tree, {BOLE_ERR_BAD_TOPOLOGY, b, node, -1}. */
bole_status bole_commit(float *S, const void *k, bole_dtype k_dtype, const float *U,
                        const float *logP, const int32_t *offsets, const int32_t *parent,
                        const int32_t *accepted, int B, int H, int dk, int dv, int N,
                        int32_t *dev_status, unsigned flags, bole_stream_t stream);

/* Unified cross-layer commit (Section IV-D and the integration notes of the
 * SGLang page: every recurrent layer writes its P, K, U factors into one
 * preallocated contiguous buffer and a single batched launch evaluates
 * Eq. (10) for all of them).  One launch commits n_layers GDN layers that
 * verified the same packed forest in this round: layer l's buffers are
 *     S    + l * s_layer_stride    [B,H,dk,dv] (or [B,H,dv,dk]) float32, in/out
 *     k    + l * k_layer_stride    [N,H,dk] k_dtype
 *     U    + l * u_layer_stride    [N,H,dv] float32
 *     logP + l * lp_layer_stride   [N,H]    float32
 * (strides in ELEMENTS of each buffer), and offsets, parent, accepted are
 * shared by all layers.  The result of each layer is exactly that of
 * bole_commit on its slices; n_layers = 1 is bole_commit.
 *   - n_layers in [0, 65535] (0 launches nothing).  With n_layers > 1 the
 *     state slices must not overlap: s_layer_stride >= B*H*dk*dv (else
 *     BOLE_ERR_INVALID_ARG); the read-only factor strides may be anything
 *     >= 0 (0 shares one factor buffer between layers).
 *   - Every stride times its element size is a multiple of 16 bytes, except
 *     lp_layer_stride (4-byte elements, any value).
 *   - flags: BOLE_FLAG_FORCE_SIMT, BOLE_FLAG_OVERLAP_LAUNCH (the previous
 *     kernel on the stream is the last layer's bole_tree_verify, or does not
 *     let dependents start early), BOLE_FLAG_STATE_VK.
 *   - Device faults go to dev_status as for bole_commit (the first fault of
 *     any layer wins; the fault record does not name the layer). */
bole_status bole_commit_layers(float *S, int64_t s_layer_stride, const void *k,
                               int64_t k_layer_stride, bole_dtype k_dtype, const float *U,
                               int64_t u_layer_stride, const float *logP, int64_t lp_layer_stride,
                               const int32_t *offsets, const int32_t *parent,
                               const int32_t *accepted, int n_layers, int B, int H, int dk, int dv,
                               int N, int32_t *dev_status, unsigned flags, bole_stream_t stream);

/* Deferred commit fused with the next verification (Eq. (10), then the
 * closed form of Section III on the committed state, in one launch).  In a
 * serving loop the commit of round r and the verification of round r + 1 both
 * stream each head's state; this call reads it once:
 *     S <- P_a S + sum over j on the path root..a of (P_a / P_j) k_j u_j^T
 * with the previous round's factors (exactly bole_commit with k_prev, U_prev,
 * logP_prev, offsets_prev, parent_prev, accepted_prev, N_prev), then this
 * round's verification from the committed S (exactly bole_tree_verify with
 * BOLE_FLAG_INLINE_TOPOLOGY: O, U, logP of this round's forest).  Both
 * rounds have the same B requests and H heads; their forests may differ.
 *   - S: [B,H,dk,dv] float32 in/out (default state layout), 16-byte aligned.
 *   - Previous round: k_prev [N_prev,H,dk] in qkv_dtype, U_prev [N_prev,H,dv],
 *     logP_prev [N_prev,H] float32, offsets_prev [B+1], parent_prev [N_prev],
 *     accepted_prev [B] (-1: that request's state is not committed).  U and
 *     logP of this call must be other buffers than U_prev and logP_prev (the
 *     same pointer returns BOLE_ERR_INVALID_ARG; partial overlaps are the
 *     caller's to avoid): keep two and alternate them between rounds.
 *   - This round: as bole_tree_verify (q, k, v, gamma, beta, offsets,
 *     parent; O, U, logP written), the topology formed in the kernel.
 *   - Supported: bf16 q/k/v (and k_prev), dk = dv = 128, max_T <= 64,
 *     max_depth <= 15; elsewhere BOLE_ERR_UNSUPPORTED with nothing launched
 *     (call bole_commit, then bole_tree_verify).  An accepted path of more than
 *     16 nodes is reported as BOLE_ERR_DEPTH {code, request, accepted node,
 *     16}; a bad accepted node, extent or parent link of the previous round
 *     as bole_commit reports it; that request's state is left uncommitted
 *     (its outputs of this round, computed from that state, are not to be
 *     used).  A request whose new tree is empty or refused is still committed.
 *   - flags: 0 or BOLE_FLAG_OVERLAP_LAUNCH (accepted and ignored: the launch
 *     always waits for the previous kernel, whose commit or verification may
 *     have written S; and no kernel after it starts before it has ended).
 *   - Device faults and the status block as for bole_tree_verify with
 *     BOLE_FLAG_INLINE_TOPOLOGY (nothing clears dev_status).
 * The last round of a sequence is committed with bole_commit. */
bole_status bole_commit_verify(float *S, const void *k_prev, const float *U_prev,
                               const float *logP_prev, const int32_t *offsets_prev,
                               const int32_t *parent_prev, const int32_t *accepted_prev,
                               int N_prev, const void *q, const void *k, const void *v,
                               bole_dtype qkv_dtype, const float *gamma, const float *beta,
                               const int32_t *offsets, const int32_t *parent, int B, int H,
                               int dk, int dv, int N, int max_T, int max_depth, void *O, float *U,
                               float *logP, int32_t *dev_status, unsigned flags,
                               bole_stream_t stream);

/* ---- Device-side proposal selection and forest build ----
 * (Section IV, hardware-aware budget: at run time each drafted candidate v
 * scores rho(v) = product over its path of the drafter's edge probabilities
 * p(u | parent(u)), and the globally highest-scoring candidates fill the
 * round's budget; a child never outscores its parent, so every request's
 * selection is ancestor-closed.  The integration keeps selection and forest
 * build on the GPU.)
 *   p [M] float32 in [0, 1]        edge probability of each candidate
 *   cand_offsets [B+1], cand_parent [M]   the drafter's trees, packed like a
 *                                  forest (request-local parents, -1 = root,
 *                                  parent before child), at most
 *                                  BOLE_MAX_CANDIDATES per request
 *   caps [B] int32 or NULL         per-request node limits (NULL: none); a
 *                                  tree never exceeds BOLE_MAX_TREE_NODES
 *   budget                         total nodes of the round
 * Rule (every decision on float32 scores accumulated root-down,
 * rho(v) = rho(parent) * p(v)): order = larger rho first, then smaller depth,
 * request, candidate index; each request with a candidate first receives its
 * best one (in that order while the budget lasts); the rest of the budget
 * goes to the best remaining candidates, skipping requests at their limit.
 * Outputs, all device:
 *   offsets [B+1]                  the packed forest's extents (offsets[B] =
 *                                  the node count, <= budget)
 *   parent [budget], src [budget]  per forest node: request-local parent and
 *                                  its candidate index (to gather its token /
 *                                  hidden state); a request's nodes in
 *                                  candidate order (parent before child)
 *   rho [M] float32 or NULL        the scores
 * The forest feeds bole_pack_forest directly with N = the node capacity
 * (offsets[B] <= N), so no host round trip is needed.  dev_status is zeroed
 * by this call (give the round's later calls their own status block, or
 * check it first); malformed candidate trees are reported as
 * BOLE_ERR_BAD_TOPOLOGY and that request gets no nodes.  B <= 4096.
 * workspace: bole_select_workspace_size(B) bytes. */
#define BOLE_MAX_CANDIDATES 1024
#define BOLE_SELECT_MAX_REQUESTS 4096
size_t bole_select_workspace_size(int B);
bole_status bole_select_forest(const float *p, const int32_t *cand_offsets,
                               const int32_t *cand_parent, const int32_t *caps, int B, int M,
                               int budget, int32_t *offsets, int32_t *parent, int32_t *src,
                               float *rho, void *workspace, size_t workspace_bytes,
                               int32_t *dev_status, unsigned flags, bole_stream_t stream);

/* ---- Stage 1 of a GDN layer: tree-parallel convolution and gates ----
 * (Section II-A: a GDN layer's short causal depthwise convolution and gates;
 * Section IV-C, the fused pipeline: stage (1) fuses the convolution, its
 * bias, SiLU and gate preparation per node along parent links, all nodes
 * concurrently.)  For every node i of every request and every head h:
 *   - window: i, its parent, grandparent, ... (nearest first); where the path
 *     reaches the committed root, the committed prefix's last W-1 tokens
 *     (conv_state rows W-2, W-3, ...);
 *   - y[c] = conv_b[c] + sum_{d<W} conv_w[c][W-1-d] * (token at distance d)[c];
 *   - SiLU; the q and k channels of each head L2-normalised (over d_k);
 *   - gamma = exp(-s_h softplus(a + c_h)), beta = sigmoid(b), with
 *     s_h = gate_scale[h] (1 if NULL) and c_h = gate_bias[h] (0 if NULL).
 * Layouts:
 *   x          [N, C] x_dtype, C = H (2 dk + dv): the q channels of every head
 *              (head-major), then k, then v -- the in-projection output
 *   conv_state [B, W-1, C] x_dtype (row W-2 the most recent committed token;
 *              may be NULL when W = 1)
 *   conv_w     [C, W] float32 (tap W-1 multiplies the current token)
 *   conv_b     [C] float32 or NULL;  a, b [N, H] float32 gate pre-activations
 *   q, k       [N, H, dk] x_dtype;  v [N, H, dv] x_dtype  (bole_tree_verify's
 *              inputs);  gamma, beta [N, H] float32
 * W in [1, 8]; dk, dv as elsewhere; max_T (1..128) bounds every tree's node
 * count (it sizes the on-chip tile of one request).  offsets / parent: the
 * packed forest (a malformed link or a tree larger than max_T is reported as
 * BOLE_ERR_BAD_TOPOLOGY in dev_status, and that request is left unwritten).
 * Stream-ordered after bole_pack_forest (which resets dev_status) and before
 * bole_tree_verify. */
#define BOLE_MAX_CONV_WIDTH 8
bole_status bole_conv_gates(const void *x, const void *conv_state, const float *conv_w,
                            const float *conv_b, const float *a, const float *b,
                            const float *gate_scale, const float *gate_bias, bole_dtype x_dtype,
                            const int32_t *offsets, const int32_t *parent, int B, int H, int dk,
                            int dv, int N, int max_T, int W, void *q, void *k, void *v,
                            float *gamma, float *beta, int32_t *dev_status, unsigned flags,
                            bole_stream_t stream);

/* Commit of the convolution state (the conv counterpart of bole_commit):
 * for every request with accepted[b] = a >= 0, conv_state[b] ([W-1, C],
 * in place) becomes the last W-1 tokens ending at a -- a's row of x in row
 * W-2, its parent's in row W-3, ..., then the old rows, most recent first.
 * accepted[b] = -1 leaves the request's state untouched.  x is the same
 * buffer bole_conv_gates read.  Exact (rows are copied).  W = 1 launches
 * nothing.  C = H (2 dk + dv) (a multiple of 16); B <= 65535. */
bole_status bole_conv_commit(void *conv_state, const void *x, bole_dtype x_dtype,
                             const int32_t *offsets, const int32_t *parent,
                             const int32_t *accepted, int B, int C, int W, int N,
                             int32_t *dev_status, unsigned flags, bole_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BOLE_H_ */
