/*
 * tv.h -- C ABI of the tree-speculative-verification library for gated-DeltaNet hybrids.
 *
 * One verify round of a hybrid model (qwen35-tree-spec post, §七 完整验证流程) runs a draft
 * tree, given by a parents[] array, through two kinds of layers:
 *
 *   - gated-DeltaNet (GDN) layers, where every node i gets its own recurrent state
 *         S_i = alpha_i * S_p @ (I - beta_i k_i k_i^T) + beta_i v_i k_i^T,   o_i = S_i q_i
 *     evolved from its parent p (the committed state S_0 for a root), either by
 *     depth-by-depth fork/checkpoint (same post, §四) or by the TreeWY form, which keeps a
 *     small pseudo-value matrix instead of per-node states (TreeWY: Speculative Verification
 *     for Gated DeltaNet Hybrids, abstract);
 *   - full-attention layers, where every node attends to the committed KV prefix plus its
 *     ancestors plus itself at RoPE position prefix_len + depth (handbook chapter
 *     投机解码进阶：树形草稿与 EAGLE, §实现, forward_with_mask and tree_mask);
 *
 * then commits the accepted path: the GDN state goes back to the last accepted node's state
 * (qwen35-tree-spec §五 用途 2) and the accepted nodes' KV moves to the contiguous slots after
 * the prefix, or whole blocks of it are taken over through the block table (handbook chapter,
 * note after the listing: the KV is reused, not recomputed).
 *
 * Conventions for every call below
 * --------------------------------
 *  - Pointers are DEVICE pointers owned by the caller, unless a comment says otherwise; the
 *    library allocates no memory.  Every tensor is dense, row-major (last index fastest) with
 *    the shape written beside it, and its base address is 16-byte aligned.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *    The return value reports only what the host can see before launch: TV_OK, or
 *    TV_ERR_INVALID_ARG (null/misaligned pointer, non-positive or inconsistent size),
 *    TV_ERR_UNSUPPORTED (a size or dtype outside the supported set) or TV_ERR_CUDA (a launch
 *    failed; tv_last_cuda_error() then holds the CUDA error code).  Nothing is launched when
 *    the return value is not TV_OK.
 *  - Data-dependent errors (a malformed tree, a bad accepted path, a block table that is too
 *    short or points outside the cache) are written per sequence to the device array
 *    err[B] (0 = that sequence is fine, else a TV_ERR_* code).  A failed sequence's outputs
 *    are left unwritten; the other sequences are unaffected.  No kernel traps or waits
 *    without bound.  Read err after synchronising the stream.
 *  - parents[b][i] is -1 (node i follows the committed state directly: a root) or an
 *    earlier node index (-1 <= parents[i] < i); anything else is TV_ERR_BAD_TREE.
 *  - Sizes: 1 <= N <= TV_MAX_NODES nodes per tree, every sequence of a call has N nodes.
 *  - dtype codes: TV_F32 (fp32) or TV_BF16 (bf16, round-to-nearest-even on store).
 *    Arithmetic is fp32 throughout.
 */
#ifndef TV_H_
#define TV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define TV_API __attribute__((visibility("default")))
#else
#define TV_API
#endif

struct CUstream_st;
typedef struct CUstream_st* tv_stream_t; /* same type as cudaStream_t */

enum tv_status {
  TV_OK = 0,
  TV_ERR_INVALID_ARG = -1,
  TV_ERR_BAD_TREE = -2,
  TV_ERR_BAD_PATH = -3,
  TV_ERR_UNSUPPORTED = -4,
  TV_ERR_CUDA = -5,
  TV_ERR_TIMEOUT = -6,
  TV_ERR_CAPACITY = -7,     /* block table too short for prefix_len + N slots */
  TV_ERR_BAD_BLOCK = -8,    /* a block-table entry outside [0, num_blocks), or (compaction)
                               two logical blocks of the tree's window on one physical block */
  TV_ERR_SCRATCH = -9       /* tv_tree_attn_static: the call needs more than
                               TV_STATIC_SCRATCH_BYTES of scratch */
};

enum tv_dtype { TV_F32 = 0, TV_BF16 = 1 };
enum tv_mode { TV_MODE_FORK = 0, TV_MODE_WY = 1 };

#define TV_MAX_NODES 256
#define TV_BLOCK_SIZE 16
#define TV_STATIC_SCRATCH_BYTES (64u << 20) /* scratch array of tv_tree_attn_static: 64 MiB */

/* Human-readable name of a tv_status code (static string, never NULL). */
TV_API const char* tv_status_string(int status);

/* CUDA error code (cudaError_t value) of the last call that returned TV_ERR_CUDA on this
 * host thread, or 0. */
TV_API int tv_last_cuda_error(void);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
TV_API int tv_version(void);

/* ------------------------------------------------------------------------------------------
 * tv_tree_prepare -- topology of B draft trees.
 *
 * Source: handbook chapter 树形草稿与 EAGLE, §实现, `depths` (depth 0 for a root, parent's
 * depth + 1 otherwise) and `tree_mask` (node i sees itself and every ancestor).
 *
 *   parents   [B, N] int32          in
 *   depth     [B, N] int32          out: depth of every node
 *   mask_bits [B, N, W] uint32      out: W = ceil(N / 32); bit (j % 32) of word j / 32 of row
 *                                   i is 1 iff node j is i or an ancestor of i
 *   paths     [B, N, path_cap] int32  out, optional (NULL: not written): row i is the root-to-i
 *                                   path (handbook §实现: the nodes a draft token's branch
 *                                   passes through), root first, then -1 up to path_cap entries
 *   path_cap  entries per path row, >= 1 when paths is given (depth + 1 entries are needed)
 *   max_depth [B] int32             out, optional (NULL: not written): the deepest node's depth
 *   err       [B] int32             out: 0, TV_ERR_BAD_TREE, or TV_ERR_UNSUPPORTED when a node's
 *                                   depth + 1 exceeds path_cap (depth, mask_bits and max_depth
 *                                   are still written; that sequence's paths are unspecified)
 * Outputs of a sequence whose tree is malformed are unspecified.  Returns TV_ERR_INVALID_ARG for
 * a null or misaligned required pointer, a misaligned optional one, or path_cap < 1 with paths.
 * ---------------------------------------------------------------------------------------- */
TV_API int tv_tree_prepare(const int32_t* parents, int B, int N, int32_t* depth, uint32_t* mask_bits,
                           int32_t* paths, int path_cap, int32_t* max_depth, int32_t* err, tv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * tv_gdn_tree_verify_fork -- one GDN layer over B draft trees, fork/checkpoint mode.
 *
 * Source: qwen35-tree-spec §四 (Fork/Checkpoint, 逐深度处理): every node evolves from its
 * parent's snapshot (S_0 for a root) and its own snapshot is kept for the commit step; the
 * per-node semantics is exactly the root-to-node path replay of the gated delta rule above.
 * The kernel keeps each node's state in fp32 on chip and walks the tree depth-first, so each
 * parent state is read from HBM once (S_0) and each node's snapshot is written once.
 *
 *   q, k        [B, N, H, dk]  io_dtype      in
 *   v           [B, N, H, dv]  io_dtype      in
 *   alpha, beta [B, N, H]      fp32          in  (decay in (0,1], write strength)
 *   S0          [B, H, dv, dk] state_dtype   in  committed state (row = value index)
 *   parents     [B, N]         int32         in
 *   q_scale                                      o_i = S_i (q_scale * q_i)
 *   out         [B, N, H, dv]  io_dtype      out o_i
 *   node_states [B, N, H, dv, dk] state_dtype out S_i of every node (the checkpoints)
 *   err         [B] int32                    out 0 or TV_ERR_BAD_TREE
 * Supported: dk, dv in {64, 128}; (io, state) in {(F32,F32), (BF16,BF16), (BF16,F32)}.
 * ---------------------------------------------------------------------------------------- */
TV_API int tv_gdn_tree_verify_fork(const void* q, const void* k, const void* v, const float* alpha,
                            const float* beta, const void* S0, const int32_t* parents, int B,
                            int N, int H, int dk, int dv, int io_dtype, int state_dtype,
                            float q_scale, void* out, void* node_states, int32_t* err,
                            tv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * tv_gdn_tree_verify_wy -- one GDN layer over B draft trees, TreeWY mode.
 *
 * Source: TreeWY abstract -- all node outputs from one triangular solve over a small
 * pseudo-value matrix, no per-node states.  Reading of the algebra (not on the page): with
 * gamma_i the product of alpha along the root-to-node path P(i), Gamma_ij = gamma_i/gamma_j,
 * and the pseudo-value w_i = beta_i (v_i - alpha_i S_parent k_i),
 *     S_i = gamma_i S_0 + sum_{j in P(i)} Gamma_ij w_j k_j^T,
 *     (I + diag(beta)(A o Gamma o K K^T)) W = diag(beta)(V - diag(gamma) K S_0^T),
 *     O = diag(gamma) (q_scale Q) S_0^T + (M o Gamma o (q_scale Q) K^T) W,
 * A the strict-ancestor mask, M = A + I the tree mask.  The system is unit lower triangular
 * because parents[i] < i; it is solved along ancestor lists (each row of A has depth(i)
 * nonzeros).
 *
 *   inputs as tv_gdn_tree_verify_fork
 *   out         [B, N, H, dv]  io_dtype   out o_i
 *   pseudo_v    [B, N, H, dv]  fp32       out W (w_i per node and head)
 *   log_gamma   [B, N, H]      fp32       out log(gamma_i)
 *   err         [B] int32                 out 0, TV_ERR_BAD_TREE, or TV_ERR_UNSUPPORTED if
 *                                         the sum over nodes of (depth+1) exceeds 4096
 * Supported: dk, dv in {64, 128}; (io, state) as for fork.
 * ---------------------------------------------------------------------------------------- */
TV_API int tv_gdn_tree_verify_wy(const void* q, const void* k, const void* v, const float* alpha,
                          const float* beta, const void* S0, const int32_t* parents, int B,
                          int N, int H, int dk, int dv, int io_dtype, int state_dtype,
                          float q_scale, void* out, float* pseudo_v, float* log_gamma,
                          int32_t* err, tv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * tv_gdn_tree_verify_wy_lazy -- TreeWY verify with the previous round's commit fused in.
 *
 * Source: TreeWY abstract (only the accepted state is rebuilt on commit).  The previous
 * round's WY commit (see tv_gdn_commit, TV_MODE_WY) is applied to S0 while it is staged for
 * this round's contraction, saving that commit's separate pass over the state:
 *   S0[b] <- gamma_a S0[b] + sum_r Gamma_{a,path[r]} w_{path[r]} k_{path[r]}^T   (written back)
 * then this round is verified exactly as tv_gdn_tree_verify_wy.  The committed S0 and all
 * outputs equal tv_gdn_commit followed by tv_gdn_tree_verify_wy, bit for bit.
 *
 *   prev_path [B, Lmax], prev_len [B]         the previous round's accepted paths (1 <= len
 *                                             <= min(Lmax, prev_N, 16))
 *   prev_parents [B, prev_N]                  the previous round's trees (the path's links are
 *                                             checked)
 *   prev_pseudo_v [B, prev_N, H, dv] fp32, prev_log_gamma [B, prev_N, H] fp32, prev_k
 *   [B, prev_N, H, dk]                        the previous round's W, log(gamma) and keys; they
 *                                             may share memory with this round's pseudo_v /
 *                                             log_gamma outputs
 *   S0                                        in/out
 *   other arguments as tv_gdn_tree_verify_wy
 *   err [B]  0, TV_ERR_BAD_TREE, TV_ERR_BAD_PATH (previous path invalid: the sequence is
 *            skipped, S0[b] untouched) or TV_ERR_UNSUPPORTED as tv_gdn_tree_verify_wy
 * Supported: bf16 I/O and state, dk = dv = 128, N <= 240 (else TV_ERR_UNSUPPORTED).
 * ---------------------------------------------------------------------------------------- */
TV_API int tv_gdn_tree_verify_wy_lazy(const int32_t* prev_path, const int32_t* prev_len, int Lmax,
                                      const int32_t* prev_parents, int prev_N, const float* prev_pseudo_v,
                                      const float* prev_log_gamma, const void* prev_k, const void* q,
                                      const void* k, const void* v, const float* alpha, const float* beta,
                                      void* S0, const int32_t* parents, int B, int N, int H, int dk, int dv,
                                      int io_dtype, int state_dtype, float q_scale, void* out,
                                      float* pseudo_v, float* log_gamma, int32_t* err, tv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * tv_gdn_commit -- write the accepted node's state back into S_0.
 *
 * Source: qwen35-tree-spec §五 用途 2 and §七 Step 4 (restore the state of the last accepted
 * token, drop the other snapshots); TreeWY abstract (rebuild only the accepted state).
 * The accepted path of sequence b is accepted_path[b][0 .. accepted_len[b]-1]: path[0] a
 * root and path[r] a child of path[r-1]; 1 <= accepted_len[b] <= Lmax.
 *
 *   mode = TV_MODE_FORK:  S0[b] <- node_states[b, path[L-1]]
 *   mode = TV_MODE_WY:    S0[b] <- gamma_a S0[b] + sum_r Gamma_{a,path[r]} w_{path[r]} k_{path[r]}^T
 *                         (a = path[L-1]), from pseudo_v, log_gamma and k of the verify call
 *
 *   accepted_path [B, Lmax] int32   in
 *   accepted_len  [B] int32         in
 *   parents       [B, N] int32      in  (to check the path)
 *   node_states   [B,N,H,dv,dk] state_dtype in  (fork mode; may be NULL in WY mode)
 *   pseudo_v      [B,N,H,dv] fp32, log_gamma [B,N,H] fp32, k [B,N,H,dk] io_dtype
 *                                   in  (WY mode; may be NULL in fork mode)
 *   S0            [B,H,dv,dk] state_dtype   in/out
 *   err           [B] int32         out 0, TV_ERR_BAD_TREE or TV_ERR_BAD_PATH (S0[b] untouched)
 * ---------------------------------------------------------------------------------------- */
TV_API int tv_gdn_commit(int mode, const int32_t* accepted_path, const int32_t* accepted_len, int Lmax,
                  const int32_t* parents, const void* node_states, const float* pseudo_v,
                  const float* log_gamma, const void* k, void* S0, int B, int N, int H, int dk,
                  int dv, int io_dtype, int state_dtype, int32_t* err, tv_stream_t stream);

/* tv_gdn_commit_layers -- the commit of a whole stack of independent layers in one launch.
 * Every layer commits the same accepted paths (the path, its length and the parents are shared),
 * once the target has accepted them; the per-layer tensors lie back to back, layer first:
 *   S0 [layers, B, H, dv, dk]; fork: node_states [layers, B, N, H, dv, dk]; TreeWY:
 *   pseudo_v [layers, B, N, H, dv], log_gamma [layers, B, N, H], k [layers, B, N, H, dk].
 * The result for each layer equals tv_gdn_commit on that layer's slices.  err [B] reports the
 * shared path check.  layers >= 1; layers * B * H must fit in an int.  The pages have no
 * counterpart: layers are independent at commit time, so one launch serves them all. */
TV_API int tv_gdn_commit_layers(int mode, const int32_t* accepted_path, const int32_t* accepted_len, int Lmax,
                                const int32_t* parents, const void* node_states, const float* pseudo_v,
                                const float* log_gamma, const void* k, void* S0, int layers, int B, int N, int H,
                                int dk, int dv, int io_dtype, int state_dtype, int32_t* err, tv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * tv_gdn_tree_verify_fork_ws -- fork mode in two passes, with a workspace.
 *
 * Same results and layouts as tv_gdn_tree_verify_fork (outputs and every node's snapshot),
 * computed differently: a TreeWY pass (TreeWY abstract: one triangular solve gives every
 * node's output and pseudo-value w_i = beta_i (v_i - alpha_i S_parent k_i)) writes the outputs
 * and w into the workspace; then every snapshot is materialized from its parent's along the
 * depth-first walk, S_i = alpha_i S_parent + w_i k_i^T -- the gated delta update
 * (qwen35-tree-spec §四) with its S_parent k_i term taken from the solve.
 *
 *   workspace   device scratch of at least tv_gdn_fork_workspace_size(B, N, H, dv) bytes,
 *               16-byte aligned, owned by the caller; contents on entry are ignored.  Calls
 *               that share a workspace must not overlap in time.
 *   err [B]     0, TV_ERR_BAD_TREE, or TV_ERR_UNSUPPORTED (also when the sum over nodes of
 *               (depth + 1) exceeds 4096, the TreeWY limit)
 * ---------------------------------------------------------------------------------------- */
TV_API size_t tv_gdn_fork_workspace_size(int B, int N, int H, int dv);
TV_API int tv_gdn_tree_verify_fork_ws(const void* q, const void* k, const void* v, const float* alpha,
                                      const float* beta, const void* S0, const int32_t* parents, int B, int N,
                                      int H, int dk, int dv, int io_dtype, int state_dtype, float q_scale,
                                      void* out, void* node_states, void* workspace, size_t workspace_bytes,
                                      int32_t* err, tv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * tv_gdn_fork_materialize -- the snapshot pass of tv_gdn_tree_verify_fork_ws as a call of its
 * own, so that it can run on a second stream.
 *
 * Source: the gated delta update of qwen35-tree-spec §四, S_i = alpha_i S_parent + w_i k_i^T,
 * with w_i from a TreeWY verify (TreeWY abstract).  Every output of fork mode, and w, come from
 * tv_gdn_tree_verify_wy on the same q, k, v, alpha, beta, S0 and parents; this call writes
 * node_states exactly as tv_gdn_tree_verify_fork_ws does.  Nothing downstream of the outputs
 * needs the snapshots until the commit, so a caller may run this pass on its own stream (after
 * an event recorded behind the verify) while the next layer's verify runs on the first.
 *
 *   k, alpha, S0, parents   as tv_gdn_tree_verify_fork (read)
 *   pseudo_v     [B, N, H, dv] fp32, the w written by tv_gdn_tree_verify_wy (read)
 *   node_states  [B, N, H, dv, dk] state_dtype, 16-byte aligned (written)
 *   err [B]      in: the verify's per-sequence status -- a sequence with err != 0 is skipped
 *                and its snapshots are left untouched; out: unchanged for the others unless
 *                the depth-first schedule fails (TV_ERR_UNSUPPORTED)
 *   max_ctas_per_sm  0: as many resident CTAs per SM as fit; > 0: at most that many, which
 *                leaves registers and shared memory for kernels of other streams
 * Returns TV_ERR_INVALID_ARG for null or misaligned pointers, B, N or H < 1, or a negative
 * max_ctas_per_sm; TV_ERR_UNSUPPORTED for sizes or dtypes without a kernel.
 * The paper has no counterpart of the split: it is a scheduling choice of this library.
 * ---------------------------------------------------------------------------------------- */
TV_API int tv_gdn_fork_materialize(const void* k, const float* alpha, const void* S0, const int32_t* parents,
                                   const float* pseudo_v, int B, int N, int H, int dk, int dv, int io_dtype,
                                   int state_dtype, int max_ctas_per_sm, void* node_states, int32_t* err,
                                   tv_stream_t stream);

/* tv_gdn_fork_materialize_selective -- the same pass keeping only the selected snapshots
 * (qwen35-tree-spec §六, 选择性 Fork): node i keeps its snapshot iff confidence[b][i] <=
 * threshold, at slot s of node_states [B, capacity, H, dv, dk], slots numbered in node order,
 * exactly as tv_gdn_tree_verify_fork_selective; its outputs come from the preceding
 * tv_gdn_tree_verify_wy.  slot [B, N] int32 out (-1: no snapshot).  A sequence that keeps
 * more than capacity snapshots reports TV_ERR_CAPACITY in err and keeps none; a sequence the
 * verify rejected (err != 0 on entry) keeps none either (all its slots -1).  The commit is
 * tv_gdn_commit_selective.  Argument errors as tv_gdn_fork_materialize, plus a null
 * confidence or slot, a non-finite threshold, or capacity outside [1, N]. */
TV_API int tv_gdn_fork_materialize_selective(const void* k, const float* alpha, const void* S0,
                                             const int32_t* parents, const float* pseudo_v,
                                             const float* confidence, float threshold, int capacity, int B,
                                             int N, int H, int dk, int dv, int io_dtype, int state_dtype,
                                             int max_ctas_per_sm, void* node_states, int32_t* slot, int32_t* err,
                                             tv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * tv_gdn_tree_verify_fork_selective / tv_gdn_commit_selective -- fork mode with selective
 * snapshots.
 *
 * Source: qwen35-tree-spec §六, 选择性 Fork: a node whose draft confidence is above a
 * threshold (0.95 on the page) is processed without keeping a snapshot -- it is almost
 * surely accepted, so it needs no rollback point -- which cuts the snapshot count.
 *
 * Verify: as tv_gdn_tree_verify_fork, except that node i keeps its snapshot only if
 * confidence[b][i] <= threshold.  Kept snapshots are numbered 0, 1, ... in node order:
 *   confidence   [B, N] fp32                 in
 *   node_states  [B, capacity, H, dv, dk]    out snapshot of the node with slot s at index s
 *   slot         [B, N] int32                out snapshot index of each node, -1 if none (all
 *                                            -1 for a sequence that reports an error)
 *   err          [B] int32                   out 0, TV_ERR_BAD_TREE, TV_ERR_UNSUPPORTED, or
 *                                            TV_ERR_CAPACITY (more than capacity kept; the
 *                                            sequence is skipped)
 *   1 <= capacity <= N.
 * Commit: S0[b] <- state of the last accepted node, resumed from the deepest node of the
 * accepted path that kept a snapshot (S0[b] itself if none did) and replayed along the rest of
 * the path with k, v, alpha, beta of the verify call.  Path rules and err as tv_gdn_commit
 * (fork mode).
 * ---------------------------------------------------------------------------------------- */
TV_API int tv_gdn_tree_verify_fork_selective(const void* q, const void* k, const void* v, const float* alpha,
                                             const float* beta, const void* S0, const int32_t* parents,
                                             const float* confidence, float threshold, int capacity, int B,
                                             int N, int H, int dk, int dv, int io_dtype, int state_dtype,
                                             float q_scale, void* out, void* node_states, int32_t* slot,
                                             int32_t* err, tv_stream_t stream);
TV_API int tv_gdn_commit_selective(const int32_t* accepted_path, const int32_t* accepted_len, int Lmax,
                                   const int32_t* parents, const void* node_states, const int32_t* slot,
                                   int capacity, const void* k, const void* v, const float* alpha,
                                   const float* beta, void* S0, int B, int N, int H, int dk, int dv,
                                   int io_dtype, int state_dtype, int32_t* err, tv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * tv_tree_attn -- tree-masked GQA attention over a paged KV prefix.
 *
 * Source: handbook chapter 树形草稿与 EAGLE, §实现, forward_with_mask: q and k of the new
 * nodes are rotated (RoPE) at position prefix_len + depth; keys/values are the cached prefix
 * followed by the nodes'; node i sees the whole prefix, its ancestors and itself; query head
 * h reads KV head h / (Hq / Hkv); softmax scale sm_scale (pass 1/sqrt(hd) for the default).
 * RoPE reading: rotate-half pairs (x_c, x_{c+hd/2}), angle pos * rope_theta^(-2c/hd), over the
 * full head dim.  Cached prefix keys are stored already rotated.
 *
 * The call first writes each node's rotated key and its value into the cache at logical slot
 * prefix_len[b] + i, then attends over logical slots [0, prefix_len[b] + N).
 *
 *   q            [B, N, Hq, hd]  bf16     in  (not rotated)
 *   k_new, v_new [B, N, Hkv, hd] bf16     in  (k not rotated)
 *   k_cache, v_cache [num_blocks, Hkv, block_size, hd] bf16  in/out
 *   block_table  [B, max_blocks] int32    in  logical slot s of sequence b lives in block
 *                                         block_table[b][s / block_size], row s % block_size
 *   prefix_len   [B] int32                in
 *   parents      [B, N] int32             in
 *   out          [B, N, Hq, hd] bf16      out
 *   workspace    device scratch of at least tv_tree_attn_workspace_size(...) bytes, 256-byte
 *                aligned, owned by the caller; contents on entry are ignored.  Calls that
 *                share a workspace must not overlap in time.
 *   err          [B] int32                out 0, TV_ERR_BAD_TREE, TV_ERR_CAPACITY
 *                                         (prefix_len + N > max_blocks * block_size or
 *                                         prefix_len < 0), TV_ERR_BAD_BLOCK, or TV_ERR_TIMEOUT
 *                                         (a bounded device wait gave up; that sequence's
 *                                         outputs are then unspecified)
 * Supported: hd in {64, 128, 256}; block_size = 16; Hq a multiple of Hkv; B <= 65535.
 * ---------------------------------------------------------------------------------------- */
TV_API size_t tv_tree_attn_workspace_size(int B, int N, int Hq, int Hkv, int hd, int max_blocks,
                                   int block_size);

TV_API int tv_tree_attn(const void* q, const void* k_new, const void* v_new, void* k_cache,
                 void* v_cache, int num_blocks, const int32_t* block_table, int max_blocks,
                 const int32_t* prefix_len, const int32_t* parents, int B, int N, int Hq,
                 int Hkv, int hd, int block_size, float rope_theta, float sm_scale, void* out,
                 void* workspace, size_t workspace_bytes, int32_t* err, tv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * tv_tree_attn_static -- tv_tree_attn without a workspace and without any allocation.
 *
 * The pages have no counterpart: this is a deployment variant of tv_tree_attn, for callers
 * that cannot hand the library a workspace (e.g. code that must not allocate).  Arguments,
 * layouts, results and the err codes are those of tv_tree_attn; the workspace is replaced by
 * one device array of TV_STATIC_SCRATCH_BYTES (64 MiB) owned by the library.
 *
 *  - Size limit: when tv_tree_attn_workspace_size(B, N, Hq, Hkv, hd, max_blocks, block_size)
 *    exceeds TV_STATIC_SCRATCH_BYTES the call returns TV_ERR_SCRATCH before any CUDA call
 *    and launches nothing; use tv_tree_attn with a workspace for such sizes.
 *  - Argument errors: every host-side check of tv_tree_attn (null or misaligned pointers,
 *    sizes) runs before any CUDA call, as does the size limit below.
 *  - Set-up: the first call in each CUDA context looks up the array's device address
 *    (cudaGetSymbolAddress; a failure returns TV_ERR_CUDA) and caches it with that context.
 *    That lookup may load a module, so make the first call on each device in set-up code,
 *    before any stream capture.  A call made in a new context of the device (e.g. after
 *    cudaDeviceReset) looks the address up again: the old one died with the old context.
 *  - Shared state: the scratch is one array per device for the whole process.  Its contents
 *    persist between calls; nothing in it has to start at zero (every call writes each
 *    scratch entry it reads).  Two calls whose execution overlaps on the same device (other
 *    streams, other host threads) race on it: serialise them, e.g. on one stream.
 * ---------------------------------------------------------------------------------------- */
TV_API int tv_tree_attn_static(const void* q, const void* k_new, const void* v_new, void* k_cache,
                        void* v_cache, int num_blocks, const int32_t* block_table, int max_blocks,
                        const int32_t* prefix_len, const int32_t* parents, int B, int N, int Hq,
                        int Hkv, int hd, int block_size, float rope_theta, float sm_scale,
                        void* out, int32_t* err, tv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * tv_kv_compact -- keep the accepted path's KV, in place.
 *
 * Source: handbook chapter 树形草稿与 EAGLE, note after the listing (the accepted nodes' KV
 * was computed at the right positions during verification and is moved to the sequence's
 * contiguous slots; rejected slots become void) and qwen35-tree-spec §七 Step 4.
 * For r < L = accepted_len[b]: logical slot prefix_len[b] + r receives what logical slot
 * prefix_len[b] + path[r] held before the call (every source is read before any write), for
 * K and V and all KV heads.  Slots at or past the new length are left as they are.
 *
 *   k_cache, v_cache [num_blocks, Hkv, block_size, hd] bf16   in/out
 *   block_table [B, max_blocks] int32, prefix_len [B] int32, parents [B, N] int32   in
 *   accepted_path [B, Lmax] int32, accepted_len [B] int32                            in
 *   slot_map    [B, Lmax] int32   out physical source slot (block * block_size + row) of
 *                                 each kept entry, -1 for r >= L
 *   new_len     [B] int32         out prefix_len + L (prefix_len on error)
 *   err         [B] int32         out 0, TV_ERR_BAD_TREE, TV_ERR_BAD_PATH, TV_ERR_CAPACITY
 *                                 or TV_ERR_BAD_BLOCK
 * Precondition, checked: the table entries of the logical blocks that hold slots prefix_len ..
 * prefix_len + N - 1 (the window every source and destination lies in) are distinct physical
 * blocks.  Were two of them the same block, a store could overwrite a source before it is read;
 * such a sequence reports TV_ERR_BAD_BLOCK and is skipped.
 * Supported: hd in {64, 128, 256}; block_size = 16.
 * ---------------------------------------------------------------------------------------- */
TV_API int tv_kv_compact(void* k_cache, void* v_cache, int num_blocks, const int32_t* block_table,
                  int max_blocks, const int32_t* prefix_len, const int32_t* parents, int N,
                  const int32_t* accepted_path, const int32_t* accepted_len, int Lmax, int B,
                  int Hkv, int hd, int block_size, int32_t* slot_map, int32_t* new_len,
                  int32_t* err, tv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * tv_kv_compact_remap -- keep the accepted path's KV, exchanging whole blocks of the block
 * table where that replaces moving them.
 *
 * Source: handbook chapter 树形草稿与 EAGLE, note after the listing (the accepted nodes' slots
 * are compacted to the sequence's positions, or only the block table is updated).  Reading,
 * per sequence with P = prefix_len[b], L = accepted_len[b], block size 16:
 *  - a logical block m with 16 m >= P that holds kept entries (P + r for r < L), all of which
 *    come from logical slot P + r + 16 j for one j >= 1, takes block m + j's physical block:
 *    entries m and m + j of the table row are exchanged, in ascending m;
 *  - every other kept entry r is moved: physical slot (new row, P + r) receives what physical
 *    slot (old row, P + path[r]) held before the call.  Every source is read before any
 *    write; an entry already in place is not written.
 * Read through block_table_out, logical slots [0, P + L) then hold what tv_kv_compact leaves
 * in them read through block_table.  The new row is a permutation of the old one; entries of
 * blocks holding prefix slots are unchanged.  Slots at or past the new length are void.
 *
 *   k_cache, v_cache [num_blocks, Hkv, block_size, hd] bf16     in/out
 *   block_table     [B, max_blocks] int32   in   the rows before the call
 *   block_table_out [B, max_blocks] int32   out  the rows after the exchanges (a copy of the
 *                                                row for a sequence with an error); must not
 *                                                overlap block_table (TV_ERR_INVALID_ARG)
 *   prefix_len, parents, accepted_path, accepted_len, slot_map, new_len, err: as for
 *                                                tv_kv_compact (slot_map under the old rows)
 *   remapped        [B] int32               out  exchanges made (0 on error)
 * Precondition, checked as for tv_kv_compact: the window's table entries are distinct (an
 * exchange of two entries naming one block would lose none but move data twice);
 * TV_ERR_BAD_BLOCK otherwise, the row copied unchanged.
 * Supported: hd in {64, 128, 256}; block_size = 16; N <= TV_MAX_NODES.
 * ---------------------------------------------------------------------------------------- */
TV_API int tv_kv_compact_remap(void* k_cache, void* v_cache, int num_blocks, const int32_t* block_table,
                        int32_t* block_table_out, int max_blocks, const int32_t* prefix_len,
                        const int32_t* parents, int N, const int32_t* accepted_path,
                        const int32_t* accepted_len, int Lmax, int B, int Hkv, int hd, int block_size,
                        int32_t* slot_map, int32_t* new_len, int32_t* remapped, int32_t* err,
                        tv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * tv_accept_walk -- greedy acceptance of B draft trees, on the device.
 *
 * Source: handbook chapter 树形草稿与 EAGLE, §实现, tree_speculative_generate: from node 0,
 * while the target model's token at the current node equals the draft token of one of its
 * children, step to the lowest-numbered such child; the target's token at the last accepted
 * node is the next token.  The walk also stops once Lmax nodes are accepted.  Its output feeds
 * tv_gdn_commit and tv_kv_compact without a host round trip.
 *
 *   parents        [B, N] int32   in
 *   draft_tokens   [B, N] int32   in  token proposed at each node
 *   target_tokens  [B, N] int32   in  token the target model chose at each node (its argmax)
 *   accepted_path  [B, Lmax] int32 out path[0] = 0, path[r] a child of path[r-1]; -1 past the
 *                                      length
 *   accepted_len   [B] int32      out 1 <= len <= Lmax (0 on error)
 *   next_token     [B] int32      out target_tokens[b][path[len-1]] (-1 on error)
 *   err            [B] int32      out 0 or TV_ERR_BAD_TREE
 * ---------------------------------------------------------------------------------------- */
TV_API int tv_accept_walk(const int32_t* parents, const int32_t* draft_tokens, const int32_t* target_tokens,
                          int B, int N, int Lmax, int32_t* accepted_path, int32_t* accepted_len,
                          int32_t* next_token, int32_t* err, tv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * tv_test_bounded_wait -- test support for the bounded device waits.
 *
 * The pages have no counterpart: this checks a property of the library.  Every wait of the
 * tensor-core kernels on a shared-memory mbarrier (copies landed, MMAs done) gives up after a
 * bounded number of polls, and the kernel then reports TV_ERR_TIMEOUT in err[b] and returns.
 * This call launches one thread that runs that same wait on a barrier nothing arrives on (no
 * copy or MMA is in flight), so a test can make it run out:
 *   max_polls   polls before giving up; 0 = the limit the library's kernels use
 *   arrive      nonzero: the thread arrives on the barrier first, so the wait succeeds
 *   status      [1] int32 out   TV_OK or TV_ERR_TIMEOUT
 *   elapsed_ns  [1] int64 out   device time the wait took (the %globaltimer clock)
 * Returns TV_ERR_INVALID_ARG for a null or misaligned pointer.
 * ---------------------------------------------------------------------------------------- */
TV_API int tv_test_bounded_wait(unsigned max_polls, int arrive, int32_t* status, int64_t* elapsed_ns,
                                tv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TV_H_ */
