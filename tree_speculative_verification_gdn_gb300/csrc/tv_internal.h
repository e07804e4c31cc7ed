// Host-side launchers of the CUDA kernels; called by the C ABI in tv_api.cu after the
// arguments have been checked.  Each returns the CUDA error of its launch(es).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "tv.h"

namespace tv {

int device_sm_count();
// TV_OK for cudaSuccess; otherwise records e for tv_last_cuda_error and returns TV_ERR_CUDA.
int cuda_status_of(cudaError_t e);

struct GdnArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* alpha;
  const float* beta;
  const void* S0;
  const int32_t* parents;
  int B, N, H, dk, dv;
  int io, state;
  float q_scale;
  void* out;
  int32_t* err;
};

cudaError_t launch_tree_prepare(const int32_t* parents, int B, int N, int32_t* depth, uint32_t* mask_bits,
                                int32_t* paths, int path_cap, int32_t* max_depth, int32_t* err, cudaStream_t s);

// Selective fork: a node keeps its snapshot only if its confidence is at most the threshold;
// kept snapshots take slots 0, 1, ... in node order.  confidence == nullptr: every node keeps
// its snapshot, at slot = node, and capacity = N.
struct ForkSelect {
  const float* confidence;  // [B, N] or nullptr
  float threshold;
  int capacity;             // snapshot slots per sequence in node_states [B, capacity, H, dv, dk]
  int32_t* slot;            // [B, N] out (slot or -1), or nullptr
};
cudaError_t launch_gdn_fork(const GdnArgs& a, void* node_states, const ForkSelect& sel, cudaStream_t s);
// Two-pass fork: the TreeWY pass writes every output and w (pseudo_v, log_gamma: caller scratch),
// then the walk materializes every snapshot from its parent's, S_i = alpha_i S_p + w_i k_i^T.
cudaError_t launch_gdn_fork_two_pass(const GdnArgs& a, void* node_states, float* pseudo_v, float* log_gamma,
                                     cudaStream_t s);
// The second pass alone (after a TreeWY verify of the same inputs wrote pseudo_v and err), every
// snapshot or (sel.confidence set) the selected ones; at most max_ctas_per_sm resident CTAs per
// SM when > 0.
cudaError_t launch_gdn_fork_materialize(const GdnArgs& a, void* node_states, const float* pseudo_v,
                                        const ForkSelect& sel, int max_ctas_per_sm, cudaStream_t s);

// TreeWY verify: tcgen05 kernel for bf16 I/O and state with dk = dv = 128, CUDA-core kernel
// for every other supported shape.
cudaError_t launch_gdn_wy(const GdnArgs& a, float* pseudo_v, float* log_gamma, cudaStream_t s);
bool gdn_wy_tc_supported(const GdnArgs& a);
// Lazy commit: the previous round's TreeWY commit applied to S_0 inside this round's verify.
// path == nullptr: no pending commit.
constexpr int kLazyMaxLen = 16;  // longest previous accepted path the fused commit takes
struct WyLazy {
  const int32_t* path;      // [B, Lmax] previous round's accepted paths
  const int32_t* len;       // [B]
  int Lmax;
  int Np;                   // previous round's nodes per tree
  const int32_t* parents;   // [B, Np] previous round's trees
  const float* pseudo_v;    // [B, Np, H, dv] previous round's W
  const float* log_gamma;   // [B, Np, H]
  const void* k;            // [B, Np, H, dk] previous round's keys
};
cudaError_t launch_gdn_wy_tc(const GdnArgs& a, float* pseudo_v, float* log_gamma, const WyLazy& lz,
                             cudaStream_t s);
bool gdn_wy_lazy_fits(int N);  // shared memory of the fused-commit kernel fits for N nodes
cudaError_t launch_gdn_wy_simt(const GdnArgs& a, float* pseudo_v, float* log_gamma, cudaStream_t s);

struct CommitArgs {
  int mode;
  const int32_t* path;
  const int32_t* path_len;
  int Lmax;
  const int32_t* parents;
  const void* node_states;
  const float* pseudo_v;
  const float* log_gamma;
  const void* k;
  void* S0;
  int B, N, H, dk, dv, io, state;
  int32_t* err;
  int layers = 1;  // S0, node_states, pseudo_v, log_gamma, k: [layers, B, ...] back to back; the
                   // path, its length, parents and err are shared by the layers
};
cudaError_t launch_gdn_commit(const CommitArgs& a, cudaStream_t s);
// Commit after a selective fork: resume from the deepest accepted node that kept a snapshot
// (or S_0) and replay the rest of the path with its inputs.
struct ReplayArgs {
  const int32_t* slot;  // [B, N] from the selective fork
  int capacity;
  const void* v;
  const float* alpha;
  const float* beta;
};
cudaError_t launch_gdn_commit_replay(const CommitArgs& a, const ReplayArgs& r, cudaStream_t s);

struct AttnArgs {
  const void* q;
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  int num_blocks;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* prefix_len;
  const int32_t* parents;
  int B, N, Hq, Hkv, hd, block_size;
  float rope_theta, sm_scale;
  void* out;
  int32_t* err;
};
size_t attn_workspace_size(int B, int N, int Hq, int Hkv, int hd, int max_blocks, int block_size);
// Host-side argument checks of tv_tree_attn other than the workspace: TV_OK or the status the
// call returns.  Makes no CUDA call.
int tree_attn_check_args(const void* q, const void* k_new, const void* v_new, const void* k_cache,
                         const void* v_cache, int num_blocks, const int32_t* block_table, int max_blocks,
                         const int32_t* prefix_len, const int32_t* parents, int B, int N, int Hq, int Hkv, int hd,
                         int block_size, float rope_theta, float sm_scale, const void* out, const int32_t* err);
// Split-KV partials on the tensor cores (head dim 128 or 256, Hq/Hkv dividing 128); the
// CUDA-core partial kernel covers every other supported shape.
bool attn_tc_supported(const AttnArgs& a);
// Tiles of 128 query rows per (sequence, KV head): one runs on single CTAs, more on CTA pairs.
int attn_tc_row_tiles(const AttnArgs& a);
cudaError_t launch_attn_partial_tc(const AttnArgs& a, const void* qrot, float* ml, float* acc, int chunk,
                                   int nsplit, cudaStream_t s);
cudaError_t launch_tree_attn(const AttnArgs& a, void* workspace, size_t workspace_bytes,
                             cudaStream_t s);

struct CompactArgs {
  void* k_cache;
  void* v_cache;
  int num_blocks;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* prefix_len;
  const int32_t* parents;
  int N;
  const int32_t* path;
  const int32_t* path_len;
  int Lmax, B, Hkv, hd, block_size;
  int32_t* slot_map;
  int32_t* new_len;
  int32_t* err;
  int32_t* table_out;   // block-table form only: the row after the exchanges
  int32_t* remapped;    // block-table form only: exchanges per sequence
};
cudaError_t launch_kv_compact(const CompactArgs& a, cudaStream_t s);
cudaError_t launch_kv_compact_remap(const CompactArgs& a, cudaStream_t s);

struct AcceptArgs {
  const int32_t* parents;
  const int32_t* draft;
  const int32_t* target;
  int B, N, Lmax;
  int32_t* path;
  int32_t* len;
  int32_t* next_token;
  int32_t* err;
};
cudaError_t launch_accept_walk(const AcceptArgs& a, cudaStream_t s);

}  // namespace tv
