// C ABI entry points (declared in include/tv.h): host-side argument checks, then the
// launchers of the individual kernels.  Nothing here allocates device memory.
#include <math.h>
#include <stdint.h>

#include "tv.h"
#include "tv_internal.h"

namespace tv {

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) cached[dev] = n;
  return n;
}

}  // namespace tv

namespace {

thread_local int g_last_cuda = 0;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return TV_OK;
  g_last_cuda = static_cast<int>(e);
  return TV_ERR_CUDA;
}

}  // namespace

int tv::cuda_status_of(cudaError_t e) { return cuda_status(e); }

namespace {

bool a16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool a4(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool dim_ok(int d) { return d == 64 || d == 128; }

// (io, state) pairs with a kernel: (F32,F32), (BF16,BF16), (BF16,F32).
int gdn_dtypes(int io, int state) {
  if ((io == TV_F32 && state == TV_F32) || (io == TV_BF16 && state == TV_BF16) ||
      (io == TV_BF16 && state == TV_F32))
    return TV_OK;
  if ((io != TV_F32 && io != TV_BF16) || (state != TV_F32 && state != TV_BF16)) return TV_ERR_INVALID_ARG;
  return TV_ERR_UNSUPPORTED;
}

int gdn_common(const void* q, const void* k, const void* v, const float* alpha, const float* beta,
               const void* S0, const int32_t* parents, int B, int N, int H, int dk, int dv, int io,
               int state, float q_scale, const void* out, const int32_t* err) {
  if (!a16(q) || !a16(k) || !a4(v) || !a4(alpha) || !a4(beta) || !a16(S0) || !a4(parents) || !a4(out) ||
      !a4(err))
    return TV_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || H < 1 || !isfinite(q_scale)) return TV_ERR_INVALID_ARG;
  if (N > TV_MAX_NODES || !dim_ok(dk) || !dim_ok(dv)) return TV_ERR_UNSUPPORTED;
  return gdn_dtypes(io, state);
}

}  // namespace

extern "C" {

const char* tv_status_string(int status) {
  switch (status) {
    case TV_OK: return "ok";
    case TV_ERR_INVALID_ARG: return "invalid argument";
    case TV_ERR_BAD_TREE: return "malformed tree (parents[i] must be -1 or an earlier node)";
    case TV_ERR_BAD_PATH: return "accepted path is not a root-to-node path";
    case TV_ERR_UNSUPPORTED: return "unsupported size or dtype";
    case TV_ERR_CUDA: return "CUDA launch error";
    case TV_ERR_TIMEOUT: return "device wait timed out";
    case TV_ERR_CAPACITY: return "block table too short for prefix_len + N slots";
    case TV_ERR_BAD_BLOCK: return "block-table entry outside the cache";
    case TV_ERR_SCRATCH: return "request needs more than the static scratch of TV_STATIC_SCRATCH_BYTES";
    default: return "unknown status";
  }
}

int tv_last_cuda_error(void) { return g_last_cuda; }

int tv_version(void) { return 100; }

int tv_tree_prepare(const int32_t* parents, int B, int N, int32_t* depth, uint32_t* mask_bits, int32_t* paths,
                    int path_cap, int32_t* max_depth, int32_t* err, tv_stream_t stream) {
  if (!a4(parents) || !a4(depth) || !a4(mask_bits) || !a4(err) || B < 1 || N < 1) return TV_ERR_INVALID_ARG;
  if ((paths != nullptr && (!a4(paths) || path_cap < 1)) || (max_depth != nullptr && !a4(max_depth)))
    return TV_ERR_INVALID_ARG;
  if (N > TV_MAX_NODES) return TV_ERR_UNSUPPORTED;
  return cuda_status(tv::launch_tree_prepare(parents, B, N, depth, mask_bits, paths, paths ? path_cap : 0, max_depth,
                                             err, stream));
}

int tv_gdn_tree_verify_fork(const void* q, const void* k, const void* v, const float* alpha,
                            const float* beta, const void* S0, const int32_t* parents, int B, int N,
                            int H, int dk, int dv, int io_dtype, int state_dtype, float q_scale,
                            void* out, void* node_states, int32_t* err, tv_stream_t stream) {
  int st = gdn_common(q, k, v, alpha, beta, S0, parents, B, N, H, dk, dv, io_dtype, state_dtype, q_scale,
                      out, err);
  if (st != TV_OK) return st;
  if (!a16(node_states)) return TV_ERR_INVALID_ARG;
  tv::GdnArgs a{q, k, v, alpha, beta, S0, parents, B, N, H, dk, dv, io_dtype, state_dtype, q_scale, out, err};
  const tv::ForkSelect all{nullptr, 0.f, N, nullptr};
  return cuda_status(tv::launch_gdn_fork(a, node_states, all, stream));
}

size_t tv_gdn_fork_workspace_size(int B, int N, int H, int dv) {
  if (B < 1 || N < 1 || H < 1 || dv < 1) return 0;
  const size_t pv = ((size_t)B * N * H * dv * 4 + 255) & ~(size_t)255;
  const size_t lg = ((size_t)B * N * H * 4 + 255) & ~(size_t)255;
  return pv + lg;
}

int tv_gdn_tree_verify_fork_ws(const void* q, const void* k, const void* v, const float* alpha, const float* beta,
                               const void* S0, const int32_t* parents, int B, int N, int H, int dk, int dv,
                               int io_dtype, int state_dtype, float q_scale, void* out, void* node_states,
                               void* workspace, size_t workspace_bytes, int32_t* err, tv_stream_t stream) {
  int st = gdn_common(q, k, v, alpha, beta, S0, parents, B, N, H, dk, dv, io_dtype, state_dtype, q_scale,
                      out, err);
  if (st != TV_OK) return st;
  if (!a16(node_states) || !a16(workspace)) return TV_ERR_INVALID_ARG;
  if (workspace_bytes < tv_gdn_fork_workspace_size(B, N, H, dv)) return TV_ERR_INVALID_ARG;
  float* pv = static_cast<float*>(workspace);
  float* lg = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                       (((size_t)B * N * H * dv * 4 + 255) & ~(size_t)255));
  tv::GdnArgs a{q, k, v, alpha, beta, S0, parents, B, N, H, dk, dv, io_dtype, state_dtype, q_scale, out, err};
  return cuda_status(tv::launch_gdn_fork_two_pass(a, node_states, pv, lg, stream));
}

int tv_gdn_fork_materialize(const void* k, const float* alpha, const void* S0, const int32_t* parents,
                            const float* pseudo_v, int B, int N, int H, int dk, int dv, int io_dtype,
                            int state_dtype, int max_ctas_per_sm, void* node_states, int32_t* err,
                            tv_stream_t stream) {
  if (!a16(k) || !a4(alpha) || !a16(S0) || !a4(parents) || !a16(pseudo_v) || !a16(node_states) || !a4(err))
    return TV_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || H < 1 || max_ctas_per_sm < 0) return TV_ERR_INVALID_ARG;
  if (N > TV_MAX_NODES || !dim_ok(dk) || !dim_ok(dv)) return TV_ERR_UNSUPPORTED;
  const int st = gdn_dtypes(io_dtype, state_dtype);
  if (st != TV_OK) return st;
  // q, v, beta and out are not read by this pass.
  tv::GdnArgs a{nullptr, k, nullptr, alpha, nullptr, S0, parents, B, N, H, dk, dv, io_dtype, state_dtype, 1.f,
                nullptr, err};
  const tv::ForkSelect all{nullptr, 0.f, N, nullptr};
  return cuda_status(tv::launch_gdn_fork_materialize(a, node_states, pseudo_v, all, max_ctas_per_sm, stream));
}

int tv_gdn_fork_materialize_selective(const void* k, const float* alpha, const void* S0, const int32_t* parents,
                                      const float* pseudo_v, const float* confidence, float threshold, int capacity,
                                      int B, int N, int H, int dk, int dv, int io_dtype, int state_dtype,
                                      int max_ctas_per_sm, void* node_states, int32_t* slot, int32_t* err,
                                      tv_stream_t stream) {
  if (!a16(k) || !a4(alpha) || !a16(S0) || !a4(parents) || !a16(pseudo_v) || !a16(node_states) || !a4(err) ||
      !a4(confidence) || !a4(slot))
    return TV_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || H < 1 || max_ctas_per_sm < 0 || !isfinite(threshold) || capacity < 1 || capacity > N)
    return TV_ERR_INVALID_ARG;
  if (N > TV_MAX_NODES || !dim_ok(dk) || !dim_ok(dv)) return TV_ERR_UNSUPPORTED;
  const int st = gdn_dtypes(io_dtype, state_dtype);
  if (st != TV_OK) return st;
  tv::GdnArgs a{nullptr, k, nullptr, alpha, nullptr, S0, parents, B, N, H, dk, dv, io_dtype, state_dtype, 1.f,
                nullptr, err};
  const tv::ForkSelect sel{confidence, threshold, capacity, slot};
  return cuda_status(tv::launch_gdn_fork_materialize(a, node_states, pseudo_v, sel, max_ctas_per_sm, stream));
}

int tv_gdn_tree_verify_fork_selective(const void* q, const void* k, const void* v, const float* alpha,
                                      const float* beta, const void* S0, const int32_t* parents,
                                      const float* confidence, float threshold, int capacity, int B, int N,
                                      int H, int dk, int dv, int io_dtype, int state_dtype, float q_scale,
                                      void* out, void* node_states, int32_t* slot, int32_t* err,
                                      tv_stream_t stream) {
  int st = gdn_common(q, k, v, alpha, beta, S0, parents, B, N, H, dk, dv, io_dtype, state_dtype, q_scale,
                      out, err);
  if (st != TV_OK) return st;
  if (!a4(confidence) || !a4(slot) || !isfinite(threshold) || capacity < 1 || capacity > N)
    return TV_ERR_INVALID_ARG;
  if (!a16(node_states)) return TV_ERR_INVALID_ARG;
  tv::GdnArgs a{q, k, v, alpha, beta, S0, parents, B, N, H, dk, dv, io_dtype, state_dtype, q_scale, out, err};
  const tv::ForkSelect sel{confidence, threshold, capacity, slot};
  return cuda_status(tv::launch_gdn_fork(a, node_states, sel, stream));
}

int tv_gdn_tree_verify_wy(const void* q, const void* k, const void* v, const float* alpha,
                          const float* beta, const void* S0, const int32_t* parents, int B, int N,
                          int H, int dk, int dv, int io_dtype, int state_dtype, float q_scale, void* out,
                          float* pseudo_v, float* log_gamma, int32_t* err, tv_stream_t stream) {
  int st = gdn_common(q, k, v, alpha, beta, S0, parents, B, N, H, dk, dv, io_dtype, state_dtype, q_scale,
                      out, err);
  if (st != TV_OK) return st;
  if (!a4(pseudo_v) || !a4(log_gamma)) return TV_ERR_INVALID_ARG;
  tv::GdnArgs a{q, k, v, alpha, beta, S0, parents, B, N, H, dk, dv, io_dtype, state_dtype, q_scale, out, err};
  return cuda_status(tv::launch_gdn_wy(a, pseudo_v, log_gamma, stream));
}

int tv_gdn_tree_verify_wy_lazy(const int32_t* prev_path, const int32_t* prev_len, int Lmax,
                               const int32_t* prev_parents, int prev_N, const float* prev_pseudo_v,
                               const float* prev_log_gamma, const void* prev_k, const void* q, const void* k,
                               const void* v, const float* alpha, const float* beta, void* S0,
                               const int32_t* parents, int B, int N, int H, int dk, int dv, int io_dtype,
                               int state_dtype, float q_scale, void* out, float* pseudo_v, float* log_gamma,
                               int32_t* err, tv_stream_t stream) {
  int st = gdn_common(q, k, v, alpha, beta, S0, parents, B, N, H, dk, dv, io_dtype, state_dtype, q_scale,
                      out, err);
  if (st != TV_OK) return st;
  if (!a4(pseudo_v) || !a4(log_gamma) || !a4(prev_path) || !a4(prev_len) || !a4(prev_parents) ||
      !a4(prev_pseudo_v) || !a4(prev_log_gamma) || !a16(prev_k) || Lmax < 1 || prev_N < 1)
    return TV_ERR_INVALID_ARG;
  if (prev_N > TV_MAX_NODES) return TV_ERR_UNSUPPORTED;
  tv::GdnArgs a{q, k, v, alpha, beta, S0, parents, B, N, H, dk, dv, io_dtype, state_dtype, q_scale, out, err};
  if (!tv::gdn_wy_tc_supported(a) || !tv::gdn_wy_lazy_fits(N)) return TV_ERR_UNSUPPORTED;
  const tv::WyLazy lz{prev_path, prev_len, Lmax, prev_N, prev_parents, prev_pseudo_v, prev_log_gamma, prev_k};
  return cuda_status(tv::launch_gdn_wy_tc(a, pseudo_v, log_gamma, lz, stream));
}

int tv_gdn_commit_layers(int mode, const int32_t* accepted_path, const int32_t* accepted_len, int Lmax,
                         const int32_t* parents, const void* node_states, const float* pseudo_v,
                         const float* log_gamma, const void* k, void* S0, int layers, int B, int N, int H, int dk,
                         int dv, int io_dtype, int state_dtype, int32_t* err, tv_stream_t stream) {
  if (!a4(accepted_path) || !a4(accepted_len) || !a4(parents) || !a16(S0) || !a4(err)) return TV_ERR_INVALID_ARG;
  if (layers < 1 || B < 1 || N < 1 || H < 1 || Lmax < 1) return TV_ERR_INVALID_ARG;
  if ((long long)layers * B * H > 0x7fffffffLL) return TV_ERR_UNSUPPORTED;
  if (mode == TV_MODE_FORK) {
    if (!a16(node_states)) return TV_ERR_INVALID_ARG;
  } else if (mode == TV_MODE_WY) {
    if (!a4(pseudo_v) || !a4(log_gamma) || !a16(k)) return TV_ERR_INVALID_ARG;
  } else {
    return TV_ERR_INVALID_ARG;
  }
  if (N > TV_MAX_NODES || !dim_ok(dk) || !dim_ok(dv)) return TV_ERR_UNSUPPORTED;
  int st = gdn_dtypes(io_dtype, state_dtype);
  if (st != TV_OK) return st;
  tv::CommitArgs a{mode, accepted_path, accepted_len, Lmax, parents, node_states, pseudo_v, log_gamma, k,
                   S0, B, N, H, dk, dv, io_dtype, state_dtype, err};
  a.layers = layers;
  if (mode == TV_MODE_FORK) a.pseudo_v = nullptr, a.log_gamma = nullptr, a.k = nullptr;
  else a.node_states = nullptr;
  return cuda_status(tv::launch_gdn_commit(a, stream));
}

int tv_gdn_commit(int mode, const int32_t* accepted_path, const int32_t* accepted_len, int Lmax,
                  const int32_t* parents, const void* node_states, const float* pseudo_v,
                  const float* log_gamma, const void* k, void* S0, int B, int N, int H, int dk, int dv,
                  int io_dtype, int state_dtype, int32_t* err, tv_stream_t stream) {
  return tv_gdn_commit_layers(mode, accepted_path, accepted_len, Lmax, parents, node_states, pseudo_v, log_gamma, k,
                              S0, 1, B, N, H, dk, dv, io_dtype, state_dtype, err, stream);
}

int tv_gdn_commit_selective(const int32_t* accepted_path, const int32_t* accepted_len, int Lmax,
                            const int32_t* parents, const void* node_states, const int32_t* slot, int capacity,
                            const void* k, const void* v, const float* alpha, const float* beta, void* S0, int B,
                            int N, int H, int dk, int dv, int io_dtype, int state_dtype, int32_t* err,
                            tv_stream_t stream) {
  if (!a4(accepted_path) || !a4(accepted_len) || !a4(parents) || !a16(S0) || !a4(err) || !a16(node_states) ||
      !a4(slot) || !a16(k) || !a4(v) || !a4(alpha) || !a4(beta))
    return TV_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || H < 1 || Lmax < 1 || capacity < 1 || capacity > N) return TV_ERR_INVALID_ARG;
  if (N > TV_MAX_NODES || !dim_ok(dk) || !dim_ok(dv)) return TV_ERR_UNSUPPORTED;
  int st = gdn_dtypes(io_dtype, state_dtype);
  if (st != TV_OK) return st;
  tv::CommitArgs a{TV_MODE_FORK, accepted_path, accepted_len, Lmax, parents, node_states, nullptr, nullptr, k,
                   S0, B, N, H, dk, dv, io_dtype, state_dtype, err};
  const tv::ReplayArgs r{slot, capacity, v, alpha, beta};
  return cuda_status(tv::launch_gdn_commit_replay(a, r, stream));
}

size_t tv_tree_attn_workspace_size(int B, int N, int Hq, int Hkv, int hd, int max_blocks, int block_size) {
  if (B < 1 || N < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || hd < 1 || max_blocks < 1 || block_size < 1) return 0;
  return tv::attn_workspace_size(B, N, Hq, Hkv, hd, max_blocks, block_size);
}

}  // extern "C"

int tv::tree_attn_check_args(const void* q, const void* k_new, const void* v_new, const void* k_cache,
                             const void* v_cache, int num_blocks, const int32_t* block_table, int max_blocks,
                             const int32_t* prefix_len, const int32_t* parents, int B, int N, int Hq, int Hkv,
                             int hd, int block_size, float rope_theta, float sm_scale, const void* out,
                             const int32_t* err) {
  if (!a16(q) || !a16(k_new) || !a16(v_new) || !a16(k_cache) || !a16(v_cache) || !a4(block_table) ||
      !a4(prefix_len) || !a4(parents) || !a16(out) || !a4(err))
    return TV_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || num_blocks < 1 || max_blocks < 1 ||
      !(rope_theta > 0.f) || !isfinite(rope_theta) || !isfinite(sm_scale))
    return TV_ERR_INVALID_ARG;
  if (N > TV_MAX_NODES || (hd != 64 && hd != 128 && hd != 256) || block_size != TV_BLOCK_SIZE)
    return TV_ERR_UNSUPPORTED;
  if (B > 65535) return TV_ERR_UNSUPPORTED;
  return TV_OK;
}

extern "C" {

int tv_tree_attn(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                 int num_blocks, const int32_t* block_table, int max_blocks, const int32_t* prefix_len,
                 const int32_t* parents, int B, int N, int Hq, int Hkv, int hd, int block_size,
                 float rope_theta, float sm_scale, void* out, void* workspace, size_t workspace_bytes,
                 int32_t* err, tv_stream_t stream) {
  const int st = tv::tree_attn_check_args(q, k_new, v_new, k_cache, v_cache, num_blocks, block_table, max_blocks,
                                          prefix_len, parents, B, N, Hq, Hkv, hd, block_size, rope_theta,
                                          sm_scale, out, err);
  if (st != TV_OK) return st;
  if (!a16(workspace)) return TV_ERR_INVALID_ARG;
  if (workspace_bytes < tv::attn_workspace_size(B, N, Hq, Hkv, hd, max_blocks, block_size))
    return TV_ERR_INVALID_ARG;
  tv::AttnArgs a{q, k_new, v_new, k_cache, v_cache, num_blocks, block_table, max_blocks, prefix_len, parents,
                 B, N, Hq, Hkv, hd, block_size, rope_theta, sm_scale, out, err};
  return cuda_status(tv::launch_tree_attn(a, workspace, workspace_bytes, stream));
}

int tv_kv_compact(void* k_cache, void* v_cache, int num_blocks, const int32_t* block_table, int max_blocks,
                  const int32_t* prefix_len, const int32_t* parents, int N, const int32_t* accepted_path,
                  const int32_t* accepted_len, int Lmax, int B, int Hkv, int hd, int block_size,
                  int32_t* slot_map, int32_t* new_len, int32_t* err, tv_stream_t stream) {
  if (!a16(k_cache) || !a16(v_cache) || !a4(block_table) || !a4(prefix_len) || !a4(parents) ||
      !a4(accepted_path) || !a4(accepted_len) || !a4(slot_map) || !a4(new_len) || !a4(err))
    return TV_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || Hkv < 1 || Lmax < 1 || num_blocks < 1 || max_blocks < 1) return TV_ERR_INVALID_ARG;
  if (N > TV_MAX_NODES || (hd != 64 && hd != 128 && hd != 256) || block_size != TV_BLOCK_SIZE)
    return TV_ERR_UNSUPPORTED;
  tv::CompactArgs a{k_cache, v_cache, num_blocks, block_table, max_blocks, prefix_len, parents, N,
                    accepted_path, accepted_len, Lmax, B, Hkv, hd, block_size, slot_map, new_len, err};
  return cuda_status(tv::launch_kv_compact(a, stream));
}

int tv_kv_compact_remap(void* k_cache, void* v_cache, int num_blocks, const int32_t* block_table,
                        int32_t* block_table_out, int max_blocks, const int32_t* prefix_len,
                        const int32_t* parents, int N, const int32_t* accepted_path,
                        const int32_t* accepted_len, int Lmax, int B, int Hkv, int hd, int block_size,
                        int32_t* slot_map, int32_t* new_len, int32_t* remapped, int32_t* err,
                        tv_stream_t stream) {
  if (!a16(k_cache) || !a16(v_cache) || !a4(block_table) || !a4(block_table_out) || !a4(prefix_len) ||
      !a4(parents) || !a4(accepted_path) || !a4(accepted_len) || !a4(slot_map) || !a4(new_len) ||
      !a4(remapped) || !a4(err))
    return TV_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || Hkv < 1 || Lmax < 1 || num_blocks < 1 || max_blocks < 1) return TV_ERR_INVALID_ARG;
  {
    const uintptr_t in0 = reinterpret_cast<uintptr_t>(block_table);
    const uintptr_t out0 = reinterpret_cast<uintptr_t>(block_table_out);
    const uintptr_t bytes = (uintptr_t)B * (uintptr_t)max_blocks * sizeof(int32_t);
    if (in0 < out0 + bytes && out0 < in0 + bytes) return TV_ERR_INVALID_ARG;
  }
  if (N > TV_MAX_NODES || (hd != 64 && hd != 128 && hd != 256) || block_size != TV_BLOCK_SIZE)
    return TV_ERR_UNSUPPORTED;
  tv::CompactArgs a{k_cache, v_cache, num_blocks, block_table, max_blocks, prefix_len, parents, N,
                    accepted_path, accepted_len, Lmax, B, Hkv, hd, block_size, slot_map, new_len, err,
                    block_table_out, remapped};
  return cuda_status(tv::launch_kv_compact_remap(a, stream));
}

int tv_accept_walk(const int32_t* parents, const int32_t* draft_tokens, const int32_t* target_tokens, int B,
                   int N, int Lmax, int32_t* accepted_path, int32_t* accepted_len, int32_t* next_token,
                   int32_t* err, tv_stream_t stream) {
  if (!a4(parents) || !a4(draft_tokens) || !a4(target_tokens) || !a4(accepted_path) || !a4(accepted_len) ||
      !a4(next_token) || !a4(err))
    return TV_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || Lmax < 1) return TV_ERR_INVALID_ARG;
  if (N > TV_MAX_NODES) return TV_ERR_UNSUPPORTED;
  tv::AcceptArgs a{parents, draft_tokens, target_tokens, B, N, Lmax, accepted_path, accepted_len, next_token, err};
  return cuda_status(tv::launch_accept_walk(a, stream));
}

}  // extern "C"
