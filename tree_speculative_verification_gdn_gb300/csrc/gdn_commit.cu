// GDN commit: write the last accepted node's state back into S_0.
//
// Fork mode (qwen35-tree-spec, §五 用途 2 and §七 Step 4): restore the accepted node's
// checkpoint, S_0[b] <- node_states[b, a], a = path[L-1].
// WY mode (TreeWY abstract: rebuild only the accepted state on commit), reading stated with
// tv_gdn_tree_verify_wy: S_a = gamma_a S_0 + sum_{r<L} (gamma_a / gamma_{path[r]}) w_{path[r]}
// k_{path[r]}^T, done in place on S_0 -- a rank-L update of a state that is read and written
// once.
#include "tv_common.cuh"
#include "tv_internal.h"

namespace tv {
namespace {

constexpr int kThreads = 256;

struct PathCheck {
  int par[TV_MAX_NODES];
  int flag;
  int status;
  int L;
  int last;
};

// Checks tree and accepted path of sequence b with the whole CTA.  Returns the status (same in
// every thread); on success pc.L / pc.last hold the length and the accepted node.
__device__ int check_path(const CommitArgs& a, int b, PathCheck& pc) {
  int st = load_and_check_tree(a.parents + (size_t)b * a.N, a.N, pc.par, &pc.flag);
  if (st) return st;
  if (threadIdx.x == 0) {
    const int L = a.path_len[b];
    int ok = (L >= 1 && L <= a.Lmax);
    int prev = -1;
    for (int r = 0; ok && r < L; ++r) {
      const int node = a.path[(size_t)b * a.Lmax + r];
      ok = (node >= 0 && node < a.N && pc.par[node] == prev);
      prev = node;
    }
    pc.status = ok ? 0 : TV_ERR_BAD_PATH;
    pc.L = L;
    pc.last = prev;
  }
  __syncthreads();
  return pc.status;
}

// One CTA per (sequence, head): copy the accepted checkpoint over S_0.
template <typename TS>
__global__ void __launch_bounds__(kThreads) commit_fork_kernel(CommitArgs a) {
  __shared__ PathCheck pc;
  const int b = blockIdx.x / a.H, h = blockIdx.x % a.H;
  const int st = check_path(a, b, pc);
  if (h == 0 && threadIdx.x == 0) a.err[b] = st;
  if (st) return;
  const size_t tile = (size_t)a.dv * a.dk * sizeof(TS);  // bytes, a multiple of 16
  const uint4* src = reinterpret_cast<const uint4*>(
      static_cast<const char*>(a.node_states) + ((((size_t)b * a.N + pc.last) * a.H + h) * tile));
  uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(a.S0) + ((size_t)b * a.H + h) * tile);
  for (size_t j = threadIdx.x; j < tile / 16; j += kThreads) dst[j] = __ldg(src + j);
}

constexpr int kLPR = 8;
constexpr int kRows = 32;  // rows of S_0 per CTA in WY mode

// One CTA per (sequence, head, 32-row slab): S_0 <- gamma_a S_0 + sum_r Gamma w k^T.
template <typename TIO, typename TS, int DK>
__global__ void __launch_bounds__(kThreads) commit_wy_kernel(CommitArgs a) {
  constexpr int CPL = DK / kLPR;
  __shared__ PathCheck pc;
  __shared__ float coef[TV_MAX_NODES];
  __shared__ int nodes[TV_MAX_NODES];
  extern __shared__ float wsm[];  // [L][kRows]
  const int slabs = a.dv / kRows;
  const int b = blockIdx.x / (a.H * slabs), h = (blockIdx.x / slabs) % a.H, slab = blockIdx.x % slabs;
  const int st = check_path(a, b, pc);
  if (h == 0 && slab == 0 && threadIdx.x == 0) a.err[b] = st;
  if (st) return;
  const int L = pc.L, N = a.N, H = a.H;
  const float lga = a.log_gamma[((size_t)b * N + pc.last) * H + h];
  for (int r = threadIdx.x; r < L; r += kThreads) {
    const int node = a.path[(size_t)b * a.Lmax + r];
    nodes[r] = node;
    coef[r] = expf(lga - a.log_gamma[((size_t)b * N + node) * H + h]);
  }
  __syncthreads();
  for (int x = threadIdx.x; x < L * kRows; x += kThreads) {
    const int r = x / kRows, row = x % kRows;
    wsm[x] = a.pseudo_v[(((size_t)b * N + nodes[r]) * H + h) * a.dv + slab * kRows + row];
  }
  __syncthreads();
  const int lane8 = threadIdx.x % kLPR, rl = threadIdx.x / kLPR;
  const int row = slab * kRows + rl;
  TS* s0 = static_cast<TS*>(a.S0) + (((size_t)b * H + h) * a.dv + row) * DK + lane8 * CPL;
  const TIO* k = static_cast<const TIO*>(a.k);
  float cur[CPL];
  load_vec_rw<CPL>(s0, cur);
  const float gam = expf(lga);
#pragma unroll
  for (int e = 0; e < CPL; ++e) cur[e] *= gam;
  for (int r = 0; r < L; ++r) {
    float kf[CPL];
    load_vec<CPL>(k + (((size_t)b * N + nodes[r]) * H + h) * DK + lane8 * CPL, kf);
    const float c = coef[r] * wsm[r * kRows + rl];
#pragma unroll
    for (int e = 0; e < CPL; ++e) cur[e] = fmaf(c, kf[e], cur[e]);
  }
  store_vec<CPL>(s0, cur);
}

template <typename TIO, typename TS, int DK>
cudaError_t launch_wy_t(const CommitArgs& a, cudaStream_t s) {
  const int max_len = a.Lmax < a.N ? a.Lmax : a.N;  // a valid path has distinct nodes
  const size_t smem = (size_t)max_len * kRows * sizeof(float);
  auto kern = commit_wy_kernel<TIO, TS, DK>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<a.B * a.H * (a.dv / kRows), kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gdn_commit(const CommitArgs& a, cudaStream_t s) {
  if (a.mode == TV_MODE_FORK) {
    if (a.state == TV_F32) commit_fork_kernel<float><<<a.B * a.H, kThreads, 0, s>>>(a);
    else commit_fork_kernel<bf16><<<a.B * a.H, kThreads, 0, s>>>(a);
    return cudaGetLastError();
  }
  if (a.io == TV_F32 && a.state == TV_F32)
    return a.dk == 64 ? launch_wy_t<float, float, 64>(a, s) : launch_wy_t<float, float, 128>(a, s);
  if (a.io == TV_BF16 && a.state == TV_BF16)
    return a.dk == 64 ? launch_wy_t<bf16, bf16, 64>(a, s) : launch_wy_t<bf16, bf16, 128>(a, s);
  return a.dk == 64 ? launch_wy_t<bf16, float, 64>(a, s) : launch_wy_t<bf16, float, 128>(a, s);
}

}  // namespace tv
