// Tree topology of B draft trees (handbook chapter 树形草稿与 EAGLE, §实现, `depths` and
// `tree_mask`): node depth, the tree-mask rows packed as bits, and optionally every node's
// root-to-node path and the tree's maximum depth.
#include "tv_common.cuh"
#include "tv_internal.h"

namespace tv {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) tree_prepare_kernel(const int32_t* __restrict__ parents, int N,
                                                                int32_t* __restrict__ depth,
                                                                uint32_t* __restrict__ mask_bits,
                                                                int32_t* __restrict__ paths, int path_cap,
                                                                int32_t* __restrict__ max_depth,
                                                                int32_t* __restrict__ err) {
  __shared__ int par[TV_MAX_NODES];
  __shared__ int flag, dmax;
  const int b = blockIdx.x;
  const int st = load_and_check_tree(parents + (size_t)b * N, N, par, &flag);
  if (st) {
    if (threadIdx.x == 0) err[b] = st;
    return;
  }
  if (threadIdx.x == 0) dmax = 0;
  __syncthreads();
  const int W = (N + 31) / 32;
  bool too_deep = false;
  for (int i = threadIdx.x; i < N; i += kThreads) {
    const int d = node_depth(par, i);
    depth[(size_t)b * N + i] = d;
    atomicMax(&dmax, d);
    if (paths != nullptr) {
      // row i: the root-to-i path, root first, then -1 up to path_cap entries
      int32_t* row = paths + ((size_t)b * N + i) * path_cap;
      if (d + 1 > path_cap) {
        too_deep = true;
      } else {
        for (int j = i, t = d; j >= 0; j = par[j], --t) row[t] = j;
        for (int t = d + 1; t < path_cap; ++t) row[t] = -1;
      }
    }
  }
  too_deep = __syncthreads_or(too_deep);
  if (threadIdx.x == 0) {
    err[b] = too_deep ? TV_ERR_UNSUPPORTED : 0;
    if (max_depth != nullptr) max_depth[b] = dmax;
  }
  // One thread per (node, word): the bits of that word on the node's root path.
  for (int x = threadIdx.x; x < N * W; x += kThreads) {
    const int i = x / W, w = x % W;
    uint32_t bits = 0;
    for (int j = i; j >= 0; j = par[j])
      if ((j >> 5) == w) bits |= 1u << (j & 31);
    mask_bits[((size_t)b * N + i) * W + w] = bits;
  }
}

}  // namespace

cudaError_t launch_tree_prepare(const int32_t* parents, int B, int N, int32_t* depth, uint32_t* mask_bits,
                                int32_t* paths, int path_cap, int32_t* max_depth, int32_t* err, cudaStream_t s) {
  tree_prepare_kernel<<<B, kThreads, 0, s>>>(parents, N, depth, mask_bits, paths, path_cap, max_depth, err);
  return cudaGetLastError();
}

}  // namespace tv
