// Tree topology of B draft trees (handbook chapter 树形草稿与 EAGLE, §实现, `depths` and
// `tree_mask`): node depth and the tree-mask rows packed as bits.
#include "tv_common.cuh"
#include "tv_internal.h"

namespace tv {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) tree_prepare_kernel(const int32_t* __restrict__ parents, int N,
                                                                int32_t* __restrict__ depth,
                                                                uint32_t* __restrict__ mask_bits,
                                                                int32_t* __restrict__ err) {
  __shared__ int par[TV_MAX_NODES];
  __shared__ int flag;
  const int b = blockIdx.x;
  const int st = load_and_check_tree(parents + (size_t)b * N, N, par, &flag);
  if (threadIdx.x == 0) err[b] = st;
  if (st) return;
  const int W = (N + 31) / 32;
  for (int i = threadIdx.x; i < N; i += kThreads) depth[(size_t)b * N + i] = node_depth(par, i);
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

cudaError_t launch_tree_prepare(const int32_t* parents, int B, int N, int32_t* depth,
                                uint32_t* mask_bits, int32_t* err, cudaStream_t s) {
  tree_prepare_kernel<<<B, kThreads, 0, s>>>(parents, N, depth, mask_bits, err);
  return cudaGetLastError();
}

}  // namespace tv
