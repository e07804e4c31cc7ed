// Greedy acceptance of B draft trees on the device (handbook chapter 树形草稿与 EAGLE, §实现,
// tree_speculative_generate): start at node 0; while the target's token at the current node
// equals the draft token of one of its children, step to the lowest-numbered such child.  The
// walk stops when no child matches or Lmax nodes are accepted; the target's token at the last
// accepted node is the next token.
//
// One warp per sequence.  Its tree (parents, draft tokens) sits in shared memory; at each step
// the lanes test 32 candidate children at once (children are numbered after their parent) and
// a ballot picks the lowest match.
#include "tv_common.cuh"
#include "tv_internal.h"

namespace tv {
namespace {

constexpr int kWarps = 4;

__global__ void __launch_bounds__(kWarps * 32) accept_walk_kernel(AcceptArgs a) {
  __shared__ int par_s[kWarps][TV_MAX_NODES];
  __shared__ int tok_s[kWarps][TV_MAX_NODES];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int b = blockIdx.x * kWarps + warp;
  if (b >= a.B) return;  // whole warps only: B is checked per warp
  const int N = a.N;
  int* par = par_s[warp];
  int* tok = tok_s[warp];
  bool bad = false;
  for (int i = lane; i < N; i += 32) {
    const int p = a.parents[(size_t)b * N + i];
    par[i] = p;
    tok[i] = a.draft[(size_t)b * N + i];
    bad |= (p < -1 || p >= i);
  }
  bad = __any_sync(0xffffffffu, bad);
  __syncwarp();
  int32_t* path = a.path + (size_t)b * a.Lmax;
  if (bad) {
    for (int r = lane; r < a.Lmax; r += 32) path[r] = -1;
    if (lane == 0) {
      a.len[b] = 0;
      a.next_token[b] = -1;
      a.err[b] = TV_ERR_BAD_TREE;
    }
    return;
  }
  const int32_t* target = a.target + (size_t)b * N;
  int node = 0, count = 1;
  while (count < a.Lmax) {
    const int want = target[node];
    int found = -1;
    for (int base = node + 1; base < N; base += 32) {
      const int c = base + lane;
      const unsigned hit = __ballot_sync(0xffffffffu, c < N && par[c] == node && tok[c] == want);
      if (hit) {
        found = base + __ffs(hit) - 1;
        break;
      }
    }
    if (found < 0) break;
    if (lane == 0) path[count] = found;
    node = found;
    ++count;
  }
  for (int r = count + lane; r < a.Lmax; r += 32) path[r] = -1;
  if (lane == 0) {
    path[0] = 0;
    a.len[b] = count;
    a.next_token[b] = target[node];
    a.err[b] = 0;
  }
}

}  // namespace

cudaError_t launch_accept_walk(const AcceptArgs& a, cudaStream_t s) {
  accept_walk_kernel<<<(a.B + kWarps - 1) / kWarps, kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace tv
