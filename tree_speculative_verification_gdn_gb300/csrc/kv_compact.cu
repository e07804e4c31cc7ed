// KV compaction of the accepted path (handbook chapter 树形草稿与 EAGLE, note after the listing:
// the accepted nodes' KV is reused by moving it to the contiguous slots after the prefix;
// qwen35-tree-spec §七 Step 4, Gather-Compact).
//
// Logical slot P + r receives logical slot P + path[r] for r < L.  Since path[r] >= r (a node
// at depth r has index >= r), a source is never a destination of an EARLIER entry; entries
// are moved in ascending chunks, and within a chunk every source is loaded before any
// destination is stored, so no entry reads a slot this call has already overwritten.
#include "tv_common.cuh"
#include "tv_internal.h"

namespace tv {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 8;   // path entries moved per load/store round
constexpr int kVecPerThread = 4;

struct CompactCheck {
  int par[TV_MAX_NODES];
  int flag, status, L, P;
};

// Tree, path, capacity and block-table checks for sequence b (whole CTA).
__device__ int check_compact(const CompactArgs& a, int b, CompactCheck& c) {
  int st = load_and_check_tree(a.parents + (size_t)b * a.N, a.N, c.par, &c.flag);
  if (st) return st;
  if (threadIdx.x == 0) {
    const int L = a.path_len[b], P = a.prefix_len[b];
    int status = 0;
    if (P < 0 || (long long)P + a.N > (long long)a.max_blocks * a.block_size) status = TV_ERR_CAPACITY;
    if (!status) {
      int ok = (L >= 1 && L <= a.Lmax), prev = -1;
      for (int r = 0; ok && r < L; ++r) {
        const int node = a.path[(size_t)b * a.Lmax + r];
        ok = (node >= 0 && node < a.N && c.par[node] == prev);
        prev = node;
      }
      if (!ok) status = TV_ERR_BAD_PATH;
    }
    if (!status) {
      const int first = P / a.block_size, last = (P + a.N - 1) / a.block_size;
      for (int lb = first; lb <= last; ++lb) {
        const int blk = a.block_table[(size_t)b * a.max_blocks + lb];
        if (blk < 0 || blk >= a.num_blocks) status = TV_ERR_BAD_BLOCK;
      }
    }
    c.status = status;
    c.L = L;
    c.P = P;
  }
  __syncthreads();
  return c.status;
}

// One CTA per (sequence, KV head).
__global__ void __launch_bounds__(kThreads) kv_compact_kernel(CompactArgs a) {
  __shared__ CompactCheck c;
  const int b = blockIdx.x / a.Hkv, kvh = blockIdx.x % a.Hkv;
  const int st = check_compact(a, b, c);
  if (kvh == 0 && threadIdx.x == 0) a.err[b] = st;
  if (kvh == 0) {
    for (int r = threadIdx.x; r < a.Lmax; r += kThreads) {
      int smap = -1;
      if (!st && r < c.L) {
        const int s = c.P + a.path[(size_t)b * a.Lmax + r];
        smap = a.block_table[(size_t)b * a.max_blocks + s / a.block_size] * a.block_size + s % a.block_size;
      }
      a.slot_map[(size_t)b * a.Lmax + r] = smap;
    }
    if (threadIdx.x == 0) a.new_len[b] = st ? a.prefix_len[b] : c.P + c.L;
  }
  if (st) return;
  // One slot row of one head: hd bf16 = hd/8 16-byte vectors.
  const int vpr = a.hd / 8;
  const int per_chunk = kChunk * vpr * 2;  // K and V
  const int* table = a.block_table + (size_t)b * a.max_blocks;
  uint4* kc = static_cast<uint4*>(a.k_cache);
  uint4* vc = static_cast<uint4*>(a.v_cache);
  auto row_base = [&](int slot) -> size_t {  // vector index of (slot, kvh, col 0)
    const int blk = table[slot / a.block_size];
    return (((size_t)blk * a.Hkv + kvh) * a.block_size + slot % a.block_size) * vpr;
  };
  for (int r0 = 0; r0 < c.L; r0 += kChunk) {
    uint4 buf[kVecPerThread];
    int dst_idx[kVecPerThread];
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      const int x = threadIdx.x + u * kThreads;
      dst_idx[u] = -1;
      if (x < per_chunk) {
        const int which = x / (kChunk * vpr);  // 0: K, 1: V
        const int rem = x % (kChunk * vpr);
        const int r = r0 + rem / vpr, col = rem % vpr;
        if (r < c.L) {
          const uint4* cache = which ? vc : kc;
          buf[u] = cache[row_base(c.P + a.path[(size_t)b * a.Lmax + r]) + col];
          dst_idx[u] = x;
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      if (dst_idx[u] >= 0) {
        const int x = dst_idx[u];
        const int which = x / (kChunk * vpr);
        const int rem = x % (kChunk * vpr);
        const int r = r0 + rem / vpr, col = rem % vpr;
        uint4* cache = which ? vc : kc;
        cache[row_base(c.P + r) + col] = buf[u];
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_kv_compact(const CompactArgs& a, cudaStream_t s) {
  kv_compact_kernel<<<a.B * a.Hkv, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace tv
