// KV compaction of the accepted path (handbook chapter 树形草稿与 EAGLE, note after the listing:
// the accepted nodes' KV is reused by moving it to the contiguous slots after the prefix, or by
// updating only the block table; qwen35-tree-spec §七 Step 4, Gather-Compact).
//
// Logical slot P + r receives logical slot P + path[r] for r < L.  Since path[r] >= r (a node
// at depth r has index >= r), a source is never a destination of an EARLIER entry; entries
// are moved in ascending rounds, and within a round every source is loaded before any
// destination is stored, so no entry reads a slot this call has already overwritten.  One round
// holds kThreads * kVecPerThread 16-byte vectors: 32 entries of K and V at hd = 256, so the
// paths of shallow trees move in one round.  An entry already in place is not written.
//
// The checks run in parallel: one thread per path entry and per block-table entry, combined
// with a barrier reduction, so a call costs a few dependent global loads, not one per entry.
#include "tv_common.cuh"
#include "tv_internal.h"

namespace tv {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 8;
constexpr int kMaxWin = TV_MAX_NODES / 16 + 2;   // logical blocks spanned by P .. P + N - 1

struct CompactCheck {
  int par[TV_MAX_NODES];
  int path[TV_MAX_NODES];
  int win[kMaxWin];        // table entries of logical blocks first .. first + nwin - 1
  int flag, L, P, first, nwin;
};

// Tree, path, capacity and block-table checks for sequence b (whole CTA; the result is the
// same in every thread).  On success c.path[0 .. L) holds the path and c.win the table entries
// of the logical blocks the tree's slots span (every source and destination lies there).
__device__ int check_compact(const CompactArgs& a, int b, CompactCheck& c) {
  if (threadIdx.x == 0) {
    c.L = a.path_len[b];
    c.P = a.prefix_len[b];
  }
  const int st = load_and_check_tree(a.parents + (size_t)b * a.N, a.N, c.par, &c.flag);
  if (st) return st;
  const int L = c.L, P = c.P;
  if (P < 0 || (long long)P + a.N > (long long)a.max_blocks * a.block_size) return TV_ERR_CAPACITY;
  // a valid path strictly increases in node index, so it holds at most N entries
  if (L < 1 || L > a.Lmax || L > a.N) return TV_ERR_BAD_PATH;
  const int* path = a.path + (size_t)b * a.Lmax;
  bool bad_path = false;
  for (int r = threadIdx.x; r < L; r += kThreads) {
    const int node = path[r];
    const int prev = r ? path[r - 1] : -1;
    const bool ok = node >= 0 && node < a.N && c.par[node] == prev;
    c.path[r] = ok ? node : 0;
    bad_path |= !ok;
  }
  const int* table = a.block_table + (size_t)b * a.max_blocks;
  const int first = P / a.block_size, last = (P + a.N - 1) / a.block_size;
  bool bad_block = false;
  for (int lb = first + threadIdx.x; lb <= last; lb += kThreads) {
    const int blk = table[lb];
    c.win[lb - first] = blk;
    bad_block |= blk < 0 || blk >= a.num_blocks;
  }
  if (threadIdx.x == 0) {
    c.first = first;
    c.nwin = last - first + 1;
  }
  if (__syncthreads_or(bad_path)) return TV_ERR_BAD_PATH;
  // The window's entries are in c.win (the barrier above).  Two logical blocks of the window on
  // one physical block would let a store overwrite a source before it is read.
  for (int i = threadIdx.x; i <= last - first; i += kThreads)
    for (int u = 0; u < i; ++u) bad_block |= c.win[u] == c.win[i];
  if (__syncthreads_or(bad_block)) return TV_ERR_BAD_BLOCK;
  return 0;
}

// Moves the kept entries of (sequence b, KV head kvh) in ascending rounds.  dst_block(lb)
// gives the physical block a destination in logical block lb is stored to, or -1 when the
// entry is not to be written (its block was taken over whole).
template <class DstBlock>
__device__ void move_entries(const CompactArgs& a, int b, int kvh, const CompactCheck& c, DstBlock dst_block) {
  const int bs = a.block_size;
  const int vpr = a.hd / 8;                                  // 16-byte vectors per row
  const int rows_per_round = kThreads * kVecPerThread / (2 * vpr);
  uint4* kc = static_cast<uint4*>(a.k_cache);
  uint4* vc = static_cast<uint4*>(a.v_cache);
  auto vec_base = [&](int blk, int row) -> size_t {
    return (((size_t)blk * a.Hkv + kvh) * bs + row) * vpr;
  };
  for (int r0 = 0; r0 < c.L; r0 += rows_per_round) {
    const int per_round = min(rows_per_round, c.L - r0) * vpr;   // vectors of K (and of V)
    uint4 buf[kVecPerThread];
    size_t dst[kVecPerThread];
    bool live[kVecPerThread];
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      const int x = threadIdx.x + u * kThreads;
      live[u] = false;
      if (x < 2 * per_round) {
        const int which = x / per_round;                     // 0: K, 1: V
        const int rem = x - which * per_round;
        const int r = r0 + rem / vpr, col = rem % vpr;
        const int ds = c.P + r, ss = c.P + c.path[r];
        const int dblk = dst_block(ds / bs);
        const int sblk = c.win[ss / bs - c.first];
        if (dblk >= 0 && (dblk != sblk || ds % bs != ss % bs)) {
          const uint4* cache = which ? vc : kc;
          buf[u] = cache[vec_base(sblk, ss % bs) + col];
          dst[u] = vec_base(dblk, ds % bs) + col;
          live[u] = true;
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      if (live[u]) {
        const int x = threadIdx.x + u * kThreads;
        uint4* cache = (x >= per_round) ? vc : kc;
        cache[dst[u]] = buf[u];
      }
    }
    __syncthreads();
  }
}

// One CTA per (sequence, KV head).
__global__ void __launch_bounds__(kThreads) kv_compact_kernel(CompactArgs a) {
  __shared__ CompactCheck c;
  const int b = blockIdx.x / a.Hkv, kvh = blockIdx.x % a.Hkv;
  const int st = check_compact(a, b, c);
  if (kvh == 0) {
    if (threadIdx.x == 0) {
      a.err[b] = st;
      a.new_len[b] = st ? a.prefix_len[b] : c.P + c.L;
    }
    for (int r = threadIdx.x; r < a.Lmax; r += kThreads) {
      int smap = -1;
      if (!st && r < c.L) {
        const int s = c.P + c.path[r];
        smap = c.win[s / a.block_size - c.first] * a.block_size + s % a.block_size;
      }
      a.slot_map[(size_t)b * a.Lmax + r] = smap;
    }
  }
  if (st) return;
  move_entries(a, b, kvh, c, [&](int lb) { return c.win[lb - c.first]; });
}

// ---------------------------------------------------------------------------------------------
// Block-table form (the same note allows updating only the block table).  A destination block
// m that lies wholly at or past the prefix (m * bs >= P) and whose kept entries r all come from
// slot P + r + j * bs (one j >= 1) is taken over by exchanging table entries m and m + j, in
// ascending m; only the other kept entries are moved.  Since path[r] - r never decreases along
// the path, the source block m + j of an exchange has not been touched by an earlier exchange.
//
// Loads use the table as it was (the checks' shared copy of its window; the input row is never
// written); stores use the new row, also held in shared memory.  A store lands in a block that is not taken over: if it was an
// exchange partner m' + j', it now holds the old block m', whose slots lie before every source
// a later round reads (sources sit at or past their destinations).  So the ascending rounds stay
// safe.  The new row goes to a separate output: the CTA of KV head 0 writes the window, and the
// sequence's CTAs share the copy of the entries outside it, which no CTA of the call changes.
__global__ void __launch_bounds__(kThreads) kv_compact_remap_kernel(CompactArgs a) {
  __shared__ CompactCheck c;
  __shared__ int win[kMaxWin];          // new table entries of logical blocks first .. last
  __shared__ int shift[kMaxWin];        // per destination block: j >= 1 to take over, else 0
  __shared__ int n_exch;
  const int b = blockIdx.x / a.Hkv, kvh = blockIdx.x % a.Hkv;
  const int bs = a.block_size;
  const int* table = a.block_table + (size_t)b * a.max_blocks;
  // This CTA's share of the row copy, loaded now so that the loads overlap the checks.
  constexpr int kPre = 4;
  const int stride = a.Hkv * kThreads, base = kvh * kThreads + threadIdx.x;
  int pre[kPre];
#pragma unroll
  for (int u = 0; u < kPre; ++u) {
    const int i = base + u * stride;
    pre[u] = i < a.max_blocks ? table[i] : 0;
  }
  const int st = check_compact(a, b, c);
  const int first = st ? 0 : c.first;
  const int nwin = st ? 0 : c.nwin;
  if (!st) {
    const int P = c.P, L = c.L;
    const int m_lo = (P + bs - 1) / bs, m_hi = (P + L - 1) / bs;
    // one thread per window block: copy its entry, and decide a destination block
    for (int i = threadIdx.x; i < nwin; i += kThreads) {
      win[i] = c.win[i];
      const int m = first + i;
      int j = 0;
      if (m >= m_lo && m <= m_hi) {
        const int r_lo = m * bs - P, r_hi = min(m * bs + bs - P, L);
        const int d = c.path[r_lo] - r_lo;
        bool ok = d > 0 && d % bs == 0;
        for (int r = r_lo + 1; ok && r < r_hi; ++r) ok = (c.path[r] - r == d);
        j = ok ? d / bs : 0;
      }
      shift[i] = j;
    }
    __syncthreads();
    if (threadIdx.x == 0) {   // the exchanges, in ascending order (at most kMaxWin)
      int cnt = 0;
      for (int i = 0; i < nwin; ++i) {
        const int j = shift[i];
        if (j) {
          const int t = win[i];
          win[i] = win[i + j];
          win[i + j] = t;
          ++cnt;
        }
      }
      n_exch = cnt;
    }
    __syncthreads();
  }
  if (kvh == 0) {
    if (threadIdx.x == 0) {
      a.err[b] = st;
      a.new_len[b] = st ? a.prefix_len[b] : c.P + c.L;
      a.remapped[b] = st ? 0 : n_exch;
    }
    for (int r = threadIdx.x; r < a.Lmax; r += kThreads) {
      int smap = -1;
      if (!st && r < c.L) {
        const int s = c.P + c.path[r];
        smap = c.win[s / bs - first] * bs + s % bs;
      }
      a.slot_map[(size_t)b * a.Lmax + r] = smap;
    }
    for (int i = threadIdx.x; i < nwin; i += kThreads) a.table_out[(size_t)b * a.max_blocks + first + i] = win[i];
  }
  if (!st) move_entries(a, b, kvh, c, [&](int lb) { return shift[lb - first] ? -1 : win[lb - first]; });
  // The rest of the row (all of it for a sequence with an error) is copied unchanged, shared
  // among the sequence's CTAs.
  int32_t* out = a.table_out + (size_t)b * a.max_blocks;
#pragma unroll
  for (int u = 0; u < kPre; ++u) {
    const int i = base + u * stride;
    if (i < a.max_blocks && (i < first || i >= first + nwin)) out[i] = pre[u];
  }
  for (int i = base + kPre * stride; i < a.max_blocks; i += stride)
    if (i < first || i >= first + nwin) out[i] = table[i];
}

}  // namespace

cudaError_t launch_kv_compact(const CompactArgs& a, cudaStream_t s) {
  kv_compact_kernel<<<a.B * a.Hkv, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_kv_compact_remap(const CompactArgs& a, cudaStream_t s) {
  kv_compact_remap_kernel<<<a.B * a.Hkv, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace tv
