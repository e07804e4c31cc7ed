// GDN commit: write the last accepted node's state back into S_0.
//
// Fork mode (qwen35-tree-spec, §五 用途 2 and §七 Step 4): restore the accepted node's
// checkpoint, S_0[b] <- node_states[b, a], a = path[L-1].
// WY mode (TreeWY abstract: rebuild only the accepted state on commit), reading stated with
// tv_gdn_tree_verify_wy: S_a = gamma_a S_0 + sum_{r<L} (gamma_a / gamma_{path[r]}) w_{path[r]}
// k_{path[r]}^T, done in place on S_0 -- a rank-L update of a state that is read and written
// once.
#include "tv_async.cuh"
#include "tv_common.cuh"
#include "tv_internal.h"

namespace tv {
namespace {

constexpr int kThreads = 256;

struct PathCheck {
  int par[TV_MAX_NODES];
  int path[TV_MAX_NODES];  // the first min(Lmax, N) entries of the sequence's path
  int flag;
  int status;
  int L;
  int last;
};

// Checks tree and accepted path of sequence b with the whole CTA.  The path entries and its
// length are loaded together with the parents, so the check itself reads shared memory only.
// Returns the status (same in every thread); on success pc.L / pc.last hold the length and
// the accepted node, and pc.path[0 .. L-1] the path.  A valid path has distinct nodes, so
// L <= N.
__device__ int check_path(const CommitArgs& a, int b, PathCheck& pc) {
  const int cap = a.Lmax < a.N ? a.Lmax : a.N;
  for (int r = threadIdx.x; r < cap; r += blockDim.x) pc.path[r] = a.path[(size_t)b * a.Lmax + r];
  if (threadIdx.x == 0) pc.L = a.path_len[b];
  int st = load_and_check_tree(a.parents + (size_t)b * a.N, a.N, pc.par, &pc.flag);  // barriers inside
  if (st) return st;
  if (threadIdx.x == 0) {
    const int L = pc.L;
    int ok = (L >= 1 && L <= cap);
    int prev = -1;
    for (int r = 0; ok && r < L; ++r) {
      const int node = pc.path[r];
      ok = (node >= 0 && node < a.N && pc.par[node] == prev);
      prev = node;
    }
    pc.status = ok ? 0 : TV_ERR_BAD_PATH;
    pc.last = prev;
  }
  __syncthreads();
  return pc.status;
}

// The per-layer view of a multi-layer commit: CTA blockIdx.x takes layer blockIdx.x / (B H) of
// (sequence, head) blockIdx.x % (B H).
__device__ __forceinline__ CommitArgs layer_view(const CommitArgs& a, int layer) {
  CommitArgs v = a;
  const size_t es = a.state == TV_F32 ? 4 : 2, eio = a.io == TV_F32 ? 4 : 2;
  const size_t bnh = (size_t)a.B * a.N * a.H;
  v.S0 = static_cast<char*>(a.S0) + layer * (size_t)a.B * a.H * a.dv * a.dk * es;
  if (a.node_states) v.node_states = static_cast<const char*>(a.node_states) + layer * bnh * a.dv * a.dk * es;
  if (a.pseudo_v) v.pseudo_v = a.pseudo_v + layer * bnh * a.dv;
  if (a.log_gamma) v.log_gamma = a.log_gamma + layer * bnh;
  if (a.k) v.k = static_cast<const char*>(a.k) + layer * bnh * a.dk * eio;
  return v;
}

constexpr int kForkThreads = 128;

// The first half of check_path: the path entries (clamped into [0, N)), its length (clamped
// into [0, min(Lmax, N)]) and the parents land in shared memory; returns the clamped length.
// The raw entries and length are kept for the check.
__device__ int path_prefetch(const CommitArgs& a, int b, PathCheck& pc) {
  const int cap = a.Lmax < a.N ? a.Lmax : a.N;
  if (threadIdx.x == 0) pc.flag = 0;
  for (int r = threadIdx.x; r < cap; r += blockDim.x) pc.path[r] = a.path[(size_t)b * a.Lmax + r];
  for (int i = threadIdx.x; i < a.N; i += blockDim.x) pc.par[i] = a.parents[(size_t)b * a.N + i];
  if (threadIdx.x == 0) pc.L = a.path_len[b];
  __syncthreads();
  const int L = pc.L;
  return L < 0 ? 0 : (L > cap ? cap : L);
}

// The second half: the tree and the path in shared memory are checked as in check_path.  The
// raw path entries are still there; the loads issued from them used clamped indices.
__device__ int check_prefetched_path(const CommitArgs& a, int b, PathCheck& pc) {
  const int cap = a.Lmax < a.N ? a.Lmax : a.N;
  for (int i = threadIdx.x; i < a.N; i += blockDim.x) {
    const int p = pc.par[i];
    if (p < -1 || p >= i) pc.flag = 1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int st = pc.flag ? TV_ERR_BAD_TREE : 0;
    if (!st) {
      const int L = pc.L;
      int ok = (L >= 1 && L <= cap);
      int prev = -1;
      for (int r = 0; ok && r < L; ++r) {
        const int node = pc.path[r];
        ok = (node >= 0 && node < a.N && pc.par[node] == prev);
        prev = node;
      }
      st = ok ? 0 : TV_ERR_BAD_PATH;
      pc.last = prev;
    }
    pc.status = st;
  }
  __syncthreads();
  return pc.status;
}

// One CTA per (sequence, head): copy the accepted checkpoint over S_0.  Thread 0 starts a bulk
// copy of the tile of the node the (not yet checked) path names, clamped into [0, N), into
// shared memory while the CTA checks the path; the tile goes out to S_0 by a bulk store only if
// the check passes, and then that node is the accepted one.
template <typename TS>
__global__ void __launch_bounds__(kForkThreads) commit_fork_kernel(CommitArgs a0) {
  __shared__ PathCheck pc;
  __shared__ __align__(8) uint64_t bar;
  __shared__ int guess_s;
  extern __shared__ __align__(128) unsigned char tile_s[];
  const int layer = blockIdx.x / (a0.B * a0.H), bh = blockIdx.x % (a0.B * a0.H);
  const CommitArgs a = layer_view(a0, layer);
  const int b = bh / a.H, h = bh % a.H;
  const uint32_t tile = (uint32_t)a.dv * a.dk * sizeof(TS);  // bytes, a multiple of 16
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
    const int L0 = a.path_len[b];
    int guess = (L0 >= 1 && L0 <= a.Lmax) ? a.path[(size_t)b * a.Lmax + L0 - 1] : 0;
    guess = guess < 0 ? 0 : (guess >= a.N ? a.N - 1 : guess);
    guess_s = guess;
    mbar_arrive_expect_tx(&bar, tile);
    bulk_g2s(tile_s, static_cast<const char*>(a.node_states) + (((size_t)b * a.N + guess) * a.H + h) * tile, tile,
             &bar);
  }
  const int st = check_path(a, b, pc);  // its barriers also publish guess_s
  if (layer == 0 && h == 0 && threadIdx.x == 0) a.err[b] = st;
  if (threadIdx.x == 0) {
    // The copy must have landed before the tile is stored -- or before the CTA may exit.
    const bool landed = mbar_wait(&bar, 0);
    if (landed && !st && pc.last == guess_s) {  // pc.last == guess whenever the path is valid
      bulk_s2g(static_cast<char*>(a.S0) + ((size_t)b * a.H + h) * tile, tile_s, tile);
      bulk_commit();
      bulk_wait_read<0>();
    } else if (!landed) {
      a.err[b] = TV_ERR_TIMEOUT;
      mbar_wait(&bar, 0);
    }
  }
}

constexpr int kLPR = 8;
constexpr int kRows = 32;          // rows of S_0 per pass of a CTA in WY mode
constexpr int kStride = 8 * kLPR;  // lane l holds columns l * 8 + j * kStride .. + 7

// One CTA per (sequence, head): S_0 <- gamma_a S_0 + sum_r Gamma w k^T.  Thread 0 starts a bulk
// copy of the head's S_0 tile into shared memory at once; the path's log(gamma), w rows and keys
// are fetched while the path is checked.  Thread (row rl, lane) then updates rows rl, rl + 32,
// ... of the tile in place, and one bulk store writes the tile back.
template <typename TIO, typename TS, int DK>
__global__ void __launch_bounds__(kThreads) commit_wy_kernel(CommitArgs a0) {
  constexpr int CPL = DK / kLPR;
  __shared__ PathCheck pc;
  __shared__ float coef[TV_MAX_NODES];
  __shared__ float lga_s;
  __shared__ __align__(8) uint64_t bar;
  // the S_0 tile [dv][DK], then w [cap][dv] fp32, then k [cap][DK]
  extern __shared__ __align__(128) unsigned char dyn[];
  const int layer = blockIdx.x / (a0.B * a0.H), bh = blockIdx.x % (a0.B * a0.H);
  const CommitArgs a = layer_view(a0, layer);
  const int passes = a.dv / kRows;
  const int b = bh / a.H, h = bh % a.H;
  const int N = a.N, H = a.H, dv = a.dv;
  const int cap = a.Lmax < N ? a.Lmax : N;
  const uint32_t tile = (uint32_t)dv * DK * sizeof(TS);  // bytes, a multiple of 16
  TS* tile_s = reinterpret_cast<TS*>(dyn);
  float* wsm = reinterpret_cast<float*>(dyn + tile);
  TIO* ksm = reinterpret_cast<TIO*>(dyn + tile + (size_t)cap * dv * sizeof(float));
  TS* s0 = static_cast<TS*>(a.S0) + ((size_t)b * H + h) * dv * DK;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
    mbar_arrive_expect_tx(&bar, tile);
    bulk_g2s(tile_s, s0, tile, &bar);
  }

  // The path's log(gamma), w rows and keys are fetched from the unchecked path (its length and
  // nodes clamped into range, so every read is in bounds) while the path is being checked; they
  // are used only if the check passes, and then they are the path's.
  const int Lu = path_prefetch(a, b, pc);  // its barrier also publishes the initialised mbarrier
  auto node_at = [&](int r) {  // the unchecked entry, clamped into [0, N)
    const int n = pc.path[r];
    return n < 0 ? 0 : (n >= N ? N - 1 : n);
  };
  for (int r = threadIdx.x; r < Lu; r += kThreads) coef[r] = a.log_gamma[((size_t)b * N + node_at(r)) * H + h];
  for (int x = threadIdx.x; x < Lu * dv; x += kThreads) {
    const int r = x / dv, rr = x % dv;
    wsm[x] = a.pseudo_v[(((size_t)b * N + node_at(r)) * H + h) * dv + rr];
  }
  constexpr int KV = DK * (int)sizeof(TIO) / 16;  // 16-byte vectors per key
  for (int x = threadIdx.x; x < Lu * KV; x += kThreads) {
    const int r = x / KV, c = x % KV;
    reinterpret_cast<uint4*>(ksm + (size_t)r * DK)[c] =
        __ldg(reinterpret_cast<const uint4*>(static_cast<const TIO*>(a.k) + (((size_t)b * N + node_at(r)) * H + h) * DK) + c);
  }
  const int st = check_prefetched_path(a, b, pc);  // barriers inside
  if (layer == 0 && h == 0 && threadIdx.x == 0) a.err[b] = st;
  // Every thread sees the tile through the barrier itself; a CTA that leaves early still waits
  // for the copy (bounded) so that it does not outlive the CTA's shared memory.
  const bool landed = mbar_wait(&bar, 0);
  if (st || !landed) {
    if (threadIdx.x == 0 && !st && !landed) a.err[b] = TV_ERR_TIMEOUT;
    return;
  }
  const int L = pc.L;
  if (threadIdx.x == 0) lga_s = coef[L - 1];
  __syncthreads();
  const float lga = lga_s;
  const float gam = expf(lga);
  const int lane8 = threadIdx.x % kLPR, rl = threadIdx.x / kLPR;
  for (int p = 0; p < passes; ++p) {
    TS* row = tile_s + (size_t)(p * kRows + rl) * DK + lane8 * 8;
    float cur[CPL];
#pragma unroll
    for (int j = 0; j < CPL / 8; ++j) load_vec_rw<8>(row + j * kStride, cur + 8 * j);
#pragma unroll
    for (int e = 0; e < CPL; ++e) cur[e] *= gam;
    for (int r = 0; r < L; ++r) {
      const float c = expf(lga - coef[r]) * wsm[r * dv + p * kRows + rl];
      const TIO* kr = ksm + (size_t)r * DK + lane8 * 8;
#pragma unroll
      for (int j = 0; j < CPL / 8; ++j) {
        float kf[8];
        if constexpr (sizeof(TIO) == 2) {
          unpack8(*reinterpret_cast<const uint4*>(kr + j * kStride), kf);
        } else {
          const float4 x0 = *reinterpret_cast<const float4*>(kr + j * kStride);
          const float4 x1 = *reinterpret_cast<const float4*>(kr + j * kStride + 4);
          kf[0] = x0.x; kf[1] = x0.y; kf[2] = x0.z; kf[3] = x0.w;
          kf[4] = x1.x; kf[5] = x1.y; kf[6] = x1.z; kf[7] = x1.w;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) cur[8 * j + e] = fmaf(c, kf[e], cur[8 * j + e]);
      }
    }
#pragma unroll
    for (int j = 0; j < CPL / 8; ++j) store_vec<8>(row + j * kStride, cur + 8 * j);
  }
  fence_async_shared();  // the bulk store reads the tile through the async proxy
  __syncthreads();
  if (threadIdx.x == 0) {
    bulk_s2g(s0, tile_s, tile);
    bulk_commit();
    bulk_wait_read<0>();
  }
}

// The same commit for paths too long to stage beside the tile: thread (row rl, lane) loads rows
// rl, rl + 32, ... of the head into registers before the path check and stores them back.
template <typename TIO, typename TS, int DK>
__global__ void __launch_bounds__(kThreads, 4) commit_wy_regs_kernel(CommitArgs a0) {
  constexpr int CPL = DK / kLPR;
  __shared__ PathCheck pc;
  __shared__ float coef[TV_MAX_NODES];
  __shared__ float lga_s;
  extern __shared__ __align__(128) unsigned char dyn[];  // w [cap][dv] fp32, then k [cap][DK]
  constexpr int P = 4;                 // passes of 32 rows: dv <= 128
  const int layer = blockIdx.x / (a0.B * a0.H), bh = blockIdx.x % (a0.B * a0.H);
  const CommitArgs a = layer_view(a0, layer);
  const int passes = a.dv / kRows;
  const int b = bh / a.H, h = bh % a.H;
  const int N = a.N, H = a.H, dv = a.dv;
  const int cap = a.Lmax < N ? a.Lmax : N;
  float* wsm = reinterpret_cast<float*>(dyn);
  TIO* ksm = reinterpret_cast<TIO*>(dyn + (size_t)cap * dv * sizeof(float));

  const int lane8 = threadIdx.x % kLPR, rl = threadIdx.x / kLPR;
  TS* s0 = static_cast<TS*>(a.S0) + (((size_t)b * H + h) * dv + rl) * DK + lane8 * 8;
  // The rows as stored (8-column chunks of 16 or 32 bytes), converted only when they are used.
  constexpr int VPC = 8 * (int)sizeof(TS) / 16;  // 16-byte vectors per chunk
  uint4 raw[P][CPL / 8][VPC];
#pragma unroll
  for (int p = 0; p < P; ++p)
    if (p < passes)
#pragma unroll
      for (int j = 0; j < CPL / 8; ++j)
#pragma unroll
        for (int u = 0; u < VPC; ++u)
          raw[p][j][u] = reinterpret_cast<const uint4*>(s0 + (size_t)p * kRows * DK + j * kStride)[u];

  // The path's log(gamma), w rows and keys are fetched from the unchecked path (its length and
  // nodes clamped into range, so every read is in bounds) while the path is being checked; they
  // are used only if the check passes, and then they are the path's.
  const int Lu = path_prefetch(a, b, pc);
  auto node_at = [&](int r) {  // the unchecked entry, clamped into [0, N)
    const int n = pc.path[r];
    return n < 0 ? 0 : (n >= N ? N - 1 : n);
  };
  for (int r = threadIdx.x; r < Lu; r += kThreads) coef[r] = a.log_gamma[((size_t)b * N + node_at(r)) * H + h];
  for (int x = threadIdx.x; x < Lu * dv; x += kThreads) {
    const int r = x / dv, rr = x % dv;
    wsm[x] = a.pseudo_v[(((size_t)b * N + node_at(r)) * H + h) * dv + rr];
  }
  constexpr int KV = DK * (int)sizeof(TIO) / 16;  // 16-byte vectors per key
  for (int x = threadIdx.x; x < Lu * KV; x += kThreads) {
    const int r = x / KV, c = x % KV;
    reinterpret_cast<uint4*>(ksm + (size_t)r * DK)[c] =
        __ldg(reinterpret_cast<const uint4*>(static_cast<const TIO*>(a.k) + (((size_t)b * N + node_at(r)) * H + h) * DK) + c);
  }
  const int st = check_prefetched_path(a, b, pc);  // barriers inside
  if (layer == 0 && h == 0 && threadIdx.x == 0) a.err[b] = st;
  if (st) return;
  const int L = pc.L;
  if (threadIdx.x == 0) lga_s = coef[L - 1];
  __syncthreads();
  const float lga = lga_s;
  const float gam = expf(lga);
#pragma unroll
  for (int p = 0; p < P; ++p) {
    if (p >= passes) break;
    float cur[CPL];
#pragma unroll
    for (int j = 0; j < CPL / 8; ++j) {
      if constexpr (sizeof(TS) == 2) {
        unpack8(raw[p][j][0], cur + 8 * j);
      } else {
        const uint4 x0 = raw[p][j][0], x1 = raw[p][j][VPC - 1];
        cur[8 * j] = __uint_as_float(x0.x); cur[8 * j + 1] = __uint_as_float(x0.y);
        cur[8 * j + 2] = __uint_as_float(x0.z); cur[8 * j + 3] = __uint_as_float(x0.w);
        cur[8 * j + 4] = __uint_as_float(x1.x); cur[8 * j + 5] = __uint_as_float(x1.y);
        cur[8 * j + 6] = __uint_as_float(x1.z); cur[8 * j + 7] = __uint_as_float(x1.w);
      }
    }
#pragma unroll
    for (int e = 0; e < CPL; ++e) cur[e] *= gam;
    for (int r = 0; r < L; ++r) {
      const float c = expf(lga - coef[r]) * wsm[r * dv + p * kRows + rl];
      const TIO* kr = ksm + (size_t)r * DK + lane8 * 8;
#pragma unroll
      for (int j = 0; j < CPL / 8; ++j) {
        float kf[8];
        if constexpr (sizeof(TIO) == 2) {
          unpack8(*reinterpret_cast<const uint4*>(kr + j * kStride), kf);
        } else {
          const float4 x0 = *reinterpret_cast<const float4*>(kr + j * kStride);
          const float4 x1 = *reinterpret_cast<const float4*>(kr + j * kStride + 4);
          kf[0] = x0.x; kf[1] = x0.y; kf[2] = x0.z; kf[3] = x0.w;
          kf[4] = x1.x; kf[5] = x1.y; kf[6] = x1.z; kf[7] = x1.w;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) cur[8 * j + e] = fmaf(c, kf[e], cur[8 * j + e]);
      }
    }
#pragma unroll
    for (int j = 0; j < CPL / 8; ++j) store_vec<8>(s0 + (size_t)p * kRows * DK + j * kStride, cur + 8 * j);
  }
}

// Commit after a selective fork (qwen35-tree-spec §六, 选择性 Fork): one CTA per (sequence,
// head).  The accepted path is resumed from its deepest node that kept a snapshot (S_0 if none)
// and the rest of the path is replayed with the gated delta rule,
//     S <- alpha_j S + w k_j^T,   w = beta_j (v_j - alpha_j S k_j),
// thread (row rl, lane) holding rows rl, rl + 32, ... in the interleaved 8-column chunks.
template <typename TIO, typename TS, int DK>
__global__ void __launch_bounds__(kThreads) commit_replay_kernel(CommitArgs a, ReplayArgs rp) {
  constexpr int CPL = DK / kLPR;
  __shared__ PathCheck pc;
  __shared__ int start_r;      // path index of the snapshot resumed from (-1: S_0)
  __shared__ int start_slot;
  __shared__ float al_s[TV_MAX_NODES], be_s[TV_MAX_NODES];
  extern __shared__ __align__(16) float ksm[];  // keys of the replayed nodes, [steps][DK]
  const int b = blockIdx.x / a.H, h = blockIdx.x % a.H;
  const int N = a.N, H = a.H, dv = a.dv;
  const int st = check_path(a, b, pc);
  if (h == 0 && threadIdx.x == 0) a.err[b] = st;
  if (st) return;
  const int L = pc.L;
  if (threadIdx.x == 0) {
    int r0 = -1, sl = -1;
    for (int r = L - 1; r >= 0; --r) {
      const int s = rp.slot[(size_t)b * N + pc.path[r]];
      if (s >= 0 && s < rp.capacity) { r0 = r; sl = s; break; }
    }
    start_r = r0;
    start_slot = sl;
  }
  __syncthreads();
  const int r0 = start_r, steps = L - 1 - r0;
  for (int x = threadIdx.x; x < steps; x += kThreads) {
    const size_t nh = ((size_t)b * N + pc.path[r0 + 1 + x]) * H + h;
    al_s[x] = rp.alpha[nh];
    be_s[x] = rp.beta[nh];
  }
  for (int x = threadIdx.x; x < steps * DK; x += kThreads) {
    const int t = x / DK, c = x % DK;
    ksm[x] = to_f32(static_cast<const TIO*>(a.k)[(((size_t)b * N + pc.path[r0 + 1 + t]) * H + h) * DK + c]);
  }
  __syncthreads();
  const int lane8 = threadIdx.x % kLPR, rl = threadIdx.x / kLPR;
  const TS* src = r0 < 0 ? static_cast<const TS*>(a.S0) + ((size_t)b * H + h) * dv * DK
                         : static_cast<const TS*>(a.node_states) + (((size_t)b * rp.capacity + start_slot) * H + h) * dv * DK;
  TS* dst = static_cast<TS*>(a.S0) + ((size_t)b * H + h) * dv * DK;
  const TIO* v = static_cast<const TIO*>(rp.v);
  for (int p = 0; p < dv / kRows; ++p) {  // the same trip count in every thread
    const int row = p * kRows + rl;
    float cur[CPL];
#pragma unroll
    for (int j = 0; j < CPL / 8; ++j) load_vec_rw<8>(src + (size_t)row * DK + lane8 * 8 + j * kStride, cur + 8 * j);
    for (int t = 0; t < steps; ++t) {
      const float* kt = ksm + t * DK + lane8 * 8;
      float pk = 0.f;
#pragma unroll
      for (int j = 0; j < CPL / 8; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) pk = fmaf(cur[8 * j + e], kt[j * kStride + e], pk);
      pk = group_sum<kLPR>(pk);
      const float al = al_s[t];
      const size_t nh = ((size_t)b * N + pc.path[r0 + 1 + t]) * H + h;
      const float w = be_s[t] * (to_f32(v[nh * dv + row]) - al * pk);
#pragma unroll
      for (int j = 0; j < CPL / 8; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) cur[8 * j + e] = fmaf(w, kt[j * kStride + e], al * cur[8 * j + e]);
    }
    __syncthreads();  // every thread has read its source rows before any S_0 row is written
#pragma unroll
    for (int j = 0; j < CPL / 8; ++j) store_vec<8>(dst + (size_t)row * DK + lane8 * 8 + j * kStride, cur + 8 * j);
  }
}

template <typename TIO, typename TS, int DK>
cudaError_t launch_replay_t(const CommitArgs& a, const ReplayArgs& r, cudaStream_t s) {
  const int cap = a.Lmax < a.N ? a.Lmax : a.N;
  const size_t smem = (size_t)cap * DK * sizeof(float);
  auto kern = commit_replay_kernel<TIO, TS, DK>;
  // (static + dynamic shared memory may pass 48 KB with a dynamic part below it)
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<a.B * a.H, kThreads, smem, s>>>(a, r);
  return cudaGetLastError();
}

template <typename TS>
cudaError_t launch_fork_commit_t(const CommitArgs& a, cudaStream_t s) {
  const size_t smem = (size_t)a.dv * a.dk * sizeof(TS);
  auto kern = commit_fork_kernel<TS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<a.layers * a.B * a.H, kForkThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <typename TIO, typename TS, int DK>
cudaError_t launch_wy_t(const CommitArgs& a, cudaStream_t s) {
  const int cap = a.Lmax < a.N ? a.Lmax : a.N;  // a valid path has distinct nodes
  const size_t rows = (size_t)cap * (a.dv * sizeof(float) + DK * sizeof(TIO));
  const size_t tile = (size_t)a.dv * DK * sizeof(TS);
  // The tile beside the path rows when both fit with the kernel's static shared memory, else
  // the tile through registers.
  cudaFuncAttributes fa;
  cudaError_t e0 = cudaFuncGetAttributes(&fa, commit_wy_kernel<TIO, TS, DK>);
  if (e0 != cudaSuccess) return e0;
  const bool staged = fa.sharedSizeBytes + tile + rows <= (size_t)227 * 1024;
  const size_t smem = staged ? tile + rows : rows;
  auto kern = staged ? commit_wy_kernel<TIO, TS, DK> : commit_wy_regs_kernel<TIO, TS, DK>;
  // (static + dynamic shared memory may pass 48 KB with a dynamic part below it)
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<a.layers * a.B * a.H, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gdn_commit_replay(const CommitArgs& a, const ReplayArgs& r, cudaStream_t s) {
  if (a.io == TV_F32 && a.state == TV_F32)
    return a.dk == 64 ? launch_replay_t<float, float, 64>(a, r, s) : launch_replay_t<float, float, 128>(a, r, s);
  if (a.io == TV_BF16 && a.state == TV_BF16)
    return a.dk == 64 ? launch_replay_t<bf16, bf16, 64>(a, r, s) : launch_replay_t<bf16, bf16, 128>(a, r, s);
  return a.dk == 64 ? launch_replay_t<bf16, float, 64>(a, r, s) : launch_replay_t<bf16, float, 128>(a, r, s);
}

cudaError_t launch_gdn_commit(const CommitArgs& a, cudaStream_t s) {
  if (a.mode == TV_MODE_FORK)
    return a.state == TV_F32 ? launch_fork_commit_t<float>(a, s) : launch_fork_commit_t<bf16>(a, s);
  if (a.io == TV_F32 && a.state == TV_F32)
    return a.dk == 64 ? launch_wy_t<float, float, 64>(a, s) : launch_wy_t<float, float, 128>(a, s);
  if (a.io == TV_BF16 && a.state == TV_BF16)
    return a.dk == 64 ? launch_wy_t<bf16, bf16, 64>(a, s) : launch_wy_t<bf16, bf16, 128>(a, s);
  return a.dk == 64 ? launch_wy_t<bf16, float, 64>(a, s) : launch_wy_t<bf16, float, 128>(a, s);
}

}  // namespace tv
