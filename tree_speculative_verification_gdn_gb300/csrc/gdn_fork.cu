// Fork/checkpoint GDN tree verify (qwen35-tree-spec, §四 Fork/Checkpoint and 逐深度处理).
//
// Every node i evolves from its parent's state (S_0 for a root):
//     S_i = alpha_i S_p (I - beta_i k_i k_i^T) + beta_i v_i k_i^T = alpha_i S_p + w_i k_i^T,
//     w_i = beta_i (v_i - alpha_i S_p k_i),   o_i = S_i (q_scale q_i),
// and every S_i is written out (the checkpoint the commit step restores).
//
// The rows of S (value index r) evolve independently: row r only needs k_i, q_i, v_i[r],
// alpha_i, beta_i.  A CTA therefore owns a slab of 16 rows of one (sequence, head), keeps
// their fp32 state on chip and walks the whole tree once, depth-first, instead of one launch
// per depth reading every parent snapshot back from HBM.  HBM traffic is the floor: S_0 read
// once per root, each checkpoint written once.  Each row is held by 8 lanes (dk/8 columns
// each), so a dot product costs 3 shuffles.  The inputs of the next 8 nodes (k, q and the
// slab's v) stream into a shared-memory ring through bulk asynchronous copies; k and q of the
// next node are converted once to fp32 for all 32 rows of the CTA.
//
// Depth-first order visits a node's light children first and its heaviest child (largest
// subtree) last.  A branching node pushes its state to a shared-memory slot that its later
// children read back; the first child takes the state straight from registers.  With
// heavy-last order a slot is at most 1 + (number of light edges above the node) and each
// light edge halves the subtree, so slots 1..7 cover every tree of <= 256 nodes (a branching
// node has >= 3 nodes in its subtree, so it sits below at most 6 light edges); the launch
// sizes the stack for the bound of its N (slots_for).
#include "tv_async.cuh"
#include "tv_common.cuh"
#include "tv_internal.h"

namespace tv {
namespace {

constexpr int kLPR = 8;                 // lanes per state row
constexpr int kRows = 32;               // state rows per CTA
constexpr int kThreads = kLPR * kRows;  // 256
constexpr int kSlots = 7;               // on-chip state slots 1..7 (S_0 is re-read for a root)
constexpr int kStages = 8;              // depth of the node-input ring

struct Sched {
  int par[TV_MAX_NODES];
  int depth[TV_MAX_NODES];
  int size[TV_MAX_NODES];
  int nchild[TV_MAX_NODES];
  int hkey[TV_MAX_NODES];    // (size << 9) | (511 - child): heaviest child, lowest index on ties
  int acc[TV_MAX_NODES];     // running offset of light children
  int before[TV_MAX_NODES];  // nodes of earlier siblings' subtrees
  int pre[TV_MAX_NODES];     // depth-first position
  int order[TV_MAX_NODES];   // node at each depth-first position
  int src[TV_MAX_NODES];     // where the parent state comes from: -1 registers, else a slot
  int push[TV_MAX_NODES];    // slot the node's own state goes to (-1: not needed later)
  int flag, maxdepth, root_acc, maxslot;
};

// Depth-first schedule of one tree, built by the whole CTA.  Returns 0, TV_ERR_BAD_TREE or
// TV_ERR_UNSUPPORTED (stack deeper than kSlots; impossible for N <= 256).
__device__ int build_schedule(const int32_t* __restrict__ parents, int N, Sched& s) {
  const int tid = threadIdx.x, nt = blockDim.x;
  int st = load_and_check_tree(parents, N, s.par, &s.flag);
  if (st) return st;
  if (tid == 0) { s.maxdepth = 0; s.root_acc = 0; s.maxslot = 0; }
  for (int i = tid; i < N; i += nt) {
    s.size[i] = 1; s.nchild[i] = 0; s.hkey[i] = 0; s.acc[i] = 0; s.order[i] = -1;
  }
  __syncthreads();
  for (int i = tid; i < N; i += nt) {
    const int d = node_depth(s.par, i);
    s.depth[i] = d;
    atomicMax(&s.maxdepth, d);
    if (s.par[i] >= 0) atomicAdd(&s.nchild[s.par[i]], 1);
  }
  __syncthreads();
  // Subtree sizes, one depth level at a time from the deepest.
  for (int d = s.maxdepth; d >= 1; --d) {
    for (int i = tid; i < N; i += nt)
      if (s.depth[i] == d) atomicAdd(&s.size[s.par[i]], s.size[i]);
    __syncthreads();
  }
  for (int i = tid; i < N; i += nt) {
    const int p = s.par[i];
    if (p >= 0) atomicMax(&s.hkey[p], (s.size[i] << 9) | (511 - i));
  }
  __syncthreads();
  // Offset of each node among its siblings: light children in arbitrary (atomic) order,
  // the heavy child after all of them; roots one after another.
  for (int i = tid; i < N; i += nt) {
    const int p = s.par[i];
    if (p < 0) {
      s.before[i] = atomicAdd(&s.root_acc, s.size[i]);
    } else {
      const int heavy = 511 - (s.hkey[p] & 511);
      s.before[i] = (i == heavy) ? s.size[p] - 1 - s.size[i] : atomicAdd(&s.acc[p], s.size[i]);
    }
  }
  __syncthreads();
  for (int i = tid; i < N; i += nt) {
    int pre = -1, light = 0;
    // pre is in [0, N) for a valid tree; the check keeps a broken invariant from indexing out.
    for (int a = i; a >= 0; a = s.par[a]) {
      pre += 1 + s.before[a];
      const int p = s.par[a];
      if (p >= 0 && a != 511 - (s.hkey[p] & 511)) ++light;
    }
    s.pre[i] = pre;
    if (pre >= 0 && pre < N) s.order[pre] = i;
    else s.flag = 1;
    const int slot = s.nchild[i] >= 2 ? 1 + light : -1;
    s.push[i] = slot;
    if (slot > 0) atomicMax(&s.maxslot, slot);
  }
  __syncthreads();
  for (int i = tid; i < N; i += nt) {
    const int p = s.par[i];
    s.src[i] = (p < 0) ? 0 : (s.pre[i] == s.pre[p] + 1 ? -1 : s.push[p]);
    if (s.order[i] < 0 || s.src[i] > kSlots) s.flag = 1;  // never expected: guards every index
  }
  __syncthreads();
  return (s.maxslot <= kSlots && !s.flag) ? 0 : TV_ERR_UNSUPPORTED;
}

// Raw inputs of one node for the CTA's (sequence, head, row slab), filled by bulk async copies.
template <typename TIO, int DK>
struct Stage {
  TIO k[DK];
  TIO q[DK];
  TIO v[kRows];
};

// Stack slots a tree of n nodes can need: a branching node below L light edges has at least
// 2^(L+2) - 1 nodes in the tree, and it pushes to slot L + 1.
__host__ __device__ constexpr int slots_for(int n) {
  int L = 0;
  while ((1 << (L + 3)) - 1 <= n) ++L;
  return L + 1;
}

template <typename TIO, typename TS, int DK>
__global__ void __launch_bounds__(kThreads) gdn_fork_kernel(GdnArgs a, TS* __restrict__ states,
                                                            int ctas_per_seq, int nslots) {
  constexpr int CPL = DK / kLPR;  // columns per lane
  constexpr int Q4 = CPL / 4;     // float4 per lane per slot
  using StageT = Stage<TIO, DK>;
  extern __shared__ __align__(128) unsigned char smem[];
  Sched& sc = *reinterpret_cast<Sched*>(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + sizeof(Sched));
  float* s_alpha = reinterpret_cast<float*>(bars + kStages);
  float* s_beta = s_alpha + TV_MAX_NODES;
  float* kq32 = s_beta + TV_MAX_NODES;                    // [2][2][DK]: k, q of two nodes in fp32
  StageT* ring = reinterpret_cast<StageT*>(kq32 + 4 * DK);
  float4* stack = reinterpret_cast<float4*>(ring + kStages);

  const int b = blockIdx.x / ctas_per_seq, g = blockIdx.x % ctas_per_seq;
  const int N = a.N, H = a.H, dv = a.dv;
  const int tid = threadIdx.x;
  const int status = build_schedule(a.parents + (size_t)b * N, N, sc);
  if (g == 0 && tid == 0) a.err[b] = (status || sc.maxslot <= nslots) ? status : TV_ERR_UNSUPPORTED;
  if (status || sc.maxslot > nslots) return;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    mbar_fence_init();
  }
  __syncthreads();

  const TIO* __restrict__ q = static_cast<const TIO*>(a.q);
  const TIO* __restrict__ k = static_cast<const TIO*>(a.k);
  const TIO* __restrict__ v = static_cast<const TIO*>(a.v);
  const TS* __restrict__ S0 = static_cast<const TS*>(a.S0);
  TIO* __restrict__ out = static_cast<TIO*>(a.out);
  const int lane = tid % kLPR, rl = tid / kLPR;
  const int slabs = dv / kRows, items = H * slabs;
  const float q_scale = a.q_scale;
  const size_t node_stride = (size_t)H * dv;     // elements between consecutive nodes (out, v)
  const size_t state_stride = node_stride * DK;  // elements between consecutive nodes (states)
  uint32_t seq = 0;      // node loads issued and consumed by this CTA before the current item
  bool timed_out = false;

  for (int item = g; item < items; item += ctas_per_seq) {
    const int h = item / slabs, r0 = (item % slabs) * kRows, r = r0 + rl;
    const size_t nh0 = (size_t)b * N * H + h;    // (b, node 0, h)
    auto issue = [&](uint32_t s, int node) {     // one thread: start the loads of node into stage s
      const size_t nh = nh0 + (size_t)node * H;
      StageT& st = ring[s % kStages];
      uint64_t* bar = &bars[s % kStages];
      mbar_arrive_expect_tx(bar, sizeof(StageT));
      bulk_g2s(st.k, k + nh * DK, DK * sizeof(TIO), bar);
      bulk_g2s(st.q, q + nh * DK, DK * sizeof(TIO), bar);
      bulk_g2s(st.v, v + nh * dv + r0, kRows * sizeof(TIO), bar);
    };
    // k and q of stage s -> fp32 buffer `buf` (every thread converts a few elements)
    auto convert = [&](uint32_t s, int buf) {
      if (!mbar_wait(&bars[s % kStages], (s / kStages) & 1u)) timed_out = true;
      const StageT& st = ring[s % kStages];
      float* dst = kq32 + buf * 2 * DK;
      for (int e = tid; e < 2 * DK; e += kThreads) dst[e] = to_f32(e < DK ? st.k[e] : st.q[e - DK]);
    };
    for (int i = tid; i < N; i += kThreads) {
      s_alpha[i] = __ldg(a.alpha + nh0 + (size_t)i * H);
      s_beta[i] = __ldg(a.beta + nh0 + (size_t)i * H);
    }
    if (tid == 0)
      for (int t = 0; t < N && t < kStages; ++t) issue(seq + t, sc.order[t]);
    convert(seq, 0);
    __syncthreads();

    const TS* s0row = S0 + (((size_t)b * H + h) * dv + r) * DK + lane * CPL;
    TIO* out_r = out + nh0 * dv + r;
    TS* st_r = states + (nh0 * dv + r) * DK + lane * CPL;
    float cur[CPL];
    for (int t = 0; t < N; ++t) {
      const int i = sc.order[t];
      const uint32_t s = seq + t;
      if (t + 1 < N) convert(s + 1, (t + 1) & 1);   // next node's k, q (read after the barrier)
      const int src = sc.src[i], push = sc.push[i];
      if (src == 0) {
        load_vec<CPL>(s0row, cur);  // a root starts from the committed state
      } else if (src > 0) {
#pragma unroll
        for (int j = 0; j < Q4; ++j) {
          const float4 f = stack[((src - 1) * Q4 + j) * kThreads + tid];
          cur[4 * j] = f.x; cur[4 * j + 1] = f.y; cur[4 * j + 2] = f.z; cur[4 * j + 3] = f.w;
        }
      }
      const float* kf = kq32 + (t & 1) * 2 * DK + lane * CPL;
      const float* qf = kf + DK;
      const float vr = to_f32(ring[s % kStages].v[rl]);
      const float al = s_alpha[i], be = s_beta[i];
      float t0 = 0.f, t1 = 0.f;
#pragma unroll
      for (int e = 0; e < CPL; e += 2) {
        t0 = fmaf(cur[e], kf[e], t0);
        t1 = fmaf(cur[e + 1], kf[e + 1], t1);
      }
      const float tk = group_sum<kLPR>(t0 + t1);      // (S_p k_i)_r
      const float w = be * (vr - al * tk);            // pseudo-value w_i[r]
      float o0 = 0.f, o1 = 0.f;
#pragma unroll
      for (int e = 0; e < CPL; e += 2) {
        cur[e] = fmaf(w, kf[e], al * cur[e]);
        cur[e + 1] = fmaf(w, kf[e + 1], al * cur[e + 1]);
        o0 = fmaf(cur[e], qf[e], o0);
        o1 = fmaf(cur[e + 1], qf[e + 1], o1);
      }
      const float ov = group_sum<kLPR>(o0 + o1);      // (S_i q_i)_r
      if (lane == 0) out_r[(size_t)i * node_stride] = from_f32<TIO>(ov * q_scale);
      store_vec_cs<CPL>(st_r + (size_t)i * state_stride, cur);
      if (push > 0) {
#pragma unroll
        for (int j = 0; j < Q4; ++j)
          stack[((push - 1) * Q4 + j) * kThreads + tid] =
              make_float4(cur[4 * j], cur[4 * j + 1], cur[4 * j + 2], cur[4 * j + 3]);
      }
      __syncthreads();  // stage s is free again; the converted next node is visible
      if (tid == 0 && t + kStages < N) issue(s + kStages, sc.order[t + kStages]);
    }
    seq += N;
  }
  if (timed_out) a.err[b] = TV_ERR_TIMEOUT;
}

template <typename TIO, typename TS, int DK>
cudaError_t launch_fork_t(const GdnArgs& a, void* states, cudaStream_t s) {
  auto kern = gdn_fork_kernel<TIO, TS, DK>;
  const int nslots = slots_for(a.N);
  const size_t smem = sizeof(Sched) + kStages * sizeof(uint64_t) + 2 * TV_MAX_NODES * sizeof(float) +
                      4 * DK * sizeof(float) + kStages * sizeof(Stage<TIO, DK>) +
                      (size_t)nslots * (DK / kLPR / 4) * kThreads * sizeof(float4);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
  if (e != cudaSuccess) return e;
  const int items = a.H * (a.dv / kRows);
  const int slots = device_sm_count() * (occ > 0 ? occ : 1);
  int per_seq = slots / a.B;
  if (per_seq < 1) per_seq = 1;
  if (per_seq > items) per_seq = items;
  kern<<<a.B * per_seq, kThreads, smem, s>>>(a, static_cast<TS*>(states), per_seq, nslots);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gdn_fork(const GdnArgs& a, void* node_states, cudaStream_t s) {
  static_assert(sizeof(Sched) % 16 == 0, "stack must start 16-byte aligned");
  if (a.io == TV_F32 && a.state == TV_F32)
    return a.dk == 64 ? launch_fork_t<float, float, 64>(a, node_states, s)
                      : launch_fork_t<float, float, 128>(a, node_states, s);
  if (a.io == TV_BF16 && a.state == TV_BF16)
    return a.dk == 64 ? launch_fork_t<bf16, bf16, 64>(a, node_states, s)
                      : launch_fork_t<bf16, bf16, 128>(a, node_states, s);
  return a.dk == 64 ? launch_fork_t<bf16, float, 64>(a, node_states, s)
                    : launch_fork_t<bf16, float, 128>(a, node_states, s);
}

}  // namespace tv
