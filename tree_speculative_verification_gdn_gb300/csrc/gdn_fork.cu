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
// once, each checkpoint written once.  Each row is held by 8 lanes (dk/8 columns each), so a
// dot product costs 3 shuffles.
//
// Depth-first order visits a node's light children first and its heaviest child (largest
// subtree) last.  A branching node pushes its state to a shared-memory slot that its later
// children read back; the first child takes the state straight from registers.  With
// heavy-last order a slot is at most 1 + (number of light edges above the node) and each
// light edge halves the subtree, so 8 slots (S_0 + 7) cover every tree of <= 256 nodes.
#include "tv_common.cuh"
#include "tv_internal.h"

namespace tv {
namespace {

constexpr int kLPR = 8;                 // lanes per state row
constexpr int kRows = 16;               // state rows per CTA
constexpr int kThreads = kLPR * kRows;  // 128
constexpr int kSlots = 8;               // on-chip state slots: S_0 + 7 branch points

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
    if (s.order[i] < 0 || s.src[i] >= kSlots) s.flag = 1;  // never expected: guards every index
  }
  __syncthreads();
  return (s.maxslot < kSlots && !s.flag) ? 0 : TV_ERR_UNSUPPORTED;
}

template <typename TIO, int CPL>
struct NodeIn {
  float k[CPL], q[CPL];
  float v, alpha, beta;
  __device__ __forceinline__ void load(const TIO* __restrict__ kp, const TIO* __restrict__ qp,
                                       const TIO* __restrict__ vp, const float* __restrict__ ap,
                                       const float* __restrict__ bp) {
    load_vec<CPL>(kp, k);
    load_vec<CPL>(qp, q);
    v = to_f32(__ldg(vp));
    alpha = __ldg(ap);
    beta = __ldg(bp);
  }
};

template <typename TIO, typename TS, int DK>
__global__ void __launch_bounds__(kThreads) gdn_fork_kernel(GdnArgs a, TS* __restrict__ states,
                                                            int ctas_per_seq) {
  constexpr int CPL = DK / kLPR;  // columns per lane
  constexpr int Q4 = CPL / 4;     // float4 per lane per slot
  extern __shared__ __align__(16) unsigned char smem[];
  Sched& sc = *reinterpret_cast<Sched*>(smem);
  float4* stack = reinterpret_cast<float4*>(smem + sizeof(Sched));

  const int b = blockIdx.x / ctas_per_seq, g = blockIdx.x % ctas_per_seq;
  const int N = a.N, H = a.H, dv = a.dv;
  const int status = build_schedule(a.parents + (size_t)b * N, N, sc);
  if (g == 0 && threadIdx.x == 0) a.err[b] = status;
  if (status) return;

  const TIO* __restrict__ q = static_cast<const TIO*>(a.q);
  const TIO* __restrict__ k = static_cast<const TIO*>(a.k);
  const TIO* __restrict__ v = static_cast<const TIO*>(a.v);
  const TS* __restrict__ S0 = static_cast<const TS*>(a.S0);
  TIO* __restrict__ out = static_cast<TIO*>(a.out);

  const int tid = threadIdx.x, lane8 = tid & (kLPR - 1), rl = tid / kLPR;
  const int slabs = dv / kRows, items = H * slabs;
  const float q_scale = a.q_scale;

  for (int item = g; item < items; item += ctas_per_seq) {
    const int h = item / slabs;
    const int r = (item % slabs) * kRows + rl;
    float cur[CPL];
    load_vec<CPL>(S0 + (((size_t)b * H + h) * dv + r) * DK + lane8 * CPL, cur);
#pragma unroll
    for (int j = 0; j < Q4; ++j)
      stack[j * kThreads + tid] = make_float4(cur[4 * j], cur[4 * j + 1], cur[4 * j + 2], cur[4 * j + 3]);

    auto in_ptrs = [&](int node, NodeIn<TIO, CPL>& x) {
      const size_t nh = ((size_t)b * N + node) * H + h;
      x.load(k + nh * DK + lane8 * CPL, q + nh * DK + lane8 * CPL, v + nh * dv + r,
             a.alpha + nh, a.beta + nh);
    };
    NodeIn<TIO, CPL> cin, nin;
    int i = sc.order[0];
    in_ptrs(i, cin);
    for (int t = 0; t < N; ++t) {
      const int inext = (t + 1 < N) ? sc.order[t + 1] : i;
      in_ptrs(inext, nin);  // prefetch the next node's inputs
      const int src = sc.src[i], push = sc.push[i];
      if (src >= 0) {
#pragma unroll
        for (int j = 0; j < Q4; ++j) {
          const float4 f = stack[(src * Q4 + j) * kThreads + tid];
          cur[4 * j] = f.x; cur[4 * j + 1] = f.y; cur[4 * j + 2] = f.z; cur[4 * j + 3] = f.w;
        }
      }
      float tk = 0.f;
#pragma unroll
      for (int e = 0; e < CPL; ++e) tk = fmaf(cur[e], cin.k[e], tk);
      tk = group_sum<kLPR>(tk);                       // (S_p k_i)_r
      const float w = cin.beta * (cin.v - cin.alpha * tk);  // pseudo-value w_i[r]
      float ov = 0.f;
#pragma unroll
      for (int e = 0; e < CPL; ++e) {
        cur[e] = fmaf(w, cin.k[e], cin.alpha * cur[e]);
        ov = fmaf(cur[e], cin.q[e], ov);
      }
      ov = group_sum<kLPR>(ov);                       // (S_i q_i)_r
      const size_t nh = ((size_t)b * N + i) * H + h;
      if (lane8 == 0) out[nh * dv + r] = from_f32<TIO>(ov * q_scale);
      store_vec_cs<CPL>(states + (nh * dv + r) * DK + lane8 * CPL, cur);
      if (push >= 0) {
#pragma unroll
        for (int j = 0; j < Q4; ++j)
          stack[(push * Q4 + j) * kThreads + tid] =
              make_float4(cur[4 * j], cur[4 * j + 1], cur[4 * j + 2], cur[4 * j + 3]);
      }
      i = inext;
      cin = nin;
    }
  }
}

template <typename TIO, typename TS, int DK>
cudaError_t launch_fork_t(const GdnArgs& a, void* states, cudaStream_t s) {
  auto kern = gdn_fork_kernel<TIO, TS, DK>;
  const size_t smem = sizeof(Sched) + (size_t)kSlots * (DK / kLPR / 4) * kThreads * sizeof(float4);
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
  kern<<<a.B * per_seq, kThreads, smem, s>>>(a, static_cast<TS*>(states), per_seq);
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
