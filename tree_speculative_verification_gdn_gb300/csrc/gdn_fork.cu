// Fork/checkpoint GDN tree verify (qwen35-tree-spec, §四 Fork/Checkpoint and 逐深度处理).
//
// Every node i evolves from its parent's state (S_0 for a root):
//     S_i = alpha_i S_p (I - beta_i k_i k_i^T) + beta_i v_i k_i^T = alpha_i S_p + w_i k_i^T,
//     w_i = beta_i (v_i - alpha_i S_p k_i),   o_i = S_i (q_scale q_i),
// and every S_i is written out (the checkpoint the commit step restores).
//
// The rows of S (value index r) evolve independently: row r only needs k_i, q_i, v_i[r],
// alpha_i, beta_i.  A CTA owns a slab of 16 rows of one (sequence, head) at a time -- a work
// unit; the grid is persistent and each CTA loops over its units (see the unit plan below) --
// keeps their fp32 state on chip and walks the whole tree once, depth-first, instead of one
// launch per depth reading every parent snapshot back from HBM.  HBM traffic is the floor: S_0
// read once per root, each checkpoint written once.  Each row is held by 8 lanes (dk/8 columns
// each, in interleaved 8-column chunks), so a row dot product costs 3 shuffles; k.q, the same
// for every row, comes from a per-unit table.  Column pairs use the paired fp32 FMA.  Every
// warp walks the tree on its own -- no barrier inside the node loop -- with the next node's k,
// q and v prefetched into registers; the CTA's warps share one (sequence, head), so k and q
// come from L1 after the first warp's read.  For bf16 inputs on small trees a lane group holds
// two rows (see RPL below).
//
// Depth-first order visits a node's leaf children first, then its light children, and its
// heaviest child (largest subtree) last.  A leaf's state only goes to its snapshot, so a leaf
// is computed from the parent state in registers without replacing it; the first non-leaf
// child then takes that state over.  A node with two or more non-leaf children pushes its
// state to a shared-memory slot that the later ones read back.  With heavy-last order a node
// pushes to slot 1 + (number of light edges above it); a pushing node has >= 5 nodes in its
// subtree (two non-leaf children) and each light edge above it at least doubles that plus
// one, so slot L + 1 needs a tree of >= g(L) nodes, g(0) = 5, g(L) = 2 g(L-1) + 1: slots
// 1..6 cover every tree of <= 256 nodes and the launch sizes the stack for the bound of its N
// (slots_for; 3 slots at N = 40).  On the k = 3, d = 3 tree an item makes 4 pushes and 8 pops
// instead of one push per branching node and one pop per later child (13 and 26).
#include "tv_common.cuh"
#include "tv_internal.h"

namespace tv {
namespace {

constexpr int kLPR = 8;                 // lanes per state row
constexpr int kRows = 16;               // state rows per CTA
constexpr int kLanes = kLPR * kRows;    // 128 lane slots: 8 per state row
constexpr int kSlots = 6;               // on-chip state slots 1..6 (S_0 is re-read for a root)
constexpr int kGroup = 16;              // CTAs that walk adjacent slabs side by side
// Column ownership: lane l of a row holds the chunks of 8 columns starting at l * 8 + j * kStride
// (j = 0 .. CPL / 8 - 1), so one chunk-wide access by the 8 lanes of a row covers kStride
// contiguous columns: full 32-byte sectors for every load and store of k, q, S_0 and states.
constexpr int kStride = 8 * kLPR;

// What the node loop needs from the schedule, plus the current item's decay / write strength.
struct Sched {
  int order[TV_MAX_NODES];   // node at each depth-first position
  // per depth-first position t: {node, (src + 1) | (push + 1) << 8 | (snapshot slot + 1) << 16,
  // alpha bits, beta bits}
  int4 ent[TV_MAX_NODES];
  float kq[TV_MAX_NODES];    // per depth-first position: k_i . q_i of the current item's head
  int flag, maxslot, pad0, pad1;
};
// Scratch of the schedule builder; it lives in the (not yet used) state-stack region.
struct BuildScratch {
  int par[TV_MAX_NODES];
  int depth[TV_MAX_NODES];
  int size[TV_MAX_NODES];
  int nchild[TV_MAX_NODES];
  int hkey[TV_MAX_NODES];    // (size << 9) | (511 - child): heaviest child, lowest index on ties
  int acc[TV_MAX_NODES];     // running offset of light non-leaf children
  int nleaf[TV_MAX_NODES];   // leaf children
  int acc_leaf[TV_MAX_NODES];  // running offset of leaf children
  int before[TV_MAX_NODES];  // nodes of earlier siblings' subtrees
  int pre[TV_MAX_NODES];     // depth-first position
  int slot[TV_MAX_NODES];    // snapshot slot of each node (selective fork), -1: none
  int src[TV_MAX_NODES];     // where the parent state comes from: -1 registers, 0 S_0, else a slot
  int push[TV_MAX_NODES];    // slot the node's own state goes to (-1: not needed later)
  int leaf[TV_MAX_NODES];    // 1: no children -- its state is stored, never kept in registers
  int maxdepth, root_acc, kept;
};

// Depth-first schedule of one tree, built by the whole CTA.  Returns 0, TV_ERR_BAD_TREE or
// TV_ERR_UNSUPPORTED (stack deeper than kSlots; impossible for N <= 256).
__device__ int build_schedule(const int32_t* __restrict__ parents, int N, Sched& s, BuildScratch& x) {
  const int tid = threadIdx.x, nt = blockDim.x;
  int st = load_and_check_tree(parents, N, x.par, &s.flag);
  if (st) return st;
  if (tid == 0) { x.maxdepth = 0; x.root_acc = 0; s.maxslot = 0; }
  for (int i = tid; i < N; i += nt) {
    x.size[i] = 1; x.nchild[i] = 0; x.hkey[i] = 0; x.acc[i] = 0; x.nleaf[i] = 0; x.acc_leaf[i] = 0;
    s.order[i] = -1;
  }
  __syncthreads();
  for (int i = tid; i < N; i += nt) {
    const int d = node_depth(x.par, i);
    x.depth[i] = d;
    atomicMax(&x.maxdepth, d);
    if (x.par[i] >= 0) atomicAdd(&x.nchild[x.par[i]], 1);
  }
  __syncthreads();
  // Subtree sizes, one depth level at a time from the deepest.
  for (int d = x.maxdepth; d >= 1; --d) {
    for (int i = tid; i < N; i += nt)
      if (x.depth[i] == d) atomicAdd(&x.size[x.par[i]], x.size[i]);
    __syncthreads();
  }
  for (int i = tid; i < N; i += nt) {
    const int p = x.par[i];
    if (p >= 0) {
      atomicMax(&x.hkey[p], (x.size[i] << 9) | (511 - i));
      if (x.nchild[i] == 0) atomicAdd(&x.nleaf[p], 1);
    }
  }
  __syncthreads();
  // Offset of each node among its siblings: leaves first, then the light non-leaf children, in
  // arbitrary (atomic) order, and the heavy child after all of them (a leaf heavy child, when
  // every child is a leaf, counts as a leaf); roots one after another.
  for (int i = tid; i < N; i += nt) {
    const int p = x.par[i];
    if (p < 0) {
      x.before[i] = atomicAdd(&x.root_acc, x.size[i]);
    } else if (x.nchild[i] == 0) {
      x.before[i] = atomicAdd(&x.acc_leaf[p], 1);
    } else {
      const int heavy = 511 - (x.hkey[p] & 511);
      x.before[i] = (i == heavy) ? x.size[p] - 1 - x.size[i] : x.nleaf[p] + atomicAdd(&x.acc[p], x.size[i]);
    }
  }
  __syncthreads();
  for (int i = tid; i < N; i += nt) {
    int pre = -1, light = 0;
    // pre is in [0, N) for a valid tree; the check keeps a broken invariant from indexing out.
    for (int a = i; a >= 0; a = x.par[a]) {
      pre += 1 + x.before[a];
      const int p = x.par[a];
      if (p >= 0 && a != 511 - (x.hkey[p] & 511)) ++light;
    }
    x.pre[i] = pre;
    if (pre >= 0 && pre < N) s.order[pre] = i;
    else s.flag = 1;
    // Leaves never disturb the parent state in registers, so a node saves its state only when
    // a second non-leaf child will need it after the first one's subtree.
    const int slot = x.nchild[i] - x.nleaf[i] >= 2 ? 1 + light : -1;
    x.push[i] = slot;
    if (slot > 0) atomicMax(&s.maxslot, slot);
  }
  __syncthreads();
  for (int i = tid; i < N; i += nt) {
    const int p = x.par[i];
    // A leaf, and the first non-leaf child (right after the leaves), find the parent state in
    // registers; a later non-leaf child pops it.
    const bool pops = p >= 0 && x.nchild[i] != 0 && x.pre[i] != x.pre[p] + 1 + x.nleaf[p];
    x.src[i] = (p < 0) ? 0 : (pops ? x.push[p] : -1);
    x.leaf[i] = x.nchild[i] == 0;
    // never expected: guards every index
    if (s.order[i] < 0 || x.src[i] > kSlots || (pops && x.push[p] <= 0)) s.flag = 1;
  }
  __syncthreads();
  return (s.maxslot <= kSlots && !s.flag) ? 0 : TV_ERR_UNSUPPORTED;
}

// Stack slots a tree of n nodes can need: a pushing node below L light edges has at least
// g(L) nodes in the tree (g(0) = 5, g(L) = 2 g(L-1) + 1), and it pushes to slot L + 1.
__host__ __device__ constexpr int slots_for(int n) {
  int L = 0, g = 5;
  while (2 * g + 1 <= n) { g = 2 * g + 1; ++L; }
  return L + 1;
}
static_assert(slots_for(TV_MAX_NODES) <= kSlots, "the stack bound covers every tree");

// A node's inputs for one lane, as stored (bf16 pairs or fp32), prefetched into registers.
template <typename TIO, int CPL>
struct Raw;
template <int CPL>
struct Raw<bf16, CPL> {
  uint32_t k[CPL / 2], q[CPL / 2];
  float v, kq;
  int4 e;  // schedule entry of the node
  __device__ __forceinline__ void load(const bf16* kp, const bf16* qp, const bf16* vp) {
#pragma unroll
    for (int j = 0; j < CPL / 8; ++j) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(kp + j * kStride));
      const uint4 c = __ldg(reinterpret_cast<const uint4*>(qp + j * kStride));
      k[4 * j] = a.x; k[4 * j + 1] = a.y; k[4 * j + 2] = a.z; k[4 * j + 3] = a.w;
      q[4 * j] = c.x; q[4 * j + 1] = c.y; q[4 * j + 2] = c.z; q[4 * j + 3] = c.w;
    }
    v = to_f32(__ldg(vp));
  }
  __device__ __forceinline__ void load_kw(const bf16* kp, const float* wp) {  // keys and a given w
#pragma unroll
    for (int j = 0; j < CPL / 8; ++j) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(kp + j * kStride));
      k[4 * j] = a.x; k[4 * j + 1] = a.y; k[4 * j + 2] = a.z; k[4 * j + 3] = a.w;
    }
    v = __ldg(wp);
  }
  __device__ __forceinline__ float kf(int e) const { return (e & 1) ? bf16hi(k[e >> 1]) : bf16lo(k[e >> 1]); }
  __device__ __forceinline__ float qf(int e) const { return (e & 1) ? bf16hi(q[e >> 1]) : bf16lo(q[e >> 1]); }
};
template <int CPL>
struct Raw<float, CPL> {
  float k[CPL], q[CPL];
  float v, kq;
  int4 e;  // schedule entry of the node
  __device__ __forceinline__ void load(const float* kp, const float* qp, const float* vp) {
#pragma unroll
    for (int j = 0; j < CPL / 8; ++j) {
      load_vec<8>(kp + j * kStride, k + 8 * j);
      load_vec<8>(qp + j * kStride, q + 8 * j);
    }
    v = __ldg(vp);
  }
  __device__ __forceinline__ void load_kw(const float* kp, const float* wp) {
#pragma unroll
    for (int j = 0; j < CPL / 8; ++j) load_vec<8>(kp + j * kStride, k + 8 * j);
    v = __ldg(wp);
  }
  __device__ __forceinline__ float kf(int e) const { return k[e]; }
  __device__ __forceinline__ float qf(int e) const { return q[e]; }
};

// FROM_W: the second pass of the two-pass fork -- w_i (and every output) already came from the
// TreeWY pass in wsrc [B, N, H, dv]; this pass only materializes the snapshots,
// S_i = alpha_i S_p + w_i k_i^T, along the same walk.
//
// RPL: state rows per lane group (1 or 2).  With two, a group of 8 lanes holds rows rg and
// rg + 8 of the slab (64 threads per CTA): the k and q loads and conversions, the schedule
// decode and the prefetch serve both rows, and the four row dot products of a node reduce
// together in four shuffles (plus two to broadcast w), so a row costs about a third fewer
// instructions than in the one-row form.
struct UnitPlan {
  int group, share, stride;  // CTAs per group, units per CTA at most, units between group starts
};

template <typename TIO, typename TS, int DK, bool FROM_W, int RPL>
__device__ __forceinline__ void gdn_fork_body(const GdnArgs& a, TS* __restrict__ states, int nslots, UnitPlan plan,
                                              const ForkSelect& sel, const float* __restrict__ wsrc) {
  const int group = plan.group, share = plan.share, stride = plan.stride;
  static_assert(RPL == 1 || (RPL == 2 && !FROM_W), "two rows per lane group in the one-pass form only");
  constexpr int CPL = DK / kLPR;  // columns per lane
  constexpr int Q4 = CPL / 4;     // float4 per lane per slot and row
  constexpr int kThreads = kLanes / RPL;
  constexpr int RG = kRows / RPL;  // row distance between a lane group's rows
  extern __shared__ __align__(128) unsigned char smem[];
  Sched& sc = *reinterpret_cast<Sched*>(smem);
  float4* stack = reinterpret_cast<float4*>(smem + sizeof(Sched));
  BuildScratch& scratch = *reinterpret_cast<BuildScratch*>(stack);

  const int N = a.N, H = a.H, dv = a.dv;
  const int tid = threadIdx.x;
  // Work units are (sequence, head, 16-row slab) in that order, U = B H dv / 16 of them.  The
  // CTAs form groups of `group`; group gamma owns the units [gamma * stride, gamma * stride +
  // min(group * share, stride)), and its CTA g takes every group-th of them from g.  So a CTA
  // gets at most `share` units, and at any moment a group's CTAs work on adjacent slabs: their
  // snapshot rows of a node land side by side in HBM.  With stride = the units of a sequence,
  // a group is one sequence; with stride = group * share, groups tile the units whatever B is
  // (the launcher picks the form with the smaller share), and a CTA's units may run through two
  // sequences.  The CTA builds the schedule of each sequence it enters; the CTA holding a
  // sequence's first unit writes its status and slot map.
  int b = -1;
  // Schedule, snapshot slots and per-position entries of sequence b; the sequence's status.
  auto setup = [&](bool first_cta) -> int {
    // A sequence the TreeWY pass rejected keeps its status and no snapshot (its slots go to -1
    // below when selecting).
    const int prior = FROM_W ? a.err[b] : 0;
    int status = prior ? prior : build_schedule(a.parents + (size_t)b * N, N, sc, scratch);
    if (!status && sc.maxslot > nslots) status = TV_ERR_UNSUPPORTED;
    // Snapshot slots (selective fork): nodes at or below the confidence threshold, numbered in
    // node order by one warp's ballot scan; otherwise slot = node.
    if (sel.confidence != nullptr) {
      if (tid < 32) {
        int carry = 0;
        for (int base = 0; base < N; base += 32) {
          const int i = base + tid;
          const bool keep = i < N && sel.confidence[(size_t)b * N + i] <= sel.threshold;
          const unsigned m = __ballot_sync(0xffffffffu, keep);
          if (i < N) scratch.slot[i] = keep ? carry + __popc(m & ((1u << tid) - 1u)) : -1;
          carry += __popc(m);
        }
        if (tid == 0) scratch.kept = carry;
      }
      __syncthreads();
      if (!status && scratch.kept > sel.capacity) status = TV_ERR_CAPACITY;
      // a sequence that is skipped keeps no snapshot: its commit then replays from S_0
      if (first_cta && sel.slot != nullptr)
        for (int i = tid; i < N; i += kThreads) sel.slot[(size_t)b * N + i] = status ? -1 : scratch.slot[i];
    } else {
      for (int i = tid; i < N; i += kThreads) scratch.slot[i] = i;
      __syncthreads();
    }
    if (first_cta && tid == 0 && (status || !FROM_W)) a.err[b] = status;
    if (status) return status;
    for (int t = tid; t < N; t += kThreads) {
      const int i = sc.order[t];
      sc.ent[t] = make_int4(i, (scratch.src[i] + 1) | ((scratch.push[i] + 1) << 8) | ((scratch.slot[i] + 1) << 16) |
                                   (scratch.leaf[i] << 28), 0, 0);
    }
    return 0;
  };

  const TIO* __restrict__ q = static_cast<const TIO*>(a.q);
  const TIO* __restrict__ k = static_cast<const TIO*>(a.k);
  const TIO* __restrict__ v = static_cast<const TIO*>(a.v);
  const TS* __restrict__ S0 = static_cast<const TS*>(a.S0);
  TIO* __restrict__ out = static_cast<TIO*>(a.out);
  const int lane = tid % kLPR, rl = tid / kLPR;
  // the row whose v this lane loads and whose output it may write: RPL = 2 splits the group
  // into lanes 0-3 (row rl) and 4-7 (row rl + 8)
  const int rmine = rl + (RPL == 2 && (lane & 4) ? RG : 0);
  const int slabs = dv / kRows, items = H * slabs;
  const float q_scale = a.q_scale;
  const size_t node_stride = (size_t)H * dv;     // elements between consecutive nodes (out, v)
  const size_t state_stride = node_stride * DK;  // elements between consecutive nodes (states)
  const size_t kq_stride = (size_t)H * DK;       // elements between consecutive nodes (q, k)
  const long long units = (long long)a.B * items;
  const long long u_base = (long long)(blockIdx.x / group) * stride;
  const long long u_begin = u_base + blockIdx.x % group;
  const long long u_end = min(units, u_base + min((long long)group * share, (long long)stride));
  // Pulls one item's inputs into L2 ahead of use: alpha, beta, k and q of every node, the
  // slab's v rows and S_0 rows.  The node loop's register prefetch then waits on L2, not HBM.
  auto prefetch_unit = [&](long long u) {
    const int bb = (int)(u / items), it = (int)(u % items);
    const int hh = it / slabs, r0 = (it % slabs) * kRows;
    const size_t n0 = (size_t)bb * N * H + hh;
    const int kq_lines = DK * (int)sizeof(TIO) / 128 > 0 ? DK * (int)sizeof(TIO) / 128 : 1;
    const int per_node = 2 * kq_lines + 1;       // k lines, q lines, the slab's v rows
    for (int x = tid; x < N * per_node; x += kThreads) {
      const int t = x / per_node, c = x % per_node;
      const size_t nh = n0 + (size_t)t * H;
      const void* p = c < kq_lines ? (const void*)(k + nh * DK + c * (128 / sizeof(TIO)))
                    : FROM_W           ? (const void*)(wsrc + nh * dv + r0)
                    : c < 2 * kq_lines ? (const void*)(q + nh * DK + (c - kq_lines) * (128 / sizeof(TIO)))
                                       : (const void*)(v + nh * dv + r0);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
    }
    const int s0_lines = kRows * DK * (int)sizeof(TS) / 128;
    for (int x = tid; x < s0_lines; x += kThreads)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(S0 + (((size_t)bb * H + hh) * dv + r0) * DK) + x * 128));
    for (int x = tid; x < (N * H + 31) / 32; x += kThreads) {  // alpha and beta of the sequence
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a.alpha + (size_t)bb * N * H + x * 32));
      if (!FROM_W) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.beta + (size_t)bb * N * H + x * 32));
    }
  };
  if (u_begin < u_end) prefetch_unit(u_begin);
  int status = 0;
  for (long long u = u_begin; u < u_end; u += group) {
    const int item = (int)(u % items);
    if ((int)(u / items) != b) {
      __syncthreads();                           // the previous sequence's walk is done with the stack
      b = (int)(u / items);
      status = setup(item == 0);
    }
    if (u + group < u_end) prefetch_unit(u + group);
    if (status) continue;                        // the same in every thread
    const int h = item / slabs, r0 = (item % slabs) * kRows, r = r0 + rl;
    const size_t nh0 = (size_t)b * N * H + h;    // (b, node 0, h)
    __syncthreads();                             // the previous item is done with alpha / beta
    for (int t = tid; t < N; t += kThreads) {
      const size_t nh = nh0 + (size_t)sc.ent[t].x * H;
      sc.ent[t].z = __float_as_int(__ldg(a.alpha + nh));
      sc.ent[t].w = FROM_W ? 0 : __float_as_int(__ldg(a.beta + nh));  // w already holds beta
    }
    // k_i . q_i is the same for every row of the head: 8 threads per node compute it once,
    // with the loads of KQB nodes in flight at a time (four when 64 threads serve the item).
    // The loop bound is warp-uniform, so every lane takes part in the shuffles.
    constexpr int kNodesPerPass = kThreads / kLPR;
    constexpr int KQB = RPL == 2 ? 4 : 1;
    for (int t0 = 0; !FROM_W && t0 < N; t0 += KQB * kNodesPerPass) {
      Raw<TIO, CPL> x[KQB];
#pragma unroll
      for (int u = 0; u < KQB; ++u) {
        const int t = t0 + u * kNodesPerPass + tid / kLPR;
        const size_t nh = nh0 + (size_t)sc.order[t < N ? t : N - 1] * H;
        x[u].load(k + nh * DK + lane * 8, q + nh * DK + lane * 8, v + nh * dv);
      }
#pragma unroll
      for (int u = 0; u < KQB; ++u) {
        const int t = t0 + u * kNodesPerPass + tid / kLPR;
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < CPL; ++e) dot = fmaf(x[u].kf(e), x[u].qf(e), dot);
        dot = group_sum<kLPR>(dot);
        if (t < N && lane == 0) sc.kq[t] = dot;
      }
    }
    __syncthreads();

    const TIO* kb = k + nh0 * DK + lane * 8;
    const TIO* qb = q + nh0 * DK + lane * 8;
    const TIO* vb = v + nh0 * dv + r0 + rmine;
    const TS* s0row = S0 + (((size_t)b * H + h) * dv + r) * DK + lane * 8;
    TIO* out_r = out + nh0 * dv + r0 + rmine;
    // snapshots of this sequence: [capacity][H][dv][dk]
    TS* st_r = states + ((((size_t)b * sel.capacity) * H + h) * dv + r) * DK + lane * 8;
    const float* wb = FROM_W ? wsrc + nh0 * dv + r0 + rmine : nullptr;
    auto fetch = [&](int t, Raw<TIO, CPL>& x) {
      x.e = sc.ent[t < N ? t : N - 1];
      const int node = x.e.x;
      if constexpr (FROM_W) {
        x.load_kw(kb + node * kq_stride, wb + node * node_stride);
      } else {
        x.kq = sc.kq[t < N ? t : N - 1];
        x.load(kb + node * kq_stride, qb + node * kq_stride, vb + node * node_stride);
      }
    };
    float2 cur[RPL][CPL / 2];  // the rows' states, column pairs (2e, 2e + 1)
    // One node: parent state -> output and S_i (kept in cur), checkpoint, optional push.  The
    // two row dot products use the parent state, so they share one reduction:
    //   (S_p k)_r, (S_p q)_r  ->  w = beta (v_r - alpha (S_p k)_r),
    //   o_r = (S_i q)_r = alpha (S_p q)_r + w (k.q),   S_i = alpha S_p + w k^T,
    // with k.q from the per-unit table.  Column pairs go through the paired fp32 FMA.
    auto body = [&](const Raw<TIO, CPL>& x) {
      const int i = x.e.x;
      const int src = (x.e.y & 255) - 1, push = ((x.e.y >> 8) & 255) - 1, slot = ((x.e.y >> 16) & 1023) - 1;
      const bool leaf = (x.e.y >> 28) & 1;
      const float al = __int_as_float(x.e.z), be = __int_as_float(x.e.w);
      if (src == 0) {
#pragma unroll
        for (int rr = 0; rr < RPL; ++rr) {
          float f[CPL];
#pragma unroll
          for (int j = 0; j < CPL / 8; ++j) load_vec<8>(s0row + rr * RG * DK + j * kStride, f + 8 * j);  // a root starts from S_0
#pragma unroll
          for (int e = 0; e < CPL / 2; ++e) cur[rr][e] = make_float2(f[2 * e], f[2 * e + 1]);
        }
      } else if (src > 0) {
#pragma unroll
        for (int rr = 0; rr < RPL; ++rr)
#pragma unroll
          for (int j = 0; j < Q4; ++j) {
            const float4 f = stack[(((src - 1) * RPL + rr) * Q4 + j) * kThreads + tid];
            cur[rr][2 * j] = make_float2(f.x, f.y);
            cur[rr][2 * j + 1] = make_float2(f.z, f.w);
          }
      }
      float2 kf[CPL / 2];
#pragma unroll
      for (int e = 0; e < CPL / 2; ++e) kf[e] = make_float2(x.kf(2 * e), x.kf(2 * e + 1));
      float w[RPL];                                         // pseudo-values w_i[r] of the rows
      if constexpr (FROM_W) {
        w[0] = x.v;
      } else {
        // Lane partials of (S_p k)_r and (S_p q)_r for each row.  With two rows they reduce in
        // one butterfly over the group's 8 lanes in which every exchange moves half of the values
        // still unreduced: lanes 0-3 / 4-7 keep row 0 / row 1, then lanes with bit 1 clear / set
        // keep the k / q product, so lane l ends with the full S_p k (bit 1 clear) or S_p q (set)
        // of row (l >> 2) & 1.
        float pk[RPL], pq[RPL];
#pragma unroll
        for (int rr = 0; rr < RPL; ++rr) {
          float2 k0 = make_float2(0.f, 0.f), q0 = k0, k1 = k0, q1 = k0;
#pragma unroll
          for (int e = 0; e < CPL / 2; e += 2) {
            const float2 qa = make_float2(x.qf(2 * e), x.qf(2 * e + 1));
            const float2 qb = make_float2(x.qf(2 * e + 2), x.qf(2 * e + 3));
            k0 = __ffma2_rn(cur[rr][e], kf[e], k0);
            q0 = __ffma2_rn(cur[rr][e], qa, q0);
            k1 = __ffma2_rn(cur[rr][e + 1], kf[e + 1], k1);
            q1 = __ffma2_rn(cur[rr][e + 1], qb, q1);
          }
          pk[rr] = (k0.x + k1.x) + (k0.y + k1.y);
          pq[rr] = (q0.x + q1.x) + (q0.y + q1.y);
        }
        if constexpr (RPL == 2) {
          const bool b2 = lane & 4, b1 = lane & 2;
          const float sk = __shfl_xor_sync(0xffffffffu, b2 ? pk[0] : pk[1], 4);
          const float sq = __shfl_xor_sync(0xffffffffu, b2 ? pq[0] : pq[1], 4);
          const float mk = (b2 ? pk[1] : pk[0]) + sk, mq = (b2 ? pq[1] : pq[0]) + sq;
          float m = (b1 ? mq : mk) + __shfl_xor_sync(0xffffffffu, b1 ? mk : mq, 2);
          m += __shfl_xor_sync(0xffffffffu, m, 1);
          // w of this lane's row, valid where m is S_p k (lanes 0 and 4), to every lane
          const float wl = be * (x.v - al * m);
          const int g0 = (tid & 31) & ~(kLPR - 1);  // the group's first lane in the warp
          w[0] = __shfl_sync(0xffffffffu, wl, g0);
          w[1] = __shfl_sync(0xffffffffu, wl, g0 + 4);
          // the output of this lane's row from lane 2 / 6, which hold S_p q
          if ((lane & 3) == 2) out_r[(size_t)i * node_stride] = from_f32<TIO>((al * m + (b2 ? w[1] : w[0]) * x.kq) * q_scale);
        } else {
          // one row: both sums to every lane in two independent chains of three shuffles
          float sk = pk[0], sq = pq[0];
#pragma unroll
          for (int o = kLPR / 2; o > 0; o >>= 1) {
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
          }
          w[0] = be * (x.v - al * sk);
          if (lane == 0) out_r[(size_t)i * node_stride] = from_f32<TIO>((al * sq + w[0] * x.kq) * q_scale);
        }
      }
      const float2 al2 = make_float2(al, al);
      if (leaf) {
        // A leaf's state only goes to its snapshot: cur keeps the parent state for the siblings.
        if (slot >= 0) {
#pragma unroll
          for (int rr = 0; rr < RPL; ++rr) {
            const float2 w2 = make_float2(w[rr], w[rr]);
            float f[CPL];
#pragma unroll
            for (int e = 0; e < CPL / 2; ++e) {
              const float2 s2 = __ffma2_rn(w2, kf[e], __fmul2_rn(al2, cur[rr][e]));
              f[2 * e] = s2.x;
              f[2 * e + 1] = s2.y;
            }
#pragma unroll
            for (int j = 0; j < CPL / 8; ++j)
              store_vec_cs<8>(st_r + (size_t)slot * state_stride + rr * RG * DK + j * kStride, f + 8 * j);
          }
        }
        return;
      }
#pragma unroll
      for (int rr = 0; rr < RPL; ++rr) {
        const float2 w2 = make_float2(w[rr], w[rr]);
#pragma unroll
        for (int e = 0; e < CPL / 2; ++e) cur[rr][e] = __ffma2_rn(w2, kf[e], __fmul2_rn(al2, cur[rr][e]));
        float f[CPL];
#pragma unroll
        for (int e = 0; e < CPL / 2; ++e) { f[2 * e] = cur[rr][e].x; f[2 * e + 1] = cur[rr][e].y; }
        if (slot >= 0) {
#pragma unroll
          for (int j = 0; j < CPL / 8; ++j)
            store_vec_cs<8>(st_r + (size_t)slot * state_stride + rr * RG * DK + j * kStride, f + 8 * j);
        }
      }
      if (push > 0) {
#pragma unroll
        for (int rr = 0; rr < RPL; ++rr)
#pragma unroll
          for (int j = 0; j < Q4; ++j)
            stack[(((push - 1) * RPL + rr) * Q4 + j) * kThreads + tid] =
                make_float4(cur[rr][2 * j].x, cur[rr][2 * j].y, cur[rr][2 * j + 1].x, cur[rr][2 * j + 1].y);
      }
    };
    // Two register buffers alternate by unrolling: node t + 1's inputs are requested before node
    // t is computed (a register copy would wait for the load).  A deeper register prefetch and a
    // cp.async ring in shared memory measured slower: the walk is bound by issue and by the
    // dependent chain of each node, not by these loads.
    Raw<TIO, CPL> ra, rb;
    fetch(0, ra);
    for (int t = 0; t < N; t += 2) {
      fetch(t + 1, rb);
      body(ra);
      if (t + 1 >= N) break;
      fetch(t + 2, ra);
      body(rb);
    }
  }
}

// Entry points over the same body.  The plain one leaves the register budget to the compiler;
// the bounded ones ask for six (80 registers) or five 128-thread CTAs per SM, which pays for
// the snapshot pass when its stack lets that many CTAs fit (at most three slots: six; four
// slots: five) -- and only then: a minimum-blocks bound that does not raise occupancy measured
// slower.
template <typename TIO, typename TS, int DK, bool FROM_W, int RPL>
__global__ void __launch_bounds__(kLanes / RPL) gdn_fork_kernel(GdnArgs a, TS* __restrict__ states, int nslots,
                                                                UnitPlan plan, ForkSelect sel,
                                                                const float* __restrict__ wsrc) {
  gdn_fork_body<TIO, TS, DK, FROM_W, RPL>(a, states, nslots, plan, sel, wsrc);
}
template <typename TIO, typename TS, int DK, int MINB>
__global__ void __launch_bounds__(kLanes, MINB) gdn_fork_snapshot_kernel(GdnArgs a, TS* __restrict__ states,
                                                                         int nslots, UnitPlan plan, ForkSelect sel,
                                                                         const float* __restrict__ wsrc) {
  gdn_fork_body<TIO, TS, DK, true, 1>(a, states, nslots, plan, sel, wsrc);
}

template <typename TIO, typename TS, int DK, bool FROM_W, int RPL>
cudaError_t launch_fork_rpl(const GdnArgs& a, void* states, const ForkSelect& sel, cudaStream_t s,
                            const float* wsrc, int max_ctas_per_sm) {
  constexpr int kThreads = kLanes / RPL;
  const int nslots = slots_for(a.N);
  void (*kern)(GdnArgs, TS*, int, UnitPlan, ForkSelect, const float*) = gdn_fork_kernel<TIO, TS, DK, FROM_W, RPL>;
  if constexpr (FROM_W) {
    if (nslots <= 3) kern = gdn_fork_snapshot_kernel<TIO, TS, DK, 6>;
    else if (nslots == 4) kern = gdn_fork_snapshot_kernel<TIO, TS, DK, 5>;
  }
  size_t stack = (size_t)nslots * (DK / kLPR / 4) * kLanes * sizeof(float4);
  if (stack < sizeof(BuildScratch)) stack = sizeof(BuildScratch);
  stack = (stack + 15) / 16 * 16;
  const size_t smem = sizeof(Sched) + stack;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (max_ctas_per_sm > 0 && occ > max_ctas_per_sm) occ = max_ctas_per_sm;
  // At most one CTA per resident slot.  Either every sequence gets the same number of CTAs (a
  // group per sequence, no CTA crosses sequences) or groups of kGroup CTAs tile the units
  // regardless of sequence boundaries (an equal share whatever B is); the form with the smaller
  // largest share (times the waves it needs) wins.  Then the fewest CTAs with that share,
  // which frees slots for other streams' work without lengthening this kernel.
  const long long items = (long long)a.H * (a.dv / kRows), units = a.B * items;
  const long long slots = (long long)device_sm_count() * (occ > 0 ? occ : 1);
  long long per_seq = slots / a.B;
  per_seq = per_seq < 1 ? 1 : (per_seq > items ? items : per_seq);
  const long long share_seq = (items + per_seq - 1) / per_seq;
  long long groups = slots / kGroup;
  if (groups < 1) groups = 1;
  const long long share_grp = (units + groups * kGroup - 1) / (groups * kGroup);
  // more sequences than slots: the per-sequence form runs in waves
  const long long waves_seq = (a.B * per_seq + slots - 1) / slots;
  UnitPlan plan;
  long long grid;
  // On a tie the groups win only when they tile each sequence exactly (measured: the strided
  // per-sequence order is faster than groups that straddle sequences, slower than ones that
  // do not).
  const bool grp_tiles = items % (share_grp * kGroup) == 0;
  if (share_seq * waves_seq < share_grp || (share_seq * waves_seq == share_grp && !grp_tiles)) {
    per_seq = (items + share_seq - 1) / share_seq;
    plan = UnitPlan{(int)per_seq, (int)share_seq, (int)items};
    grid = a.B * per_seq;
  } else {
    groups = (units + share_grp * kGroup - 1) / (share_grp * kGroup);
    plan = UnitPlan{kGroup, (int)share_grp, (int)(share_grp * kGroup)};
    grid = groups * kGroup;
  }
  kern<<<(unsigned)grid, kThreads, smem, s>>>(a, static_cast<TS*>(states), nslots, plan, sel, wsrc);
  return cudaGetLastError();
}

// The one-pass form takes two rows per lane group for bf16 inputs when the tree needs at most
// three stack slots (N <= 46): its 64-thread CTAs then fit six to an SM and issue about a third
// fewer instructions per row.  Deeper stacks, fp32 inputs (twice the registers per row) and the
// snapshot pass (no dot products to share) keep one row per group.
template <typename TIO, typename TS, int DK, bool FROM_W = false>
cudaError_t launch_fork_t(const GdnArgs& a, void* states, const ForkSelect& sel, cudaStream_t s,
                          const float* wsrc = nullptr, int max_ctas_per_sm = 0) {
  if constexpr (!FROM_W && sizeof(TIO) == 2) {
    if (slots_for(a.N) <= 3) return launch_fork_rpl<TIO, TS, DK, FROM_W, 2>(a, states, sel, s, wsrc, max_ctas_per_sm);
  }
  return launch_fork_rpl<TIO, TS, DK, FROM_W, 1>(a, states, sel, s, wsrc, max_ctas_per_sm);
}

}  // namespace

cudaError_t launch_gdn_fork(const GdnArgs& a, void* node_states, const ForkSelect& sel, cudaStream_t s) {
  static_assert(sizeof(Sched) % 16 == 0, "stack must start 16-byte aligned");
  if (a.io == TV_F32 && a.state == TV_F32)
    return a.dk == 64 ? launch_fork_t<float, float, 64>(a, node_states, sel, s)
                      : launch_fork_t<float, float, 128>(a, node_states, sel, s);
  if (a.io == TV_BF16 && a.state == TV_BF16)
    return a.dk == 64 ? launch_fork_t<bf16, bf16, 64>(a, node_states, sel, s)
                      : launch_fork_t<bf16, bf16, 128>(a, node_states, sel, s);
  return a.dk == 64 ? launch_fork_t<bf16, float, 64>(a, node_states, sel, s)
                    : launch_fork_t<bf16, float, 128>(a, node_states, sel, s);
}

cudaError_t launch_gdn_fork_materialize(const GdnArgs& a, void* node_states, const float* pseudo_v,
                                        const ForkSelect& all, int max_ctas_per_sm, cudaStream_t s) {
  const int m = max_ctas_per_sm;
  if (a.io == TV_F32 && a.state == TV_F32)
    return a.dk == 64 ? launch_fork_t<float, float, 64, true>(a, node_states, all, s, pseudo_v, m)
                      : launch_fork_t<float, float, 128, true>(a, node_states, all, s, pseudo_v, m);
  if (a.io == TV_BF16 && a.state == TV_BF16)
    return a.dk == 64 ? launch_fork_t<bf16, bf16, 64, true>(a, node_states, all, s, pseudo_v, m)
                      : launch_fork_t<bf16, bf16, 128, true>(a, node_states, all, s, pseudo_v, m);
  return a.dk == 64 ? launch_fork_t<bf16, float, 64, true>(a, node_states, all, s, pseudo_v, m)
                    : launch_fork_t<bf16, float, 128, true>(a, node_states, all, s, pseudo_v, m);
}

cudaError_t launch_gdn_fork_two_pass(const GdnArgs& a, void* node_states, float* pseudo_v, float* log_gamma,
                                     cudaStream_t s) {
  cudaError_t e = launch_gdn_wy(a, pseudo_v, log_gamma, s);  // every output, and w
  if (e != cudaSuccess) return e;
  const ForkSelect all{nullptr, 0.f, a.N, nullptr};
  return launch_gdn_fork_materialize(a, node_states, pseudo_v, all, 0, s);
}

}  // namespace tv
