// TreeWY GDN tree verify, CUDA-core form (TreeWY: Speculative Verification for Gated DeltaNet
// Hybrids, abstract: every node's output from one triangular solve over a pseudo-value
// matrix, no per-node states).
//
// Reading of the algebra (the page gives only the abstract).  With gamma_i the product of
// alpha along the root-to-node path P(i) and Gamma_ij = gamma_i / gamma_j,
//     S_i = gamma_i S_0 + sum_{j in P(i)} Gamma_ij w_j k_j^T,
//     w_i = beta_i (v_i - gamma_i S_0 k_i) - sum_{j in P(i), j != i} beta_i Gamma_ij (k_i.k_j) w_j,
//     o_i = gamma_i S_0 (q_scale q_i) + sum_{j in P(i)} Gamma_ij q_scale (q_i.k_j) w_j.
// The second line is forward substitution of the unit lower-triangular system
// (I + diag(beta)(A o Gamma o K K^T)) W = diag(beta)(V - diag(gamma) K S_0^T), solved along
// each node's ancestor list (parents[i] < i, so ancestors come first).
//
// A CTA owns 32 rows of S_0 for one (sequence, head).  It first computes the scalar
// coefficients c_ij = beta_i Gamma_ij (k_i.k_j) and e_ij = q_scale Gamma_ij (q_i.k_j) for
// every (node, path entry) pair, then walks the nodes in index order: each row computes
// (S_0 k_i)_r and (S_0 q_i)_r with 8 lanes, and lane 0 of the row does the two short sums over
// the ancestors' w, kept in shared memory.
#include "tv_common.cuh"
#include "tv_internal.h"

namespace tv {
namespace {

constexpr int kLPR = 8;
constexpr int kRows = 32;
constexpr int kThreads = kLPR * kRows;  // 256
constexpr int kPathCap = 4096;          // max sum over nodes of (depth + 1)

struct WyHead {
  int par[TV_MAX_NODES];
  int depth[TV_MAX_NODES];
  int off[TV_MAX_NODES + 1];
  float lg[TV_MAX_NODES];
  int flag, total;
};

template <typename TIO, typename TS, int DK>
__global__ void __launch_bounds__(kThreads) gdn_wy_simt_kernel(GdnArgs a, float* __restrict__ pseudo_v,
                                                               float* __restrict__ log_gamma, int cap) {
  constexpr int CPL = DK / kLPR;
  extern __shared__ __align__(16) unsigned char smem[];
  WyHead& s = *reinterpret_cast<WyHead*>(smem);
  int* pidx = reinterpret_cast<int*>(smem + sizeof(WyHead));
  float* cK = reinterpret_cast<float*>(pidx + cap);
  float* cQ = cK + cap;
  float* wsm = cQ + cap;  // [N][kRows]

  const int N = a.N, H = a.H, dv = a.dv;
  const int slabs = dv / kRows;
  const int b = blockIdx.x / (H * slabs);
  const int h = (blockIdx.x / slabs) % H;
  const int slab = blockIdx.x % slabs;
  const int tid = threadIdx.x, nt = blockDim.x;
  const bool writer = (h == 0 && slab == 0 && tid == 0);

  int status = load_and_check_tree(a.parents + (size_t)b * N, N, s.par, &s.flag);
  if (status) {
    if (writer) a.err[b] = status;
    return;
  }
  const float* __restrict__ alpha = a.alpha;
  const float* __restrict__ beta = a.beta;
  for (int i = tid; i < N; i += nt) {
    s.depth[i] = node_depth(s.par, i);
    float lg = 0.f;
    for (int j = i; j >= 0; j = s.par[j]) lg += logf(__ldg(alpha + ((size_t)b * N + j) * H + h));
    s.lg[i] = lg;
  }
  __syncthreads();
  if (tid < 32) {  // exclusive scan of (depth + 1)
    int carry = 0;
    for (int base = 0; base < N; base += 32) {
      const int i = base + tid;
      int x = (i < N) ? s.depth[i] + 1 : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (tid >= o) x += y;
      }
      if (i < N) s.off[i + 1] = carry + x;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (tid == 0) { s.off[0] = 0; s.total = carry; }
  }
  __syncthreads();
  status = s.total > cap ? TV_ERR_UNSUPPORTED : 0;
  if (writer) a.err[b] = status;
  if (status) return;

  const TIO* __restrict__ q = static_cast<const TIO*>(a.q);
  const TIO* __restrict__ k = static_cast<const TIO*>(a.k);
  const TIO* __restrict__ v = static_cast<const TIO*>(a.v);
  const TS* __restrict__ S0 = static_cast<const TS*>(a.S0);
  TIO* __restrict__ out = static_cast<TIO*>(a.out);
  const float q_scale = a.q_scale;

  for (int i = tid; i < N; i += nt) {  // path entries, root first
    int j = i;
    for (int u = s.depth[i]; u >= 0; --u) { pidx[s.off[i] + u] = j; j = s.par[j]; }
    if (slab == 0) log_gamma[((size_t)b * N + i) * H + h] = s.lg[i];
  }
  __syncthreads();

  // Coefficients: one warp per node, lanes split the key dimension.
  constexpr int EPL = DK / 32;
  const int warp = tid / 32, lane = tid % 32;
  for (int i = warp; i < N; i += nt / 32) {
    const size_t ni = ((size_t)b * N + i) * H + h;
    float ki[EPL], qi[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      ki[e] = to_f32(k[ni * DK + lane * EPL + e]);
      qi[e] = to_f32(q[ni * DK + lane * EPL + e]);
    }
    const float bi = __ldg(beta + ni), lgi = s.lg[i];
    const int d = s.depth[i], o = s.off[i];
    for (int t = 0; t <= d; ++t) {
      const int j = pidx[o + t];
      const size_t nj = ((size_t)b * N + j) * H + h;
      float kk = 0.f, qk = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const float kj = to_f32(k[nj * DK + lane * EPL + e]);
        kk = fmaf(ki[e], kj, kk);
        qk = fmaf(qi[e], kj, qk);
      }
      kk = group_sum<32>(kk);
      qk = group_sum<32>(qk);
      if (lane == 0) {
        const float G = expf(lgi - s.lg[j]);
        cK[o + t] = (t < d) ? bi * G * kk : 0.f;
        cQ[o + t] = q_scale * G * qk;
      }
    }
  }
  __syncthreads();

  // Forward substitution per row.
  const int lane8 = tid & (kLPR - 1), rl = tid / kLPR;
  const int r = slab * kRows + rl;
  float s0[CPL];
  load_vec<CPL>(S0 + (((size_t)b * H + h) * dv + r) * DK + lane8 * CPL, s0);
  for (int i = 0; i < N; ++i) {
    const size_t ni = ((size_t)b * N + i) * H + h;
    float kf[CPL], qf[CPL];
    load_vec<CPL>(k + ni * DK + lane8 * CPL, kf);
    load_vec<CPL>(q + ni * DK + lane8 * CPL, qf);
    float tk = 0.f, uq = 0.f;
#pragma unroll
    for (int e = 0; e < CPL; ++e) {
      tk = fmaf(s0[e], kf[e], tk);
      uq = fmaf(s0[e], qf[e], uq);
    }
    tk = group_sum<kLPR>(tk);
    uq = group_sum<kLPR>(uq);
    if (lane8 == 0) {
      const float gam = expf(s.lg[i]);
      const int d = s.depth[i], o = s.off[i];
      float w = __ldg(beta + ni) * (to_f32(v[ni * dv + r]) - gam * tk);
      for (int t = 0; t < d; ++t) w -= cK[o + t] * wsm[pidx[o + t] * kRows + rl];
      wsm[i * kRows + rl] = w;
      float ov = q_scale * gam * uq;
      for (int t = 0; t <= d; ++t) ov = fmaf(cQ[o + t], wsm[pidx[o + t] * kRows + rl], ov);
      out[ni * dv + r] = from_f32<TIO>(ov);
      pseudo_v[ni * dv + r] = w;
    }
  }
}

template <typename TIO, typename TS, int DK>
cudaError_t launch_wy_t(const GdnArgs& a, float* pseudo_v, float* log_gamma, cudaStream_t s) {
  auto kern = gdn_wy_simt_kernel<TIO, TS, DK>;
  int cap = a.N * (a.N + 1) / 2;
  if (cap > kPathCap) cap = kPathCap;
  const size_t smem = sizeof(WyHead) + (size_t)cap * 12 + (size_t)a.N * kRows * 4;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = a.B * a.H * (a.dv / kRows);
  kern<<<grid, kThreads, smem, s>>>(a, pseudo_v, log_gamma, cap);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gdn_wy(const GdnArgs& a, float* pseudo_v, float* log_gamma, cudaStream_t s) {
  if (gdn_wy_tc_supported(a)) return launch_gdn_wy_tc(a, pseudo_v, log_gamma, WyLazy{}, s);
  return launch_gdn_wy_simt(a, pseudo_v, log_gamma, s);
}

cudaError_t launch_gdn_wy_simt(const GdnArgs& a, float* pseudo_v, float* log_gamma, cudaStream_t s) {
  if (a.io == TV_F32 && a.state == TV_F32)
    return a.dk == 64 ? launch_wy_t<float, float, 64>(a, pseudo_v, log_gamma, s)
                      : launch_wy_t<float, float, 128>(a, pseudo_v, log_gamma, s);
  if (a.io == TV_BF16 && a.state == TV_BF16)
    return a.dk == 64 ? launch_wy_t<bf16, bf16, 64>(a, pseudo_v, log_gamma, s)
                      : launch_wy_t<bf16, bf16, 128>(a, pseudo_v, log_gamma, s);
  return a.dk == 64 ? launch_wy_t<bf16, float, 64>(a, pseudo_v, log_gamma, s)
                    : launch_wy_t<bf16, float, 128>(a, pseudo_v, log_gamma, s);
}

}  // namespace tv
