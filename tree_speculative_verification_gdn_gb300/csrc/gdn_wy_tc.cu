// TreeWY GDN tree verify on the 5th-generation tensor cores (bf16 I/O and state, dk = dv = 128).
//
// Same algebra as the CUDA-core kernel in gdn_wy.cu (TreeWY: Speculative Verification for
// Gated DeltaNet Hybrids, abstract; reading stated there).  The one dense contraction of the
// method -- S_0 times every node's key and query, [S_0 K^T | S_0 Q^T], a 128 x 2N x 128 product
// per (sequence, head) -- runs as tcgen05 MMAs: TMA stages S_0 (A operand, 128 x 128) and the
// node keys and queries (B operands, N x 128 each, zero rows past N) into shared memory in the
// 128-byte swizzle layout, one thread issues 16 MMAs (M = 128, N = Npad, K = 16) that
// accumulate in fp32 in TMEM, and the epilogue reads row r of both products back with
// tcgen05.ld, 16 columns per load -- row r belongs to TMEM lane r.  The (node, path entry)
// coefficients come from the same shared-memory tiles, 8 lanes per entry, while the MMAs run.
// The forward substitution then runs depth level by depth level: within a level every node is
// independent, so groups of threads split it, 8 nodes at a time, and every per-node load
// serves all of a thread's rows (two per thread while the products fit in shared memory).
#include "tv_async.cuh"
#include "tv_common.cuh"
#include "tv_internal.h"
#include "tv_tc.cuh"
#include "tv_tma_host.h"

namespace tv {
namespace {

constexpr int kThreads = 256;   // two warp groups; warp w reads TMEM lanes 32 (w % 4) .. + 31
constexpr int kD = 128;         // dk = dv
constexpr int kPathCap = 4096;  // max sum over nodes of (depth + 1)
constexpr int kBatch = 8;       // nodes per warp in flight during the solve
constexpr uint32_t kTileA = kD * kD * 2;  // S_0 tile bytes

// tcgen05.wait::ld with the destination registers of the loads it waits for as operands:
// every later use of them depends on the wait.
__device__ __forceinline__ void tmem_wait_ld8(uint32_t* a) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld16x2(uint32_t* a, uint32_t* c) {
  tmem_wait_ld8(a);  // one wait covers every load issued so far; the others only tie registers
  asm volatile("" : "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
               "+r"(a[15]));
  asm volatile("" : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3]), "+r"(c[4]), "+r"(c[5]), "+r"(c[6]), "+r"(c[7]));
  asm volatile("" : "+r"(c[8]), "+r"(c[9]), "+r"(c[10]), "+r"(c[11]), "+r"(c[12]), "+r"(c[13]), "+r"(c[14]),
               "+r"(c[15]));
}

// After tcgen05.wait::ld: every later use of r[0..N) depends on the wait (the empty asm
// statements are volatile, so they stay after it, and each "writes" its register).
template <int NR>
__device__ __forceinline__ void tie_after_wait(uint32_t* r) {
#pragma unroll
  for (int k = 0; k < NR; ++k) asm volatile("" : "+r"(r[k]));
}

struct TcHead {
  uint64_t tma_bar;
  uint64_t mma_bar;
  uint32_t tmem_base;
  int flag, total, fail, maxdepth;
  int par[TV_MAX_NODES];
  int depth[TV_MAX_NODES];
  int off[TV_MAX_NODES + 1];
  float lg[TV_MAX_NODES];
  float gam[TV_MAX_NODES];
  float beta[TV_MAX_NODES];
  int lvl_cnt[TV_MAX_NODES + 1];   // nodes per depth, then start of each depth level
  int lvl_fill[TV_MAX_NODES];
  int lvl_nodes[TV_MAX_NODES];     // nodes grouped by depth
  // lazy commit: the previous round's accepted path, gamma ratios, log(gamma) of its last node
  int lz_nodes[kLazyMaxLen];
  float lz_g[kLazyMaxLen];
  float lz_lga;
  int lz_L, lz_status, lz_pad;
};

static_assert(sizeof(TcHead) % 16 == 0, "the path-entry table after the head is 16-byte aligned");
static_assert(TV_MAX_NODES <= kThreads, "one node per thread in the prologue");

// LAZY: the previous round's commit is applied to S_0 first (lz); a separate instantiation, so
// the plain kernel keeps its own register allocation.
template <bool LAZY>
__global__ void __launch_bounds__(kThreads) gdn_wy_tc_kernel(GdnArgs a, float* __restrict__ pseudo_v,
                                                             float* __restrict__ log_gamma, int cap, int Npad,
                                                             uint32_t tmem_cols, int v_in_smem,
                                                             const __grid_constant__ CUtensorMap mS0,
                                                             const __grid_constant__ CUtensorMap mK,
                                                             const __grid_constant__ CUtensorMap mQ,
                                                             const __grid_constant__ CUtensorMap mV,
                                                             const __grid_constant__ WyLazy lz) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);  // 1024-byte aligned tiles
  unsigned char* sA = smem;                                  // S_0: 2 k-blocks x 128 rows x 128 B
  unsigned char* sKQ = smem + kTileA;                        // K: 2 x Npad x 128 B, then Q: same
  const uint32_t kq_bytes = (uint32_t)Npad * 128u;           // one k-block of K or Q
  unsigned char* sV = sKQ + 4 * kq_bytes;                    // V: 2 x Npad x 128 B (when it fits)
  TcHead& hd = *reinterpret_cast<TcHead*>(sV + (v_in_smem ? 2 * kq_bytes : 0));
  // Per (node, path entry) pair e, root first: coef[e] = {c_ij, e_ij} and pent[e] = (node << 8) |
  // path node.
  float2* coef = reinterpret_cast<float2*>(&hd + 1);
  int* pent = reinterpret_cast<int*>(coef + cap);
  float* wsm = reinterpret_cast<float*>(sKQ);                // [N][128], after the MMAs are done

  const int N = a.N, H = a.H;
  const int b = blockIdx.x / H, h = blockIdx.x % H;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

  // One node per thread (N <= kThreads): its parent, alpha and beta are requested before any
  // barrier, so the three loads overlap each other and the set-up below.
  const bool own = tid < N;
  const size_t nh_own = ((size_t)b * N + tid) * H + h;
  const int par_own = own ? __ldg(a.parents + (size_t)b * N + tid) : -1;
  const float alpha_own = own ? __ldg(a.alpha + nh_own) : 1.f;
  const float beta_own = own ? __ldg(a.beta + nh_own) : 0.f;

  if (tid == 0) {
    mbar_init(&hd.tma_bar, 1);
    mbar_init(&hd.mma_bar, 1);
    hd.fail = 0;
    hd.flag = 0;
    hd.maxdepth = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(&hd.tmem_base, tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = hd.tmem_base;

  if (tid == 0) {
    mbar_arrive_expect_tx(&hd.tma_bar, kTileA + (v_in_smem ? 6 : 4) * kq_bytes);
    for (int kb = 0; kb < 2; ++kb) {
      tma_load_2d(sA + kb * (kTileA / 2), &mS0, kb * 64, (b * H + h) * kD, &hd.tma_bar);
      tma_load_4d(sKQ + kb * kq_bytes, &mK, kb * 64, h, 0, b, &hd.tma_bar);
      tma_load_4d(sKQ + (2 + kb) * kq_bytes, &mQ, kb * 64, h, 0, b, &hd.tma_bar);
      if (v_in_smem) tma_load_4d(sV + kb * kq_bytes, &mV, kb * 64, h, 0, b, &hd.tma_bar);
    }
  }

  // Topology, log(gamma), gamma, beta, depth levels and path lists while the tiles are in flight.
  // A parent must be -1 or an earlier node.
  if (own) {
    hd.par[tid] = par_own;
    if (par_own < -1 || par_own >= tid) hd.flag = 1;
    hd.gam[tid] = logf(alpha_own);
    hd.beta[tid] = beta_own;
  }
  for (int i = tid; i <= N; i += kThreads) hd.lvl_cnt[i] = 0;
  __syncthreads();
  int status = hd.flag ? TV_ERR_BAD_TREE : 0;

  // Lazy commit (TreeWY abstract: rebuild only the accepted state): the previous round's
  // accepted path, its log(gamma), w rows and keys, staged while the tiles are in flight.
  // Thread 0 checks the path's own links in the previous tree.
  int* lz_nodes = hd.lz_nodes;
  float* lz_g = hd.lz_g;
  float& lz_lga = hd.lz_lga;
  int& lz_L = hd.lz_L;
  int& lz_status = hd.lz_status;
  float* lz_w = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(pent + cap) + 15) & ~uintptr_t(15));  // [L][128]
  bf16* lz_k = reinterpret_cast<bf16*>(lz_w + kLazyMaxLen * kD);      // [L][128]
  constexpr bool lazy = LAZY;
  if (lazy) {
    // Every thread stages its rows of the path's w and keys from the unchecked entries, clamped
    // into range so every read is in bounds, while warp 0 checks the path, one entry per lane:
    // node in range, its parent the previous entry (-1 for the first).  The rows are used only
    // if the check passes, and then they are the path's.
    const int Lraw = lz.len[b];
    const int Lc = Lraw < 0 ? 0 : min(Lraw, min(kLazyMaxLen, min(lz.Lmax, lz.Np)));
    for (int x = tid; x < Lc * kD; x += kThreads) {
      const int e = lz.path[(size_t)b * lz.Lmax + x / kD];
      const int node = e < 0 ? 0 : (e >= lz.Np ? lz.Np - 1 : e);
      const size_t nh = ((size_t)b * lz.Np + node) * H + h;
      lz_w[x] = lz.pseudo_v[nh * kD + x % kD];
      lz_k[x] = static_cast<const bf16*>(lz.k)[nh * kD + x % kD];
    }
    if (warp == 0) {
      const bool len_ok = Lraw >= 1 && Lraw <= lz.Lmax && Lraw <= lz.Np && Lraw <= kLazyMaxLen;
      int node = -1, pn = -1;
      float lgt = 0.f;
      if (len_ok && lane < Lraw) {
        node = lz.path[(size_t)b * lz.Lmax + lane];
        if (node >= 0 && node < lz.Np) {
          pn = lz.parents[(size_t)b * lz.Np + node];
          lgt = lz.log_gamma[((size_t)b * lz.Np + node) * H + h];
        }
      }
      int prev = __shfl_up_sync(0xffffffffu, node, 1);
      if (lane == 0) prev = -1;
      const bool mine = lane >= Lraw || (node >= 0 && node < lz.Np && pn == prev);
      const bool ok = len_ok && __all_sync(0xffffffffu, mine);
      const float lga = __shfl_sync(0xffffffffu, lgt, ok ? Lraw - 1 : 0);
      if (ok && lane < Lraw) {
        lz_nodes[lane] = node;
        lz_g[lane] = lgt;  // log(gamma) of the entry for now; the ratio below
      }
      if (lane == 0) {
        lz_L = ok ? Lraw : 0;
        lz_status = ok ? 0 : TV_ERR_BAD_PATH;
        lz_lga = lga;
      }
    }
    __syncthreads();
    if (!status) status = lz_status;
    if (!status)
      for (int t = tid; t < lz_L; t += kThreads) lz_g[t] = expf(lz_lga - lz_g[t]);
  }
  if (!status) {
    for (int i = tid; i < N; i += kThreads) {
      int d = 0;
      float lg = hd.gam[i];
      for (int j = hd.par[i]; j >= 0; j = hd.par[j]) { lg += hd.gam[j]; ++d; }
      hd.depth[i] = d;
      atomicMax(&hd.maxdepth, d);
      atomicAdd(&hd.lvl_cnt[d], 1);
      hd.lg[i] = lg;
    }
    __syncthreads();
    for (int i = tid; i < N; i += kThreads) hd.gam[i] = expf(hd.lg[i]);
    if (warp == 0) {  // exclusive scans of (depth + 1) over nodes and of node counts over depths
      int carry = 0;
      for (int base = 0; base < N; base += 32) {
        const int i = base + lane;
        int x = (i < N) ? hd.depth[i] + 1 : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        if (i < N) hd.off[i + 1] = carry + x;
        carry += __shfl_sync(0xffffffffu, x, 31);
      }
      if (lane == 0) { hd.off[0] = 0; hd.total = carry; }
      carry = 0;
      const int nl = hd.maxdepth + 1;
      for (int base = 0; base < nl; base += 32) {
        const int d = base + lane;
        int x = (d < nl) ? hd.lvl_cnt[d] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        if (d < nl) hd.lvl_cnt[d] = carry + x;  // inclusive prefix count
        carry += __shfl_sync(0xffffffffu, x, 31);
      }
    }
    __syncthreads();
    if (hd.total > cap) status = TV_ERR_UNSUPPORTED;
  }
  if (!status) {
    // lvl_cnt now holds inclusive prefix counts: level d spans [lvl_cnt[d-1], lvl_cnt[d]).
    for (int d = tid; d <= hd.maxdepth; d += kThreads) hd.lvl_fill[d] = 0;
    __syncthreads();
    for (int i = tid; i < N; i += kThreads) {
      const int d = hd.depth[i];
      const int start = d ? hd.lvl_cnt[d - 1] : 0;
      hd.lvl_nodes[start + atomicAdd(&hd.lvl_fill[d], 1)] = i;
      int j = i;
      for (int u = d; u >= 0; --u) { pent[hd.off[i] + u] = (i << 8) | j; j = hd.par[j]; }
    }
  }
  // The tiles must have landed before anything reads them -- or before the CTA may exit.
  if (!mbar_wait(&hd.tma_bar, 0)) hd.fail = 1;
  __syncthreads();
  const bool run = !status && !hd.fail;

  if (run && lazy) {
    // S_0 <- gamma_a S_0 + sum_t (gamma_a / gamma_t) w_t k_t^T on the swizzled tile, in the
    // operation order of the commit kernel; the committed state also goes back to HBM.
    // Thread (row, half) takes the 64 columns of one k-block of one row.
    // All 64 columns stay in registers while the path entries stream past, each entry's
    // coefficient formed once; every element still sees gamma_a first, then the entries in order.
    const int row = tid >> 1, kb = tid & 1, L = lz_L;
    const float gam = expf(lz_lga);
    unsigned char* rowp = sA + kb * (kTileA / 2) + row * 128;
    uint4* g = reinterpret_cast<uint4*>(static_cast<bf16*>(const_cast<void*>(a.S0)) +
                                        (((size_t)b * H + h) * kD + row) * kD + kb * 64);
    float x[8][8];
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      unpack8(*reinterpret_cast<const uint4*>(rowp + ((ch ^ (row & 7)) << 4)), x[ch]);
#pragma unroll
      for (int e = 0; e < 8; ++e) x[ch][e] *= gam;
    }
    for (int t = 0; t < L; ++t) {
      const float c = lz_g[t] * lz_w[t * kD + row];
      const uint4* kr = reinterpret_cast<const uint4*>(lz_k + t * kD + kb * 64);
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        float kf[8];
        unpack8(kr[ch], kf);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[ch][e] = fmaf(c, kf[e], x[ch][e]);
      }
    }
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      const uint4 pk = pack8(x[ch]);
      *reinterpret_cast<uint4*>(rowp + ((ch ^ (row & 7)) << 4)) = pk;
      g[ch] = pk;
    }
    fence_proxy_async();  // the MMA reads the tile through the async proxy
  }
  __syncthreads();

  if (run && tid == 0) {
    tc_fence_after();
    const uint32_t idesc = idesc_bf16_f32(128, Npad);
    const uint32_t a0 = smem_addr(sA), kq0 = smem_addr(sKQ);
    for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint64_t ad = sw128_desc(a0 + kb * (kTileA / 2) + ks * 32);
        const uint64_t bk = sw128_desc(kq0 + kb * kq_bytes + ks * 32);
        const uint64_t bq = sw128_desc(kq0 + (2 + kb) * kq_bytes + ks * 32);
        const uint32_t acc = (kb | ks) ? 1u : 0u;
        mma_bf16(tmem, ad, bk, idesc, acc);
        mma_bf16(tmem + (uint32_t)Npad, ad, bq, idesc, acc);
      }
    }
    mma_commit(&hd.mma_bar);
  }

  if (run) {
    // Coefficients c_ij = beta_i Gamma_ij (k_i.k_j) (strict ancestors) and
    // e_ij = q_scale Gamma_ij (q_i.k_j) (path incl. i): 8 lanes per (node, path entry) pair, each
    // lane 16 of the 128 elements, read from the swizzled tiles.
    const int grp = tid / 8, gl = tid % 8;
    auto chunk8 = [&](int region, int n, int g16, float* x) {  // elements 8*g16 .. 8*g16+7 of row n
      const int kb = g16 / 8, ch = g16 % 8;
      const unsigned char* p = sKQ + (region * 2 + kb) * kq_bytes + n * 128 + ((ch ^ (n & 7)) << 4);
      unpack8(*reinterpret_cast<const uint4*>(p), x);
    };
    for (int e0 = 0; e0 < hd.total; e0 += kThreads / 8) {
      const int e = e0 + grp;
      const bool valid = e < hd.total;
      const int pk = valid ? pent[e] : 0;
      const int i = pk >> 8, j = pk & 255;
      float kk = 0.f, qk = 0.f;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        float ki[8], qi[8], kj[8];
        chunk8(0, i, 2 * gl + u, ki);
        chunk8(1, i, 2 * gl + u, qi);
        chunk8(0, j, 2 * gl + u, kj);
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          kk = fmaf(ki[x], kj[x], kk);
          qk = fmaf(qi[x], kj[x], qk);
        }
      }
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) {
        kk += __shfl_xor_sync(0xffffffffu, kk, o);
        qk += __shfl_xor_sync(0xffffffffu, qk, o);
      }
      if (valid && gl == 0) {
        const int t = e - hd.off[i];
        const float G = expf(hd.lg[i] - hd.lg[j]);
        coef[e] = make_float2((t < hd.depth[i]) ? hd.beta[i] * G * kk : 0.f, a.q_scale * G * qk);
      }
    }
  }
  __syncthreads();
  if (run && !mbar_wait(&hd.mma_bar, 0)) hd.fail = 1;
  tc_fence_after();
  __syncthreads();

  if (run && !hd.fail) {
    // Thread (row r, warp group wg): r = TMEM lane.  First every node's MMA results leave TMEM
    // 16 columns per load: a_i[r] = beta_i (v_i[r] - gamma_i (S_0 k_i)_r) into wsm, and, when it
    // fits in the S_0 tile (free once the MMAs are done; N <= 64), b_i[r] = q_scale gamma_i
    // (S_0 q_i)_r into bsm.  Then the forward substitution runs depth level by depth level:
    // within a level every node is independent, so each warp takes kBatch of them at a time and
    // walks their (equal-length) ancestor lists together, one read of each ancestor's w feeding
    // both w_i = a_i - sum c_{i,t} w_t and o_i = b_i + sum e_{i,t} w_t; the two warp groups split
    // a level and meet at a barrier before the next.  Without bsm, b_i comes from single-column
    // TMEM loads requested one batch ahead.
    const bf16* __restrict__ v = static_cast<const bf16*>(a.v);
    bf16* __restrict__ out = static_cast<bf16*>(a.out);
    const int q = warp % 4, wg = warp / 4;
    const int r = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const float q_scale = a.q_scale;
    const int maxd = hd.maxdepth;
    const bool use_bsm = (uint32_t)N * kD * 4 <= kTileA;
    float* bsm = reinterpret_cast<float*>(sA);
    for (int c = wg; c < Npad / 16; c += 2) {
      uint32_t dk[16], dq[16];
      tmem_ld16_nowait(tmem + lane_base + (uint32_t)(16 * c), dk);
      if (use_bsm) tmem_ld16_nowait(tmem + lane_base + (uint32_t)(Npad + 16 * c), dq);
      tmem_wait_ld16x2(dk, dq);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = 16 * c + u;
        if (i < N) {
          float vv;
          if (v_in_smem) {  // v[i][r] from the swizzled V tile
            const int cc = r % 64;
            vv = to_f32(*(reinterpret_cast<const bf16*>(sV + (r / 64) * kq_bytes + i * 128 +
                                                         (((cc / 8) ^ (i & 7)) << 4)) + (cc % 8)));
          } else {
            vv = to_f32(v[(((size_t)b * N + i) * H + h) * kD + r]);
          }
          const float gam = hd.gam[i];
          wsm[i * kD + r] = hd.beta[i] * (vv - gam * __uint_as_float(dk[u]));
          if (use_bsm) bsm[i * kD + r] = q_scale * gam * __uint_as_float(dq[u]);
        }
      }
    }
    __syncthreads();
    // (ld_d, ld_base): the next batch whose (S_0 q) columns to request, in the order the loop
    // below consumes them (only without bsm).
    uint32_t nq[kBatch];
    int ld_d = 0, ld_base = wg * kBatch;
    auto request_next = [&]() {
      while (ld_d <= maxd && ld_base >= hd.lvl_cnt[ld_d]) {
        ++ld_d;
        if (ld_d <= maxd) ld_base = hd.lvl_cnt[ld_d - 1] + wg * kBatch;
      }
      if (ld_d > maxd) return;
      const int s1 = hd.lvl_cnt[ld_d];
#pragma unroll
      for (int x = 0; x < kBatch; ++x) {
        const int pos = ld_base + x;
        const int col = pos < s1 ? hd.lvl_nodes[pos] : 0;
        nq[x] = tmem_ld1_nowait(tmem + lane_base + (uint32_t)(Npad + col));
      }
      ld_base += 2 * kBatch;
    };
    if (use_bsm) {
      // Thread (row pair, group): rows r0 and r0 + 64 (the walk reads shared memory only, so a
      // thread's rows need not be its TMEM lane), node group g of 4 splitting each level; each
      // per-node load serves both rows.
      const int r0 = tid & 63, g = tid >> 6;
      bf16* __restrict__ outb = out + ((size_t)b * N * H + h) * kD;
      float* __restrict__ pvb = pseudo_v + ((size_t)b * N * H + h) * kD;
      for (int d = 0; d <= maxd; ++d) {
        const int s0 = d ? hd.lvl_cnt[d - 1] : 0, s1 = hd.lvl_cnt[d];
        for (int base = s0 + g * kBatch; base < s1; base += 4 * kBatch) {
          float w0[kBatch], w1[kBatch], ov0[kBatch], ov1[kBatch];
          int nodes[kBatch], o[kBatch];
#pragma unroll
          for (int x = 0; x < kBatch; ++x) {
            const int pos = base + x;
            nodes[x] = pos < s1 ? hd.lvl_nodes[pos] : -1;
            const int i = nodes[x] < 0 ? 0 : nodes[x];
            o[x] = hd.off[i];
            w0[x] = wsm[i * kD + r0];
            w1[x] = wsm[i * kD + r0 + 64];
            ov0[x] = bsm[i * kD + r0];
            ov1[x] = bsm[i * kD + r0 + 64];
          }
          for (int t = 0; t < d; ++t) {
#pragma unroll
            for (int x = 0; x < kBatch; ++x) {
              if (nodes[x] < 0) continue;
              const float2 c = coef[o[x] + t];
              const float* wj = wsm + (pent[o[x] + t] & 255) * kD + r0;
              const float a0 = wj[0], a1 = wj[64];
              w0[x] = fmaf(-c.x, a0, w0[x]);
              ov0[x] = fmaf(c.y, a0, ov0[x]);
              w1[x] = fmaf(-c.x, a1, w1[x]);
              ov1[x] = fmaf(c.y, a1, ov1[x]);
            }
          }
#pragma unroll
          for (int x = 0; x < kBatch; ++x) {
            const int i = nodes[x];
            if (i < 0) continue;
            wsm[i * kD + r0] = w0[x];
            wsm[i * kD + r0 + 64] = w1[x];
            const float e = coef[o[x] + d].y;
            const size_t ni = (size_t)i * H * kD;
            outb[ni + r0] = from_f32<bf16>(fmaf(e, w0[x], ov0[x]));
            outb[ni + r0 + 64] = from_f32<bf16>(fmaf(e, w1[x], ov1[x]));
            pvb[ni + r0] = w0[x];
            pvb[ni + r0 + 64] = w1[x];
          }
        }
        __syncthreads();
      }
    }
    if (!use_bsm) request_next();
    for (int d = 0; d <= (use_bsm ? -1 : maxd); ++d) {
      const int s0 = d ? hd.lvl_cnt[d - 1] : 0, s1 = hd.lvl_cnt[d];
      for (int base = s0 + wg * kBatch; base < s1; base += 2 * kBatch) {
        uint32_t dq[kBatch];
        if (!use_bsm) {
          tmem_wait_ld8(nq);  // the wait names the registers, so no use moves above it
#pragma unroll
          for (int x = 0; x < kBatch; ++x) dq[x] = nq[x];
          request_next();
        }
        float w[kBatch], ov[kBatch];
        int nodes[kBatch], o[kBatch];
#pragma unroll
        for (int x = 0; x < kBatch; ++x) {
          const int pos = base + x;
          nodes[x] = pos < s1 ? hd.lvl_nodes[pos] : -1;
          const int i = nodes[x] < 0 ? 0 : nodes[x];
          o[x] = hd.off[i];
          w[x] = wsm[i * kD + r];
          ov[x] = use_bsm ? bsm[i * kD + r] : q_scale * hd.gam[i] * __uint_as_float(dq[x]);
        }
        for (int t = 0; t < d; ++t) {
#pragma unroll
          for (int x = 0; x < kBatch; ++x) {
            if (nodes[x] < 0) continue;
            const float2 c = coef[o[x] + t];
            const float wj = wsm[(pent[o[x] + t] & 255) * kD + r];
            w[x] = fmaf(-c.x, wj, w[x]);
            ov[x] = fmaf(c.y, wj, ov[x]);
          }
        }
#pragma unroll
        for (int x = 0; x < kBatch; ++x) {
          const int i = nodes[x];
          if (i < 0) continue;
          wsm[i * kD + r] = w[x];
          const float ovx = fmaf(coef[o[x] + d].y, w[x], ov[x]);
          const size_t ni = ((size_t)b * N + i) * H + h;
          out[ni * kD + r] = from_f32<bf16>(ovx);
          pseudo_v[ni * kD + r] = w[x];
        }
      }
      __syncthreads();
    }
    for (int i = tid; i < N; i += kThreads) log_gamma[((size_t)b * N + i) * H + h] = hd.lg[i];
  }
  if (h == 0 && tid == 0) a.err[b] = status ? status : (hd.fail ? TV_ERR_TIMEOUT : 0);
  if (hd.fail && tid == 0) {  // a wait gave up: let in-flight copies and MMAs drain (bounded)
    mbar_wait(&hd.tma_bar, 0);
    if (!status) mbar_wait(&hd.mma_bar, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, tmem_cols);
}

// ---------------------------------------------------------------------------------------------
// Trees of at most 64 nodes: one thread per state row, the root path's pseudo-values in
// registers.
//
// 128 threads; thread r owns state row r, which is TMEM lane r of the S_0 contraction.  The key
// and query tiles are staged stacked, [K; Q] per 64-column k-block, so that two groups of
// tcgen05 MMAs run from the same shared memory at once:
//   D1 = S_0 [K; Q]^T   (M = 128 rows, N = 2 Npad)  -> (S_0 k_i)_r and (S_0 q_i)_r in lane r;
//   D2 = [K; Q] K^T     (M = 128, N = Npad)         -> k_m.k_j (lane m < Npad) and q_m.k_j
//                                                      (lane Npad + m) for every node pair.
// Warp 2 issues the copies and, as soon as they land, the MMAs, while warps 0-1 analyse the tree:
// depths, log(gamma), and the depth-first pre-order of the nodes.  Lane m of D2 then forms the
// coefficients of its node's root path, beta_i Gamma_ij (k_i.k_j) and q_scale Gamma_ij (q_i.k_j),
// and every thread turns its row of D1 into a_i and b_i, stored by pre-order position.
//
// The solve visits the nodes in pre-order.  When a node at depth d is visited, the last node
// visited at each depth t < d is its ancestor at depth t, so a thread keeps the pseudo-values
// of the current root path in registers, w_i = a_i - sum_t c_{i,t} w_t and o_i = b_i +
// sum_t e_{i,t} w_t + e_{i,i} w_i read no shared memory but a_i, b_i and the coefficients, and
// no thread ever waits for another.  Trees deeper than the register path (15) keep every w in
// shared memory instead and read the ancestors' from there.  The operation order per element is
// the kernel's above, except that the dot products come from the tensor cores.
constexpr int kSmallN = 64;
constexpr int kSThreads = 128;

struct TcHeadS {
  uint64_t tma_bar;
  uint64_t mma_bar;
  uint32_t tmem_base;
  int flag, total, fail, maxdepth, mma_issued;
  int par[kSmallN];
  int depth[kSmallN];
  int size[kSmallN];     // nodes in the subtree
  int sib[kSmallN];      // nodes in the subtrees of earlier siblings
  int pos[kSmallN];      // pre-order position of each node
  int2 meta[kSmallN];    // per position: {node | depth << 8, e_ii (register walk) or first entry (deep)}
  unsigned long long key[kSmallN];  // root-to-node path, 7 bits per level, root in the top bits
  float4 np[kSmallN];    // per node: {beta, gamma, position, -}
  float lg[kSmallN];
  float beta[kSmallN];
  float gam[kSmallN];
  int lz_nodes[kLazyMaxLen];
  float lz_g[kLazyMaxLen];
  float lz_lga;
  int lz_L, lz_status;
  int lz_store;          // a TMA store is reading the committed tile
  int lz_pad;
};
static_assert(sizeof(TcHeadS) % 16 == 0, "the entry table after the head is 16-byte aligned");

struct WySmallLayout {
  uint32_t kq, v, head, ent, anc, lz_w, lz_k, total;
};
// Byte offsets from the 1024-byte aligned base: S_0 tile, stacked [K; Q] tiles, V tile (when it
// fits), head, path-entry coefficients (cap float2 {c, e}), the entries' ancestor positions
// (cap int, deep trees only), lazy-commit rows (w and keys, fp32).  The second k-block's
// D2 A operand reads 128 rows from its start, so the allocation extends at least 16 KB past it.
__host__ __device__ inline WySmallLayout wy_small_layout(int Npad, int cap, bool lazy, bool v_in_smem) {
  WySmallLayout L{};
  L.kq = kTileA;
  const uint32_t region = (uint32_t)(2 * Npad) * 128u;   // [K; Q] rows of one k-block
  L.v = L.kq + 2 * region;
  L.head = L.v + (v_in_smem ? 2u * (uint32_t)Npad * 128u : 0u);
  L.ent = L.head + (uint32_t)sizeof(TcHeadS);
  L.anc = L.ent + (uint32_t)cap * 8u;
  uint32_t end = (L.anc + (uint32_t)cap * 4u + 15u) & ~15u;
  L.lz_w = end;
  L.lz_k = L.lz_w + (lazy ? (uint32_t)kLazyMaxLen * kD * 4u : 0u);
  end = L.lz_k + (lazy ? (uint32_t)kLazyMaxLen * kD * 4u : 0u);
  const uint32_t overrun = L.kq + region + 128u * 128u;
  L.total = end > overrun ? end : overrun;
  return L;
}

__device__ __forceinline__ void bar_sync_named(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// The solve with the root path in registers (every depth < D, D even); see above.  ab[p][r]
// holds {a, b} of the node at position p, ce[p][t] its {c, e} of the ancestor at depth t, zero
// for t >= depth (those terms vanish), and meta[p] = {node | depth << 8, e_ii}.  Every load of
// an iteration depends on p alone, so the loads of the next nodes run ahead of the arithmetic.
template <int D>
__device__ __forceinline__ void wy_small_walk_regs(const float2* __restrict__ ab, const int2* __restrict__ meta,
                                                   const float2* __restrict__ ce, int N, int H, int r,
                                                   bf16* __restrict__ outb, float* __restrict__ pvb) {
  float pw[D];
#pragma unroll
  for (int t = 0; t < D; ++t) pw[t] = 0.f;
#pragma unroll 2
  for (int p = 0; p < N; ++p) {
    const int2 m = meta[p];
    const float2 x = ab[p * kD + r];
    float w = x.x, o = x.y;
#pragma unroll
    for (int t = 0; t < D; t += 2) {
      const float4 q = *reinterpret_cast<const float4*>(ce + p * D + t);   // entries t and t + 1
      w = fmaf(-q.x, pw[t], w);
      o = fmaf(q.y, pw[t], o);
      w = fmaf(-q.z, pw[t + 1], w);
      o = fmaf(q.w, pw[t + 1], o);
    }
    o = fmaf(__int_as_float(m.y), w, o);
    const int d = m.x >> 8;
#pragma unroll
    for (int t = 0; t < D; ++t)
      if (t == d) pw[t] = w;
    const size_t ni = (size_t)(m.x & 255) * H * kD;
    outb[ni + r] = from_f32<bf16>(o);
    pvb[ni + r] = w;
  }
}

// One thread: D1 = S_0 [K; Q]^T and D2 = [K; Q] K^T, committed to hd.mma_bar.
__device__ __forceinline__ void wy_small_issue_mma(uint32_t tmem, const unsigned char* sA, const unsigned char* sKQ,
                                                   uint32_t region, int Npad, TcHeadS& hd) {
  tc_fence_after();
  const uint32_t id1 = idesc_bf16_f32(128, 2 * Npad), id2 = idesc_bf16_f32(128, Npad);
  const uint32_t a0 = smem_addr(sA), kq0 = smem_addr(sKQ);
  for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t ad = sw128_desc(a0 + kb * (kTileA / 2) + ks * 32);
      const uint64_t kq = sw128_desc(kq0 + kb * region + ks * 32);
      const uint32_t acc = (kb | ks) ? 1u : 0u;
      mma_bf16(tmem, ad, kq, id1, acc);
      mma_bf16(tmem + (uint32_t)(2 * Npad), kq, kq, id2, acc);
    }
  }
  mma_commit(&hd.mma_bar);
  hd.mma_issued = 1;
}

template <bool LAZY>
__global__ void __launch_bounds__(kSThreads, 1) gdn_wy_tc_small_kernel(
    GdnArgs a, float* __restrict__ pseudo_v, float* __restrict__ log_gamma, int cap, int Npad, uint32_t tmem_cols,
    int v_in_smem, const __grid_constant__ CUtensorMap mS0, const __grid_constant__ CUtensorMap mK,
    const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mV,
    const __grid_constant__ WyLazy lz) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const WySmallLayout Ly = wy_small_layout(Npad, cap, LAZY, v_in_smem != 0);
  unsigned char* sA = smem;
  unsigned char* sKQ = smem + Ly.kq;
  unsigned char* sV = smem + Ly.v;
  TcHeadS& hd = *reinterpret_cast<TcHeadS*>(smem + Ly.head);
  float2* ce = reinterpret_cast<float2*>(smem + Ly.ent);    // per path entry: {c, e}
  int* anc = reinterpret_cast<int*>(smem + Ly.anc);         // per path entry: the ancestor's position
  const uint32_t region = (uint32_t)(2 * Npad) * 128u;

  const int N = a.N, H = a.H;
  const int b = blockIdx.x / H, h = blockIdx.x % H;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

  // Lazy commit: warps 2-3 start the previous path's loads at once (its length and every entry
  // up to the row length); the staging below waits for them.
  int lz_len = 0, lz_ent[kLazyMaxLen];
  if (LAZY && warp >= 2) {
    lz_len = lz.len[b];
#pragma unroll
    for (int t = 0; t < kLazyMaxLen; ++t) lz_ent[t] = t < lz.Lmax ? lz.path[(size_t)b * lz.Lmax + t] : 0;
  }
  const bool own = tid < N;   // warps 0-1 analyse the tree, one node per thread
  const size_t nh_own = ((size_t)b * N + tid) * H + h;
  const int par_own = own ? __ldg(a.parents + (size_t)b * N + tid) : -1;
  const float alpha_own = own ? __ldg(a.alpha + nh_own) : 1.f;
  const float beta_own = own ? __ldg(a.beta + nh_own) : 0.f;

  if (tid == 0) {
    mbar_init(&hd.tma_bar, 1);
    mbar_init(&hd.mma_bar, 1);
    hd.fail = 0;
    hd.flag = 0;
    hd.maxdepth = 0;
    hd.mma_issued = 0;
    hd.lz_store = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(&hd.tmem_base, tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = hd.tmem_base;

  int* lz_nodes = hd.lz_nodes;
  float* lz_g = hd.lz_g;
  float* lz_w = reinterpret_cast<float*>(smem + Ly.lz_w);  // [L][128]
  float* lz_k = reinterpret_cast<float*>(smem + Ly.lz_k);  // [L][128], converted once for every row

  if (warp >= 2) {
    auto issue_tiles = [&]() {
      mbar_arrive_expect_tx(&hd.tma_bar, kTileA + (uint32_t)(v_in_smem ? 6 : 4) * (uint32_t)Npad * 128u);
      for (int kb = 0; kb < 2; ++kb) {
        tma_load_2d(sA + kb * (kTileA / 2), &mS0, kb * 64, (b * H + h) * kD, &hd.tma_bar);
        tma_load_4d(sKQ + kb * region, &mK, kb * 64, h, 0, b, &hd.tma_bar);
        tma_load_4d(sKQ + kb * region + Npad * 128, &mQ, kb * 64, h, 0, b, &hd.tma_bar);
        if (v_in_smem) tma_load_4d(sV + kb * Npad * 128, &mV, kb * 64, h, 0, b, &hd.tma_bar);
      }
    };
    if (tid == 64 && !LAZY) {
      issue_tiles();
      if (mbar_wait(&hd.tma_bar, 0)) wy_small_issue_mma(tmem, sA, sKQ, region, Npad, hd);
      else hd.fail = 1;
    }
    if (LAZY) {
      // The previous round's accepted path (TreeWY abstract: rebuild only the accepted state):
      // warps 2-3 stage the path's w and key rows from the unchecked entries, clamped into
      // range, while warp 2 checks the links, one entry per lane.  Those loads go out before
      // the tiles are requested (thread 64), so they do not queue behind them.
      const int Lraw = lz_len;
      const int Lc = Lraw < 0 ? 0 : min(Lraw, min(kLazyMaxLen, min(lz.Lmax, lz.Np)));
      // Every path entry first, then every row element (columns u and u + 64 of each entry), so
      // the loads of each kind are in flight together.
      const int u = tid - 64;
      int node[kLazyMaxLen];
#pragma unroll
      for (int t = 0; t < kLazyMaxLen; ++t) {
        const int e = t < Lc ? lz_ent[t] : 0;
        node[t] = e < 0 ? 0 : (e >= lz.Np ? lz.Np - 1 : e);
      }
      float w0[kLazyMaxLen], w1[kLazyMaxLen];
      bf16 k0[kLazyMaxLen], k1[kLazyMaxLen];
#pragma unroll
      for (int t = 0; t < kLazyMaxLen; ++t) {
        if (t < Lc) {
          const size_t nh = ((size_t)b * lz.Np + node[t]) * H + h;
          const float* w = lz.pseudo_v + nh * kD;
          const bf16* k = static_cast<const bf16*>(lz.k) + nh * kD;
          w0[t] = w[u];
          w1[t] = w[u + 64];
          k0[t] = k[u];
          k1[t] = k[u + 64];
        }
      }
      const bool len_ok = Lraw >= 1 && Lraw <= lz.Lmax && Lraw <= lz.Np && Lraw <= kLazyMaxLen;
      int lnode = -1, pn = -1;
      float lgt = 0.f;
      if (warp == 2 && len_ok && lane < Lraw) {
#pragma unroll
        for (int t = 0; t < kLazyMaxLen; ++t)
          if (t == lane) lnode = lz_ent[t];
        if (lnode >= 0 && lnode < lz.Np) {
          pn = lz.parents[(size_t)b * lz.Np + lnode];
          lgt = lz.log_gamma[((size_t)b * lz.Np + lnode) * H + h];
        }
      }
      if (tid == 64) issue_tiles();
#pragma unroll
      for (int t = 0; t < kLazyMaxLen; ++t) {
        if (t < Lc) {
          lz_w[t * kD + u] = w0[t];
          lz_w[t * kD + u + 64] = w1[t];
          lz_k[t * kD + u] = to_f32(k0[t]);
          lz_k[t * kD + u + 64] = to_f32(k1[t]);
        }
      }
      if (warp == 2) {  // the path's links, one entry per lane
        const int node = lnode;
        int prev = __shfl_up_sync(0xffffffffu, node, 1);
        if (lane == 0) prev = -1;
        const bool mine = lane >= Lraw || (node >= 0 && node < lz.Np && pn == prev);
        const bool ok = len_ok && __all_sync(0xffffffffu, mine);
        const float lga = __shfl_sync(0xffffffffu, lgt, ok ? Lraw - 1 : 0);
        if (ok && lane < Lraw) {
          lz_nodes[lane] = node;
          lz_g[lane] = expf(lga - lgt);   // gamma_a / gamma_t
        }
        if (lane == 0) {
          hd.lz_L = ok ? Lraw : 0;
          hd.lz_status = ok ? 0 : TV_ERR_BAD_PATH;
          hd.lz_lga = lga;
        }
      }
      bar_sync_named(2, 64);
    }
  } else {
    // Tree analysis, warps 0-1 (named barrier 1): a parent must be -1 or an earlier node.
    if (own) {
      hd.par[tid] = par_own;
      if (par_own < -1 || par_own >= tid) hd.flag = 1;
      hd.lg[tid] = logf(alpha_own);
      hd.beta[tid] = beta_own;
      hd.size[tid] = 0;
    }
    bar_sync_named(1, 64);
    if (!hd.flag) {
      if (own) {  // depth, log(gamma) and the path key along the root path
        int d = 0;
        float lg = hd.lg[tid];
        unsigned long long key = (unsigned long long)(tid + 1) << 56;
        for (int j = par_own; j >= 0; j = hd.par[j]) {
          lg += hd.lg[j];
          ++d;
          key = (key >> 7) | ((unsigned long long)(j + 1) << 56);
        }
        hd.depth[tid] = d;
        atomicMax(&hd.maxdepth, d);
        hd.gam[tid] = lg;  // log(gamma) for now, moved to lg below
        hd.key[tid] = key;
      }
      bar_sync_named(1, 64);
      if (hd.maxdepth <= 8) {
        // Pre-order with children in index order is the lexicographic order of the root-to-node
        // index paths; up to depth 8 a path is one 64-bit key, so a node's position is the
        // number of smaller keys.
        if (own) {
          const unsigned long long k = hd.key[tid];
          int p = 0;
#pragma unroll 8
          for (int j = 0; j < N; ++j) p += hd.key[j] < k ? 1 : 0;
          hd.pos[tid] = p;
          hd.meta[p].x = tid | (hd.depth[tid] << 8);
          hd.lg[tid] = hd.gam[tid];
          hd.gam[tid] = expf(hd.gam[tid]);
        }
      } else {
        if (own) {  // deeper trees: every node counts in its own and its ancestors' subtrees
          atomicAdd(&hd.size[tid], 1);
          for (int j = par_own; j >= 0; j = hd.par[j]) atomicAdd(&hd.size[j], 1);
        }
        bar_sync_named(1, 64);
        if (own) {
          int sib = 0;  // the subtrees of earlier siblings come first in pre-order
#pragma unroll 8
          for (int s = 0; s < tid; ++s) sib += (hd.par[s] == par_own) ? hd.size[s] : 0;
          hd.sib[tid] = sib;
          hd.lg[tid] = hd.gam[tid];
          hd.gam[tid] = expf(hd.gam[tid]);
        }
        bar_sync_named(1, 64);
        if (own) {  // pre-order position: depth + the earlier-sibling counts along the root path
          int p = hd.depth[tid];
          for (int j = tid; j >= 0; j = hd.par[j]) p += hd.sib[j];
          hd.pos[tid] = p;
          hd.meta[p].x = tid | (hd.depth[tid] << 8);
        }
      }
      bar_sync_named(1, 64);
      const int maxd = hd.maxdepth;
      if (maxd < 16) {
        // Register walk: position p's entries at ce[p * D + t], D = the walk's path length;
        // zero-filled, so the entries past a node's depth contribute nothing.
        const int D = maxd < 4 ? 4 : (maxd < 10 ? 10 : 16);
        for (int x = tid; x < N * D; x += 64) ce[x] = make_float2(0.f, 0.f);
      } else {
        if (warp == 0) {  // path entries per position: exclusive scan of (depth + 1) in pre-order
          int carry = 0;
          for (int base = 0; base < N; base += 32) {
            const int p = base + lane;
            const int x0 = (p < N) ? (hd.meta[p].x >> 8) + 1 : 0;
            int x = x0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const int y = __shfl_up_sync(0xffffffffu, x, o);
              if (lane >= o) x += y;
            }
            if (p < N) hd.meta[p].y = carry + x - x0;
            carry += __shfl_sync(0xffffffffu, x, 31);
          }
          if (lane == 0) hd.total = carry;
        }
        bar_sync_named(1, 64);
        if (own) {  // entries root first, with the ancestor's position
          const int d = hd.depth[tid], e0 = hd.meta[hd.pos[tid]].y;
          int j = tid;
          for (int t = d; t >= 0; --t) {
            anc[e0 + t] = hd.pos[j];
            j = hd.par[j];
          }
        }
      }
      if (own) hd.np[tid] = make_float4(hd.beta[tid], hd.gam[tid], __int_as_float(hd.pos[tid]), 0.f);
    }
  }
  __syncthreads();
  int status = hd.flag ? TV_ERR_BAD_TREE : 0;
  if (LAZY && !status) status = hd.lz_status;

  if constexpr (LAZY) {
    // The commit, once the analysis and the staging are both done: every thread takes one row,
    // S_0[r] <- gamma_a S_0[r] + sum_t (gamma_a / gamma_t) w_t[r] k_t, in the commit kernel's
    // operation order (paired FMAs are two plain ones), and writes it into the tile; thread 64
    // then starts the MMAs on it and two TMA stores that write it back to HBM.  A sequence that
    // does not run (bad tree or path) keeps its state.
    if (!status && !hd.fail) {
      const int row = tid, L = hd.lz_L;
      const float gam = expf(hd.lz_lga);
      if (mbar_wait(&hd.tma_bar, 0)) {
        const float2 gam2 = make_float2(gam, gam);
        for (int kb = 0; kb < 2; ++kb) {
          unsigned char* rowp = sA + kb * (kTileA / 2) + row * 128;
          float2 x[32];
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            float f[8];
            unpack8(*reinterpret_cast<const uint4*>(rowp + ((ch ^ (row & 7)) << 4)), f);
#pragma unroll
            for (int e = 0; e < 4; ++e) x[4 * ch + e] = __fmul2_rn(make_float2(f[2 * e], f[2 * e + 1]), gam2);
          }
          for (int t = 0; t < L; ++t) {
            const float c = lz_g[t] * lz_w[t * kD + row];
            const float2 c2 = make_float2(c, c);
            const float4* kr = reinterpret_cast<const float4*>(lz_k + t * kD + kb * 64);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float4 k4 = kr[q];
              x[2 * q] = __ffma2_rn(c2, make_float2(k4.x, k4.y), x[2 * q]);
              x[2 * q + 1] = __ffma2_rn(c2, make_float2(k4.z, k4.w), x[2 * q + 1]);
            }
          }
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) { f[2 * e] = x[4 * ch + e].x; f[2 * e + 1] = x[4 * ch + e].y; }
            *reinterpret_cast<uint4*>(rowp + ((ch ^ (row & 7)) << 4)) = pack8(f);
          }
        }
        fence_proxy_async();  // the MMAs read the tile through the async proxy
      } else {
        hd.fail = 1;
      }
    }
    __syncthreads();  // the tile is committed (and hd.fail settled)
    if (tid == 64 && !status && !hd.fail) {
      wy_small_issue_mma(tmem, sA, sKQ, region, Npad, hd);
      for (int kb = 0; kb < 2; ++kb)
        asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                     ::"l"(&mS0), "r"(kb * 64), "r"((b * H + h) * kD), "r"(smem_addr(sA + kb * (kTileA / 2)))
                     : "memory");
      bulk_commit();
      hd.lz_store = 1;
    }
  }
  const bool run = !status && !hd.fail;
  if (run && !mbar_wait(&hd.mma_bar, 0)) hd.fail = 1;
  if (LAZY && tid == 64 && hd.lz_store) bulk_wait_read<0>();  // the tile is free once the store has read it
  tc_fence_after();
  __syncthreads();

  if (run && !hd.fail) {
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const int r = tid;
    // Path-entry coefficients.  Lane m of D2 holds row m of [K; Q] K^T; its Npad dot products go
    // to a padded shared-memory row (the S_0 and [K; Q] tiles are free now), then the thread
    // forms the entries of its node: c = beta_i Gamma_ij (k_i.k_j) for strict ancestors (K
    // lanes), e = q_scale Gamma_ij (q_i.k_j) for the path including i (Q lanes).
    const int rs = Npad + 4;                     // row stride in floats (16-byte rows, no conflicts)
    float* d2 = reinterpret_cast<float*>(sA);    // [2 Npad][rs]
    {
      uint32_t v64[64];                          // every thread of the warp takes part in each load
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (c < Npad / 16) tmem_ld16_nowait(tmem + lane_base + (uint32_t)(2 * Npad + 16 * c), v64 + 16 * c);
      tmem_wait_ld();
      tie_after_wait<64>(v64);
      if (r < 2 * Npad) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (c < Npad / 16) {
#pragma unroll
            for (int u = 0; u < 16; u += 4)
              *reinterpret_cast<float4*>(d2 + r * rs + 16 * c + u) =
                  make_float4(__uint_as_float(v64[16 * c + u]), __uint_as_float(v64[16 * c + u + 1]),
                              __uint_as_float(v64[16 * c + u + 2]), __uint_as_float(v64[16 * c + u + 3]));
          }
      }
    }
    const int maxd = hd.maxdepth;
    const int D = maxd < 4 ? 4 : (maxd < 10 ? 10 : 16);
    {
      const bool is_k = r < Npad;
      const int i = is_k ? r : r - Npad;
      if (r < 2 * Npad && i < N) {
        const int d = hd.depth[i], p = hd.pos[i];
        const float lgi = hd.lg[i];
        const float pre = is_k ? hd.beta[i] : a.q_scale;
        // register walk: strided entries, e_ii in meta; deep trees: the packed list, e_ii at t = d
        float* dst = reinterpret_cast<float*>(ce + (maxd < 16 ? p * D : hd.meta[p].y)) + (is_k ? 0 : 1);
        int j = is_k ? hd.par[i] : i;
        for (int t = is_k ? d - 1 : d; t >= 0; --t) {   // root path, i (or its parent) first
          const float v = pre * expf(lgi - hd.lg[j]) * d2[r * rs + j];
          if (maxd < 16 && t == d) hd.meta[p].y = __float_as_int(v);
          else dst[2 * t] = v;
          j = hd.par[j];
        }
      }
    }
    tc_fence_before();
    __syncthreads();  // the entries are complete; the tiles' space is free for a and b
    tc_fence_after();

    // a_i[r] = beta_i (v_i[r] - gamma_i (S_0 k_i)_r) and b_i[r] = q_scale gamma_i (S_0 q_i)_r ->
    // ab[pos(i)][r]; 16 nodes per load pair.  The tiles are free: ab spans the S_0 tile and as
    // much of the [K; Q] tiles as it needs.
    float2* ab = reinterpret_cast<float2*>(sA);
    const bf16* __restrict__ v = static_cast<const bf16*>(a.v);
    const float q_scale = a.q_scale;
    for (int c = 0; c < Npad / 16; ++c) {
      uint32_t dk[16], dq[16];
      tmem_ld16_nowait(tmem + lane_base + (uint32_t)(16 * c), dk);
      tmem_ld16_nowait(tmem + lane_base + (uint32_t)(Npad + 16 * c), dq);
      tmem_wait_ld16x2(dk, dq);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = 16 * c + u;
        if (i < N) {
          float vv;
          if (v_in_smem) {
            const int cc = r % 64;
            vv = to_f32(*(reinterpret_cast<const bf16*>(sV + (r / 64) * Npad * 128 + i * 128 +
                                                         (((cc / 8) ^ (i & 7)) << 4)) + (cc % 8)));
          } else {
            vv = to_f32(v[(((size_t)b * N + i) * H + h) * kD + r]);
          }
          const float4 q = hd.np[i];   // {beta, gamma, position}
          ab[__float_as_int(q.z) * kD + r] =
              make_float2(q.x * (vv - q.y * __uint_as_float(dk[u])), q_scale * q.y * __uint_as_float(dq[u]));
        }
      }
    }
    bf16* __restrict__ outb = static_cast<bf16*>(a.out) + ((size_t)b * N * H + h) * kD;
    float* __restrict__ pvb = pseudo_v + ((size_t)b * N * H + h) * kD;
    if (maxd < 4) {
      wy_small_walk_regs<4>(ab, hd.meta, ce, N, H, r, outb, pvb);
    } else if (maxd < 10) {
      wy_small_walk_regs<10>(ab, hd.meta, ce, N, H, r, outb, pvb);
    } else if (maxd < 16) {
      wy_small_walk_regs<16>(ab, hd.meta, ce, N, H, r, outb, pvb);
    } else {
      // Deep trees: every w stays in ab (in place of a) and the ancestors' are read from there.
      for (int p = 0; p < N; ++p) {
        const int2 m = hd.meta[p];
        const int nid = m.x & 255, d = m.x >> 8, e0 = m.y;
        float2 x = ab[p * kD + r];
        float w = x.x, o = x.y;
        for (int t = 0; t < d; ++t) {
          const float2 q = ce[e0 + t];
          const float wj = ab[anc[e0 + t] * kD + r].x;
          w = fmaf(-q.x, wj, w);
          o = fmaf(q.y, wj, o);
        }
        o = fmaf(ce[e0 + d].y, w, o);
        ab[p * kD + r].x = w;
        const size_t ni = (size_t)nid * H * kD;
        outb[ni + r] = from_f32<bf16>(o);
        pvb[ni + r] = w;
      }
    }
    for (int i = tid; i < N; i += kSThreads) log_gamma[((size_t)b * N + i) * H + h] = hd.lg[i];
  }
  if (h == 0 && tid == 0) a.err[b] = status ? status : (hd.fail ? TV_ERR_TIMEOUT : 0);
  if (tid == 0) {  // nothing in flight may outlive the CTA's shared memory and TMEM (bounded waits)
    if (hd.fail || status) mbar_wait(&hd.tma_bar, 0);
    if (hd.mma_issued && (hd.fail || status)) mbar_wait(&hd.mma_bar, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, tmem_cols);
}

}  // namespace

bool gdn_wy_tc_supported(const GdnArgs& a) {
  return a.io == TV_BF16 && a.state == TV_BF16 && a.dk == kD && a.dv == kD;
}

bool gdn_wy_lazy_fits(int N) {
  const int Npad = (N + 15) / 16 * 16;
  int cap = N * (N + 1) / 2;
  if (cap > kPathCap) cap = kPathCap;
  if (N <= kSmallN)
    return 1024 + wy_small_layout(Npad, N * (N + 1) / 2 > 16 * N ? N * (N + 1) / 2 : 16 * N, true, false).total <=
           227 * 1024;
  return 1024 + kTileA + (size_t)4 * Npad * 128 + sizeof(TcHead) + (size_t)cap * 12 + 16 +
             (size_t)kLazyMaxLen * kD * 6 <= 227 * 1024;
}

namespace {

// The row-per-thread kernel for trees of at most 64 nodes.
cudaError_t launch_gdn_wy_tc_small(const GdnArgs& a, float* pseudo_v, float* log_gamma, const WyLazy& lz,
                                   cudaStream_t s) {
  const int Npad = (a.N + 15) / 16 * 16;
  const uint32_t cols = 3 * Npad <= 128 ? 128u : 256u;   // D1 (2 Npad columns) and D2 (Npad)
  // path entries: the packed lists of a deep tree (sum of depth + 1 <= N (N + 1) / 2) or the
  // position-strided table of the register walk (N x 16)
  const int cap = a.N * (a.N + 1) / 2 > 16 * a.N ? a.N * (a.N + 1) / 2 : 16 * a.N;
  const bool lazy = lz.path != nullptr;
  size_t smem = 1024 + wy_small_layout(Npad, cap, lazy, true).total;
  const int v_in_smem = smem <= 227 * 1024;
  if (!v_in_smem) smem = 1024 + wy_small_layout(Npad, cap, lazy, false).total;
  auto kern = lazy ? gdn_wy_tc_small_kernel<true> : gdn_wy_tc_small_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e != cudaSuccess) return e;
  // TMEM: the CTAs resident on one SM must fit in its 512 columns; pad shared memory if needed.
  for (;;) {
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kSThreads, smem);
    if (e != cudaSuccess) return e;
    if ((uint32_t)occ * cols <= 512u || smem >= 227 * 1024) break;
    smem += 8 * 1024;
    if (smem > 227 * 1024) smem = 227 * 1024;
  }
  CUtensorMap mS0, mK, mQ, mV;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)a.B * a.H * kD};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64, 128};
    if (!make_map_bf16_sw128(&mS0, a.S0, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)a.H, (cuuint64_t)a.N, (cuuint64_t)a.B};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)a.H * kD * 2, (cuuint64_t)a.N * a.H * kD * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)Npad, 1};
    if (!make_map_bf16_sw128(&mK, a.k, 4, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_map_bf16_sw128(&mQ, a.q, 4, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_map_bf16_sw128(&mV, a.v, 4, dims, strides, box)) return cudaErrorInvalidValue;
  }
  kern<<<a.B * a.H, kSThreads, smem, s>>>(a, pseudo_v, log_gamma, cap, Npad, cols, v_in_smem, mS0, mK, mQ, mV, lz);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gdn_wy_tc(const GdnArgs& a, float* pseudo_v, float* log_gamma, const WyLazy& lz,
                             cudaStream_t s) {
  if (a.N <= kSmallN) return launch_gdn_wy_tc_small(a, pseudo_v, log_gamma, lz, s);
  const int Npad = (a.N + 15) / 16 * 16;
  uint32_t cols = 32;
  while (cols < (uint32_t)(2 * Npad)) cols <<= 1;
  int cap = a.N * (a.N + 1) / 2;
  if (cap > kPathCap) cap = kPathCap;
  const size_t lazy_bytes = lz.path != nullptr ? 16 + (size_t)kLazyMaxLen * kD * (4 + 2) : 0;
  const size_t base = 1024 + kTileA + (size_t)4 * Npad * 128 + sizeof(TcHead) + (size_t)cap * 12 + lazy_bytes;
  const int v_in_smem = base + (size_t)2 * Npad * 128 <= 227 * 1024;
  size_t smem = base + (v_in_smem ? (size_t)2 * Npad * 128 : 0);
  auto kern = lz.path != nullptr ? gdn_wy_tc_kernel<true> : gdn_wy_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e != cudaSuccess) return e;
  // TMEM: the CTAs resident on one SM must fit in its 512 columns; pad shared memory if needed.
  for (;;) {
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    if ((uint32_t)occ * cols <= 512u || smem >= 227 * 1024) break;
    smem += 8 * 1024;
    if (smem > 227 * 1024) smem = 227 * 1024;
  }
  CUtensorMap mS0, mK, mQ, mV;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)a.B * a.H * kD};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64, 128};
    if (!make_map_bf16_sw128(&mS0, a.S0, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)a.H, (cuuint64_t)a.N, (cuuint64_t)a.B};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)a.H * kD * 2, (cuuint64_t)a.N * a.H * kD * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)Npad, 1};
    if (!make_map_bf16_sw128(&mK, a.k, 4, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_map_bf16_sw128(&mQ, a.q, 4, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_map_bf16_sw128(&mV, a.v, 4, dims, strides, box)) return cudaErrorInvalidValue;
  }
  kern<<<a.B * a.H, kThreads, smem, s>>>(a, pseudo_v, log_gamma, cap, Npad, cols, v_in_smem, mS0, mK, mQ, mV, lz);
  return cudaGetLastError();
}

}  // namespace tv
