// Tree-masked GQA attention over a paged KV prefix (handbook chapter 树形草稿与 EAGLE, §实现,
// forward_with_mask / tree_mask; positions prefix_len + depth from the chapter's summary).
//
// Four launches on the caller's stream:
//   1. check   -- per sequence: tree, capacity (prefix_len + N slots in the block table) and
//                 every block-table entry the call touches; err[b] is final after it.
//   2. rope    -- per node: rotate q (into the workspace, bf16) and k at prefix_len + depth,
//                 write rotated k and v into the node's cache slot prefix_len + i.
//   3. partial -- split-KV: each CTA takes one (sequence, KV head, key chunk, query-row tile)
//                 and runs an online softmax over its chunk of logical slots, masking the node
//                 slots with the tree mask; writes (max, sum, unnormalised output) per row.
//                 Head dims 128 and 256 run on the tensor cores (tree_attn_tc.cu); the CUDA-core
//                 kernel below covers the rest.
//   4. combine -- merges the chunks of every (sequence, node, query head).
// Query rows of one KV head are (node, group member) pairs, so K/V of a chunk is shared by
// every query head of the group.
#include "tv_common.cuh"
#include "tv_internal.h"

namespace tv {
namespace {

constexpr int kRowsPerCta = 32;
constexpr int kPartialThreads = 256;  // 8 warps x 4 rows
constexpr float kLog2e = 1.4426950408889634f;

struct AttnPlan {
  int chunk, nsplit, R, RG;
  size_t off_qrot, off_ml, off_acc, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

AttnPlan plan_attn(int B, int N, int Hq, int Hkv, int hd, int max_blocks, int bs) {
  AttnPlan p;
  const long long slots = (long long)max_blocks * bs;
  const long long work = (long long)B * Hkv * slots;
  // Items with one tile of 128 query rows run on single CTAs: about 1536 of them, ten per SM,
  // chunks of 128 .. 8192 keys (a sweep over 512 .. 2048 items picked it).  Items with more row
  // tiles run on CTA pairs, whose set-up and pipeline fill cost about as much as several key
  // tiles, so they take far fewer, longer chunks: whole sequences when those alone give at least
  // four waves of CTAs on a 152-SM GPU (then only sequences past 16384 keys split), otherwise
  // about 152 CTAs with no chunk longer than 6912 keys, so that sequences of unequal length
  // still spread evenly (a sweep over 1536 .. 152 CTAs and caps of 6912 .. 32768 keys picked
  // these).  The chunk count comes first and the capacity is then split evenly, so no chunk is
  // a short remainder.  The plan depends on the sizes alone, and so does the workspace size.
  const long long mtiles = ((long long)(Hq / Hkv) * N + 127) / 128;
  const long long whole_ctas = (long long)B * Hkv * 2 * ((mtiles + 1) / 2);
  long long chunk;
  if (mtiles == 1) {
    chunk = (work + 1535) / 1536;
    if (chunk > 8192) chunk = 8192;
  } else if (whole_ctas >= 4 * 152) {
    chunk = 16384;
  } else {
    chunk = (work * mtiles + 151) / 152;
    if (chunk > 6912) chunk = 6912;
  }
  if (chunk < 128) chunk = 128;
  const long long nsplit = (slots + chunk - 1) / chunk;
  chunk = (slots + nsplit - 1) / nsplit;
  chunk = (chunk + 127) / 128 * 128;
  p.chunk = (int)chunk;
  p.nsplit = (int)((slots + chunk - 1) / chunk);
  p.R = (Hq / Hkv) * N;
  p.RG = (p.R + kRowsPerCta - 1) / kRowsPerCta;
  p.off_qrot = 0;
  p.off_ml = align256((size_t)B * N * Hq * hd * sizeof(bf16));
  p.off_acc = p.off_ml + align256((size_t)B * Hkv * p.nsplit * p.R * 2 * sizeof(float));
  p.total = p.off_acc + align256((size_t)B * Hkv * p.nsplit * p.R * hd * sizeof(float));
  return p;
}

// Inverse frequencies theta^(-2c/hd), c < hd/2, computed once per call in fp64 on the host and
// passed as fp32 (hi, lo) pairs: hi + lo carries about 48 bits.
struct RopeTable {
  float2 inv[128];
};

// One CTA per (sequence, node).  Every CTA first checks its sequence -- the tree, the cache
// capacity for prefix + N slots, and the block ids those slots use -- so that nothing is written
// for a sequence that fails; the CTA of node 0 records the status.  The angle pos * inv is formed as a double-float product
// (the FMA gives the rounding error of pos * hi exactly) and reduced modulo 2 pi with the
// three-part Cody-Waite split 2 pi = C1 + C2 + C3, C1 = 25/4 having 5 significant bits so that
// k * C1 is exact for every k < 2^19 (positions below 2^21); the reduced angle is then within a
// few ulp before the fp32 sincos.
__global__ void attn_rope_kernel(AttnArgs a, bf16* __restrict__ qrot, const __grid_constant__ RopeTable tab) {
  constexpr float C1 = 6.25f, C2 = 3.318530693650246e-2f, C3 = 2.430837753308879e-10f;
  constexpr float kInv2Pi = 0.15915494309189535f;
  __shared__ float2 cs[128];  // (cos, sin) of each pair index c
  __shared__ int par[TV_MAX_NODES];
  __shared__ int flag, bad_block;
  const int b = blockIdx.x / a.N, i = blockIdx.x % a.N;
  int st = load_and_check_tree(a.parents + (size_t)b * a.N, a.N, par, &flag);
  if (!st) {
    const int P = a.prefix_len[b];
    if (P < 0 || (long long)P + a.N > (long long)a.max_blocks * a.block_size) st = TV_ERR_CAPACITY;
  }
  if (!st) {
    if (threadIdx.x == 0) bad_block = 0;
    __syncthreads();
    const int nblk = (a.prefix_len[b] + a.N + a.block_size - 1) / a.block_size;
    for (int lb = threadIdx.x; lb < nblk; lb += blockDim.x) {
      const int blk = a.block_table[(size_t)b * a.max_blocks + lb];
      if (blk < 0 || blk >= a.num_blocks) bad_block = 1;
    }
    __syncthreads();
    if (bad_block) st = TV_ERR_BAD_BLOCK;
  }
  if (i == 0 && threadIdx.x == 0) a.err[b] = st;
  if (st) return;
  const int depth = node_depth(par, i);
  const int P = a.prefix_len[b];
  const float pos = (float)(P + depth);  // exact: positions stay below 2^24
  const int hd = a.hd, half = hd / 2, bs = a.block_size;
  for (int c = threadIdx.x; c < half; c += blockDim.x) {
    const float2 iv = tab.inv[c];
    const float hi = pos * iv.x;
    const float lo = fmaf(pos, iv.x, -hi) + pos * iv.y;
    const float k = rintf(hi * kInv2Pi);
    float r = fmaf(-k, C1, hi);
    r = fmaf(-k, C2, r);
    r = fmaf(-k, C3, r);
    r += lo;
    float sn, cn;
    sincosf(r, &sn, &cn);
    cs[c] = make_float2(cn, sn);
  }
  __syncthreads();
  const int slot = P + i;
  const int blk = a.block_table[(size_t)b * a.max_blocks + slot / bs];
  const bf16* q = static_cast<const bf16*>(a.q) + ((size_t)b * a.N + i) * a.Hq * hd;
  const bf16* kn = static_cast<const bf16*>(a.k_new) + ((size_t)b * a.N + i) * a.Hkv * hd;
  const bf16* vn = static_cast<const bf16*>(a.v_new) + ((size_t)b * a.N + i) * a.Hkv * hd;
  bf16* qo = qrot + ((size_t)b * a.N + i) * a.Hq * hd;
  bf16* kc = static_cast<bf16*>(a.k_cache);
  bf16* vc = static_cast<bf16*>(a.v_cache);
  // Every (head, column pair c, c + 1) of q and k: rotate-half pairs (x_c, x_{c + half}).
  const int hp = half / 2;
  for (int x = threadIdx.x; x < (a.Hq + a.Hkv) * hp; x += blockDim.x) {
    const int h = x / hp, c = 2 * (x % hp);
    const float2 t0 = cs[c], t1 = cs[c + 1];
    const bf16* src;
    bf16* dst;
    if (h < a.Hq) {
      src = q + (size_t)h * hd;
      dst = qo + (size_t)h * hd;
    } else {
      const int g = h - a.Hq;
      const size_t row = (((size_t)blk * a.Hkv + g) * bs + slot % bs) * hd;
      src = kn + (size_t)g * hd;
      dst = kc + row;
      *reinterpret_cast<uint32_t*>(vc + row + c) = *reinterpret_cast<const uint32_t*>(vn + (size_t)g * hd + c);
      *reinterpret_cast<uint32_t*>(vc + row + c + half) =
          *reinterpret_cast<const uint32_t*>(vn + (size_t)g * hd + c + half);
    }
    const uint32_t u1 = *reinterpret_cast<const uint32_t*>(src + c);
    const uint32_t u2 = *reinterpret_cast<const uint32_t*>(src + c + half);
    const float a0 = bf16lo(u1), a1 = bf16hi(u1), b0 = bf16lo(u2), b1 = bf16hi(u2);
    float o1[2] = {a0 * t0.x - b0 * t0.y, a1 * t1.x - b1 * t1.y};
    float o2[2] = {b0 * t0.x + a0 * t0.y, b1 * t1.x + a1 * t1.y};
    *reinterpret_cast<uint32_t*>(dst + c) = pack_bf16x2(o1[0], o1[1]);
    *reinterpret_cast<uint32_t*>(dst + c + half) = pack_bf16x2(o2[0], o2[1]);
  }
}

// Split-KV partial attention on CUDA cores.  grid.x = nsplit * Hkv * RG, grid.y = B.
template <int HD>
__global__ void __launch_bounds__(kPartialThreads) attn_partial_simt_kernel(AttnArgs a, const bf16* __restrict__ qrot,
                                                                            float* __restrict__ ml,
                                                                            float* __restrict__ acc, int chunk,
                                                                            int nsplit, int RG) {
  constexpr int DPL = HD / 32;  // head dims per lane
  __shared__ __align__(16) bf16 Ks[16][HD];
  __shared__ __align__(16) bf16 Vs[16][HD];
  __shared__ uint32_t maskw[kRowsPerCta][TV_MAX_NODES / 32];
  __shared__ int par[TV_MAX_NODES];

  const int b = blockIdx.y;
  const int split = blockIdx.x % nsplit;
  const int rest = blockIdx.x / nsplit;
  const int kvh = rest % a.Hkv, rg = rest / a.Hkv;
  if (a.err[b]) return;
  const int N = a.N, P = a.prefix_len[b], total = P + N;
  const int lo = split * chunk;
  if (lo >= total) return;
  const int hi = min(total, lo + chunk);
  const int G = a.Hq / a.Hkv, R = G * N, W = (N + 31) / 32;

  for (int x = threadIdx.x; x < N; x += blockDim.x) par[x] = a.parents[(size_t)b * N + x];
  __syncthreads();
  for (int x = threadIdx.x; x < kRowsPerCta * W; x += blockDim.x) {
    const int rr = rg * kRowsPerCta + x / W, w = x % W;
    uint32_t bits = 0;
    if (rr < R)
      for (int j = rr / G; j >= 0; j = par[j])
        if ((j >> 5) == w) bits |= 1u << (j & 31);
    maskw[x / W][w] = bits;
  }

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const float scale = a.sm_scale * kLog2e;
  float qv[4][DPL], o[4][DPL], m[4], l[4];
  bool active[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int rr = rg * kRowsPerCta + warp * 4 + j;
    active[j] = rr < R;
    m[j] = -INFINITY;
    l[j] = 0.f;
    const int node = active[j] ? rr / G : 0, h = kvh * G + (active[j] ? rr % G : 0);
    const bf16* qp = qrot + (((size_t)b * N + node) * a.Hq + h) * HD + lane * DPL;
#pragma unroll
    for (int d = 0; d < DPL; ++d) {
      qv[j][d] = active[j] ? to_f32(qp[d]) : 0.f;
      o[j][d] = 0.f;
    }
  }
  const bf16* kc = static_cast<const bf16*>(a.k_cache);
  const bf16* vc = static_cast<const bf16*>(a.v_cache);
  const int* table = a.block_table + (size_t)b * a.max_blocks;
  constexpr int VPB = 16 * HD / 8;  // 16-byte vectors per block tile
  for (int s0 = lo; s0 < hi; s0 += 16) {
    __syncthreads();
    const int blk = table[s0 / 16];
    const uint4* ksrc = reinterpret_cast<const uint4*>(kc + ((size_t)blk * a.Hkv + kvh) * 16 * HD);
    const uint4* vsrc = reinterpret_cast<const uint4*>(vc + ((size_t)blk * a.Hkv + kvh) * 16 * HD);
    for (int x = threadIdx.x; x < VPB; x += blockDim.x) {
      reinterpret_cast<uint4*>(&Ks[0][0])[x] = ksrc[x];
      reinterpret_cast<uint4*>(&Vs[0][0])[x] = vsrc[x];
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (!active[j]) continue;
      const int xr = warp * 4 + j;
      float sc[16];
      float mx = -INFINITY;
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        float part = 0.f;
#pragma unroll
        for (int d = 0; d < DPL; ++d) part = fmaf(qv[j][d], to_f32(Ks[kk][lane * DPL + d]), part);
        part = group_sum<32>(part) * scale;
        const int slot = s0 + kk;
        bool vis = slot < hi;
        if (vis && slot >= P) {
          const int n = slot - P;
          vis = (maskw[xr][n >> 5] >> (n & 31)) & 1u;
        }
        sc[kk] = vis ? part : -INFINITY;
        mx = fmaxf(mx, sc[kk]);
      }
      const float m_new = fmaxf(m[j], mx);
      if (m_new == -INFINITY) continue;
      const float corr = (m[j] == -INFINITY) ? 0.f : exp2f(m[j] - m_new);
      l[j] *= corr;
#pragma unroll
      for (int d = 0; d < DPL; ++d) o[j][d] *= corr;
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const float p = (sc[kk] == -INFINITY) ? 0.f : exp2f(sc[kk] - m_new);
        l[j] += p;
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[j][d] = fmaf(p, to_f32(Vs[kk][lane * DPL + d]), o[j][d]);
      }
      m[j] = m_new;
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (!active[j]) continue;
    const int rr = rg * kRowsPerCta + warp * 4 + j;
    const size_t row = (((size_t)b * a.Hkv + kvh) * nsplit + split) * R + rr;
    if (lane == 0) {
      ml[row * 2] = m[j];
      ml[row * 2 + 1] = l[j];
    }
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[row * HD + lane * DPL + d] = o[j][d];
  }
}

// A thread merges four head dims (16 bytes) of one (sequence, node, query head) at a time:
// o = sum_s 2^(m_s - M) acc_s / l,
// l = sum_s 2^(m_s - M) l_s, M = max_s m_s.  The chunks' (m_s, l_s) and outputs are all loaded
// before any is used -- up to kBatch chunks in one round trip of loads -- and the arithmetic
// then runs chunk by chunk in order.  With `per_node`, CTA x takes the units of (sequence, node)
// x (used when those CTAs fill the GPU); otherwise one wave of CTAs takes all units grid-stride.
constexpr int kCombineThreads = 256;
constexpr int kBatch = 8;

__global__ void __launch_bounds__(kCombineThreads) attn_combine_kernel(AttnArgs a, const float* __restrict__ ml,
                                                                       const float* __restrict__ acc, int chunk,
                                                                       int nsplit, int per_node) {
  const int Hq = a.Hq, hd = a.hd, v4 = hd / 4;
  const int G = Hq / a.Hkv, R = G * a.N;
  const long long node_units = (long long)Hq * v4;
  const long long units = per_node ? node_units * (blockIdx.x + 1) : (long long)a.B * a.N * node_units;
  const long long first = per_node ? node_units * blockIdx.x + threadIdx.x : (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long step = per_node ? blockDim.x : (long long)gridDim.x * blockDim.x;
  for (long long u = first; u < units; u += step) {
    const int c = (int)(u % v4) * 4;
    const long long bih = u / v4;  // (sequence, node, query head)
    const int h = (int)(bih % Hq), i = (int)(bih / Hq % a.N), b = (int)(bih / Hq / a.N);
    if (a.err[b]) continue;
    const int total = a.prefix_len[b] + a.N;
    const int nsp = (total + chunk - 1) / chunk;
    bf16* out = static_cast<bf16*>(a.out) + ((size_t)b * a.N + i) * Hq * hd;
    // partial row of (sequence b, node i, query head h) in chunk 0; chunk s is s * R rows on
    const size_t row0 = (((size_t)b * a.Hkv + h / G) * nsplit) * R + (size_t)i * G + h % G;
    if (nsp <= kBatch) {
      float2 m_l[kBatch];
      float4 p[kBatch];
#pragma unroll
      for (int s = 0; s < kBatch; ++s)
        if (s < nsp) {
          const size_t row = row0 + (size_t)s * R;
          m_l[s] = *reinterpret_cast<const float2*>(ml + row * 2);
          p[s] = *reinterpret_cast<const float4*>(acc + row * hd + c);
        }
      float M = -INFINITY;
#pragma unroll
      for (int s = 0; s < kBatch; ++s)
        if (s < nsp) M = fmaxf(M, m_l[s].x);
      float lsum = 0.f;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s = 0; s < kBatch; ++s)
        if (s < nsp && m_l[s].x != -INFINITY) {
          const float wgt = exp2f(m_l[s].x - M);
          lsum = fmaf(m_l[s].y, wgt, lsum);
          o.x = fmaf(p[s].x, wgt, o.x);
          o.y = fmaf(p[s].y, wgt, o.y);
          o.z = fmaf(p[s].z, wgt, o.z);
          o.w = fmaf(p[s].w, wgt, o.w);
        }
      bf16* dst = out + (size_t)h * hd + c;
      dst[0] = from_f32<bf16>(o.x / lsum);
      dst[1] = from_f32<bf16>(o.y / lsum);
      dst[2] = from_f32<bf16>(o.z / lsum);
      dst[3] = from_f32<bf16>(o.w / lsum);
    } else {
      float M = -INFINITY;
      for (int s = 0; s < nsp; ++s) M = fmaxf(M, ml[(row0 + (size_t)s * R) * 2]);
      float lsum = 0.f;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < nsp; ++s) {
        const size_t row = row0 + (size_t)s * R;
        const float ms = ml[row * 2];
        if (ms == -INFINITY) continue;
        const float wgt = exp2f(ms - M);
        lsum = fmaf(ml[row * 2 + 1], wgt, lsum);
        const float4 pp = *reinterpret_cast<const float4*>(acc + row * hd + c);
        o.x = fmaf(pp.x, wgt, o.x);
        o.y = fmaf(pp.y, wgt, o.y);
        o.z = fmaf(pp.z, wgt, o.z);
        o.w = fmaf(pp.w, wgt, o.w);
      }
      bf16* dst = out + (size_t)h * hd + c;
      dst[0] = from_f32<bf16>(o.x / lsum);
      dst[1] = from_f32<bf16>(o.y / lsum);
      dst[2] = from_f32<bf16>(o.z / lsum);
      dst[3] = from_f32<bf16>(o.w / lsum);
    }
  }
}

template <int HD>
cudaError_t launch_partial(const AttnArgs& a, const AttnPlan& p, char* ws, cudaStream_t s) {
  dim3 grid(p.nsplit * a.Hkv * p.RG, a.B);
  attn_partial_simt_kernel<HD><<<grid, kPartialThreads, 0, s>>>(
      a, reinterpret_cast<const bf16*>(ws + p.off_qrot), reinterpret_cast<float*>(ws + p.off_ml),
      reinterpret_cast<float*>(ws + p.off_acc), p.chunk, p.nsplit, p.RG);
  return cudaGetLastError();
}

// One wave of combine CTAs on the current device: SMs times the resident CTAs of 256 threads
// (cached per device ordinal).
int combine_grid() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1216;
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_combine_kernel, kCombineThreads, 0) != cudaSuccess ||
      sms * per_sm <= 0)
    return 1216;
  if (dev >= 0 && dev < 64) cached[dev] = sms * per_sm;
  return sms * per_sm;
}

}  // namespace

size_t attn_workspace_size(int B, int N, int Hq, int Hkv, int hd, int max_blocks, int block_size) {
  return plan_attn(B, N, Hq, Hkv, hd, max_blocks, block_size).total;
}

cudaError_t launch_tree_attn(const AttnArgs& a, void* workspace, size_t workspace_bytes, cudaStream_t s) {
  const AttnPlan p = plan_attn(a.B, a.N, a.Hq, a.Hkv, a.hd, a.max_blocks, a.block_size);
  if (workspace_bytes < p.total) return cudaErrorInvalidValue;
  char* ws = static_cast<char*>(workspace);
  RopeTable tab;
  for (int c = 0; c < a.hd / 2; ++c) {
    const double inv = pow((double)a.rope_theta, -2.0 * c / a.hd);
    tab.inv[c].x = (float)inv;
    tab.inv[c].y = (float)(inv - (double)tab.inv[c].x);
  }
  attn_rope_kernel<<<a.B * a.N, 256, 0, s>>>(a, reinterpret_cast<bf16*>(ws + p.off_qrot), tab);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (attn_tc_supported(a))
    e = launch_attn_partial_tc(a, ws + p.off_qrot, reinterpret_cast<float*>(ws + p.off_ml),
                               reinterpret_cast<float*>(ws + p.off_acc), p.chunk, p.nsplit, s);
  else if (a.hd == 64) e = launch_partial<64>(a, p, ws, s);
  else if (a.hd == 128) e = launch_partial<128>(a, p, ws, s);
  else e = launch_partial<256>(a, p, ws, s);
  if (e != cudaSuccess) return e;
  const int wave = combine_grid();
  const int per_node = a.B * a.N >= wave ? 1 : 0;
  attn_combine_kernel<<<per_node ? a.B * a.N : wave, kCombineThreads, 0, s>>>(
      a, reinterpret_cast<const float*>(ws + p.off_ml), reinterpret_cast<const float*>(ws + p.off_acc), p.chunk,
      p.nsplit, per_node);
  return cudaGetLastError();
}

}  // namespace tv
