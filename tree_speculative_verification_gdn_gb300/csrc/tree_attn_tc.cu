// Split-KV tree attention partials on the 5th-generation tensor cores (bf16, head dim 128/256),
// run by pairs of CTAs on pairs of SMs with M = 256 MMAs (cta_group::2).
//
// Same contract as the CUDA-core partial kernel in tree_attn.cu (handbook chapter
// 树形草稿与 EAGLE, §实现, forward_with_mask): for one (sequence, KV head, key chunk) and the
// query rows of that KV head -- (node, group member) pairs -- the kernel leaves the chunk's
// running max, sum and unnormalised output per row for the combine kernel.  The tree mask is
// applied on the node slots, the running max is kept in log2 units and raised lazily (only when
// a tile's max exceeds it by more than 2^8, the output in tensor memory then rescaled), and
// value rows past the sequence end are zeroed in shared memory before PV so that unused cache
// contents never reach the accumulator.
#include "tv_async.cuh"
#include "tv_common.cuh"
#include "tv_internal.h"
#include "tv_tc.cuh"
#include "tv_tma_host.h"

namespace tv {
namespace {

constexpr int kRows = 128;        // query rows per CTA (TMEM lanes)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale = 8.0f;  // log2 headroom of the lazily raised running max

// ---------------------------------------------------------------------------------------------
// Single-CTA form, for items with one tile of query rows (where a pair would leave one SM's
// softmax idle): one CTA takes one (sequence, KV head, key chunk, tile of 128 query rows) and
// runs M = 128 MMAs on key tiles of 64.
//   warp 4      TMA producer: the rotated queries once, then K and V tiles of 64 keys (four
//               16-token pages per tile, reached through the block table) into a 2-stage and
//               a 3-stage ring;
//   warp 5      MMA issuer: S = Q K^T (M=128, N=64, K=head dim) into one of two TMEM S buffers,
//               then O += P V (M=128, N=head dim, K=64, V read as an MN-major operand);
//   warps 0-3   softmax, one query row per thread (TMEM lane = row).
constexpr int KT = 64;            // keys per tile
constexpr int kThreads = 192;     // warps 0-3 softmax, warp 4 TMA, warp 5 MMA
constexpr int kKStages = 2;       // key tiles in the ring
constexpr int kVStages = 3;       // value tiles in the ring

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kKStages];
  uint64_t k_empty[kKStages];
  uint64_t v_full[kVStages];
  uint64_t v_empty[kVStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

static_assert(sizeof(Bars) <= 256, "barriers fit their reserved region");

template <int HD>
struct Layout {
  static constexpr uint32_t QCHUNK = kRows * 128;    // one 64-column chunk of Q
  static constexpr uint32_t KVCHUNK = KT * 128;      // one 64-column chunk of a K or V tile
  static constexpr uint32_t KVB = HD / 64 * KVCHUNK; // one K (or V) tile
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t K0 = Q + HD / 64 * QCHUNK;  // kKStages key tiles
  static constexpr uint32_t V0 = K0 + kKStages * KVB;   // kVStages value tiles
  static constexpr uint32_t BARS = V0 + kVStages * KVB;
  static constexpr uint32_t TOTAL = BARS + 256;
  static constexpr uint32_t TMEM_COLS = (HD + 2 * KT <= 256) ? 256 : 512;
};

// Bounded mbarrier wait that also gives up once another role has flagged an abort.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort) {
  for (uint32_t it = 0; it < (1u << 22); ++it) {
    if (mbar_test(bar, parity)) return true;
    if (it > 64) {
      __nanosleep(64);
      if ((it & 255) == 0 && *abort) return false;
    }
  }
  *abort = 1;
  return false;
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    attn_partial_tc_kernel(AttnArgs a, float* __restrict__ ml, float* __restrict__ acc, int chunk, int nsplit,
                           int mtiles, int npt, const __grid_constant__ CUtensorMap mQ,
                           const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV) {
  using L = Layout<HD>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  Bars& bar = *reinterpret_cast<Bars*>(sm + L::BARS);
  volatile int* abort = &bar.abort;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

  // Query-row tiles of one (KV head, chunk) are adjacent so their K/V reads meet in L2.
  const int b = blockIdx.y;
  int x = blockIdx.x;
  const int mt = x % mtiles;
  x /= mtiles;
  const int split = x % nsplit;
  const int kvh = x / nsplit;
  if (a.err[b]) return;
  const int N = a.N, P = a.prefix_len[b], total = P + N;
  const int lo = split * chunk;
  if (lo >= total) return;
  const int hi = min(total, lo + chunk);
  const int T = (hi - lo + KT - 1) / KT;
  const int G = a.Hq / a.Hkv, R = G * N;
  // Softmax warps with at least one query row of this tile (rows r < active_rows); the others
  // have nothing to compute and sit the tile loop out.
  const int active_rows = G * max(0, min(npt, N - mt * npt));
  const int active_warps = (active_rows + 31) / 32;

  if (tid == 0) {
    mbar_init(&bar.q_full, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&bar.k_full[s], 1);
      mbar_init(&bar.k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bar.v_full[s], 1);
      mbar_init(&bar.v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar.s_full[s], 1);
      mbar_init(&bar.p_full[s], 32 * active_warps);
      mbar_init(&bar.pv_done[s], 1);
    }
    mbar_init(&bar.drain, 1);
    bar.abort = 0;
    mbar_fence_init();
  }
  if (warp == 5) tmem_alloc(&bar.tmem_base, L::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tO = bar.tmem_base;          // columns [0, HD): output accumulator
  const uint32_t tS = bar.tmem_base + HD;     // columns [HD, HD + 2 KT): two S buffers
  unsigned char* sQ = sm + L::Q;
  int issued_k = 0, issued_v = 0;  // K and V tiles whose loads the producer started

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer (whole warp)
    // Lane 0 posts a tile's expected bytes; then lane p < KT / 16 issues the boxes of the tile's
    // page p.  Each of those lanes reads the block ids of its page of the next key tile and of
    // the next value tile as soon as the current ones are issued, so no table read waits.
    const int last_lb = (total - 1) / 16;
    const int* table = a.block_table + (size_t)b * a.max_blocks;
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar.q_full, (uint32_t)(HD * G * npt * 2));
      for (int c = 0; c < HD / 64; ++c) tma_load_5d(sQ + c * L::QCHUNK, &mQ, c * 64, 0, kvh, mt * npt, b, &bar.q_full);
    }
    auto page_blk = [&](int j) {  // block id of this lane's page of tile j
      return (lane < KT / 16 && j < T) ? table[min((lo + j * KT) / 16 + lane, last_lb)] : 0;
    };
    // K (or V) tile j into stage st from block id blk of this lane's page: four 16-token pages,
    // each HD / 64 boxes of 64 columns.
    auto load_tile = [&](const CUtensorMap* map, uint32_t region, int st, int blk, uint64_t* full) {
      if (lane == 0) mbar_arrive_expect_tx(full, L::KVB);
      __syncwarp();
      if (lane < KT / 16)
        for (int c = 0; c < HD / 64; ++c)
          tma_load_4d(sm + region + st * L::KVB + c * L::KVCHUNK + lane * 2048, map, c * 64, 0, kvh, blk, full);
    };
    auto wait_all = [&](uint64_t* w, uint32_t parity) {
      return __all_sync(0xffffffffu, wait_or_abort(w, parity, abort));
    };
    // Keys run kKStages - 1 tiles ahead of values: a key stage frees when S of its previous
    // tile is done, a value stage when the PV of its previous tile is done.
    int kblk = page_blk(0), vblk = kblk;
    for (int jk = 0; jk < kKStages - 1 && jk < T; ++jk) {
      load_tile(&mK, L::K0, jk, kblk, &bar.k_full[jk]);
      issued_k = jk + 1;
      kblk = page_blk(jk + 1);
    }
    for (int j = 0; j < T; ++j) {
      const int jk = j + kKStages - 1;
      if (jk < T) {
        if (jk >= kKStages && !wait_all(&bar.k_empty[jk % kKStages], ((jk - kKStages) / kKStages) & 1)) break;
        load_tile(&mK, L::K0, jk % kKStages, kblk, &bar.k_full[jk % kKStages]);
        issued_k = jk + 1;
        kblk = page_blk(jk + 1);
      }
      if (j >= kVStages && !wait_all(&bar.v_empty[j % kVStages], ((j - kVStages) / kVStages) & 1)) break;
      load_tile(&mV, L::V0, j % kVStages, vblk, &bar.v_full[j % kVStages]);
      issued_v = j + 1;
      vblk = page_blk(j + 1);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // Event-driven: S of the next tile as soon as its keys have landed and its TMEM buffer is
    // free -- the PV of the tile two back, which reads that tile's P from the same columns, has
    // been issued (MMAs run in issue order, so it reads P before this S overwrites it); PV of the
    // oldest tile as soon as its P and values are ready.
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(128, KT), idO = idesc_bf16_f32(128, HD, true);
      const uint32_t q0 = smem_addr(sQ);
      bool ok = wait_or_abort(&bar.q_full, 0, abort);
      int ns = 0, np = 0;
      uint32_t idle = 0;
      while (ok && np < T) {
        bool progressed = false;
        if (ns < T && ns < np + 2 && mbar_test(&bar.k_full[ns % kKStages], (ns / kKStages) & 1)) {
          tc_fence_after();
          const int st = ns & 1, ks3 = ns % kKStages;
          const uint32_t k0 = smem_addr(sm + L::K0 + ks3 * L::KVB);
          for (int c = 0; c < HD / 64; ++c) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_bf16(tS + st * KT, sw128_desc(q0 + c * L::QCHUNK + ks * 32),
                       sw128_desc(k0 + c * L::KVCHUNK + ks * 32), idS, (c | ks) ? 1u : 0u);
          }
          mma_commit(&bar.s_full[st]);
          mma_commit(&bar.k_empty[ks3]);
          ++ns;
          progressed = true;
        }
        if (np < ns && mbar_test(&bar.p_full[np & 1], (np >> 1) & 1) &&
            mbar_test(&bar.v_full[np % kVStages], (np / kVStages) & 1)) {
          tc_fence_after();
          const int ps = np & 1, vs = np % kVStages;
          // P of the tile sits in TMEM over the first KT / 2 columns of its S buffer.
          const uint32_t v0 = smem_addr(sm + L::V0 + vs * L::KVB);
#pragma unroll
          for (int kk = 0; kk < KT / 16; ++kk)
            mma_bf16_tmem_a(tO, tS + ps * KT + kk * 8, sw128_mn_desc(v0 + kk * 2048, L::KVCHUNK), idO,
                            (np > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bar.pv_done[ps]);
          mma_commit(&bar.v_empty[vs]);
          ++np;
          progressed = true;
        }
        if (progressed) {
          idle = 0;
        } else if (++idle > (1u << 22)) {
          *abort = 1;
          ok = false;
        } else if (idle > 64) {
          __nanosleep(64);
          if ((idle & 255) == 0 && *abort) ok = false;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax, one row per thread
    const int r = tid;
    const int node = mt * npt + r / G, g = r % G;
    const bool active = (r < G * npt) && node < N;
    const bool warp_idle = warp >= active_warps;
    uint32_t mb[TV_MAX_NODES / 32];
#pragma unroll
    for (int w = 0; w < TV_MAX_NODES / 32; ++w) mb[w] = 0;
    if (active) {
      const int32_t* par = a.parents + (size_t)b * N;
      for (int j = node; j >= 0; j = par[j]) {
#pragma unroll
        for (int w = 0; w < TV_MAX_NODES / 32; ++w)
          if ((j >> 5) == w) mb[w] |= 1u << (j & 31);
      }
    }
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const float scale = a.sm_scale * kLog2e;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < T && !warp_idle; ++j) {
      const int st = j & 1;
      if (!__all_sync(0xffffffffu, wait_or_abort(&bar.s_full[st], (j >> 1) & 1, abort))) { ok = false; break; }
      tc_fence_after();
      float s[KT];
      {
        uint32_t raw[KT];
#pragma unroll
        for (int q4 = 0; q4 < KT / 16; ++q4) tmem_ld16_nowait(tS + lane_base + st * KT + q4 * 16, raw + q4 * 16);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < KT; ++c) s[c] = __uint_as_float(raw[c]);
      }
      const int base = lo + j * KT;
      // Visible columns of this tile for this row: the prefix part and, on node slots, the row
      // node's ancestors and itself.
      uint64_t vis = 0;
      if (active) {
        const int nprefix = min(max(min(hi, P) - base, 0), KT);     // prefix slots in the tile
        vis = nprefix >= 64 ? ~0ull : ((1ull << nprefix) - 1ull);
        const int node_end = min(hi - base, KT);
        for (int c = max(nprefix, 0); c < node_end; ++c) {
          const int n = base + c - P;
          uint32_t word = 0;
#pragma unroll
          for (int w = 0; w < TV_MAX_NODES / 32; ++w) word = ((n >> 5) == w) ? mb[w] : word;
          vis |= (uint64_t)((word >> (n & 31)) & 1u) << c;
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < KT; ++c) {
        s[c] = ((vis >> c) & 1ull) ? s[c] * scale : -INFINITY;
        mx = fmaxf(mx, s[c]);
      }
      const bool raise = mx > m_used + kRescale;
      const bool rescale_o = raise && m_used != -INFINITY;
      if (__any_sync(0xffffffffu, rescale_o)) {
        // O holds earlier tiles: wait for the last PV, then scale this warp's rows in TMEM.
        if (!__all_sync(0xffffffffu, wait_or_abort(&bar.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float f = rescale_o ? ex2_approx(m_used - mx) : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < HD; c0 += 16) {
          float o16[16];
          tmem_ld16(tO + lane_base + c0, o16);
#pragma unroll
          for (int e = 0; e < 16; ++e) o16[e] *= f;
          tmem_st16(tO + lane_base + c0, o16);
        }
      }
      if (raise) {
        l = rescale_o ? l * ex2_approx(m_used - mx) : 0.f;
        m_used = mx;
      }
      // P in bf16 pairs over the first KT / 2 columns of this tile's S buffer (already read).
      uint32_t pk[KT / 2];
      float psum = 0.f;
#pragma unroll
      for (int e = 0; e < KT / 2; ++e) {
        // masked keys: 2^(-inf) = 0; a row with nothing visible yet keeps m_used = -inf
        const float p0 = (m_used == -INFINITY) ? 0.f : ex2_approx(s[2 * e] - m_used);
        const float p1 = (m_used == -INFINITY) ? 0.f : ex2_approx(s[2 * e + 1] - m_used);
        pk[e] = pack_bf16x2(p0, p1);
        psum += bf16lo(pk[e]) + bf16hi(pk[e]);  // the sum of what PV will use
      }
      tmem_st32(tS + lane_base + st * KT, pk);
      l += psum;
      if (base + KT > hi) {  // zero V rows past the chunk end: their P is 0 but contents are unknown
        if (!__all_sync(0xffffffffu, wait_or_abort(&bar.v_full[j % kVStages], (j / kVStages) & 1, abort))) {
          ok = false;
          break;
        }
        const int first = hi - base;
        unsigned char* v0 = sm + L::V0 + (j % kVStages) * L::KVB;
        for (int idx = r; idx < (KT - first) * (HD / 8); idx += 32 * active_warps) {
          const int kr = first + idx / (HD / 8), rem = idx % (HD / 8);
          *reinterpret_cast<uint4*>(v0 + (rem / 8) * L::KVCHUNK + kr * 128 + (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
      }
      tc_fence_before();
      mbar_arrive(&bar.p_full[st]);
    }
    if (ok && !warp_idle && __all_sync(0xffffffffu, wait_or_abort(&bar.pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1, abort))) {
      tc_fence_after();
      const size_t row = (((size_t)b * a.Hkv + kvh) * nsplit + split) * R + (size_t)node * G + g;
#pragma unroll 1
      for (int c0 = 0; c0 < HD; c0 += 16) {
        float o16[16];
        tmem_ld16(tO + lane_base + c0, o16);
        if (active) {
          float4* dst = reinterpret_cast<float4*>(acc + row * HD + c0);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_float4(o16[4 * e], o16[4 * e + 1], o16[4 * e + 2], o16[4 * e + 3]);
        }
      }
      if (active) {
        ml[row * 2] = m_used;
        ml[row * 2 + 1] = l;
      }
    }
  }
  __syncthreads();
  if (bar.abort) {  // drain everything this CTA started before its TMEM and shared memory go away
    if (warp == 5 && lane == 0) {
      mma_commit(&bar.drain);
      mbar_wait(&bar.drain, 0);
    }
    if (warp == 4 && lane == 0) {
      mbar_wait(&bar.q_full, 0);
      for (int j = issued_k - kKStages < 0 ? 0 : issued_k - kKStages; j < issued_k; ++j)
        mbar_wait(&bar.k_full[j % kKStages], (j / kKStages) & 1);
      for (int j = issued_v - kVStages < 0 ? 0 : issued_v - kVStages; j < issued_v; ++j)
        mbar_wait(&bar.v_full[j % kVStages], (j / kVStages) & 1);
    }
    if (tid == 0) a.err[b] = TV_ERR_TIMEOUT;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(bar.tmem_base, L::TMEM_COLS);
}

// ---------------------------------------------------------------------------------------------
// Two CTAs on two SMs take query-row tiles 2p (rank 0) and 2p + 1 (rank 1) of one (sequence,
// KV head, key chunk) and run M = 256 MMAs over both, on key tiles of 128.  A key tile's 128
// keys split 64 per CTA and a value tile's head dim splits in halves, so each SM loads half of
// every K/V tile and the pair reads the chunk once (one CTA per row tile would read it once per
// row tile).  S = Q K^T runs with N = 128: an MMA of N = 64 costs about as
// much as one of N = 128 here, since both read the same A slice.
//   rank 0, warp 5   MMA issuer for the pair: S = Q K^T (M=256, N=128) and O += P V (M=256, N=hd);
//                    each commit arrives on the barrier in both CTAs;
//   rank 1, warp 5   relay: tells rank 0 when this CTA's Q, K and V tiles have landed, zeroing
//                    value rows past the sequence end first;
//   warps 4 and 6    TMA producers of the CTA's own Q tile and key half (warp 4) and value half
//                    (warp 6), apart, so a value load never waits behind a key stage;
//   warps 0-3        softmax, one query row per thread, the tile's 128 scores in registers;
//                    rank 1 arrives on rank 0's barriers.  At the end each thread moves its
//                    output row from tensor memory into the (then idle) stage region and copies
//                    it out with one bulk copy.
// Every wait is bounded; a CTA that gives up raises the abort flag in both CTAs, and both still
// reach the closing cluster barrier and free the pair's tensor memory together.
constexpr int PKT = 128;  // keys per tile
constexpr int kPairThreads = 224;

template <int HD>
struct PairLayout {
  static constexpr int KS = HD == 256 ? 2 : 4;         // half key tiles in the ring
  static constexpr int VS = HD == 256 ? 3 : 6;         // half value tiles in the ring
  static constexpr uint32_t QCHUNK = kRows * 128;      // one 64-column chunk of Q
  static constexpr uint32_t KH_CHUNK = PKT / 2 * 128;  // 64 keys of one 64-column chunk
  static constexpr uint32_t KHB = HD / 64 * KH_CHUNK;  // this CTA's half of a key tile
  static constexpr uint32_t VCHUNK = PKT * 128;        // 128 keys of one 64-column chunk
  static constexpr uint32_t VHB = HD / 128 * VCHUNK;   // this CTA's half of a value tile
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t K0 = Q + HD / 64 * QCHUNK;
  static constexpr uint32_t V0 = K0 + KS * KHB;
  static constexpr uint32_t BARS = V0 + VS * VHB;
  static constexpr uint32_t TOTAL = BARS + 512;
  // O [0, HD), two S buffers [HD, HD + 2 PKT) (P over the first PKT / 2 columns of each)
  static constexpr uint32_t TMEM_COLS = (HD + 2 * PKT <= 256) ? 256 : 512;
  static_assert(KS <= 4 && VS <= 6, "the barrier arrays hold the rings");
  static_assert(kRows * (HD + 4) * 4 <= BARS - K0, "the padded output rows fit the stage region");
};

struct PairBars {
  uint64_t q_land, q_peer;
  uint64_t k_land[4], k_peer[4], k_empty[4];
  uint64_t v_land[6], v_peer[6], v_empty[6];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  uint32_t go;
};
static_assert(sizeof(PairBars) <= 512, "pair barriers fit their reserved region");

// Bounded wait with cluster-scope acquire: the thread sleeps in the barrier unit until the phase
// completes or about a microsecond passes.
__device__ __forceinline__ bool mbar_try_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(1000u)
      : "memory");
  return done != 0;
}

template <int HD>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    attn_partial_pair_kernel(AttnArgs a, float* __restrict__ ml, float* __restrict__ acc, int chunk, int nsplit,
                             int npairs, int npt, const __grid_constant__ CUtensorMap mQ,
                             const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV) {
  using L = PairLayout<HD>;
  constexpr int KS = L::KS, VS = L::VS;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  PairBars& bar = *reinterpret_cast<PairBars*>(sm + L::BARS);
  volatile int* abort = &bar.abort;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;

  const int b = blockIdx.y;
  int x = blockIdx.x >> 1;
  const int pair = x % npairs;
  x /= npairs;
  const int split = x % nsplit;
  const int kvh = x / nsplit;
  const int mt = 2 * pair + (int)rank;
  const int N = a.N, P = a.prefix_len[b], total = P + N;
  const int lo = split * chunk;
  if (lo >= total) return;  // the same for both CTAs of the pair
  const int hi = min(total, lo + chunk);
  const int T = (hi - lo + PKT - 1) / PKT;
  const int G = a.Hq / a.Hkv, R = G * N;
  auto warps_of = [&](int t) { return (G * max(0, min(npt, N - t * npt)) + 31) / 32; };
  const int active_warps = warps_of(mt);

  if (tid == 0) {
    const uint32_t pair_warps = (uint32_t)(warps_of(2 * pair) + warps_of(2 * pair + 1));
    mbar_init(&bar.q_land, 1);
    mbar_init(&bar.q_peer, 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(&bar.k_land[s], 1);
      mbar_init(&bar.k_peer[s], 1);
      mbar_init(&bar.k_empty[s], 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&bar.v_land[s], 1);
      mbar_init(&bar.v_peer[s], 1);
      mbar_init(&bar.v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar.s_full[s], 1);
      mbar_init(&bar.p_full[s], pair_warps);
      mbar_init(&bar.pv_done[s], 1);
    }
    mbar_init(&bar.drain, 1);
    bar.abort = 0;
    bar.go = a.err[b] == 0 ? 1u : 0u;
    mbar_fence_init();
  }
  // Both CTAs' barriers exist before either signals the other.  Rank 0's reading of the status
  // word decides for the pair, so both take the same branch even if another CTA writes it.
  cluster_sync();
  if (!cluster_ld_u32(cluster_map(smem_addr(&bar.go), 0))) {
    cluster_sync();  // rank 0 stays until rank 1 has read its flag
    return;
  }
  if (warp == 5) tmem_alloc_pair(&bar.tmem_base, L::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tO = bar.tmem_base;        // output accumulator
  const uint32_t tS = bar.tmem_base + HD;   // two S buffers
  const uint32_t peer_abort = cluster_map(smem_addr((const void*)&bar.abort), peer);
  auto fail = [&]() {
    *abort = 1;
    cluster_st_u32(peer_abort, 1u);
  };
  auto pwait = [&](uint64_t* w, uint32_t parity) -> bool {
    for (uint32_t it = 0; it < (1u << 20); ++it) {
      if (mbar_try_cluster(w, parity)) return true;
      if (*abort) return false;
    }
    fail();
    return false;
  };
  auto to_rank0 = [&](uint64_t* w) { return cluster_map(smem_addr(w), 0); };
  int issued_k = 0, issued_v = 0;

  if (warp == 4 || warp == 6) {
    // ------------------------------------------------------------ TMA producers (whole warps)
    // Warp 4 loads this CTA's keys, pages 4 rank .. 4 rank + 3 of a tile (lanes 0-3); warp 6
    // loads its values, the head-dim half `rank` of all eight pages (lanes 0-7).
    const int last_lb = (total - 1) / 16;
    const int* table = a.block_table + (size_t)b * a.max_blocks;
    auto wait_all = [&](uint64_t* w, uint32_t parity) { return __all_sync(0xffffffffu, pwait(w, parity)); };
    if (warp == 4) {
      if (lane == 0) {  // this CTA's 128 query rows (padding rows past N read as zeros)
        mbar_arrive_expect_tx(&bar.q_land, (uint32_t)(HD * G * npt * 2));
        for (int c = 0; c < HD / 64; ++c)
          tma_load_5d(sm + L::Q + c * L::QCHUNK, &mQ, c * 64, 0, kvh, mt * npt, b, &bar.q_land);
      }
      auto kpage = [&](int j) {
        return (lane < 4 && j < T) ? table[min((lo + j * PKT) / 16 + 4 * (int)rank + lane, last_lb)] : 0;
      };
      int blk = kpage(0);
      for (int j = 0; j < T; ++j) {
        const int st = j % KS;
        if (j >= KS && !wait_all(&bar.k_empty[st], ((j - KS) / KS) & 1)) break;
        if (lane == 0) mbar_arrive_expect_tx(&bar.k_land[st], L::KHB);
        __syncwarp();
        if (lane < 4)
          for (int c = 0; c < HD / 64; ++c)
            tma_load_4d(sm + L::K0 + st * L::KHB + c * L::KH_CHUNK + lane * 2048, &mK, c * 64, 0, kvh, blk,
                        &bar.k_land[st]);
        issued_k = j + 1;
        blk = kpage(j + 1);
      }
    } else {
      auto vpage = [&](int j) { return (lane < 8 && j < T) ? table[min((lo + j * PKT) / 16 + lane, last_lb)] : 0; };
      int blk = vpage(0);
      for (int j = 0; j < T; ++j) {
        const int st = j % VS;
        if (j >= VS && !wait_all(&bar.v_empty[st], ((j - VS) / VS) & 1)) break;
        if (lane == 0) mbar_arrive_expect_tx(&bar.v_land[st], L::VHB);
        __syncwarp();
        if (lane < 8)
          for (int cc = 0; cc < HD / 128; ++cc)
            tma_load_4d(sm + L::V0 + st * L::VHB + cc * L::VCHUNK + lane * 2048, &mV,
                        ((int)rank * (HD / 128) + cc) * 64, 0, kvh, blk, &bar.v_land[st]);
        issued_v = j + 1;
        blk = vpage(j + 1);
      }
    }
  } else if (warp == 5 && rank == 0) {
    // ------------------------------------------------------------ MMA issuer for the pair
    // Event-driven: S of the next tile once both halves of its keys have landed and its S buffer
    // is free (the PV that reads the buffer's P has been issued, and MMAs run in issue order);
    // PV of the oldest tile once its P (both CTAs) and both halves of its values are ready.
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(256, PKT), idO = idesc_bf16_f32(256, HD, true);
      const uint32_t q0 = smem_addr(sm + L::Q);
      bool ok = pwait(&bar.q_land, 0) && pwait(&bar.q_peer, 0);
      int ns = 0, np = 0;
      uint32_t idle = 0;
      while (ok && np < T) {
        bool progressed = false;
        const int ks = ns % KS, kph = (ns / KS) & 1;
        if (ns < T && ns < np + 2 && mbar_test(&bar.k_land[ks], kph) && mbar_test_cluster(&bar.k_peer[ks], kph)) {
          tc_fence_after();
          const int st = ns & 1;
          const uint32_t k0 = smem_addr(sm + L::K0 + ks * L::KHB);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk)
            mma_bf16_pair(tS + st * PKT, sw128_desc(q0 + (kk / 4) * L::QCHUNK + (kk % 4) * 32),
                          sw128_desc(k0 + (kk / 4) * L::KH_CHUNK + (kk % 4) * 32), idS, kk ? 1u : 0u);
          mma_commit_pair(&bar.s_full[st], 3);
          mma_commit_pair(&bar.k_empty[ks], 3);
          ++ns;
          progressed = true;
        }
        const int vs = np % VS, vph = (np / VS) & 1;
        if (np < ns && mbar_test_cluster(&bar.p_full[np & 1], (np >> 1) & 1) && mbar_test(&bar.v_land[vs], vph) &&
            mbar_test_cluster(&bar.v_peer[vs], vph)) {
          tc_fence_after();
          const int ps = np & 1;
          const uint32_t v0 = smem_addr(sm + L::V0 + vs * L::VHB);
#pragma unroll
          for (int kk = 0; kk < PKT / 16; ++kk)
            mma_bf16_tmem_a_pair(tO, tS + ps * PKT + kk * 8, sw128_mn_desc(v0 + kk * 2048, L::VCHUNK), idO,
                                 (np > 0 || kk > 0) ? 1u : 0u);
          mma_commit_pair(&bar.pv_done[ps], 3);
          mma_commit_pair(&bar.v_empty[vs], 3);
          ++np;
          progressed = true;
        }
        if (progressed) {
          idle = 0;
        } else if (++idle > (1u << 20)) {
          fail();
          ok = false;
        } else {
          // sleep in the barrier unit on what the oldest tile still lacks, else on the keys of
          // the next one
          if (np < ns && !mbar_test_cluster(&bar.p_full[np & 1], (np >> 1) & 1))
            mbar_try_cluster(&bar.p_full[np & 1], (np >> 1) & 1);
          else if (np < ns && !mbar_test(&bar.v_land[vs], vph))
            mbar_try_cluster(&bar.v_land[vs], vph);
          else if (np < ns)
            mbar_try_cluster(&bar.v_peer[vs], vph);
          else
            mbar_try_cluster(&bar.k_land[ks], kph);
          if (*abort) ok = false;
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ relay (rank 1, whole warp)
    bool ok = __all_sync(0xffffffffu, pwait(&bar.q_land, 0));
    if (ok && lane == 0) mbar_arrive_cluster_relaxed(to_rank0(&bar.q_peer));
    int nk = 0, nv = 0;
    uint32_t idle = 0;
    while (ok && (nk < T || nv < T)) {
      bool progressed = false;
      if (nk < T && __shfl_sync(0xffffffffu, lane == 0 && mbar_test(&bar.k_land[nk % KS], (nk / KS) & 1), 0)) {
        if (lane == 0) mbar_arrive_cluster_relaxed(to_rank0(&bar.k_peer[nk % KS]));
        ++nk;
        progressed = true;
      }
      if (nv < T && __shfl_sync(0xffffffffu, lane == 0 && mbar_test(&bar.v_land[nv % VS], (nv / VS) & 1), 0)) {
        const int base = lo + nv * PKT;
        if (base + PKT > hi) {  // value rows past the chunk end: their P is 0 but contents are unknown
          const int first = hi - base;
          unsigned char* v0 = sm + L::V0 + (nv % VS) * L::VHB;
          for (int idx = lane; idx < (PKT - first) * (HD / 16); idx += 32) {
            const int kr = first + idx / (HD / 16), rem = idx % (HD / 16);
            *reinterpret_cast<uint4*>(v0 + (rem / 8) * L::VCHUNK + kr * 128 + (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async();
          __syncwarp();
        }
        if (lane == 0) mbar_arrive_cluster_relaxed(to_rank0(&bar.v_peer[nv % VS]));
        ++nv;
        progressed = true;
      }
      if (progressed) {
        idle = 0;
      } else if (++idle > (1u << 20)) {
        if (lane == 0) fail();
        ok = false;
      } else {
        if (lane == 0) {
          if (nk < T)
            mbar_try_cluster(&bar.k_land[nk % KS], (nk / KS) & 1);
          else
            mbar_try_cluster(&bar.v_land[nv % VS], (nv / VS) & 1);
        }
        ok = __shfl_sync(0xffffffffu, *abort == 0, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax, one row per thread
    const int r = tid;
    const int node = mt * npt + r / G, g = r % G;
    const bool active = (r < G * npt) && node < N;
    const bool warp_idle = warp >= active_warps;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    bool ok = true;
    uint32_t mb[TV_MAX_NODES / 32];
#pragma unroll
    for (int w = 0; w < TV_MAX_NODES / 32; ++w) mb[w] = 0;
    if (active) {
      const int32_t* par = a.parents + (size_t)b * N;
      for (int j = node; j >= 0; j = par[j]) {
#pragma unroll
        for (int w = 0; w < TV_MAX_NODES / 32; ++w)
          if ((j >> 5) == w) mb[w] |= 1u << (j & 31);
      }
    }
    const float scale = a.sm_scale * kLog2e;
    // Visible keys of the 64-key half starting at slot `base` for this row: the prefix part and,
    // on node slots, the row node's ancestors and itself.
    auto visible = [&](int base) -> uint64_t {
      if (!active) return 0;
      const int nprefix = min(max(min(hi, P) - base, 0), 64);
      uint64_t vis = nprefix >= 64 ? ~0ull : ((1ull << nprefix) - 1ull);
      const int node_end = min(hi - base, 64);
      for (int c = max(nprefix, 0); c < node_end; ++c) {
        const int n = base + c - P;
        uint32_t word = 0;
#pragma unroll
        for (int w = 0; w < TV_MAX_NODES / 32; ++w) word = ((n >> 5) == w) ? mb[w] : word;
        vis |= (uint64_t)((word >> (n & 31)) & 1u) << c;
      }
      return vis;
    };
    float m_used = -INFINITY, l = 0.f;
    for (int j = 0; j < T && !warp_idle; ++j) {
      const int st = j & 1;
      if (!__all_sync(0xffffffffu, pwait(&bar.s_full[st], (j >> 1) & 1))) { ok = false; break; }
      tc_fence_after();
      const int base = lo + j * PKT;
      const uint32_t sbuf = tS + lane_base + st * PKT;
      // the whole tile's S in registers, one load
      float s[PKT];
      {
        uint32_t rawv[PKT];
#pragma unroll
        for (int q4 = 0; q4 < PKT / 16; ++q4) tmem_ld16_nowait(sbuf + q4 * 16, rawv + q4 * 16);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < PKT; ++c) s[c] = __uint_as_float(rawv[c]) * scale;  // log2 units
      }
      // tiles wholly inside the prefix need no mask; others set invisible keys to -inf
      if (!__all_sync(0xffffffffu, active && base + PKT <= min(hi, P))) {
        const uint64_t vis0 = visible(base), vis1 = visible(base + 64);
#pragma unroll
        for (int c = 0; c < PKT; ++c)
          if (!((((c < 64) ? vis0 : vis1) >> (c & 63)) & 1ull)) s[c] = -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < PKT; ++c) mx = fmaxf(mx, s[c]);
      const bool raise = mx > m_used + kRescale;
      const bool rescale_o = raise && m_used != -INFINITY;
      if (__any_sync(0xffffffffu, rescale_o)) {
        if (!__all_sync(0xffffffffu, pwait(&bar.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float f = rescale_o ? ex2_approx(m_used - mx) : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < HD; c0 += 16) {
          float o16[16];
          tmem_ld16(tO + lane_base + c0, o16);
#pragma unroll
          for (int e = 0; e < 16; ++e) o16[e] *= f;
          tmem_st16(tO + lane_base + c0, o16);
        }
      }
      if (raise) {
        l = rescale_o ? l * ex2_approx(m_used - mx) : 0.f;
        m_used = mx;
      }
      // P in bf16 pairs over the first PKT / 2 columns of the S buffer (already read); a row
      // with nothing visible yet keeps m_used = -inf and gives 0, masked keys give 2^-inf = 0
      const float mneg = m_used == -INFINITY ? 0.f : -m_used;
      const bool none = m_used == -INFINITY;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
        float psum = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float p0 = none ? 0.f : ex2_approx(s[64 * h + 2 * e] + mneg);
          const float p1 = none ? 0.f : ex2_approx(s[64 * h + 2 * e + 1] + mneg);
          pk[e] = pack_bf16x2(p0, p1);
          psum += bf16lo(pk[e]) + bf16hi(pk[e]);
        }
        tmem_st32(sbuf + h * 32, pk);
        l += psum;
      }
      if (rank == 0 && base + PKT > hi) {  // rank 0's value rows past the chunk end (rank 1's relay zeroes its own)
        if (!__all_sync(0xffffffffu, pwait(&bar.v_land[j % VS], (j / VS) & 1))) {
          ok = false;
          break;
        }
        const int first = hi - base;
        unsigned char* v0 = sm + L::V0 + (j % VS) * L::VHB;
        for (int idx = r; idx < (PKT - first) * (HD / 16); idx += 32 * active_warps) {
          const int kr = first + idx / (HD / 16), rem = idx % (HD / 16);
          *reinterpret_cast<uint4*>(v0 + (rem / 8) * L::VCHUNK + kr * 128 + (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(&bar.p_full[st]);
        else
          mbar_arrive_cluster_relaxed(to_rank0(&bar.p_full[st]));
      }
    }
    if (ok && !warp_idle && __all_sync(0xffffffffu, pwait(&bar.pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1))) {
      tc_fence_after();
      // Every key and value stage has been consumed: the row goes through the stage region,
      // padded by 16 bytes per row so that a warp's 16-byte stores meet all banks, and out with
      // one bulk copy.
      const size_t row = (((size_t)b * a.Hkv + kvh) * nsplit + split) * R + (size_t)node * G + g;
      float* stage = reinterpret_cast<float*>(sm + L::K0) + (size_t)r * (HD + 4);
#pragma unroll 1
      for (int c0 = 0; c0 < HD; c0 += 64) {
        uint32_t o[64];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) tmem_ld16_nowait(tO + lane_base + c0 + q4 * 16, o + q4 * 16);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e)
          *reinterpret_cast<uint4*>(stage + c0 + 4 * e) = make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
      }
      fence_proxy_async();
      if (active) {
        bulk_s2g(acc + row * HD, stage, HD * 4);
        bulk_commit();
        ml[row * 2] = m_used;
        ml[row * 2 + 1] = l;
        bulk_wait_read<0>();
      }
    }
  }
  __syncthreads();
  // Close: rank 0's last commit reaches both CTAs once every pair MMA has completed; each CTA
  // then lets its own loads land, and neither leaves or frees tensor memory before the other.
  if (warp == 5 && lane == 0) {
    if (rank == 0) mma_commit_pair(&bar.drain, 3);
    if (!mbar_wait(&bar.drain, 0)) *abort = 1;
  }
  __syncthreads();
  if (*abort) {
    if (warp == 4 && lane == 0) {
      mbar_wait(&bar.q_land, 0);
      for (int j = issued_k - KS < 0 ? 0 : issued_k - KS; j < issued_k; ++j)
        mbar_wait(&bar.k_land[j % KS], (j / KS) & 1);
    }
    if (warp == 6 && lane == 0)
      for (int j = issued_v - VS < 0 ? 0 : issued_v - VS; j < issued_v; ++j)
        mbar_wait(&bar.v_land[j % VS], (j / VS) & 1);
    if (tid == 0) a.err[b] = TV_ERR_TIMEOUT;
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 5) tmem_dealloc_pair(bar.tmem_base, L::TMEM_COLS);
}

template <int HD>
cudaError_t launch_pair_t(const AttnArgs& a, const void* qrot, float* ml, float* acc, int chunk, int nsplit,
                          cudaStream_t s) {
  using L = PairLayout<HD>;
  const int G = a.Hq / a.Hkv;
  const int npt = kRows / G;
  const int mtiles = (a.N + npt - 1) / npt;
  const int npairs = (mtiles + 1) / 2;
  CUtensorMap mQ, mK, mV;
  {
    // rotated queries [B][N][Hkv][G][hd]
    const cuuint64_t dims[5] = {(cuuint64_t)HD, (cuuint64_t)G, (cuuint64_t)a.Hkv, (cuuint64_t)a.N, (cuuint64_t)a.B};
    const cuuint64_t strides[4] = {(cuuint64_t)HD * 2, (cuuint64_t)G * HD * 2, (cuuint64_t)a.Hq * HD * 2,
                                   (cuuint64_t)a.N * a.Hq * HD * 2};
    const cuuint32_t box[5] = {64, (cuuint32_t)G, 1, (cuuint32_t)npt, 1};
    if (!make_map_bf16_sw128(&mQ, qrot, 5, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[4] = {(cuuint64_t)HD, 16, (cuuint64_t)a.Hkv, (cuuint64_t)a.num_blocks};
    const cuuint64_t strides[3] = {(cuuint64_t)HD * 2, (cuuint64_t)16 * HD * 2, (cuuint64_t)a.Hkv * 16 * HD * 2};
    const cuuint32_t box[4] = {64, 16, 1, 1};
    if (!make_map_bf16_sw128(&mK, a.k_cache, 4, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_map_bf16_sw128(&mV, a.v_cache, 4, dims, strides, box)) return cudaErrorInvalidValue;
  }
  const size_t smem = L::TOTAL + 1024;
  auto kern = attn_partial_pair_kernel<HD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(nsplit * npairs * 2 * a.Hkv, a.B);
  kern<<<grid, kPairThreads, smem, s>>>(a, ml, acc, chunk, nsplit, npairs, npt, mQ, mK, mV);
  return cudaGetLastError();
}

template <int HD>
cudaError_t launch_t(const AttnArgs& a, const void* qrot, float* ml, float* acc, int chunk, int nsplit,
                     cudaStream_t s) {
  using L = Layout<HD>;
  const int G = a.Hq / a.Hkv;
  const int npt = kRows / G;                     // nodes per tile of 128 query rows
  const int mtiles = (a.N + npt - 1) / npt;
  CUtensorMap mQ, mK, mV;
  {
    // rotated queries [B][N][Hkv][G][hd]
    const cuuint64_t dims[5] = {(cuuint64_t)HD, (cuuint64_t)G, (cuuint64_t)a.Hkv, (cuuint64_t)a.N, (cuuint64_t)a.B};
    const cuuint64_t strides[4] = {(cuuint64_t)HD * 2, (cuuint64_t)G * HD * 2, (cuuint64_t)a.Hq * HD * 2,
                                   (cuuint64_t)a.N * a.Hq * HD * 2};
    const cuuint32_t box[5] = {64, (cuuint32_t)G, 1, (cuuint32_t)npt, 1};
    if (!make_map_bf16_sw128(&mQ, qrot, 5, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    // caches [num_blocks][Hkv][16][hd]
    const cuuint64_t dims[4] = {(cuuint64_t)HD, 16, (cuuint64_t)a.Hkv, (cuuint64_t)a.num_blocks};
    const cuuint64_t strides[3] = {(cuuint64_t)HD * 2, (cuuint64_t)16 * HD * 2, (cuuint64_t)a.Hkv * 16 * HD * 2};
    const cuuint32_t box[4] = {64, 16, 1, 1};
    if (!make_map_bf16_sw128(&mK, a.k_cache, 4, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_map_bf16_sw128(&mV, a.v_cache, 4, dims, strides, box)) return cudaErrorInvalidValue;
  }
  const size_t smem = L::TOTAL + 1024;
  auto kern = attn_partial_tc_kernel<HD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(nsplit * mtiles * a.Hkv, a.B);
  kern<<<grid, kThreads, smem, s>>>(a, ml, acc, chunk, nsplit, mtiles, npt, mQ, mK, mV);
  return cudaGetLastError();
}

}  // namespace

int attn_tc_row_tiles(const AttnArgs& a) { return (a.Hq / a.Hkv * a.N + kRows - 1) / kRows; }

bool attn_tc_supported(const AttnArgs& a) {
  const int G = a.Hq / a.Hkv;
  return (a.hd == 128 || a.hd == 256) && G >= 1 && G <= 128 && (128 % G) == 0 && a.block_size == 16;
}

cudaError_t launch_attn_partial_tc(const AttnArgs& a, const void* qrot, float* ml, float* acc, int chunk,
                                   int nsplit, cudaStream_t s) {
  if (chunk % PKT) return cudaErrorInvalidValue;
  if (attn_tc_row_tiles(a) == 1)
    return a.hd == 128 ? launch_t<128>(a, qrot, ml, acc, chunk, nsplit, s)
                       : launch_t<256>(a, qrot, ml, acc, chunk, nsplit, s);
  return a.hd == 128 ? launch_pair_t<128>(a, qrot, ml, acc, chunk, nsplit, s)
                     : launch_pair_t<256>(a, qrot, ml, acc, chunk, nsplit, s);
}

}  // namespace tv
