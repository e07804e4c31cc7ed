// Shared device helpers of the CUDA library: dtype conversion, vector loads/stores,
// warp reductions and the per-CTA tree schedule used by the GDN kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tv.h"

namespace tv {

typedef __nv_bfloat16 bf16;

// ------------------------------------------------------------------ conversions
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }

template <class T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// Two bf16 packed in a 32-bit word -> two floats (exact).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// ------------------------------------------------------------------ vector memory ops
// NE contiguous elements <-> NE floats.  NE is a multiple of 4; the address is aligned to
// 4 * sizeof(T) bytes (16 for fp32, 8 for bf16) and, for bf16 with NE >= 8, to 16 bytes.
__device__ __forceinline__ void unpack8(uint4 t, float* o) {
  o[0] = bf16lo(t.x); o[1] = bf16hi(t.x); o[2] = bf16lo(t.y); o[3] = bf16hi(t.y);
  o[4] = bf16lo(t.z); o[5] = bf16hi(t.z); o[6] = bf16lo(t.w); o[7] = bf16hi(t.w);
}
__device__ __forceinline__ void unpack4(uint2 t, float* o) {
  o[0] = bf16lo(t.x); o[1] = bf16hi(t.x); o[2] = bf16lo(t.y); o[3] = bf16hi(t.y);
}
__device__ __forceinline__ uint4 pack8(const float* i) {
  return make_uint4(pack_bf16x2(i[0], i[1]), pack_bf16x2(i[2], i[3]), pack_bf16x2(i[4], i[5]),
                    pack_bf16x2(i[6], i[7]));
}
__device__ __forceinline__ uint2 pack4(const float* i) {
  return make_uint2(pack_bf16x2(i[0], i[1]), pack_bf16x2(i[2], i[3]));
}

template <int NE>
__device__ __forceinline__ void load_vec(const float* __restrict__ p, float* out) {
  static_assert(NE % 4 == 0, "vector of 4");
#pragma unroll
  for (int j = 0; j < NE / 4; ++j) {
    float4 t = __ldg(reinterpret_cast<const float4*>(p) + j);
    out[4 * j + 0] = t.x; out[4 * j + 1] = t.y; out[4 * j + 2] = t.z; out[4 * j + 3] = t.w;
  }
}
template <int NE>
__device__ __forceinline__ void load_vec(const bf16* __restrict__ p, float* out) {
  static_assert(NE % 4 == 0, "vector of 4");
#pragma unroll
  for (int j = 0; j < NE / 8; ++j) unpack8(__ldg(reinterpret_cast<const uint4*>(p) + j), out + 8 * j);
  if constexpr (NE % 8 == 4) unpack4(__ldg(reinterpret_cast<const uint2*>(p + NE - 4)), out + NE - 4);
}
// Plain (coherent) loads, for data written earlier by the same kernel or call sequence.
template <int NE>
__device__ __forceinline__ void load_vec_rw(const float* p, float* out) {
  static_assert(NE % 4 == 0, "vector of 4");
#pragma unroll
  for (int j = 0; j < NE / 4; ++j) {
    float4 t = reinterpret_cast<const float4*>(p)[j];
    out[4 * j + 0] = t.x; out[4 * j + 1] = t.y; out[4 * j + 2] = t.z; out[4 * j + 3] = t.w;
  }
}
template <int NE>
__device__ __forceinline__ void load_vec_rw(const bf16* p, float* out) {
  static_assert(NE % 4 == 0, "vector of 4");
#pragma unroll
  for (int j = 0; j < NE / 8; ++j) unpack8(reinterpret_cast<const uint4*>(p)[j], out + 8 * j);
  if constexpr (NE % 8 == 4) unpack4(*reinterpret_cast<const uint2*>(p + NE - 4), out + NE - 4);
}

// Streaming stores (evict-first): outputs that are not re-read by this kernel.
template <int NE>
__device__ __forceinline__ void store_vec_cs(float* p, const float* in) {
  static_assert(NE % 4 == 0, "vector of 4");
#pragma unroll
  for (int j = 0; j < NE / 4; ++j)
    __stcs(reinterpret_cast<float4*>(p) + j, make_float4(in[4 * j], in[4 * j + 1], in[4 * j + 2], in[4 * j + 3]));
}
template <int NE>
__device__ __forceinline__ void store_vec_cs(bf16* p, const float* in) {
  static_assert(NE % 4 == 0, "vector of 4");
#pragma unroll
  for (int j = 0; j < NE / 8; ++j) __stcs(reinterpret_cast<uint4*>(p) + j, pack8(in + 8 * j));
  if constexpr (NE % 8 == 4) __stcs(reinterpret_cast<uint2*>(p + NE - 4), pack4(in + NE - 4));
}
template <int NE>
__device__ __forceinline__ void store_vec(float* p, const float* in) {
  static_assert(NE % 4 == 0, "vector of 4");
#pragma unroll
  for (int j = 0; j < NE / 4; ++j)
    reinterpret_cast<float4*>(p)[j] = make_float4(in[4 * j], in[4 * j + 1], in[4 * j + 2], in[4 * j + 3]);
}
template <int NE>
__device__ __forceinline__ void store_vec(bf16* p, const float* in) {
  static_assert(NE % 4 == 0, "vector of 4");
#pragma unroll
  for (int j = 0; j < NE / 8; ++j) reinterpret_cast<uint4*>(p)[j] = pack8(in + 8 * j);
  if constexpr (NE % 8 == 4) *reinterpret_cast<uint2*>(p + NE - 4) = pack4(in + NE - 4);
}

// ------------------------------------------------------------------ reductions
// Sum over groups of G consecutive lanes (G a power of two <= 32); every lane of the group
// receives the total.
template <int G>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ------------------------------------------------------------------ tree topology
// Validity of one tree (parents[i] in [-1, i)), checked by the whole block.  Loads parents
// into s_par.  Returns 0 or TV_ERR_BAD_TREE, identically in every thread.  Contains
// __syncthreads().
__device__ __forceinline__ int load_and_check_tree(const int32_t* __restrict__ parents, int N,
                                                   int* s_par, int* s_flag) {
  if (threadIdx.x == 0) *s_flag = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    int p = parents[i];
    s_par[i] = p;
    if (p < -1 || p >= i) *s_flag = 1;
  }
  __syncthreads();
  int bad = *s_flag;
  __syncthreads();
  return bad ? TV_ERR_BAD_TREE : 0;
}

__device__ __forceinline__ int node_depth(const int* s_par, int i) {
  int d = 0;
  for (int j = s_par[i]; j >= 0; j = s_par[j]) ++d;
  return d;
}

}  // namespace tv
