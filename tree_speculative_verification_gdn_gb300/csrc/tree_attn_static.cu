// Tree attention that allocates nothing and takes no workspace: the scratch the split-KV
// kernels need (rotated queries, per-chunk max/sum, partial outputs) lives in one file-scope
// device array of TV_STATIC_SCRATCH_BYTES.  The attention itself is the one tv_tree_attn
// runs; this entry point only supplies the scratch pointer.
//
// Every host-side argument check of tv_tree_attn, and the size check against the array, runs
// before any CUDA call.  The device address of the array is then looked up with
// cudaGetSymbolAddress on the first call made in each CUDA context (the current device's
// context at the time of the call) and cached together with that context.  A call in another
// context of the same device -- after cudaDeviceReset, say, which tears down the module that
// held the array -- looks the address up again instead of using a stale one.  A lookup may
// load this file's module, so the first call on each device belongs in set-up code, before any
// stream capture.  Later calls in the same context do no lookup.
#include <cuda.h>
#include <mutex>
#include <stddef.h>
#include <stdint.h>

#include "tv.h"
#include "tv_internal.h"

namespace {

__device__ __align__(256) unsigned char g_attn_scratch[TV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// cuCtxGetCurrent through the driver entry point the runtime hands out (no link-time
// dependency on the driver library); nullptr if the driver does not provide it.
CtxGetCurrentFn ctx_get_current_fn() {
  static const CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  return fn;
}

// Device address of g_attn_scratch in the current context; cudaSuccess or the lookup's error.
cudaError_t scratch_in_current_context(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (get_ctx == nullptr) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (ctx == nullptr || g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    // No context current on this thread yet, or a different one: the lookup makes the
    // device's context current if needed; the cache then records that context.
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

int tv_tree_attn_static(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                        int num_blocks, const int32_t* block_table, int max_blocks, const int32_t* prefix_len,
                        const int32_t* parents, int B, int N, int Hq, int Hkv, int hd, int block_size,
                        float rope_theta, float sm_scale, void* out, int32_t* err, tv_stream_t stream) {
  // Host-only checks first: a bad argument or a request over the maximum is refused before
  // any CUDA call.
  const size_t need = tv_tree_attn_workspace_size(B, N, Hq, Hkv, hd, max_blocks, block_size);
  if (need > (size_t)TV_STATIC_SCRATCH_BYTES) return TV_ERR_SCRATCH;
  const int st = tv::tree_attn_check_args(q, k_new, v_new, k_cache, v_cache, num_blocks, block_table, max_blocks,
                                          prefix_len, parents, B, N, Hq, Hkv, hd, block_size, rope_theta,
                                          sm_scale, out, err);
  if (st != TV_OK) return st;
  if (need == 0) return TV_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const cudaError_t e = scratch_in_current_context(&scratch);
  if (e != cudaSuccess) return tv::cuda_status_of(e);
  return tv_tree_attn(q, k_new, v_new, k_cache, v_cache, num_blocks, block_table, max_blocks, prefix_len,
                      parents, B, N, Hq, Hkv, hd, block_size, rope_theta, sm_scale, out, scratch,
                      (size_t)TV_STATIC_SCRATCH_BYTES, err, stream);
}

}  // extern "C"
