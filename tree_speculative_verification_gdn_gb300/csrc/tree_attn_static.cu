// Tree attention that allocates nothing and takes no workspace: the scratch the split-KV
// kernels need (rotated queries, per-chunk max/sum, partial outputs) lives in one file-scope
// device array of TV_STATIC_SCRATCH_BYTES.  The attention itself is the one tv_tree_attn
// runs; this entry point only supplies the scratch pointer.
//
// The device address of the array is looked up with cudaGetSymbolAddress on the first call
// made on each device (the current device at the time of the call) and cached per device.
// That first call may load this file's module, so it belongs in set-up code, before any
// stream capture.  Later calls do no lookup.
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

// Device address of g_attn_scratch on the current device; cudaSuccess or the lookup's error.
cudaError_t scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
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
  // Host-only size check first: a request over the maximum is refused before any CUDA call.
  const size_t need = tv_tree_attn_workspace_size(B, N, Hq, Hkv, hd, max_blocks, block_size);
  if (need > (size_t)TV_STATIC_SCRATCH_BYTES) return TV_ERR_SCRATCH;
  void* scratch = nullptr;
  const cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) return tv::cuda_status_of(e);
  return tv_tree_attn(q, k_new, v_new, k_cache, v_cache, num_blocks, block_table, max_blocks, prefix_len,
                      parents, B, N, Hq, Hkv, hd, block_size, rope_theta, sm_scale, out, scratch,
                      (size_t)TV_STATIC_SCRATCH_BYTES, err, stream);
}

}  // extern "C"
