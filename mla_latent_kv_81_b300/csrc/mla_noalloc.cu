// mla_compress_append_noalloc: the cache append without a caller-provided workspace.
//
// The append needs scratch for the fp32 k-split partials of the down-projection.
// This variant takes that scratch from a fixed array compiled into the library
// instead of from the caller, for callers that cannot allocate device memory
// (see include/mla.h).  It runs exactly the same kernels as mla_compress_append.
#include <mutex>

#include "mla_common.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;   // 16 MiB per device that loads the library

// In host code this name is only a stand-in for the device array; its device
// address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_append_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device.
mla_status scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_append_scratch) != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" mla_status mla_compress_append_noalloc(const mla_config* cfg, const void* x, const void* W_DKV,
                                                  const void* W_KR, const int32_t* seq_idx, const int32_t* pos,
                                                  const mla_rope_table* rope, const mla_paged_cache* cache, int T,
                                                  mla_stream_t stream) {
  // the same argument checks as mla_compress_append, in the same order
  const mla_status v = mla::validate_append(cfg, x, W_DKV, W_KR, seq_idx, pos, rope, cache, T);
  if (v != MLA_OK || T == 0) return v;
  // the scratch this call would need must fit in the fixed array; larger calls are refused before
  // anything touches the GPU
  if (mla::append_scratch_bytes(cfg, T) > kScratchBytes) return MLA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const mla_status s = scratch_on_current_device(&scratch);
  if (s != MLA_OK) return s;
  // Every scratch element the kernels read is written earlier in the same call, so the array needs
  // no clearing between calls.  Device-side flags go to the library's own status word (read with
  // mla_get_device_status(NULL, ...)): there is no caller workspace to hold them.
  return mla::run_append(cfg, x, W_DKV, W_KR, seq_idx, pos, rope, cache, T, scratch, nullptr, stream);
}
