// gqa_attn_decode_static: the split-KV decode for callers that cannot
// allocate device memory.
//
// Some callers have no allocator to hand: code that runs where cudaMalloc is
// off limits (a plugin inside a host framework that owns all device memory,
// or a path that must not allocate once serving has started) and plain C
// callers with no tensor library at all. This entry point takes the decode's
// scratch from a fixed array in this library's own device memory instead of
// asking the caller for a workspace.
//
// The array is a file-scope __device__ variable. Host code cannot use its
// name as a device address (on the host it is only a stand-in symbol), so the
// first call on each device, with that device current, looks the address up
// with cudaGetSymbolAddress and keeps it for later calls.
#include <mutex>

#include "../../include/gqa_attn.h"
#include "kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;   // GQA_ATTN_STATIC_SCRATCH_BYTES
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (set up once).
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" int gqa_attn_decode_static(const float* q, const float* k_cache,
                                      const float* v_cache, const int32_t* cache_len,
                                      int32_t max_cache_len, float* out, int B, int H, int Hkv,
                                      int D, int capacity, int window, float softcap,
                                      float scale, int32_t* status, void* stream) {
  if (B > 0 && max_cache_len >= 1 && Hkv >= 1 && H >= 1 && H % Hkv == 0 && D >= 2) {
    const size_t need = gqa_attn_decode_workspace_size(B, H, Hkv, D, max_cache_len, window);
    if (need > kStaticScratchBytes) return ATTN_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != ATTN_OK) return rc;
  return gqa_attn_decode(q, k_cache, v_cache, cache_len, max_cache_len, out, B, H, Hkv, D,
                         capacity, window, softcap, scale, scratch, kStaticScratchBytes, status,
                         stream);
}
