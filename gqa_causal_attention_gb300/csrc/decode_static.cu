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
// with cudaGetSymbolAddress and keeps it for later calls. The kept address is
// tied to the device's current context (by the context's process-unique id):
// after cudaDeviceReset the module is loaded again, possibly elsewhere, and
// the next call looks the address up again.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <map>
#include <mutex>

#include "../../include/gqa_attn.h"
#include "kernels.h"

// Process-unique id of the calling thread's current context, or 0 when the
// driver does not offer the query or no context is current.
unsigned long long gqa::current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    cudaGetLastError();
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;   // GQA_ATTN_STATIC_SCRATCH_BYTES
static_assert(kStaticScratchBytes == GQA_ATTN_STATIC_SCRATCH_BYTES, "header and array agree");

__device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

struct Entry {
  unsigned long long ctx_id;   // process-unique id of the context the address belongs to
  void* addr;
};

std::mutex g_mutex;
std::map<int, Entry> g_scratch;   // device ordinal -> address in its current context

// Device address of g_decode_scratch on the current device: looked up on the
// first call in the device's current context, then reused.
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) {
    cudaGetLastError();
    return gqa::record_cuda_error(e);
  }
  // Before the runtime's first use on this device no context is current (id 0);
  // the symbol lookup below creates it, and the id is read again after it.
  unsigned long long id = gqa::current_context_id();
  std::lock_guard<std::mutex> lock(g_mutex);
  auto it = g_scratch.find(dev);
  if (id != 0 && it != g_scratch.end() && it->second.ctx_id == id) {
    *out = it->second.addr;
    return ATTN_OK;
  }
  void* p = nullptr;
  if (cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch); e != cudaSuccess || !p) {
    cudaGetLastError();
    return gqa::record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
  }
  if (id == 0) id = gqa::current_context_id();   // the lookup has made the context current
  if (id != 0) g_scratch[dev] = Entry{id, p};
  *out = p;
  return ATTN_OK;
}

}  // namespace

extern "C" int gqa_attn_decode_static(const float* q, const float* k_cache,
                                      const float* v_cache, const int32_t* cache_len,
                                      int32_t max_cache_len, float* out, int B, int H, int Hkv,
                                      int D, int capacity, int window, float softcap,
                                      float scale, int32_t* status, void* stream) {
  // gqa_attn_decode's own host checks come first, so refusals match it exactly.
  const int rc = gqa::decode_host_check(q, k_cache, v_cache, cache_len, max_cache_len, out, B, H,
                                        Hkv, D, capacity, window, softcap, scale);
  if (rc != ATTN_OK || B == 0) return rc;
  const size_t need = gqa::decode_partial_bytes(B, H, Hkv, D, max_cache_len, window, false);
  if (need == 0 || need > kStaticScratchBytes) return ATTN_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (const int r = scratch_for_current_device(&scratch); r != ATTN_OK) return r;
  return gqa_attn_decode(q, k_cache, v_cache, cache_len, max_cache_len, out, B, H, Hkv, D,
                         capacity, window, softcap, scale, scratch, kStaticScratchBytes, status,
                         stream);
}
