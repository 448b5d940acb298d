// gqa_attn_prefill_from_host: one prefill step whose q, k, v and output live in
// host memory ("mojolearn.transformer", TransformerBlock.forward: the caller
// hands in the step's tensors and reads the attention result back).
//
// The step is split into chunks of batch rows. Each chunk's q, k, v rows go to
// the device on one copy stream, its k/v cache append and its attention run on
// the caller's stream once they have landed, and its output rows go back to
// the host on a second copy stream once they are written. Host-to-device
// copies, kernels and device-to-host copies of different chunks overlap, so
// the step costs about the slower of the two copy directions rather than the
// sum of copies and compute. Batch rows are independent in every kernel of the
// path, so each row gets the same result as in one call over the whole batch.
//
// The two copy streams belong to the library: one pair per device, created by
// the first call on that device (with it current) and kept until exit.
#include <math.h>

#include <mutex>

#include "../../include/gqa_attn.h"
#include "kernels.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 8;

std::mutex g_mutex;
cudaStream_t g_copy[kMaxDevices][2] = {};   // [device][0: host->device, 1: device->host]

int copy_streams(cudaStream_t* h2d, cudaStream_t* d2h) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return gqa::record_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  for (int i = 0; i < 2; ++i) {
    if (!g_copy[dev][i]) {
      e = cudaStreamCreateWithFlags(&g_copy[dev][i], cudaStreamNonBlocking);
      if (e != cudaSuccess) {
        g_copy[dev][i] = nullptr;
        return gqa::record_cuda_error(e);
      }
    }
  }
  *h2d = g_copy[dev][0];
  *d2h = g_copy[dev][1];
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Batch rows per chunk: at most kMaxChunks chunks. Chunk offsets must keep every
// device pointer 16-byte aligned; when a row of k or of the cache is not a whole
// number of 16-byte units the step runs as one chunk.
int rows_per_chunk(int B, int Hkv, int L, int D, int capacity) {
  const long long kv_row = (long long)Hkv * L * D;
  const long long cache_row = (long long)Hkv * capacity * D;
  if (B <= 0 || kv_row % 4 != 0 || cache_row % 4 != 0) return B > 0 ? B : 1;
  return (B + kMaxChunks - 1) / kMaxChunks;
}

}  // namespace

extern "C" {

size_t gqa_attn_prefill_from_host_workspace_size(int B, int H, int Hkv, int L, int D,
                                                 int capacity, const attn_rope_params* rp) {
  if (B < 0 || capacity < 1) return 0;
  const int rows = rows_per_chunk(B, Hkv, L, D, capacity);
  return gqa_attn_prefill_rope_workspace_size(rows, H, Hkv, L, D, rp);
}

int gqa_attn_prefill_from_host(const float* q_host, const float* k_host, const float* v_host,
                               float* out_host, float* q, float* k, float* v, float* out, int B,
                               int H, int Hkv, int L, int D, const int32_t* start,
                               int32_t max_start, const attn_rope_params* rp, const float* table,
                               const float* q_norm_w, const float* k_norm_w, float norm_eps,
                               float* k_cache, float* v_cache, int capacity, int window,
                               float softcap, float scale, void* workspace,
                               size_t workspace_bytes, int32_t* status, void* stream) {
  // Every check that the per-chunk calls below would make, made first for the
  // whole batch, so that an invalid call returns before any copy is enqueued.
  if (B < 0 || H < 1 || Hkv < 1 || H % Hkv != 0 || L < 0 || D < 2 || D % 2 != 0 ||
      D > gqa::kMaxHeadDim || window < 0 || capacity < 1 || (window > 0 && capacity != window))
    return ATTN_ERR_SHAPE;
  if (!isfinite(softcap) || !isfinite(scale)) return ATTN_ERR_PARAM;
  if (B == 0 || L == 0) return ATTN_OK;
  if (!q_host || !k_host || !v_host || !out_host || !q || !k || !v || !out || !start || !rp ||
      !table || !k_cache || !v_cache)
    return ATTN_ERR_NULL;
  if (attn_rope_table_bytes(rp, D) == 0 || !(norm_eps >= 0.f)) return ATTN_ERR_PARAM;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(table) ||
      !aligned16(k_cache) || !aligned16(v_cache) || (q_norm_w && !aligned16(q_norm_w)) ||
      (k_norm_w && !aligned16(k_norm_w)))
    return ATTN_ERR_ALIGN;
  const int max_positions = rp->max_positions > 0 ? rp->max_positions : 8192;
  if (max_start < 0 || (int64_t)max_start + L - 1 >= (int64_t)max_positions)
    return ATTN_ERR_POSITION;
  if (window == 0 && (int64_t)max_start + L > (int64_t)capacity) return ATTN_ERR_CAPACITY;
  const int rows = rows_per_chunk(B, Hkv, L, D, capacity);
  const size_t need = gqa_attn_prefill_rope_workspace_size(rows, H, Hkv, L, D, rp);
  if (need == 0) return ATTN_ERR_SHAPE;
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_ALIGN;

  cudaStream_t h2d = nullptr, d2h = nullptr;
  if (int rc = copy_streams(&h2d, &d2h); rc != ATTN_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int nchunks = (B + rows - 1) / rows;

  // events: [0] entry, [1] host->device done, [2] device->host done,
  // [3 + c] chunk c landed, [3 + nchunks + c] chunk c's output written
  cudaEvent_t ev[3 + 2 * kMaxChunks] = {};
  const int nev = 3 + 2 * nchunks;
  int rc = ATTN_OK;
  for (int i = 0; i < nev && rc == ATTN_OK; ++i)
    rc = gqa::record_cuda_error(cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming));
  auto release = [&]() {
    for (int i = 0; i < nev; ++i)
      if (ev[i]) cudaEventDestroy(ev[i]);
  };
  if (rc != ATTN_OK) {
    release();
    return rc;
  }

  // Both copy streams start after the caller's earlier work on its stream.
  rc = gqa::record_cuda_error(cudaEventRecord(ev[0], s));
  if (rc == ATTN_OK) rc = gqa::record_cuda_error(cudaStreamWaitEvent(h2d, ev[0], 0));
  if (rc == ATTN_OK) rc = gqa::record_cuda_error(cudaStreamWaitEvent(d2h, ev[0], 0));

  const size_t q_row = (size_t)H * L * D, kv_row = (size_t)Hkv * L * D;
  const size_t cache_row = (size_t)Hkv * capacity * D;
  for (int c = 0; c < nchunks && rc == ATTN_OK; ++c) {
    const size_t b0 = (size_t)c * rows;
    const size_t nb = (size_t)((B - (int)b0) < rows ? (B - (int)b0) : rows);
    rc = gqa::record_cuda_error(cudaMemcpyAsync(q + b0 * q_row, q_host + b0 * q_row,
                                                nb * q_row * sizeof(float),
                                                cudaMemcpyHostToDevice, h2d));
    if (rc == ATTN_OK)
      rc = gqa::record_cuda_error(cudaMemcpyAsync(k + b0 * kv_row, k_host + b0 * kv_row,
                                                  nb * kv_row * sizeof(float),
                                                  cudaMemcpyHostToDevice, h2d));
    if (rc == ATTN_OK)
      rc = gqa::record_cuda_error(cudaMemcpyAsync(v + b0 * kv_row, v_host + b0 * kv_row,
                                                  nb * kv_row * sizeof(float),
                                                  cudaMemcpyHostToDevice, h2d));
    if (rc == ATTN_OK) rc = gqa::record_cuda_error(cudaEventRecord(ev[3 + c], h2d));
  }
  for (int c = 0; c < nchunks && rc == ATTN_OK; ++c) {
    const size_t b0 = (size_t)c * rows;
    const int nb = (B - (int)b0) < rows ? (B - (int)b0) : rows;
    rc = gqa::record_cuda_error(cudaStreamWaitEvent(s, ev[3 + c], 0));
    if (rc == ATTN_OK)
      rc = kv_cache_append(k + b0 * kv_row, v + b0 * kv_row, nb, Hkv, L, D, start + b0,
                           max_start, rp, table, k_norm_w, norm_eps, k_cache + b0 * cache_row,
                           v_cache + b0 * cache_row, capacity, window, status, s);
    if (rc == ATTN_OK)
      rc = gqa_attn_prefill_rope(q + b0 * q_row, k + b0 * kv_row, v + b0 * kv_row,
                                 out + b0 * q_row, nb, H, Hkv, L, D, start + b0, max_start, rp,
                                 table, q_norm_w, norm_eps, window, softcap, scale, workspace,
                                 workspace_bytes, status, s);
    if (rc == ATTN_OK) rc = gqa::record_cuda_error(cudaEventRecord(ev[3 + nchunks + c], s));
    if (rc == ATTN_OK)
      rc = gqa::record_cuda_error(cudaStreamWaitEvent(d2h, ev[3 + nchunks + c], 0));
    if (rc == ATTN_OK)
      rc = gqa::record_cuda_error(cudaMemcpyAsync(out_host + b0 * q_row, out + b0 * q_row,
                                                  (size_t)nb * q_row * sizeof(float),
                                                  cudaMemcpyDeviceToHost, d2h));
  }

  // Join: the caller's stream continues after every copy this call enqueued,
  // also when a step above failed after some copies were already in flight.
  int jrc = gqa::record_cuda_error(cudaEventRecord(ev[1], h2d));
  if (jrc == ATTN_OK) jrc = gqa::record_cuda_error(cudaEventRecord(ev[2], d2h));
  if (jrc == ATTN_OK) jrc = gqa::record_cuda_error(cudaStreamWaitEvent(s, ev[1], 0));
  if (jrc == ATTN_OK) jrc = gqa::record_cuda_error(cudaStreamWaitEvent(s, ev[2], 0));
  release();
  return rc != ATTN_OK ? rc : jrc;
}

}  // extern "C"
