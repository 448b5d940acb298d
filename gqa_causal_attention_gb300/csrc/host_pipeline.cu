// gqa_attn_prefill_from_host: one prefill step whose q, k, v and output live in
// host memory ("mojolearn.transformer", TransformerBlock.forward: the caller
// hands in the step's tensors and reads the attention result back).
//
// The step is split into chunks: groups of batch rows, or slices of one row's kv
// heads (with their query heads) when there are few rows. Each chunk's q, k, v go to
// the device on one copy stream, its k/v cache append and its attention run on
// the caller's stream once they have landed, and its output goes back to
// the host on a second copy stream once it is written. Host-to-device copies,
// kernels and device-to-host copies of different chunks overlap, so the step
// costs about the copies alone rather than copies plus compute. Batch rows and kv-head groups are independent in
// every kernel of the path, so each gets the same result as in one call over
// the whole batch.
//
// The two copy streams belong to the library: one pair per device, created by
// the first call on that device (with it current) and kept until exit.
#include <math.h>

#include <mutex>

#include "../../include/gqa_attn.h"
#include "kernels.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 16;

// The two copy streams of a device ([0] host to device, [1] device to host), made
// by the first call in the device's current context (streams belong to it).
struct CopyStreams {
  cudaStream_t s[2];
  cudaError_t err;
};
gqa::PerContext<CopyStreams> g_copy;

int copy_streams(cudaStream_t* h2d, cudaStream_t* d2h) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return gqa::record_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  const CopyStreams cs = g_copy.get(
      [] {
        CopyStreams c{};
        for (int i = 0; i < 2 && c.err == cudaSuccess; ++i)
          c.err = cudaStreamCreateWithFlags(&c.s[i], cudaStreamNonBlocking);
        if (c.err != cudaSuccess) {
          // nothing half made is kept: the next call tries again in a clean state
          for (int i = 0; i < 2; ++i)
            if (c.s[i]) cudaStreamDestroy(c.s[i]);
          c.s[0] = c.s[1] = nullptr;
        }
        return c;
      },
      CopyStreams{}, [](const CopyStreams& c) { return c.err == cudaSuccess; });
  if (cs.err != cudaSuccess) return gqa::record_cuda_error(cs.err);
  if (!cs.s[0] || !cs.s[1]) return ATTN_ERR_CUDA;
  *h2d = cs.s[0];
  *d2h = cs.s[1];
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A chunk is nb whole batch rows from b0 (all kv heads), or, when there are
// fewer rows than kMaxChunks, kv heads [h0, h0 + nh) of one row with their query
// heads: in [B, heads, L, D] and [B, Hkv, capacity, D] either is one contiguous
// run of memory, and either is a valid call of the kernels (B = nb, Hkv = nh).
// Chunk offsets keep every device pointer 16-byte aligned only when one head's
// rows (L * D and capacity * D floats) are whole 16-byte units; otherwise the
// step runs as one chunk.
struct Plan {
  int rows;      // batch rows per chunk (1 when rows are sliced by heads)
  int heads;     // kv heads per chunk
  int slices;    // chunks per row
  int chunks;
};

Plan plan_chunks(int B, int Hkv, int L, int D, int capacity) {
  Plan p{B > 0 ? B : 1, Hkv, 1, 1};
  if (B <= 0 || ((long long)L * D) % 4 != 0 || ((long long)capacity * D) % 4 != 0) return p;
  if (B >= kMaxChunks) {
    p.rows = (B + kMaxChunks - 1) / kMaxChunks;
    p.chunks = (B + p.rows - 1) / p.rows;
    return p;
  }
  p.rows = 1;
  const int want = kMaxChunks / B;                      // slices per row, >= 1
  p.heads = (Hkv + want - 1) / want;
  p.slices = (Hkv + p.heads - 1) / p.heads;
  p.chunks = B * p.slices;
  return p;
}

}  // namespace

extern "C" {

size_t gqa_attn_prefill_from_host_workspace_size(int B, int H, int Hkv, int L, int D,
                                                 int capacity, const attn_rope_params* rp) {
  if (B < 0 || capacity < 1 || Hkv < 1 || H % Hkv != 0) return 0;
  const Plan p = plan_chunks(B, Hkv, L, D, capacity);
  return gqa_attn_prefill_rope_workspace_size(p.rows, p.heads * (H / Hkv), p.heads, L, D, rp);
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
  const int G = H / Hkv;
  const Plan plan = plan_chunks(B, Hkv, L, D, capacity);
  const size_t need =
      gqa_attn_prefill_rope_workspace_size(plan.rows, plan.heads * G, plan.heads, L, D, rp);
  if (need == 0) return ATTN_ERR_SHAPE;
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
  // The non-finite check, when on, runs inside each chunk's calls and needs a status word.
  if (gqa::check_finite_enabled() && !status) return ATTN_ERR_NULL;

  cudaStream_t h2d = nullptr, d2h = nullptr;
  if (int rc = copy_streams(&h2d, &d2h); rc != ATTN_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int nchunks = plan.chunks;

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

  // chunk c: rows [b0, b0 + nb), kv heads [h0, h0 + nh); element offsets of its
  // q/out, k/v and cache runs
  struct Chunk {
    int b0, nb, h0, nh;
    size_t q_off, kv_off, cache_off;
  };
  auto chunk = [&](int c) {
    Chunk r{};
    r.b0 = (c / plan.slices) * plan.rows;
    r.nb = B - r.b0 < plan.rows ? B - r.b0 : plan.rows;
    r.h0 = (c % plan.slices) * plan.heads;
    r.nh = Hkv - r.h0 < plan.heads ? Hkv - r.h0 : plan.heads;
    const size_t head = (size_t)L * D;
    r.q_off = ((size_t)r.b0 * H + (size_t)r.h0 * G) * head;
    r.kv_off = ((size_t)r.b0 * Hkv + r.h0) * head;
    r.cache_off = ((size_t)r.b0 * Hkv + r.h0) * (size_t)capacity * D;
    return r;
  };
  const size_t head_bytes = (size_t)L * D * sizeof(float);
  for (int c = 0; c < nchunks && rc == ATTN_OK; ++c) {
    const Chunk ch = chunk(c);
    const size_t kv_bytes = (size_t)ch.nb * ch.nh * head_bytes;
    rc = gqa::record_cuda_error(cudaMemcpyAsync(q + ch.q_off, q_host + ch.q_off, kv_bytes * G,
                                                cudaMemcpyHostToDevice, h2d));
    if (rc == ATTN_OK)
      rc = gqa::record_cuda_error(cudaMemcpyAsync(k + ch.kv_off, k_host + ch.kv_off, kv_bytes,
                                                  cudaMemcpyHostToDevice, h2d));
    if (rc == ATTN_OK)
      rc = gqa::record_cuda_error(cudaMemcpyAsync(v + ch.kv_off, v_host + ch.kv_off, kv_bytes,
                                                  cudaMemcpyHostToDevice, h2d));
    if (rc == ATTN_OK) rc = gqa::record_cuda_error(cudaEventRecord(ev[3 + c], h2d));
  }
  for (int c = 0; c < nchunks && rc == ATTN_OK; ++c) {
    const Chunk ch = chunk(c);
    rc = gqa::record_cuda_error(cudaStreamWaitEvent(s, ev[3 + c], 0));
    if (rc == ATTN_OK)
      rc = kv_cache_append(k + ch.kv_off, v + ch.kv_off, ch.nb, ch.nh, L, D, start + ch.b0,
                           max_start, rp, table, k_norm_w, norm_eps, k_cache + ch.cache_off,
                           v_cache + ch.cache_off, capacity, window, status, s);
    if (rc == ATTN_OK)
      rc = gqa_attn_prefill_rope(q + ch.q_off, k + ch.kv_off, v + ch.kv_off, out + ch.q_off,
                                 ch.nb, ch.nh * G, ch.nh, L, D, start + ch.b0, max_start, rp,
                                 table, q_norm_w, norm_eps, window, softcap, scale, workspace,
                                 workspace_bytes, status, s);
    if (rc == ATTN_OK) rc = gqa::record_cuda_error(cudaEventRecord(ev[3 + nchunks + c], s));
    if (rc == ATTN_OK)
      rc = gqa::record_cuda_error(cudaStreamWaitEvent(d2h, ev[3 + nchunks + c], 0));
    if (rc == ATTN_OK)
      rc = gqa::record_cuda_error(cudaMemcpyAsync(
          out_host + ch.q_off, out + ch.q_off, (size_t)ch.nb * ch.nh * G * head_bytes,
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
