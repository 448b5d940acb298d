// Internal launch interface between the C ABI (api.cu) and the kernels.
// Host-side only; every launcher enqueues on `stream` and returns the launch
// status. Arguments have been validated by the caller.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace gqa {

// Process-unique id of the calling thread's current CUDA context; 0 when the
// driver does not offer the query or no context is current yet.
unsigned long long current_context_id();

// A value worked out once per device and context. Function attributes set with
// cudaFuncSetAttribute, occupancy answers and streams belong to a device's
// context: another device, or the context created again after cudaDeviceReset,
// works them out again. (Without the context query the value is kept per
// device.) compute() runs with the device current; a value that keep() turns
// down is returned but not kept (the next call computes again); on_error is
// returned when the current device cannot be read.
template <class T>
class PerContext {
 public:
  template <class F, class K>
  T get(F compute, T on_error, K keep) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kSlots) {
      cudaGetLastError();
      return on_error;
    }
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(mu_);
    if (!known_[dev] || (id != 0 && id != ctx_[dev])) {
      const T v = compute();
      if (!keep(v)) return v;
      value_[dev] = v;
      ctx_[dev] = id != 0 ? id : current_context_id();   // compute() may have made it
      known_[dev] = true;
    }
    return value_[dev];
  }
  template <class F>
  T get(F compute, T on_error) {
    return get(compute, on_error, [](const T&) { return true; });
  }

 private:
  static constexpr int kSlots = 64;
  std::mutex mu_;
  unsigned long long ctx_[kSlots] = {};
  T value_[kSlots] = {};
  bool known_[kSlots] = {};
};

constexpr int kMaxHeadDim = 256;
constexpr int kMaxRopeHalf = kMaxHeadDim / 2;

struct InvFreq {
  double v[kMaxRopeHalf];   // rotary frequencies theta_i, i < R/2
};

struct RopeJob {
  float* x;                 // [B, NH, L, D], rotated in place (or read only, see y)
  float* y;                 // nullptr: in place; else rotated rows go here ([B, NH, L, D])
  int B, NH, L, D, R;
  const int32_t* start;     // [B], or nullptr: every row starts at 0
  int max_positions;
  const float2* table;      // [max_positions][R/2] (cos, sin), or nullptr: no rotation
  const float* norm_w;      // [D] or nullptr
  float norm_eps;
  int32_t* status;
  // cache append (k rows only); k_cache == nullptr: plain rotation
  const float* v;
  float* k_cache;
  float* v_cache;
  int capacity;
  int window;
  const int32_t* skip = nullptr;   // non-finite check on: return if *skip has ATTN_DEV_NONFINITE
};

// ATTN_OK for cudaSuccess; otherwise remembers e for attn_last_cuda_error on this host
// thread and returns ATTN_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// The host checks of gqa_attn_decode other than its workspace (api.cu): ATTN_OK,
// also when B == 0 (nothing to do), or the ATTN_ERR_* that call would return.
int decode_host_check(const float* q, const float* k_cache, const float* v_cache,
                      const int32_t* cache_len, int32_t max_cache_len, const float* out, int B,
                      int H, int Hkv, int D, int capacity, int window, float softcap,
                      float scale);

cudaError_t launch_rope_table(const InvFreq& inv, int R, int max_positions, float2* table,
                              cudaStream_t stream);
cudaError_t launch_rope_rows(const RopeJob& job, cudaStream_t stream);

// Fused q RMSNorm + RoPE inside the tensor-core prefill (q is then the raw query).
struct QRope {
  const float2* table;      // [max_positions][R/2] (cos, sin); nullptr: q already rotated
  const int32_t* start;     // [B], or nullptr: every row starts at 0
  const float* norm_w;      // [D] or nullptr
  float norm_eps;
  int R, max_positions;
};

struct AttnShape {
  const float* q;           // [B, H, L, D]
  const float* k;           // [B, Hkv, L, D]
  const float* v;           // [B, Hkv, L, D]
  float* out;               // [B, H, L, D]
  float* vt;                // workspace: V^T [B, Hkv, D, vt_pitch] (tensor-core path)
  int vt_pitch;
  int B, H, Hkv, L, D;
  int window;               // 0: causal
  float softcap;            // <= 0: off
  float scale;              // > 0
  int32_t* status;
  QRope rope;               // rope.table == nullptr: q already rotated
  // Continuing a cached prefix (persistent kernel, D <= 256): k and vt then hold Lk
  // key rows per head, kv_off[b] of them before query row 0 of row b.
  const int32_t* kv_off = nullptr;
  int Lk = 0;               // 0: the chunk's own keys (Lk = L)
  // Ragged batch: row b is real at query (and key) positions [0, lengths[b]);
  // padding rows of out are written as +0.0 and padding keys are never seen.
  // nullptr: every row has length L. Not combined with kv_off.
  const int32_t* lengths = nullptr;
  const int32_t* skip = nullptr;   // as RopeJob::skip
  // Rows between consecutive heads of k (0: Lk, i.e. contiguous heads); lets the
  // kernel read rotated keys from a cache whose heads hold `capacity` rows.
  int k_head_rows = 0;
};

cudaError_t launch_prefill_simt(const AttnShape& a, cudaStream_t stream);
// Returns cudaErrorNotSupported (nothing launched) for shapes it does not take.
cudaError_t launch_prefill_tc(const AttnShape& a, cudaStream_t stream);      // V^T pre-pass + kernel
cudaError_t launch_prefill_tc_vt(const AttnShape& a, cudaStream_t stream);   // a.vt already written
// lengths (optional, [BHkv / Hkv]): columns m >= lengths[bh / Hkv] of vt are
// written as 0, so padding values (even inf or NaN) never meet a zero weight
// in P V.
cudaError_t launch_transpose_v(const float* v, float* vt, int BHkv, int L, int D, int vt_pitch,
                               cudaStream_t stream, const int32_t* lengths = nullptr,
                               int Hkv = 1, int32_t* status = nullptr,
                               const int32_t* skip = nullptr);
bool prefill_tc_supports(int D);
// Keys for continuing a cached prefix: per (b, kv head), rows [0, pre_b) from the
// cache (positions start[b] - pre_b .. start[b] - 1; slot = position, or position
// mod window for a ring), then the chunk's L rows of k / v, then zeros up to Lk.
// K goes to kg [B, Hkv, Lk, D], V transposed to vtg [B, Hkv, D, vt_pitch].
// pre_b = start[b] (window 0) or min(start[b], window - 1); written to pre[b].
struct GatherJob {
  const float* k;           // [B, Hkv, L, D] rotated chunk keys
  const float* v;
  const float* k_cache;     // [B, Hkv, capacity, D]
  const float* v_cache;
  const int32_t* start;     // [B]
  int32_t* pre;             // [B] out: prefix keys per row
  float* kg;
  float* vtg;
  int B, Hkv, L, D, capacity, window, Lk, vt_pitch, max_start;
  int32_t* status;
  const int32_t* skip = nullptr;
};
cudaError_t launch_gather_kv(const GatherJob& j, cudaStream_t stream);
bool prefill_tq_supports_kv_off(int D);
int prefill_vt_pitch(int L);   // row pitch (floats) of the V^T workspace
cudaError_t launch_prefill_tq(const AttnShape& a, cudaStream_t stream);  // 32 <= D <= 256
bool prefill_fuses_rope(int D);  // the kernel taking D applies a.rope itself

struct DecodeJob {
  const float* q;           // [B, H, D]
  const float* k_cache;     // [B, Hkv, capacity, D]
  const float* v_cache;
  const int32_t* cache_len; // [B]
  int max_cache_len;
  float* out;               // [B, H, D]
  int B, H, Hkv, D, capacity, window;
  float softcap, scale;
  float* partial;           // workspace [B, H, nsplit, D + 2]
  int nsplit, chunk;
  int32_t* status;
  const int32_t* skip = nullptr;
};
// (Kept at this size: the split kernels read it through references, and
// growing it by 72 bytes measured 20 % slower on the long carried decode.)

// A whole decode step in the head-pair split kernel (decode_step_fuses): q and
// the new k, v raw, positions pos[b]; each block rotates its heads' q, the block
// whose slots hold position pos[b] writes the rotated k and v there before
// reading them, and one block per row writes cache_len[b] = pos[b] + 1 (0 for a
// position without a table row or slot) for the combine. DecodeJob::q is unused.
struct DecodeStepArgs {
  const float* q_raw;       // [B, H, D]
  const float* k_new;       // [B, Hkv, D]
  const float* v_new;
  const int32_t* pos;       // [B]
  const float2* table;      // [max_positions][R / 2] (cos, sin)
  const float* q_norm_w;
  const float* k_norm_w;
  float norm_eps;
  int R, max_positions;
  int32_t* cache_len;       // [B], written (DecodeJob::cache_len points here too)
};
// Whether a decode step of this shape runs as one split pass (+ combine) with
// the prep fused in: D = 128 and rotary dims R % 8 == 0 (64 or 128 with 8 query
// heads per KV head).
bool decode_step_fuses(int H, int Hkv, int D, int R);

// One decode step's prep pass (decode.cu): q RMSNorm + RoPE into qrot, k RMSNorm +
// RoPE and v into their cache slots, cache_len[b] = pos[b] + 1 (0 for a row whose
// position fails the device check).
struct DecodePrepJob {
  const float* q;           // [B, H, D] raw
  const float* k;           // [B, Hkv, D] raw
  const float* v;
  float* qrot;              // [B, H, D]
  float* k_cache;           // [B, Hkv, capacity, D]
  float* v_cache;
  int32_t* cache_len;       // [B]
  int B, H, Hkv, D, R;
  const int32_t* pos;       // [B] tokens already cached = the new token's position
  int max_positions, capacity, window;
  const float2* table;
  const float* q_norm_w;
  const float* k_norm_w;
  float norm_eps;
  int32_t* status;
  const int32_t* skip = nullptr;
};
cudaError_t launch_decode_prep(const DecodePrepJob& j, cudaStream_t stream);

// The identical numeric mode: one warp per query row, fixed arithmetic order
// (identical.cu). Keys at positions >= s0 come from k / v (the chunk), below
// s0 from the cache. Prefill: s0 = start[b] (nullptr: 0), query row l at
// position s0 + l. Decode (cache_len != nullptr): L = 1, position
// cache_len[b] - 1, every key from the cache.
struct IdentJob {
  const float* q;           // [B, H, L, D] rotated
  const float* k;           // [B, Hkv, L, D] rotated chunk keys, or nullptr (decode)
  const float* v;
  const float* k_cache;     // [B, Hkv, capacity, D] or nullptr (no cached prefix)
  const float* v_cache;
  const int32_t* start;     // [B] or nullptr
  const int32_t* cache_len; // [B], decode only
  int max_start, max_len;
  float* out;               // [B, H, L, D]
  int B, H, Hkv, L, D, capacity, window;
  float softcap, scale;
  int32_t* status;
  const int32_t* skip = nullptr;
};
cudaError_t launch_identical(const IdentJob& j, cudaStream_t stream);

// The decoder block around the attention (block.cu).
cudaError_t launch_rmsnorm_rows(const float* x, const float* w, float* y, long T, int n,
                                float eps, bool offset, bool round_out, cudaStream_t stream,
                                const int32_t* skip = nullptr);
cudaError_t launch_swap_mid(const float* in, float* out, int B, int P, int Q, int D,
                            cudaStream_t stream,
                            const int32_t* skip = nullptr);   // [B, P, Q, D] -> [B, Q, P, D]

// Projections on the tensor cores (gemm_tc.cu): Y = X W^T, W in torch's [out, in]
// layout, TF32 operands, fp32 accumulation. Up to three segments share X.
struct GemmSegment {
  const float* w;           // [n, K]; SwiGLU: gate_proj
  const float* w_up;        // SwiGLU only: up_proj [n, K]
  int n;                    // output columns
  int mode;                 // 0 store, 1 out = res + X W^T, 2 out = SiLU(X Wg^T) * (X Wu^T)
  int round_out;            // round outputs to the nearest TF32 value
  float* out;               // row-major [T, ldo] (out_heads == 0) or head-major
  long ldo;
  int out_heads;            // > 0: out [T / L, out_heads, L, D], column h * D + d
  const float* res;         // mode 1: [T, ldr] (may equal out)
  long ldr;
};
struct GemmJob {
  const float* x;           // [T, K] token-major, or head-major (x_heads > 0)
  long T;
  int K;
  int x_heads;              // > 0: x is [T / L, x_heads, L, D] with K = x_heads * D, D % 32 == 0
  int L, D;                 // tokens per batch row and head dim (head-major x or out)
  int nseg;
  GemmSegment seg[3];       // SwiGLU: one segment only
  int32_t* status;
  const int32_t* skip = nullptr;
};
bool gemm_tc_supports(const GemmJob& j);
cudaError_t launch_gemm_tc(const GemmJob& j, cudaStream_t stream);

// The memory pass of a prefill step (step.cu): k RMSNorm + RoPE into the cache
// (and into kr when given), v into the cache, V^T into vt; k and v are read only.
struct AppendVtJob {
  const float* k;           // [B, Hkv, L, D]
  const float* v;
  float* k_cache;           // [B, Hkv, capacity, D]: slot = position, or position mod window
  float* v_cache;
  float* kr;                // [B, Hkv, L, D] rotated keys (may be k itself), or nullptr
  float* vt;                // [B * Hkv, D, vt_pitch], or nullptr
  int B, Hkv, L, D, R;
  const float2* table;      // [max_positions][R/2] (cos, sin); nullptr: no rotation
  const float* norm_w;      // [D] or nullptr
  float norm_eps;
  const int32_t* start;     // [B] or nullptr (0)
  int max_positions, capacity, window, vt_pitch;
  int32_t* status;
  const int32_t* skip = nullptr;
};
bool append_vt_supports(int D);
cudaError_t launch_append_vt(const AppendVtJob& j, cudaStream_t stream);

// The opt-in non-finite input check (finite.cu). A region is B * NH blocks of R
// rows, C values of each row checked, rows ld floats apart (blocks R * ld apart);
// the rows checked depend on the mode (info[b] per batch row b = block / NH).
enum { kFiniteAll = 0,       // every row
       kFiniteLen = 1,       // rows < info[b] (a ragged row's length)
       kFiniteCache = 2,     // cache slots live at cache length info[b]: rows < min(info[b], R)
       kFinitePrefix = 3 };  // slots of the positions a chunk at start info[b] reads from the
                             // cache: all below it, or the last window - 1 of them in a ring
struct FiniteRegion {
  const float* p;
  int B, NH;
  long R, C, ld;
  int mode;
  const int32_t* info;
  int window;
};
constexpr int kMaxFiniteRegions = 12;
struct FiniteJob {
  int n;
  FiniteRegion r[kMaxFiniteRegions];
  int32_t* status;
};
int check_finite_enabled();              // the process-wide switch (ATTN_CHECK_FINITE at first use)
int set_check_finite(int on);            // on < 0: query only; returns the previous value
cudaError_t launch_finite_check(const FiniteJob& j, cudaStream_t stream);

void decode_split_plan(int B, int Hkv, int max_cache_len, int window, int* nsplit, int* chunk);
// Split partials in bytes: for exactly this max_cache_len (what a call uses), or
// (bound) the largest over every max_cache_len up to it (what a caller allocates).
size_t decode_partial_bytes(int B, int H, int Hkv, int D, int max_cache_len, int window,
                            bool bound);
cudaError_t launch_decode(const DecodeJob& j, cudaStream_t stream,
                          const DecodeStepArgs* step = nullptr);
int decode_launches(const DecodeJob& j, bool step);   // kernels launch_decode launches

}  // namespace gqa
