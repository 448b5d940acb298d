// C ABI of libgqa_attn.so: argument checks on the host, then kernel launches.
// Nothing here allocates device memory or synchronises a stream.
#include <math.h>
#include <stdint.h>

#include "../../include/gqa_attn.h"
#include "kernels.h"

namespace {

constexpr double kPi = 3.14159265358979323846;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int max_pos_of(const attn_rope_params* rp) {
  return rp->max_positions > 0 ? rp->max_positions : 8192;
}

int rope_dim_of(const attn_rope_params* rp, int D) { return rp->rope_dim > 0 ? rp->rope_dim : D; }

bool rope_params_ok(const attn_rope_params* rp, int D) {
  if (!rp) return false;
  if (!(rp->theta > 0.0) || !isfinite(rp->theta)) return false;
  if (rp->rope_dim < 0 || rp->max_positions < 0) return false;
  const int R = rope_dim_of(rp, D);
  if (R % 2 != 0 || R > D || R < 2) return false;
  switch (rp->scaling_type) {
    case ATTN_ROPE_SCALING_NONE:
      return true;
    case ATTN_ROPE_SCALING_LINEAR:
      return rp->factor > 0.0 && isfinite(rp->factor);
    case ATTN_ROPE_SCALING_LLAMA3:
      return rp->factor > 0.0 && isfinite(rp->factor) && rp->low_freq_factor > 0.0 &&
             rp->high_freq_factor > rp->low_freq_factor && isfinite(rp->high_freq_factor) &&
             rp->original_max_positions > 0;
    default:
      return false;
  }
}

// theta_i = theta^(-2i/R), then the scaling rule of attn_rope_params.
void inv_freq(const attn_rope_params* rp, int R, gqa::InvFreq* out) {
  for (int i = 0; i < R / 2; ++i) {
    double f = pow(rp->theta, -2.0 * i / (double)R);
    if (rp->scaling_type == ATTN_ROPE_SCALING_LINEAR) {
      f /= rp->factor;
    } else if (rp->scaling_type == ATTN_ROPE_SCALING_LLAMA3) {
      const double orig = (double)rp->original_max_positions;
      const double wl = 2.0 * kPi / f;
      if (wl > orig / rp->low_freq_factor) {
        f /= rp->factor;
      } else if (wl >= orig / rp->high_freq_factor) {
        const double s = (orig / wl - rp->low_freq_factor) /
                         (rp->high_freq_factor - rp->low_freq_factor);
        f = (1.0 - s) * f / rp->factor + s * f;
      }
    }
    out->v[i] = f;
  }
}

bool dims_ok(int B, int Hx, int L, int D) {
  return B >= 0 && Hx >= 1 && L >= 0 && D >= 2 && D <= gqa::kMaxHeadDim && D % 2 == 0;
}

// The CUDA error behind the last ATTN_ERR_CUDA returned on this host thread.
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return ATTN_OK;
  g_last_cuda_error = e;
  return ATTN_ERR_CUDA;
}

}  // namespace

int gqa::record_cuda_error(cudaError_t e) { return cuda_status(e); }

namespace {
// The opt-in non-finite check. add() lists what a call reads; gate() then, with
// the check on, requires a status word, enqueues the check and hands back the
// status word as the kernels' skip flag (nullptr and nothing enqueued when off).
struct Finite {
  gqa::FiniteJob j{};
  void add(const float* p, int B, int NH, long R, long C, int mode = gqa::kFiniteAll,
           const int32_t* info = nullptr, int window = 0, long ld = 0) {
    if (!p || B < 1 || NH < 1 || R < 1 || C < 1 || j.n >= gqa::kMaxFiniteRegions) return;
    gqa::FiniteRegion& r = j.r[j.n++];
    r.p = p; r.B = B; r.NH = NH; r.R = R; r.C = C; r.ld = ld > 0 ? ld : C;
    r.mode = mode; r.info = info; r.window = window;
  }
  int gate(int32_t* status, cudaStream_t s, const int32_t** skip) {
    *skip = nullptr;
    if (!gqa::check_finite_enabled()) return ATTN_OK;
    if (!status) return ATTN_ERR_NULL;
    j.status = status;
    *skip = status;
    return cuda_status(gqa::launch_finite_check(j, s));
  }
};
}  // namespace

// Every host check of gqa_attn_decode except the workspace's: ATTN_OK (also for
// B == 0, when there is nothing to do) or the ATTN_ERR_* the call would return.
int gqa::decode_host_check(const float* q, const float* k_cache, const float* v_cache,
                           const int32_t* cache_len, int32_t max_cache_len, const float* out,
                           int B, int H, int Hkv, int D, int capacity, int window, float softcap,
                           float scale) {
  if (!dims_ok(B, H, 1, D) || Hkv < 1 || H % Hkv != 0 || window < 0 || capacity < 1)
    return ATTN_ERR_SHAPE;
  if (window > 0 && capacity != window) return ATTN_ERR_SHAPE;
  if (!isfinite(softcap) || !isfinite(scale)) return ATTN_ERR_PARAM;
  if (B == 0) return ATTN_OK;
  if (max_cache_len < 1) return ATTN_ERR_SHAPE;
  if (window == 0 && max_cache_len > capacity) return ATTN_ERR_CAPACITY;
  if (!q || !k_cache || !v_cache || !cache_len || !out) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return ATTN_ERR_ALIGN;
  return ATTN_OK;
}

extern "C" {

const char* attn_version(void) { return "0.2.0"; }

int attn_set_check_finite(int on) { return gqa::set_check_finite(on); }

const char* attn_last_cuda_error(void) {
  return g_last_cuda_error == cudaSuccess ? "no CUDA error" : cudaGetErrorString(g_last_cuda_error);
}

const char* attn_status_string(int code) {
  switch (code) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULL: return "a required pointer is NULL";
    case ATTN_ERR_SHAPE: return "sizes break the shape rules";
    case ATTN_ERR_POSITION: return "a position reaches max_positions";
    case ATTN_ERR_CAPACITY: return "a position has no cache slot";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
    case ATTN_ERR_PARAM: return "invalid RoPE parameters or table";
    case ATTN_ERR_CUDA: return "a CUDA launch failed";
    default: return "unknown status";
  }
}

size_t attn_rope_table_bytes(const attn_rope_params* rp, int D) {
  if (!rope_params_ok(rp, D) || D > gqa::kMaxHeadDim) return 0;
  return (size_t)max_pos_of(rp) * (size_t)(rope_dim_of(rp, D) / 2) * 2 * sizeof(float);
}

int attn_rope_table_init(const attn_rope_params* rp, int D, float* table, size_t table_bytes,
                         void* stream) {
  if (!rp || !table) return ATTN_ERR_NULL;
  if (D < 2 || D > gqa::kMaxHeadDim || D % 2) return ATTN_ERR_SHAPE;
  const size_t need = attn_rope_table_bytes(rp, D);
  if (need == 0 || table_bytes < need) return ATTN_ERR_PARAM;
  if (!aligned16(table)) return ATTN_ERR_ALIGN;
  gqa::InvFreq inv;
  const int R = rope_dim_of(rp, D);
  inv_freq(rp, R, &inv);
  return cuda_status(gqa::launch_rope_table(inv, R, max_pos_of(rp), reinterpret_cast<float2*>(table),
                                            static_cast<cudaStream_t>(stream)));
}

int attn_rope_apply(float* x, int B, int Hx, int L, int D, const int32_t* start,
                    int32_t max_start, const attn_rope_params* rp, const float* table,
                    const float* norm_w, float norm_eps, int32_t* status, void* stream) {
  if (!rp || !table) return ATTN_ERR_NULL;
  if (!dims_ok(B, Hx, L, D)) return ATTN_ERR_SHAPE;
  if (B == 0 || L == 0) return ATTN_OK;
  if (!x || !start) return ATTN_ERR_NULL;
  if (!rope_params_ok(rp, D) || !(norm_eps >= 0.f)) return ATTN_ERR_PARAM;
  if (!aligned16(x) || !aligned16(table) || (norm_w && !aligned16(norm_w))) return ATTN_ERR_ALIGN;
  if (max_start < 0 || (int64_t)max_start + L - 1 >= (int64_t)max_pos_of(rp))
    return ATTN_ERR_POSITION;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Finite fin;
  fin.add(x, B, Hx, L, D);
  fin.add(norm_w, 1, 1, 1, D);
  const int32_t* skip = nullptr;
  if (const int rc = fin.gate(status, s, &skip)) return rc;
  gqa::RopeJob j{};
  j.x = x; j.B = B; j.NH = Hx; j.L = L; j.D = D; j.R = rope_dim_of(rp, D);
  j.start = start; j.max_positions = max_pos_of(rp);
  j.table = reinterpret_cast<const float2*>(table);
  j.norm_w = norm_w; j.norm_eps = norm_eps; j.status = status; j.skip = skip;
  return cuda_status(gqa::launch_rope_rows(j, s));
}

int kv_cache_append(float* k, const float* v, int B, int Hkv, int L, int D,
                    const int32_t* start, int32_t max_start, const attn_rope_params* rp,
                    const float* table, const float* k_norm_w, float norm_eps, float* k_cache,
                    float* v_cache, int capacity, int window, int32_t* status, void* stream) {
  if (!dims_ok(B, Hkv, L, D) || capacity < 1 || window < 0) return ATTN_ERR_SHAPE;
  if (window > 0 && capacity != window) return ATTN_ERR_SHAPE;
  if (B == 0 || L == 0) return ATTN_OK;
  if (!k || !v || !start || !k_cache || !v_cache) return ATTN_ERR_NULL;
  if (rp ? !table : (table || k_norm_w)) return rp ? ATTN_ERR_NULL : ATTN_ERR_PARAM;
  if (rp && !rope_params_ok(rp, D)) return ATTN_ERR_PARAM;
  if (!(norm_eps >= 0.f)) return ATTN_ERR_PARAM;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (table && !aligned16(table)) || (k_norm_w && !aligned16(k_norm_w)))
    return ATTN_ERR_ALIGN;
  const int max_positions = rp ? max_pos_of(rp) : 0x7fffffff;
  if (max_start < 0 || (int64_t)max_start + L - 1 >= (int64_t)max_positions)
    return ATTN_ERR_POSITION;
  if (window == 0 && (int64_t)max_start + L > (int64_t)capacity) return ATTN_ERR_CAPACITY;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Finite fin;
  fin.add(k, B, Hkv, L, D);
  fin.add(v, B, Hkv, L, D);
  fin.add(k_norm_w, 1, 1, 1, D);
  const int32_t* skip = nullptr;
  if (const int rc = fin.gate(status, s, &skip)) return rc;
  if (gqa::append_vt_supports(D) && (int64_t)B * Hkv <= 65535) {
    // 32-row tiles through shared memory: the rotated keys go to the cache and back
    // over k (each tile is read whole before any of it is written)
    gqa::AppendVtJob aj{};
    aj.k = k; aj.v = v; aj.k_cache = k_cache; aj.v_cache = v_cache; aj.kr = k; aj.vt = nullptr;
    aj.B = B; aj.Hkv = Hkv; aj.L = L; aj.D = D; aj.R = rp ? rope_dim_of(rp, D) : D;
    aj.table = reinterpret_cast<const float2*>(table);
    aj.norm_w = k_norm_w; aj.norm_eps = norm_eps; aj.start = start;
    aj.max_positions = max_positions; aj.capacity = capacity; aj.window = window;
    aj.vt_pitch = 0; aj.status = status; aj.skip = skip;
    return cuda_status(gqa::launch_append_vt(aj, s));
  }
  gqa::RopeJob j{};
  j.x = k; j.B = B; j.NH = Hkv; j.L = L; j.D = D; j.R = rp ? rope_dim_of(rp, D) : D;
  j.start = start; j.max_positions = max_positions;
  j.table = reinterpret_cast<const float2*>(table);
  j.norm_w = k_norm_w; j.norm_eps = norm_eps; j.status = status; j.skip = skip;
  j.v = v; j.k_cache = k_cache; j.v_cache = v_cache; j.capacity = capacity; j.window = window;
  return cuda_status(gqa::launch_rope_rows(j, s));
}

size_t gqa_attn_prefill_workspace_size(int B, int Hkv, int L, int D) {
  if (B < 0 || Hkv < 1 || L < 0 || D < 2 || D > gqa::kMaxHeadDim || D % 2) return 0;
  if (!gqa::prefill_tc_supports(D) || B == 0 || L == 0) return 16;
  return (size_t)B * Hkv * D * gqa::prefill_vt_pitch(L) * sizeof(float);
}

namespace {
// gqa_attn_prefill, and gqa_attn_prefill_ragged without RoPE (lengths != NULL).
int prefill_impl(const float* q, const float* k, const float* v, float* out, int B, int H,
                 int Hkv, int L, int D, int window, float softcap, float scale, void* workspace,
                 size_t workspace_bytes, int32_t* status, void* stream,
                 const int32_t* lengths) {
  if (!dims_ok(B, H, L, D) || Hkv < 1 || H % Hkv != 0 || window < 0) return ATTN_ERR_SHAPE;
  if (!isfinite(softcap) || !isfinite(scale)) return ATTN_ERR_PARAM;
  if (B == 0 || L == 0) return ATTN_OK;
  if (!q || !k || !v || !out) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return ATTN_ERR_ALIGN;
  gqa::AttnShape a{};
  a.q = q; a.k = k; a.v = v; a.out = out;
  a.B = B; a.H = H; a.Hkv = Hkv; a.L = L; a.D = D;
  a.window = window; a.softcap = softcap > 0.f ? softcap : 0.f;
  a.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
  a.status = status;
  a.lengths = lengths;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (gqa::prefill_tc_supports(D)) {
    if (!workspace || workspace_bytes < gqa_attn_prefill_workspace_size(B, Hkv, L, D))
      return ATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
  }
  {
    Finite fin;
    const int mode = lengths ? gqa::kFiniteLen : gqa::kFiniteAll;
    fin.add(q, B, H, L, D, mode, lengths);
    fin.add(k, B, Hkv, L, D, mode, lengths);
    fin.add(v, B, Hkv, L, D, mode, lengths);
    if (const int rc = fin.gate(status, s, &a.skip)) return rc;
  }
  if (gqa::prefill_tc_supports(D)) {
    a.vt = static_cast<float*>(workspace);
    a.vt_pitch = gqa::prefill_vt_pitch(L);
    return cuda_status(gqa::launch_prefill_tc(a, s));
  }
  return cuda_status(gqa::launch_prefill_simt(a, s));
}
}  // namespace

int gqa_attn_prefill(const float* q, const float* k, const float* v, float* out, int B, int H,
                     int Hkv, int L, int D, int window, float softcap, float scale,
                     void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
  return prefill_impl(q, k, v, out, B, H, Hkv, L, D, window, softcap, scale, workspace,
                      workspace_bytes, status, stream, nullptr);
}

namespace {
// The fused path applies q's RMSNorm + RoPE inside the tensor-core kernel.
bool rope_fused(int D, int R) {
  return gqa::prefill_tc_supports(D) && gqa::prefill_fuses_rope(D) && R % 64 == 0;
}
size_t round256(size_t n) { return (n + 255) / 256 * 256; }
}  // namespace

size_t gqa_attn_prefill_rope_workspace_size(int B, int H, int Hkv, int L, int D,
                                            const attn_rope_params* rp) {
  const size_t base = gqa_attn_prefill_workspace_size(B, Hkv, L, D);
  if (base == 0 || H < 1 || (rp && !rope_params_ok(rp, D))) return 0;
  if (!rp || rope_fused(D, rope_dim_of(rp, D))) return base;
  return round256(base) + (size_t)B * H * L * D * sizeof(float);
}

int gqa_attn_vt_pitch(int L) { return L < 0 ? 0 : gqa::prefill_vt_pitch(L); }

int gqa_attn_v_transpose(const float* v, float* vt, int B, int Hkv, int L, int D, void* stream) {
  if (B < 0 || Hkv < 1 || L < 0 || !gqa::prefill_tc_supports(D)) return ATTN_ERR_SHAPE;
  if (B == 0 || L == 0) return ATTN_OK;
  if (!v || !vt) return ATTN_ERR_NULL;
  if (!aligned16(v) || !aligned16(vt)) return ATTN_ERR_ALIGN;
  return cuda_status(gqa::launch_transpose_v(v, vt, B * Hkv, L, D, gqa::prefill_vt_pitch(L),
                                             static_cast<cudaStream_t>(stream)));
}

size_t gqa_attn_prefill_rope_vt_workspace_size(int B, int H, int L, int D,
                                               const attn_rope_params* rp) {
  if (B < 0 || H < 1 || L < 0 || !gqa::prefill_tc_supports(D) || (rp && !rope_params_ok(rp, D)))
    return 0;
  if (!rp || rope_fused(D, rope_dim_of(rp, D)) || B == 0 || L == 0) return 16;
  return (size_t)B * H * L * D * sizeof(float);
}

namespace {
// Shared by gqa_attn_prefill_rope (vt == NULL: V^T is built in the workspace)
// and gqa_attn_prefill_rope_vt (vt given; the workspace holds only rotated q).
int prefill_rope_impl(const float* q, const float* k, const float* v, const float* vt, float* out,
                      int B, int H, int Hkv, int L, int D, const int32_t* start,
                      int32_t max_start, const attn_rope_params* rp, const float* table,
                      const float* q_norm_w, float norm_eps, int window, float softcap,
                      float scale, void* workspace, size_t workspace_bytes, int32_t* status,
                      void* stream, const int32_t* lengths = nullptr) {
  if (!dims_ok(B, H, L, D) || Hkv < 1 || H % Hkv != 0 || window < 0) return ATTN_ERR_SHAPE;
  if (vt && !gqa::prefill_tc_supports(D)) return ATTN_ERR_SHAPE;
  if (!isfinite(softcap) || !isfinite(scale)) return ATTN_ERR_PARAM;
  if (B == 0 || L == 0) return ATTN_OK;
  if (!q || !k || !(v || vt) || !out) return ATTN_ERR_NULL;
  if (!rp && (table || q_norm_w)) return ATTN_ERR_PARAM;     // no RoPE: q arrives rotated
  if (rp && (!start || !table)) return ATTN_ERR_NULL;
  if ((rp && !rope_params_ok(rp, D)) || !(norm_eps >= 0.f)) return ATTN_ERR_PARAM;
  if (!aligned16(q) || !aligned16(k) || (v && !aligned16(v)) || (vt && !aligned16(vt)) ||
      !aligned16(out) || (table && !aligned16(table)) || (q_norm_w && !aligned16(q_norm_w)))
    return ATTN_ERR_ALIGN;
  if (rp && (max_start < 0 || (int64_t)max_start + L - 1 >= (int64_t)max_pos_of(rp)))
    return ATTN_ERR_POSITION;
  const size_t need = vt ? gqa_attn_prefill_rope_vt_workspace_size(B, H, L, D, rp)
                         : gqa_attn_prefill_rope_workspace_size(B, H, Hkv, L, D, rp);
  const int R = rp ? rope_dim_of(rp, D) : 0;
  const bool fused = !rp || rope_fused(D, R);
  const bool needs_ws = !vt || !fused;
  if (needs_ws) {
    if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  gqa::AttnShape a{};
  a.k = k; a.v = v; a.out = out;
  a.B = B; a.H = H; a.Hkv = Hkv; a.L = L; a.D = D;
  a.window = window; a.softcap = softcap > 0.f ? softcap : 0.f;
  a.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
  a.status = status;
  a.lengths = lengths;
  {
    Finite fin;
    const int mode = lengths ? gqa::kFiniteLen : gqa::kFiniteAll;
    fin.add(q, B, H, L, D, mode, lengths);
    fin.add(k, B, Hkv, L, D, mode, lengths);
    if (v) fin.add(v, B, Hkv, L, D, mode, lengths);
    else fin.add(vt, B, Hkv, D, L, gqa::kFiniteAll, nullptr, 0, gqa::prefill_vt_pitch(L));
    fin.add(q_norm_w, 1, 1, 1, D);
    if (const int rc = fin.gate(status, s, &a.skip)) return rc;
  }
  if (gqa::prefill_tc_supports(D)) {
    a.vt = vt ? const_cast<float*>(vt) : static_cast<float*>(workspace);
    a.vt_pitch = gqa::prefill_vt_pitch(L);
  }
  // The kernels that launch after the V^T pre-pass (when this call builds V^T).
  auto attend = [&]() -> int {
    if (!gqa::prefill_tc_supports(D)) return cuda_status(gqa::launch_prefill_simt(a, s));
    return cuda_status(vt ? gqa::launch_prefill_tc_vt(a, s) : gqa::launch_prefill_tc(a, s));
  };
  if (!rp) {
    a.q = q;
    return attend();
  }
  if (fused) {
    a.q = q;
    a.rope.table = reinterpret_cast<const float2*>(table);
    a.rope.start = start;
    a.rope.norm_w = q_norm_w;
    a.rope.norm_eps = norm_eps;
    a.rope.R = R;
    a.rope.max_positions = max_pos_of(rp);
    return attend();
  }
  // Other shapes: rotate q out of place into the workspace, then the plain kernels.
  float* qrot = vt ? static_cast<float*>(workspace)
                   : reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                              round256(gqa_attn_prefill_workspace_size(B, Hkv, L,
                                                                                       D)));
  gqa::RopeJob j{};
  j.x = const_cast<float*>(q); j.y = qrot;
  j.B = B; j.NH = H; j.L = L; j.D = D; j.R = R;
  j.start = start; j.max_positions = max_pos_of(rp);
  j.table = reinterpret_cast<const float2*>(table);
  j.norm_w = q_norm_w; j.norm_eps = norm_eps; j.status = status; j.skip = a.skip;
  if (cudaError_t e = gqa::launch_rope_rows(j, s); e != cudaSuccess) return cuda_status(e);
  a.q = qrot;
  return attend();
}
}  // namespace

int gqa_attn_prefill_rope(const float* q, const float* k, const float* v, float* out, int B,
                          int H, int Hkv, int L, int D, const int32_t* start, int32_t max_start,
                          const attn_rope_params* rp, const float* table, const float* q_norm_w,
                          float norm_eps, int window, float softcap, float scale,
                          void* workspace, size_t workspace_bytes, int32_t* status,
                          void* stream) {
  return prefill_rope_impl(q, k, v, nullptr, out, B, H, Hkv, L, D, start, max_start, rp, table,
                           q_norm_w, norm_eps, window, softcap, scale, workspace, workspace_bytes,
                           status, stream);
}

int gqa_attn_prefill_rope_vt(const float* q, const float* k, const float* vt, float* out, int B,
                             int H, int Hkv, int L, int D, const int32_t* start,
                             int32_t max_start, const attn_rope_params* rp, const float* table,
                             const float* q_norm_w, float norm_eps, int window, float softcap,
                             float scale, void* workspace, size_t workspace_bytes,
                             int32_t* status, void* stream) {
  return prefill_rope_impl(q, k, nullptr, vt, out, B, H, Hkv, L, D, start, max_start, rp, table,
                           q_norm_w, norm_eps, window, softcap, scale, workspace, workspace_bytes,
                           status, stream);
}

namespace {
// Workspace of gqa_attn_prefill_step, in order: V^T | rotated keys (a ring shorter
// than the chunk) | rotated q (shapes whose kernel does not rotate q) -- or, for
// head dims the tensor cores do not take, rotated keys | rotated q.
struct StepLayout {
  bool tc;
  size_t vt, kr, qrot, total;
};
StepLayout step_layout(int B, int H, int Hkv, int L, int D, int window,
                       const attn_rope_params* rp) {
  StepLayout y{};
  y.tc = gqa::prefill_tc_supports(D) && gqa::append_vt_supports(D);
  const size_t kv = (size_t)B * Hkv * L * D * sizeof(float);
  size_t p = 0;
  if (y.tc) {
    y.vt = p;
    p += round256((size_t)B * Hkv * D * gqa::prefill_vt_pitch(L) * sizeof(float));
    y.kr = p;
    if (window > 0 && L > window) p += round256(kv);
    y.qrot = p;
    if (!rope_fused(D, rope_dim_of(rp, D))) p += round256((size_t)B * H * L * D * sizeof(float));
  } else {
    y.kr = p;
    p += round256(kv);
    y.qrot = p;
    p += round256((size_t)B * H * L * D * sizeof(float));
  }
  y.total = p;
  return y;
}
}  // namespace

size_t gqa_attn_prefill_step_workspace_size(int B, int H, int Hkv, int L, int D, int window,
                                            const attn_rope_params* rp) {
  if (!dims_ok(B, H, L, D) || Hkv < 1 || H % Hkv != 0 || window < 0 || !rope_params_ok(rp, D))
    return 0;
  if (B == 0 || L == 0) return 16;
  return step_layout(B, H, Hkv, L, D, window, rp).total;
}

int gqa_attn_prefill_step(const float* q, const float* k, const float* v, float* out, int B,
                          int H, int Hkv, int L, int D, const attn_rope_params* rp,
                          const float* table, const float* q_norm_w, const float* k_norm_w,
                          float norm_eps, float* k_cache, float* v_cache, int capacity,
                          int window, float softcap, float scale, void* workspace,
                          size_t workspace_bytes, int32_t* status, void* stream) {
  if (!dims_ok(B, H, L, D) || Hkv < 1 || H % Hkv != 0 || window < 0 || capacity < 1)
    return ATTN_ERR_SHAPE;
  if (window > 0 && capacity != window) return ATTN_ERR_SHAPE;
  if (!isfinite(softcap) || !isfinite(scale)) return ATTN_ERR_PARAM;
  if (!rp) return ATTN_ERR_NULL;
  if (!rope_params_ok(rp, D) || !(norm_eps >= 0.f)) return ATTN_ERR_PARAM;
  if (B == 0 || L == 0) return ATTN_OK;
  if (!q || !k || !v || !out || !table || !k_cache || !v_cache) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(table) ||
      !aligned16(k_cache) || !aligned16(v_cache) || (q_norm_w && !aligned16(q_norm_w)) ||
      (k_norm_w && !aligned16(k_norm_w)))
    return ATTN_ERR_ALIGN;
  if ((int64_t)L - 1 >= (int64_t)max_pos_of(rp)) return ATTN_ERR_POSITION;
  if (window == 0 && L > capacity) return ATTN_ERR_CAPACITY;
  if ((int64_t)B * Hkv > 65535) return ATTN_ERR_SHAPE;
  const StepLayout lay = step_layout(B, H, Hkv, L, D, window, rp);
  if (!workspace || workspace_bytes < lay.total) return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const int R = rope_dim_of(rp, D);
  const int32_t* skip = nullptr;
  {
    Finite fin;
    fin.add(q, B, H, L, D);
    fin.add(k, B, Hkv, L, D);
    fin.add(v, B, Hkv, L, D);
    fin.add(q_norm_w, 1, 1, 1, D);
    fin.add(k_norm_w, 1, 1, 1, D);
    if (const int rc = fin.gate(status, s, &skip)) return rc;
  }
  // RoPE jobs at positions 0 .. L-1 (no start array)
  auto rope_job = [&](float* x, float* y, int NH, const float* nw) {
    gqa::RopeJob j{};
    j.x = x; j.y = y; j.B = B; j.NH = NH; j.L = L; j.D = D; j.R = R;
    j.start = nullptr; j.max_positions = max_pos_of(rp);
    j.table = reinterpret_cast<const float2*>(table);
    j.norm_w = nw; j.norm_eps = norm_eps; j.status = status; j.skip = skip;
    return j;
  };
  gqa::AttnShape a{};
  a.out = out; a.v = v;
  a.B = B; a.H = H; a.Hkv = Hkv; a.L = L; a.D = D;
  a.window = window; a.softcap = softcap > 0.f ? softcap : 0.f;
  a.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
  a.status = status;
  a.skip = skip;
  if (!lay.tc) {
    // head dims off the tensor cores: rotate a copy of k (into the cache as well) and
    // q, then the CUDA-core prefill
    float* kr = reinterpret_cast<float*>(ws + lay.kr);
    float* qrot = reinterpret_cast<float*>(ws + lay.qrot);
    if (cudaError_t e = cudaMemcpyAsync(kr, k, (size_t)B * Hkv * L * D * sizeof(float),
                                        cudaMemcpyDeviceToDevice, s);
        e != cudaSuccess)
      return cuda_status(e);
    gqa::RopeJob kj = rope_job(kr, nullptr, Hkv, k_norm_w);
    kj.v = v; kj.k_cache = k_cache; kj.v_cache = v_cache; kj.capacity = capacity;
    kj.window = window;
    if (cudaError_t e = gqa::launch_rope_rows(kj, s); e != cudaSuccess) return cuda_status(e);
    const gqa::RopeJob qj = rope_job(const_cast<float*>(q), qrot, H, q_norm_w);
    if (cudaError_t e = gqa::launch_rope_rows(qj, s); e != cudaSuccess) return cuda_status(e);
    a.q = qrot; a.k = kr;
    return cuda_status(gqa::launch_prefill_simt(a, s));
  }
  // one memory pass: rotated k into the cache (and kr for a ring shorter than the
  // chunk), v into the cache, V^T into the workspace; then the tensor-core kernel
  // reads the rotated keys from the cache
  float* vt = reinterpret_cast<float*>(ws + lay.vt);
  float* kr = window > 0 && L > window ? reinterpret_cast<float*>(ws + lay.kr) : nullptr;
  gqa::AppendVtJob aj{};
  aj.k = k; aj.v = v; aj.k_cache = k_cache; aj.v_cache = v_cache; aj.kr = kr; aj.vt = vt;
  aj.B = B; aj.Hkv = Hkv; aj.L = L; aj.D = D; aj.R = R;
  aj.table = reinterpret_cast<const float2*>(table);
  aj.norm_w = k_norm_w; aj.norm_eps = norm_eps; aj.start = nullptr;
  aj.max_positions = max_pos_of(rp); aj.capacity = capacity; aj.window = window;
  aj.vt_pitch = gqa::prefill_vt_pitch(L); aj.status = status; aj.skip = skip;
  if (cudaError_t e = gqa::launch_append_vt(aj, s); e != cudaSuccess) return cuda_status(e);
  a.k = kr ? kr : k_cache;
  a.k_head_rows = kr ? 0 : capacity;
  a.vt = vt; a.vt_pitch = aj.vt_pitch;
  if (rope_fused(D, R)) {
    a.q = q;
    a.rope.table = reinterpret_cast<const float2*>(table);
    a.rope.start = nullptr;
    a.rope.norm_w = q_norm_w;
    a.rope.norm_eps = norm_eps;
    a.rope.R = R;
    a.rope.max_positions = max_pos_of(rp);
  } else {
    float* qrot = reinterpret_cast<float*>(ws + lay.qrot);
    const gqa::RopeJob qj = rope_job(const_cast<float*>(q), qrot, H, q_norm_w);
    if (cudaError_t e = gqa::launch_rope_rows(qj, s); e != cudaSuccess) return cuda_status(e);
    a.q = qrot;
  }
  return cuda_status(gqa::launch_prefill_tc_vt(a, s));
}

size_t gqa_attn_prefill_ragged_workspace_size(int B, int H, int Hkv, int L, int D,
                                              const attn_rope_params* rp) {
  const size_t base = rp ? gqa_attn_prefill_rope_workspace_size(B, H, Hkv, L, D, rp)
                         : gqa_attn_prefill_workspace_size(B, Hkv, L, D);
  if (base == 0 || H < 1) return 0;
  return round256((size_t)B * sizeof(int32_t)) + round256(base);
}

int gqa_attn_prefill_ragged(const float* q, const float* k, const float* v, float* out, int B,
                            int H, int Hkv, int L, int D, const int32_t* lengths,
                            const attn_rope_params* rp, const float* table,
                            const float* q_norm_w, float norm_eps, int window, float softcap,
                            float scale, void* workspace, size_t workspace_bytes,
                            int32_t* status, void* stream) {
  if (!dims_ok(B, H, L, D) || Hkv < 1 || H % Hkv != 0 || window < 0) return ATTN_ERR_SHAPE;
  if (rp && !rope_params_ok(rp, D)) return ATTN_ERR_PARAM;
  if (B == 0 || L == 0) return ATTN_OK;
  if (!lengths) return ATTN_ERR_NULL;
  const size_t need = gqa_attn_prefill_ragged_workspace_size(B, H, Hkv, L, D, rp);
  if (need == 0) return ATTN_ERR_SHAPE;
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
  // [start = 0 per row (B int32) | the plain or RoPE prefill's workspace]
  const size_t zb = round256((size_t)B * sizeof(int32_t));
  char* rest = static_cast<char*>(workspace) + zb;
  if (!rp)
    return prefill_impl(q, k, v, out, B, H, Hkv, L, D, window, softcap, scale, rest,
                        workspace_bytes - zb, status, stream, lengths);
  int32_t* zero_start = static_cast<int32_t*>(workspace);
  if (cudaError_t e = cudaMemsetAsync(zero_start, 0, (size_t)B * sizeof(int32_t),
                                      static_cast<cudaStream_t>(stream));
      e != cudaSuccess)
    return cuda_status(e);
  return prefill_rope_impl(q, k, v, nullptr, out, B, H, Hkv, L, D, zero_start, 0, rp, table,
                           q_norm_w, norm_eps, window, softcap, scale, rest,
                           workspace_bytes - zb, status, stream, lengths);
}

namespace {
// Key rows per head of the continued prefill's key buffer.
int64_t cached_lk(int32_t max_start, int window, int L) {
  const int64_t pre = window > 0 ? (max_start < window - 1 ? max_start : window - 1) : max_start;
  return pre + L;
}
struct CachedLayout {
  size_t pre, kg, vtg, qrot, total;
};
CachedLayout cached_layout(int B, int H, int Hkv, int L, int D, int32_t max_start, int window,
                           bool rotate_q_first) {
  const int64_t Lk = cached_lk(max_start, window, L);
  CachedLayout c{};
  c.pre = 0;
  c.kg = round256((size_t)B * sizeof(int32_t));
  c.vtg = c.kg + round256((size_t)B * Hkv * Lk * D * sizeof(float));
  c.qrot = c.vtg + round256((size_t)B * Hkv * D * gqa::prefill_vt_pitch((int)Lk) * sizeof(float));
  c.total = c.qrot + (rotate_q_first ? (size_t)B * H * L * D * sizeof(float) : 0);
  return c;
}
}  // namespace

size_t gqa_attn_prefill_cached_workspace_size(int B, int H, int Hkv, int L, int D,
                                              int32_t max_start, int window,
                                              const attn_rope_params* rp) {
  if (B < 0 || H < 1 || Hkv < 1 || L < 0 || max_start < 0 || window < 0 ||
      !gqa::prefill_tq_supports_kv_off(D))
    return 0;
  if (rp && !rope_params_ok(rp, D)) return 0;
  if (cached_lk(max_start, window, L) > (int64_t)1 << 30) return 0;
  const bool rotate_first = rp && !rope_fused(D, rope_dim_of(rp, D));
  return cached_layout(B, H, Hkv, L, D, max_start, window, rotate_first).total;
}

int gqa_attn_prefill_cached(const float* q, const float* k, const float* v, const float* k_cache,
                            const float* v_cache, int capacity, float* out, int B, int H,
                            int Hkv, int L, int D, const int32_t* start, int32_t max_start,
                            const attn_rope_params* rp, const float* table,
                            const float* q_norm_w, float norm_eps, int window, float softcap,
                            float scale, void* workspace, size_t workspace_bytes,
                            int32_t* status, void* stream) {
  if (!dims_ok(B, H, L, D) || Hkv < 1 || H % Hkv != 0 || window < 0 || capacity < 1)
    return ATTN_ERR_SHAPE;
  if (!gqa::prefill_tq_supports_kv_off(D)) return ATTN_ERR_SHAPE;
  if (window > 0 && capacity != window) return ATTN_ERR_SHAPE;
  if (!isfinite(softcap) || !isfinite(scale)) return ATTN_ERR_PARAM;
  if (B == 0 || L == 0) return ATTN_OK;
  if (!q || !k || !v || !k_cache || !v_cache || !out || !start) return ATTN_ERR_NULL;
  if (rp && (!table || !rope_params_ok(rp, D) || !(norm_eps >= 0.f))) return ATTN_ERR_PARAM;
  if (!rp && (table || q_norm_w)) return ATTN_ERR_PARAM;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(out) || (table && !aligned16(table)) ||
      (q_norm_w && !aligned16(q_norm_w)))
    return ATTN_ERR_ALIGN;
  if (max_start < 0) return ATTN_ERR_POSITION;
  if (rp && (int64_t)max_start + L - 1 >= (int64_t)max_pos_of(rp)) return ATTN_ERR_POSITION;
  if (window == 0 && max_start > capacity) return ATTN_ERR_CAPACITY;
  const size_t need =
      gqa_attn_prefill_cached_workspace_size(B, H, Hkv, L, D, max_start, window, rp);
  if (need == 0) return ATTN_ERR_SHAPE;
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int R = rp ? rope_dim_of(rp, D) : 0;
  const bool fused = rp && rope_fused(D, R);
  const CachedLayout lay = cached_layout(B, H, Hkv, L, D, max_start, window, rp && !fused);
  char* ws = static_cast<char*>(workspace);
  const int Lk = (int)cached_lk(max_start, window, L);
  const int32_t* skip = nullptr;
  {
    Finite fin;
    fin.add(q, B, H, L, D);
    fin.add(k, B, Hkv, L, D);
    fin.add(v, B, Hkv, L, D);
    fin.add(k_cache, B, Hkv, capacity, D, gqa::kFinitePrefix, start, window);
    fin.add(v_cache, B, Hkv, capacity, D, gqa::kFinitePrefix, start, window);
    fin.add(q_norm_w, 1, 1, 1, D);
    if (const int rc = fin.gate(status, s, &skip)) return rc;
  }

  gqa::GatherJob gj{};
  gj.k = k; gj.v = v; gj.k_cache = k_cache; gj.v_cache = v_cache; gj.start = start;
  gj.pre = reinterpret_cast<int32_t*>(ws + lay.pre);
  gj.kg = reinterpret_cast<float*>(ws + lay.kg);
  gj.vtg = reinterpret_cast<float*>(ws + lay.vtg);
  gj.B = B; gj.Hkv = Hkv; gj.L = L; gj.D = D; gj.capacity = capacity; gj.window = window;
  gj.Lk = Lk; gj.vt_pitch = gqa::prefill_vt_pitch(Lk); gj.max_start = max_start;
  gj.status = status;
  gj.skip = skip;
  if (cudaError_t e = gqa::launch_gather_kv(gj, s); e != cudaSuccess) return cuda_status(e);

  gqa::AttnShape a{};
  a.k = gj.kg; a.v = nullptr; a.out = out;
  a.vt = gj.vtg; a.vt_pitch = gj.vt_pitch;
  a.B = B; a.H = H; a.Hkv = Hkv; a.L = L; a.D = D;
  a.window = window; a.softcap = softcap > 0.f ? softcap : 0.f;
  a.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
  a.status = status;
  a.kv_off = gj.pre;
  a.Lk = Lk;
  a.q = q;
  a.skip = skip;
  if (fused) {
    a.rope.table = reinterpret_cast<const float2*>(table);
    a.rope.start = start;
    a.rope.norm_w = q_norm_w;
    a.rope.norm_eps = norm_eps;
    a.rope.R = R;
    a.rope.max_positions = max_pos_of(rp);
  } else if (rp) {
    float* qrot = reinterpret_cast<float*>(ws + lay.qrot);
    gqa::RopeJob j{};
    j.x = const_cast<float*>(q); j.y = qrot;
    j.B = B; j.NH = H; j.L = L; j.D = D; j.R = R;
    j.start = start; j.max_positions = max_pos_of(rp);
    j.table = reinterpret_cast<const float2*>(table);
    j.norm_w = q_norm_w; j.norm_eps = norm_eps; j.status = status; j.skip = skip;
    if (cudaError_t e = gqa::launch_rope_rows(j, s); e != cudaSuccess) return cuda_status(e);
    a.q = qrot;
  }
  return cuda_status(gqa::launch_prefill_tq(a, s));
}

size_t gqa_attn_decode_workspace_size(int B, int H, int Hkv, int D, int max_cache_len,
                                      int window) {
  if (B < 1 || H < 1 || Hkv < 1 || H % Hkv || D < 2 || max_cache_len < 1 || window < 0) return 0;
  return gqa::decode_partial_bytes(B, H, Hkv, D, max_cache_len, window, true);
}

namespace {
// Workspace of gqa_block_forward, in order (each part 256-byte aligned):
// zero start [B] | normed rows [T, d_model] | q [B, H, L, D] | k, v [B, Hkv, L, D] |
// attention output [B, H, L, D] | its token-major copy [T, d_model] (only when
// D % 32 != 0) | SwiGLU activations [T, IT] | the attention's own workspace.
struct BlockLayout {
  size_t zs, nrm, qh, kh, vh, ao, aot, act, attn, total;
};
BlockLayout block_layout(int B, int L, int H, int Hkv, int D, int IT, size_t attn_bytes) {
  const size_t T = (size_t)B * L, QW = (size_t)H * D, KW = (size_t)Hkv * D;
  BlockLayout y{};
  size_t p = 0;
  auto take = [&](size_t bytes) { const size_t r = p; p += round256(bytes); return r; };
  y.zs = take((size_t)B * 4);
  y.nrm = take(T * QW * 4);
  y.qh = take(T * QW * 4);
  y.kh = take(T * KW * 4);
  y.vh = take(T * KW * 4);
  y.ao = take(T * QW * 4);
  y.aot = D % 32 ? take(T * QW * 4) : p;
  y.act = take(T * (size_t)IT * 4);
  y.attn = take(attn_bytes);
  y.total = p;
  return y;
}
}  // namespace

size_t gqa_block_forward_workspace_size(int B, int L, int H, int Hkv, int D, int IT,
                                        const attn_rope_params* rp) {
  if (B < 0 || L < 0 || H < 1 || Hkv < 1 || H % Hkv != 0 || IT < 1 || !rope_params_ok(rp, D))
    return 0;
  const size_t attn = gqa_attn_prefill_rope_workspace_size(B, H, Hkv, L, D, rp);
  if (attn == 0) return 0;
  return block_layout(B, L, H, Hkv, D, IT, attn).total;
}

int gqa_block_forward(const float* x, float* out, int B, int L, int H, int Hkv, int D, int IT,
                      const attn_block_weights* w, int norm_offset, float norm_eps,
                      const attn_rope_params* rp, const float* table, int window, float softcap,
                      float scale, void* workspace, size_t workspace_bytes, int32_t* status,
                      void* stream) {
  if (!dims_ok(B, H, L, D) || Hkv < 1 || H % Hkv != 0 || IT < 1 || window < 0)
    return ATTN_ERR_SHAPE;
  if ((H * D) % 4 || IT % 4) return ATTN_ERR_SHAPE;   // 16-byte rows for the projections
  if (!isfinite(softcap) || !isfinite(scale) || !(norm_eps >= 0.f)) return ATTN_ERR_PARAM;
  if (!rp || !rope_params_ok(rp, D)) return rp ? ATTN_ERR_PARAM : ATTN_ERR_NULL;
  if (B == 0 || L == 0) return ATTN_OK;
  if (!x || !out || !w || !table || !w->input_norm || !w->post_norm || !w->wq || !w->wk ||
      !w->wv || !w->wo || !w->w_gate || !w->w_up || !w->w_down)
    return ATTN_ERR_NULL;
  if (x == out) return ATTN_ERR_SHAPE;
  if ((int64_t)L - 1 >= (int64_t)max_pos_of(rp)) return ATTN_ERR_POSITION;
  const size_t need = gqa_block_forward_workspace_size(B, L, H, Hkv, D, IT, rp);
  if (need == 0) return ATTN_ERR_SHAPE;
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  const float* ptrs[] = {x, out, table, w->input_norm, w->post_norm, w->wq, w->wk, w->wv,
                         w->wo, w->w_gate, w->w_up, w->w_down, w->q_norm, w->k_norm};
  for (const float* pp : ptrs)
    if (pp && !aligned16(pp)) return ATTN_ERR_ALIGN;
  if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long T = (long)B * L;
  const int QW = H * D, KW = Hkv * D;
  const size_t attn_need = gqa_attn_prefill_rope_workspace_size(B, H, Hkv, L, D, rp);
  const BlockLayout lay = block_layout(B, L, H, Hkv, D, IT, attn_need);
  char* ws = static_cast<char*>(workspace);
  int32_t* zero_start = reinterpret_cast<int32_t*>(ws + lay.zs);
  float* nrm = reinterpret_cast<float*>(ws + lay.nrm);
  float* qh = reinterpret_cast<float*>(ws + lay.qh);
  float* kh = reinterpret_cast<float*>(ws + lay.kh);
  float* vh = reinterpret_cast<float*>(ws + lay.vh);
  float* ao = reinterpret_cast<float*>(ws + lay.ao);
  float* aot = reinterpret_cast<float*>(ws + lay.aot);
  float* act = reinterpret_cast<float*>(ws + lay.act);
  const bool offset = norm_offset != 0;
  const int32_t* skip = nullptr;
  {
    Finite fin;
    fin.add(x, 1, 1, T, QW);
    fin.add(w->input_norm, 1, 1, 1, QW);
    fin.add(w->post_norm, 1, 1, 1, QW);
    fin.add(w->wq, 1, 1, QW, QW);
    fin.add(w->wk, 1, 1, KW, QW);
    fin.add(w->wv, 1, 1, KW, QW);
    fin.add(w->wo, 1, 1, QW, QW);
    fin.add(w->w_gate, 1, 1, IT, QW);
    fin.add(w->w_up, 1, 1, IT, QW);
    fin.add(w->w_down, 1, 1, QW, IT);
    fin.add(w->q_norm, 1, 1, 1, D);
    fin.add(w->k_norm, 1, 1, 1, D);
    if (const int rc = fin.gate(status, s, &skip)) return rc;
  }
  auto chk = [&](cudaError_t e) { return e == cudaSuccess ? ATTN_OK : cuda_status(e); };
  auto gemm = [&](gqa::GemmJob& j) {
    j.skip = skip;
    return gqa::gemm_tc_supports(j) ? chk(gqa::launch_gemm_tc(j, s)) : ATTN_ERR_SHAPE;
  };
  int rc;
  if ((rc = chk(cudaMemsetAsync(zero_start, 0, (size_t)B * 4, s)))) return rc;
  // attention half: n1 = RMSNorm(x); q, k, v = n1 W^T written head-major
  if ((rc = chk(gqa::launch_rmsnorm_rows(x, w->input_norm, nrm, T, QW, norm_eps, offset, true,
                                         s, skip))))
    return rc;
  {
    gqa::GemmJob j{};
    j.x = nrm; j.T = T; j.K = QW; j.L = L; j.D = D; j.status = status;
    j.nseg = 3;
    const float* wts[3] = {w->wq, w->wk, w->wv};
    float* outs[3] = {qh, kh, vh};
    const int ns[3] = {QW, KW, KW}, heads[3] = {H, Hkv, Hkv};
    for (int i = 0; i < 3; ++i) {
      j.seg[i].w = wts[i]; j.seg[i].n = ns[i]; j.seg[i].mode = 0;
      j.seg[i].out = outs[i]; j.seg[i].out_heads = heads[i];
    }
    if ((rc = gemm(j))) return rc;
  }
  gqa::RopeJob rj{};
  rj.x = kh; rj.B = B; rj.NH = Hkv; rj.L = L; rj.D = D; rj.R = rope_dim_of(rp, D);
  rj.start = zero_start; rj.max_positions = max_pos_of(rp);
  rj.table = reinterpret_cast<const float2*>(table);
  rj.norm_w = w->k_norm; rj.norm_eps = norm_eps; rj.status = status; rj.skip = skip;
  if ((rc = chk(gqa::launch_rope_rows(rj, s)))) return rc;
  rc = gqa_attn_prefill_rope(qh, kh, vh, ao, B, H, Hkv, L, D, zero_start, 0, rp, table,
                             w->q_norm, norm_eps, window, softcap, scale, ws + lay.attn,
                             workspace_bytes - lay.attn, status, stream);
  if (rc != ATTN_OK) return rc;
  // h = x + o_proj(attention): the projection reads the head-major attention output
  // directly when a 32-wide K block stays inside one head
  {
    gqa::GemmJob j{};
    j.T = T; j.K = QW; j.L = L; j.D = D; j.status = status; j.nseg = 1;
    if (D % 32 == 0) {
      j.x = ao; j.x_heads = H;
    } else {
      if ((rc = chk(gqa::launch_swap_mid(ao, aot, B, H, L, D, s, skip)))) return rc;
      j.x = aot;
    }
    j.seg[0].w = w->wo; j.seg[0].n = QW; j.seg[0].mode = 1;
    j.seg[0].out = out; j.seg[0].ldo = QW; j.seg[0].res = x; j.seg[0].ldr = QW;
    if ((rc = gemm(j))) return rc;
  }
  // MLP half: n2 = RMSNorm(h); act = SiLU(n2 Wg^T) * (n2 Wu^T); out = h + act Wd^T
  if ((rc = chk(gqa::launch_rmsnorm_rows(out, w->post_norm, nrm, T, QW, norm_eps, offset, true,
                                         s, skip))))
    return rc;
  {
    gqa::GemmJob j{};
    j.x = nrm; j.T = T; j.K = QW; j.L = L; j.D = D; j.status = status; j.nseg = 1;
    j.seg[0].w = w->w_gate; j.seg[0].w_up = w->w_up; j.seg[0].n = IT; j.seg[0].mode = 2;
    j.seg[0].round_out = 1; j.seg[0].out = act; j.seg[0].ldo = IT;
    if ((rc = gemm(j))) return rc;
  }
  {
    gqa::GemmJob j{};
    j.x = act; j.T = T; j.K = IT; j.L = L; j.D = D; j.status = status; j.nseg = 1;
    j.seg[0].w = w->w_down; j.seg[0].n = QW; j.seg[0].mode = 1;
    j.seg[0].out = out; j.seg[0].ldo = QW; j.seg[0].res = out; j.seg[0].ldr = QW;
    if ((rc = gemm(j))) return rc;
  }
  return ATTN_OK;
}

int attn_linear(const float* x, const float* w, const float* residual, float* y, long T, int N,
                int K, int32_t* status, void* stream) {
  if (T < 0 || N < 1 || K < 1) return ATTN_ERR_SHAPE;
  if (K % 4 || N % 4) return ATTN_ERR_SHAPE;
  if (T == 0) return ATTN_OK;
  if (T > 0x7fffffffL) return ATTN_ERR_SHAPE;
  if (!x || !w || !y) return ATTN_ERR_NULL;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (residual && !aligned16(residual)))
    return ATTN_ERR_ALIGN;
  gqa::GemmJob j{};
  j.x = x; j.T = T; j.K = K; j.L = 1; j.D = 1; j.status = status; j.nseg = 1;
  j.seg[0].w = w; j.seg[0].n = N; j.seg[0].mode = residual ? 1 : 0;
  j.seg[0].out = y; j.seg[0].ldo = N; j.seg[0].res = residual; j.seg[0].ldr = N;
  if (!gqa::gemm_tc_supports(j)) return ATTN_ERR_SHAPE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Finite fin;
  fin.add(x, 1, 1, T, K);
  fin.add(w, 1, 1, N, K);
  fin.add(residual, 1, 1, T, N);
  if (const int rc = fin.gate(status, s, &j.skip)) return rc;
  return cuda_status(gqa::launch_gemm_tc(j, s));
}

int gqa_attn_prefill_identical(const float* q, const float* k, const float* v,
                               const float* k_cache, const float* v_cache, int capacity,
                               float* out, int B, int H, int Hkv, int L, int D,
                               const int32_t* start, int32_t max_start, int window,
                               float softcap, float scale, int32_t* status, void* stream) {
  if (!dims_ok(B, H, L, D) || Hkv < 1 || H % Hkv != 0 || window < 0) return ATTN_ERR_SHAPE;
  const bool cached = k_cache || v_cache;
  if (cached && (capacity < 1 || (window > 0 && capacity != window))) return ATTN_ERR_SHAPE;
  if (!isfinite(softcap) || !isfinite(scale)) return ATTN_ERR_PARAM;
  if (B == 0 || L == 0) return ATTN_OK;
  if (!q || !k || !v || !out || (cached && !(k_cache && v_cache && start))) return ATTN_ERR_NULL;
  if (max_start < 0 || (!start && max_start != 0)) return ATTN_ERR_POSITION;
  if (cached && window == 0 && max_start > capacity) return ATTN_ERR_CAPACITY;
  gqa::IdentJob j{};
  j.q = q; j.k = k; j.v = v; j.k_cache = k_cache; j.v_cache = v_cache;
  j.start = start; j.max_start = max_start; j.out = out;
  j.B = B; j.H = H; j.Hkv = Hkv; j.L = L; j.D = D; j.capacity = capacity; j.window = window;
  j.softcap = softcap > 0.f ? softcap : 0.f;
  j.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
  j.status = status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Finite fin;
  fin.add(q, B, H, L, D);
  fin.add(k, B, Hkv, L, D);
  fin.add(v, B, Hkv, L, D);
  if (cached) {
    fin.add(k_cache, B, Hkv, capacity, D, gqa::kFinitePrefix, start, window);
    fin.add(v_cache, B, Hkv, capacity, D, gqa::kFinitePrefix, start, window);
  }
  if (const int rc = fin.gate(status, s, &j.skip)) return rc;
  return cuda_status(gqa::launch_identical(j, s));
}

int gqa_attn_decode_identical(const float* q, const float* k_cache, const float* v_cache,
                              const int32_t* cache_len, int32_t max_cache_len, float* out, int B,
                              int H, int Hkv, int D, int capacity, int window, float softcap,
                              float scale, int32_t* status, void* stream) {
  if (!dims_ok(B, H, 1, D) || Hkv < 1 || H % Hkv != 0 || window < 0 || capacity < 1)
    return ATTN_ERR_SHAPE;
  if (window > 0 && capacity != window) return ATTN_ERR_SHAPE;
  if (!isfinite(softcap) || !isfinite(scale)) return ATTN_ERR_PARAM;
  if (B == 0) return ATTN_OK;
  if (max_cache_len < 1) return ATTN_ERR_SHAPE;
  if (window == 0 && max_cache_len > capacity) return ATTN_ERR_CAPACITY;
  if (!q || !k_cache || !v_cache || !cache_len || !out) return ATTN_ERR_NULL;
  gqa::IdentJob j{};
  j.q = q; j.k_cache = k_cache; j.v_cache = v_cache; j.cache_len = cache_len;
  j.max_len = max_cache_len; j.out = out;
  j.B = B; j.H = H; j.Hkv = Hkv; j.L = 1; j.D = D; j.capacity = capacity; j.window = window;
  j.softcap = softcap > 0.f ? softcap : 0.f;
  j.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
  j.status = status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Finite fin;
  fin.add(q, B, H, 1, D);
  fin.add(k_cache, B, Hkv, capacity, D, gqa::kFiniteCache, cache_len);
  fin.add(v_cache, B, Hkv, capacity, D, gqa::kFiniteCache, cache_len);
  if (const int rc = fin.gate(status, s, &j.skip)) return rc;
  return cuda_status(gqa::launch_identical(j, s));
}

int gqa_attn_decode(const float* q, const float* k_cache, const float* v_cache,
                    const int32_t* cache_len, int32_t max_cache_len, float* out, int B, int H,
                    int Hkv, int D, int capacity, int window, float softcap, float scale,
                    void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
  const int rc = gqa::decode_host_check(q, k_cache, v_cache, cache_len, max_cache_len, out, B, H,
                                        Hkv, D, capacity, window, softcap, scale);
  if (rc != ATTN_OK || B == 0) return rc;
  gqa::DecodeJob j{};
  j.q = q; j.k_cache = k_cache; j.v_cache = v_cache; j.cache_len = cache_len;
  j.max_cache_len = max_cache_len; j.out = out;
  j.B = B; j.H = H; j.Hkv = Hkv; j.D = D; j.capacity = capacity; j.window = window;
  j.softcap = softcap > 0.f ? softcap : 0.f;
  j.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
  j.status = status;
  gqa::decode_split_plan(B, Hkv, max_cache_len, window, &j.nsplit, &j.chunk);
  if (j.nsplit > 1) {
    const size_t need = gqa::decode_partial_bytes(B, H, Hkv, D, max_cache_len, window, false);
    if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
  }
  j.partial = static_cast<float*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Finite fin;
  fin.add(q, B, H, 1, D);
  fin.add(k_cache, B, Hkv, capacity, D, gqa::kFiniteCache, cache_len);
  fin.add(v_cache, B, Hkv, capacity, D, gqa::kFiniteCache, cache_len);
  if (const int rc = fin.gate(status, s, &j.skip)) return rc;
  return cuda_status(gqa::launch_decode(j, s));
}

int gqa_attn_decode_launches(int B, int H, int Hkv, int D, int32_t max_cache_len, int window,
                             int step_rope_dim) {
  if (B < 1 || H < 1 || Hkv < 1 || H % Hkv || D < 2 || D % 2 || D > gqa::kMaxHeadDim ||
      max_cache_len < 1 || window < 0 ||
      (step_rope_dim >= 0 && (step_rope_dim > D || step_rope_dim % 2)))
    return ATTN_ERR_SHAPE;
  gqa::DecodeJob j{};
  j.B = B; j.H = H; j.Hkv = Hkv; j.D = D; j.window = window; j.max_cache_len = max_cache_len;
  gqa::decode_split_plan(B, Hkv, max_cache_len, window, &j.nsplit, &j.chunk);
  if (step_rope_dim < 0) return gqa::decode_launches(j, false);
  const bool fused = gqa::decode_step_fuses(H, Hkv, D, step_rope_dim ? step_rope_dim : D);
  return (fused ? 0 : 1) + gqa::decode_launches(j, fused);
}

namespace {
// Workspace of gqa_attn_decode_step: rotated q [B, H, D] | cache lengths [B] | the
// split partials.
struct DecodeStepLayout {
  size_t qrot, cl, part, total;
};
DecodeStepLayout decode_step_layout(int B, int H, int Hkv, int D, int max_len, int window,
                                    bool bound) {
  DecodeStepLayout y{};
  size_t p = 0;
  y.qrot = p;
  p += round256((size_t)B * H * D * sizeof(float));
  y.cl = p;
  p += round256((size_t)B * sizeof(int32_t));
  y.part = p;
  p += round256(gqa::decode_partial_bytes(B, H, Hkv, D, max_len, window, bound));
  y.total = p;
  return y;
}
}  // namespace

size_t gqa_attn_decode_step_workspace_size(int B, int H, int Hkv, int D, int32_t max_pos,
                                           int window) {
  if (B < 1 || H < 1 || Hkv < 1 || H % Hkv || D < 2 || D % 2 || D > gqa::kMaxHeadDim ||
      max_pos < 0 || max_pos == 0x7fffffff || window < 0)
    return 0;
  return decode_step_layout(B, H, Hkv, D, max_pos + 1, window, true).total;
}

int gqa_attn_decode_step(const float* q, const float* k, const float* v, float* out, int B,
                         int H, int Hkv, int D, const int32_t* pos, int32_t max_pos,
                         const attn_rope_params* rp, const float* table, const float* q_norm_w,
                         const float* k_norm_w, float norm_eps, float* k_cache, float* v_cache,
                         int capacity, int window, float softcap, float scale, void* workspace,
                         size_t workspace_bytes, int32_t* status, void* stream) {
  if (!dims_ok(B, H, 1, D) || Hkv < 1 || H % Hkv != 0 || window < 0 || capacity < 1)
    return ATTN_ERR_SHAPE;
  if (window > 0 && capacity != window) return ATTN_ERR_SHAPE;
  if (!isfinite(softcap) || !isfinite(scale)) return ATTN_ERR_PARAM;
  if (!rp) return ATTN_ERR_NULL;
  if (!rope_params_ok(rp, D) || !(norm_eps >= 0.f)) return ATTN_ERR_PARAM;
  if (B == 0) return ATTN_OK;
  if (!q || !k || !v || !out || !pos || !table || !k_cache || !v_cache) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(table) ||
      !aligned16(k_cache) || !aligned16(v_cache) || (q_norm_w && !aligned16(q_norm_w)) ||
      (k_norm_w && !aligned16(k_norm_w)))
    return ATTN_ERR_ALIGN;
  if (max_pos < 0 || (int64_t)max_pos >= (int64_t)max_pos_of(rp)) return ATTN_ERR_POSITION;
  if (window == 0 && max_pos >= capacity) return ATTN_ERR_CAPACITY;
  const DecodeStepLayout lay = decode_step_layout(B, H, Hkv, D, max_pos + 1, window, false);
  if (!workspace || workspace_bytes < lay.total) return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const int32_t* skip = nullptr;
  {
    Finite fin;
    fin.add(q, B, H, 1, D);
    fin.add(k, B, Hkv, 1, D);
    fin.add(v, B, Hkv, 1, D);
    fin.add(k_cache, B, Hkv, capacity, D, gqa::kFiniteCache, pos);
    fin.add(v_cache, B, Hkv, capacity, D, gqa::kFiniteCache, pos);
    fin.add(q_norm_w, 1, 1, 1, D);
    fin.add(k_norm_w, 1, 1, 1, D);
    if (const int rc = fin.gate(status, s, &skip)) return rc;
  }
  gqa::DecodePrepJob pj{};
  pj.q = q; pj.k = k; pj.v = v;
  pj.qrot = reinterpret_cast<float*>(ws + lay.qrot);
  pj.k_cache = k_cache; pj.v_cache = v_cache;
  pj.cache_len = reinterpret_cast<int32_t*>(ws + lay.cl);
  pj.B = B; pj.H = H; pj.Hkv = Hkv; pj.D = D; pj.R = rope_dim_of(rp, D);
  pj.pos = pos; pj.max_positions = max_pos_of(rp); pj.capacity = capacity; pj.window = window;
  pj.table = reinterpret_cast<const float2*>(table);
  pj.q_norm_w = q_norm_w; pj.k_norm_w = k_norm_w; pj.norm_eps = norm_eps;
  pj.status = status; pj.skip = skip;
  gqa::DecodeJob j{};
  // The split kernel rotates q and appends k, v itself where it can (one launch fewer).
  const bool fused = gqa::decode_step_fuses(H, Hkv, D, pj.R);
  gqa::DecodeStepArgs st{};
  if (fused) {
    st.q_raw = q; st.k_new = k; st.v_new = v; st.pos = pos;
    st.table = pj.table; st.R = pj.R; st.max_positions = pj.max_positions;
    st.q_norm_w = q_norm_w; st.k_norm_w = k_norm_w; st.norm_eps = norm_eps;
    st.cache_len = pj.cache_len;
  } else if (cudaError_t e = gqa::launch_decode_prep(pj, s); e != cudaSuccess) {
    return cuda_status(e);
  }
  j.q = pj.qrot; j.k_cache = k_cache; j.v_cache = v_cache; j.cache_len = pj.cache_len;
  j.max_cache_len = max_pos + 1; j.out = out;
  j.B = B; j.H = H; j.Hkv = Hkv; j.D = D; j.capacity = capacity; j.window = window;
  j.softcap = softcap > 0.f ? softcap : 0.f;
  j.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
  j.status = status;
  j.skip = skip;
  gqa::decode_split_plan(B, Hkv, max_pos + 1, window, &j.nsplit, &j.chunk);
  j.partial = reinterpret_cast<float*>(ws + lay.part);
  return cuda_status(gqa::launch_decode(j, s, fused ? &st : nullptr));
}

}  // extern "C"
