// The "identical" numeric mode ("mojolearn.transformer", TransformerBlock:
// numeric_mode 'identical'; in that mode decoding token by token, or a prefill
// continued from a carried cache, gives the same bits as one prefill over the
// whole sequence).
//
// One kernel serves all three calls, so the arithmetic is the same machine
// code whichever call runs it. A warp owns one query row (b, h, position p)
// and does, in a fixed order that depends only on p and on the visible key
// positions:
//   s_m  = scale * (q . k_m): lane t accumulates dims t, t + 32, ... with fmaf,
//          then an xor butterfly adds the 32 partial sums (each step adds two
//          values in either order, so every lane holds the same bits);
//          softcap: c * tanh(s_m / c);
//   M    = max over the visible m (exact, so order-free);
//   l, o = sums over m in ascending position order of w_m = exp(s_m - M) and
//          w_m v_m (fmaf per dim);
//   out  = o / l.
// Key and value rows come from the caller's chunk (positions start[b] ..) or,
// below the chunk, from the cache (slot = position, or position mod window for
// a ring): the cache holds the same bits kv_cache_append wrote for those rows.
// Explicit _rn operations keep the compiler from contracting or reordering.
// Slow by design (scores computed twice, CUDA cores): a reproducibility mode.
#include "common.cuh"
#include "kernels.h"

namespace gqa {

namespace {

constexpr int kWarps = 4;

__global__ void __launch_bounds__(kWarps * 32) identical_attn_kernel(IdentJob j) {
  if (gated_off(j.skip)) return;
  const int lane = threadIdx.x & 31;
  const long rows = static_cast<long>(j.B) * j.H * j.L;
  const long nwarps = static_cast<long>(gridDim.x) * kWarps;
  const int G = j.H / j.Hkv;
  for (long row = static_cast<long>(blockIdx.x) * kWarps + threadIdx.x / 32; row < rows;
       row += nwarps) {
    const int l = static_cast<int>(row % j.L);
    const long bh = row / j.L;
    const int h = static_cast<int>(bh % j.H), b = static_cast<int>(bh / j.H);
    const long kvh = static_cast<long>(b) * j.Hkv + h / G;
    // The query's position p and the first position held by the chunk (s0).
    int p, s0;
    if (j.cache_len) {                          // decode: every key is in the cache
      const int n = j.cache_len[b];
      if (n < 1 || n > j.max_len || (j.window == 0 && n > j.capacity)) {
        if (lane == 0 && h == 0) report(j.status, ATTN_DEV_LENGTH);
        continue;
      }
      p = n - 1;
      s0 = n;
    } else {
      s0 = j.start ? j.start[b] : 0;
      if (s0 < 0 || s0 > j.max_start || (j.k_cache && j.window == 0 && s0 > j.capacity)) {
        if (lane == 0 && h == 0 && l == 0)
          report(j.status, s0 < 0 || s0 > j.max_start ? ATTN_DEV_POSITION : ATTN_DEV_CAPACITY);
        continue;
      }
      p = s0 + l;
    }
    int lo = j.window > 0 ? max(0, p - j.window + 1) : 0;
    if (!j.k_cache) lo = max(lo, s0);           // no cache: the chunk's own keys only
    auto key_row = [&](int m, bool value) -> const float* {
      if (m >= s0)
        return (value ? j.v : j.k) + (kvh * j.L + (m - s0)) * j.D;
      const long slot = j.window > 0 ? m % j.window : m;
      return (value ? j.v_cache : j.k_cache) + (kvh * j.capacity + slot) * j.D;
    };
    float qv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int d = lane + 32 * i;
      qv[i] = d < j.D ? j.q[row * j.D + d] : 0.f;
    }
    auto score = [&](int m) -> float {
      const float* kp = key_row(m, false);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int d = lane + 32 * i;
        if (d < j.D) acc = fmaf(qv[i], kp[d], acc);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
      float s = __fmul_rn(acc, j.scale);
      if (j.softcap > 0.f) s = __fmul_rn(j.softcap, tanhf(__fdiv_rn(s, j.softcap)));
      return s;
    };
    float M = -INFINITY;
    for (int m = lo; m <= p; ++m) M = fmaxf(M, score(m));
    float lsum = 0.f, o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = 0.f;
    for (int m = lo; m <= p; ++m) {
      const float w = expf(__fsub_rn(score(m), M));
      lsum = __fadd_rn(lsum, w);
      const float* vp = key_row(m, true);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int d = lane + 32 * i;
        if (d < j.D) o[i] = fmaf(w, vp[d], o[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int d = lane + 32 * i;
      if (d < j.D) j.out[row * j.D + d] = __fdiv_rn(o[i], lsum);
    }
  }
}

}  // namespace

cudaError_t launch_identical(const IdentJob& j, cudaStream_t stream) {
  const long rows = static_cast<long>(j.B) * j.H * j.L;
  if (rows == 0) return cudaSuccess;
  long blocks = (rows + kWarps - 1) / kWarps;
  if (blocks > 152L * 16) blocks = 152L * 16;
  identical_attn_kernel<<<static_cast<unsigned>(blocks), kWarps * 32, 0, stream>>>(j);
  return cudaGetLastError();
}

}  // namespace gqa
