// RoPE table, q/k RMSNorm + RoPE, and the fused K rotation + KV-cache append.
//
// Rotary position embedding follows "Core Layers -- Deep Reference", section
// "RoPE": the pair (a, b) at position p turns by p * theta_i. Pairs are
// rotate-half (i, i + R/2) and dims R..D-1 pass through (partial rotary,
// "mojolearn.transformer" rope_dim). RMSNorm ("Core Layers -- Deep Reference",
// "RMSNorm") runs before the rotation ("mojolearn.transformer", qk_norm).
// The cache rules are those of "mojolearn.transformer", TransformerState:
// slot = position, or position mod W in a ring of W slots.
//
// These passes are HBM-bound elementwise work: one warp per head row, with
// every access coalesced across the warp.
#include "common.cuh"
#include "kernels.h"

namespace gqa {

// table[pos][i] = (cos, sin)(pos * theta_i): angle and both functions in fp64,
// one rounding to fp32 at the end.
__global__ void rope_table_kernel(InvFreq inv, int half, int max_positions, float2* table) {
  const long n = (long)max_positions * half;
  for (long t = blockIdx.x * (long)blockDim.x + threadIdx.x; t < n;
       t += (long)gridDim.x * blockDim.x) {
    const int pos = (int)(t / half);
    const int i = (int)(t % half);
    const double ang = (double)pos * inv.v[i];
    double sn, cs;
    sincos(ang, &sn, &cs);
    table[t] = make_float2((float)cs, (float)sn);
  }
}

cudaError_t launch_rope_table(const InvFreq& inv, int R, int max_positions, float2* table,
                              cudaStream_t stream) {
  const int half = R / 2;
  const long n = (long)max_positions * half;
  const int threads = 256;
  const long blocks = (n + threads - 1) / threads;
  rope_table_kernel<<<(unsigned)(blocks < 65535 * 8 ? blocks : 65535 * 8), threads, 0, stream>>>(
      inv, half, max_positions, table);
  return cudaGetLastError();
}

template <int VEC>
struct VecT;
template <>
struct VecT<1> { using T = float; };
template <>
struct VecT<2> { using T = float2; };
template <>
struct VecT<4> { using T = float4; };

template <int VEC>
__device__ __forceinline__ void load_vec(const float* p, float* r) {
  using T = typename VecT<VEC>::T;
  T t = *reinterpret_cast<const T*>(p);
  const float* f = reinterpret_cast<const float*>(&t);
#pragma unroll
  for (int e = 0; e < VEC; ++e) r[e] = f[e];
}

template <int VEC>
__device__ __forceinline__ void store_vec(float* p, const float* r) {
  using T = typename VecT<VEC>::T;
  T t;
  float* f = reinterpret_cast<float*>(&t);
#pragma unroll
  for (int e = 0; e < VEC; ++e) f[e] = r[e];
  *reinterpret_cast<T*>(p) = t;
}

// One warp per row of x [B, NH, L, D]. Lane `lane` holds the rotary pairs
// i = (lane + 32 k) * VEC .. + VEC - 1 (and their partners i + R/2), and the
// float2 pairs of the pass-through part at R + 2 (lane + 32 k).
// With k_cache set, the row is a key row: after its rotation it is stored at
// its cache slot, and the matching value row is copied beside it.
template <int VEC>
__global__ void __launch_bounds__(256) rope_rows_kernel(RopeJob j) {
  constexpr int NP = 4 / VEC;            // R/2 <= 128  ->  <= 4/VEC vectors per lane
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const long rows = (long)j.B * j.NH * j.L;
  const int D = j.D, R = j.R, half = R / 2;
  const int ntail = (D - R) / 2;
  const bool append = j.k_cache != nullptr;
  const bool need_tail = append || j.norm_w != nullptr;

  for (long row = (long)blockIdx.x * wpb + (threadIdx.x >> 5); row < rows;
       row += (long)gridDim.x * wpb) {
    const int b = (int)(row / ((long)j.NH * j.L));
    const int l = (int)(row % j.L);
    const int s0 = j.start[b];
    // Device-side re-check of the positions the host could not see.
    if (s0 < 0 || (long)s0 + j.L - 1 >= (long)j.max_positions) {
      if (lane == 0 && l == 0) report(j.status, ATTN_DEV_POSITION);
      continue;
    }
    if (append && j.window == 0 && (long)s0 + j.L > (long)j.capacity) {
      if (lane == 0 && l == 0) report(j.status, ATTN_DEV_CAPACITY);
      continue;
    }
    const int p = s0 + l;
    float* x = j.x + row * D;

    float lo[NP * VEC], hi[NP * VEC];
    float2 tl[4];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < NP; ++k) {
      const int i = (lane + 32 * k) * VEC;
      if (i < half) {
        load_vec<VEC>(x + i, lo + k * VEC);
        load_vec<VEC>(x + i + half, hi + k * VEC);
#pragma unroll
        for (int e = 0; e < VEC; ++e)
          ss += lo[k * VEC + e] * lo[k * VEC + e] + hi[k * VEC + e] * hi[k * VEC + e];
      }
    }
    if (need_tail) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int t = lane + 32 * k;
        if (t < ntail) {
          tl[k] = *reinterpret_cast<const float2*>(x + R + 2 * t);
          ss += tl[k].x * tl[k].x + tl[k].y * tl[k].y;
        }
      }
    }

    if (j.norm_w) {
      ss = warp_sum(ss);
      const float inv_rms = 1.0f / sqrtf(ss / (float)D + j.norm_eps);
#pragma unroll
      for (int k = 0; k < NP; ++k) {
        const int i = (lane + 32 * k) * VEC;
        if (i < half) {
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            lo[k * VEC + e] = lo[k * VEC + e] * inv_rms * j.norm_w[i + e];
            hi[k * VEC + e] = hi[k * VEC + e] * inv_rms * j.norm_w[i + half + e];
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int t = lane + 32 * k;
        if (t < ntail) {
          tl[k].x = tl[k].x * inv_rms * j.norm_w[R + 2 * t];
          tl[k].y = tl[k].y * inv_rms * j.norm_w[R + 2 * t + 1];
        }
      }
    }

    if (j.table) {
      const float2* tab = j.table + (long)p * half;
#pragma unroll
      for (int k = 0; k < NP; ++k) {
        const int i = (lane + 32 * k) * VEC;
        if (i < half) {
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            const float2 cs = tab[i + e];
            const float a = lo[k * VEC + e], bb = hi[k * VEC + e];
            lo[k * VEC + e] = fmaf(a, cs.x, -bb * cs.y);
            hi[k * VEC + e] = fmaf(a, cs.y, bb * cs.x);
          }
        }
      }
    }

    // Write back the rotated row (in place) ...
    if (j.table || j.norm_w) {
#pragma unroll
      for (int k = 0; k < NP; ++k) {
        const int i = (lane + 32 * k) * VEC;
        if (i < half) {
          store_vec<VEC>(x + i, lo + k * VEC);
          store_vec<VEC>(x + i + half, hi + k * VEC);
        }
      }
      if (j.norm_w) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int t = lane + 32 * k;
          if (t < ntail) *reinterpret_cast<float2*>(x + R + 2 * t) = tl[k];
        }
      }
    }

    // ... and, for key rows, into the cache next to the value row.
    if (append) {
      // Of a chunk longer than the ring only its last W positions survive;
      // writing the earlier ones would race on the same slots.
      if (j.window > 0 && l < j.L - j.window) continue;
      const long slot = j.window > 0 ? (long)(p % j.window) : (long)p;
      const long hrow = row / j.L;                      // b * NH + head
      const long dst = (hrow * j.capacity + slot) * D;
      float* kc = j.k_cache + dst;
#pragma unroll
      for (int k = 0; k < NP; ++k) {
        const int i = (lane + 32 * k) * VEC;
        if (i < half) {
          store_vec<VEC>(kc + i, lo + k * VEC);
          store_vec<VEC>(kc + i + half, hi + k * VEC);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int t = lane + 32 * k;
        if (t < ntail) *reinterpret_cast<float2*>(kc + R + 2 * t) = tl[k];
      }
      const float2* vs = reinterpret_cast<const float2*>(j.v + row * D);
      float2* vd = reinterpret_cast<float2*>(j.v_cache + dst);
      for (int t = lane; t < D / 2; t += 32) vd[t] = vs[t];
    }
  }
}

cudaError_t launch_rope_rows(const RopeJob& j, cudaStream_t stream) {
  const int half = j.R / 2;
  const long rows = (long)j.B * j.NH * j.L;
  if (rows == 0) return cudaSuccess;
  const int threads = 256, wpb = threads / 32;
  long blocks = (rows + wpb - 1) / wpb;
  const long cap = 152L * 16;                   // up to 16 resident blocks per SM
  if (blocks > cap) blocks = cap;
  if (half % 4 == 0 && half >= 128)
    rope_rows_kernel<4><<<(unsigned)blocks, threads, 0, stream>>>(j);
  else if (half % 2 == 0)
    rope_rows_kernel<2><<<(unsigned)blocks, threads, 0, stream>>>(j);
  else
    rope_rows_kernel<1><<<(unsigned)blocks, threads, 0, stream>>>(j);
  return cudaGetLastError();
}

}  // namespace gqa
