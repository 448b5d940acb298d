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

// Warps own groups of RPW consecutive rows of x [B, NH, L, D] and load all of
// a group before using any of it, so each warp keeps RPW rows of reads in
// flight. Lane `lane` holds the rotary pairs i = (lane + 32 k) * VEC .. + VEC - 1
// (and their partners i + R/2), and the float2 pairs of the pass-through part
// at R + 2 (lane + 32 k). With k_cache set, the rows are key rows: after their
// rotation they are stored at their cache slots, and the matching value rows
// are copied beside them.
template <int VEC, int RPW, bool APPEND, bool TAIL>
__global__ void __launch_bounds__(256) rope_rows_kernel(RopeJob j) {
  constexpr int NP = 4 / VEC;            // R/2 <= 128  ->  <= 4/VEC vectors per lane
  if (gated_off(j.skip)) return;
  const int lane = threadIdx.x & 31;
  const long warps = (long)gridDim.x * (blockDim.x >> 5);
  const long gwarp = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long rows = (long)j.B * j.NH * j.L;
  const int D = j.D, R = j.R, half = R / 2;
  const int ntail = (D - R) / 2;
  constexpr bool append = APPEND;             // key rows: also store k and v in the cache
  // The norm weights of this lane's dims, loaded once (every row uses the same).
  float wlo[NP * VEC], whi[NP * VEC];
  float2 wtl[TAIL ? 4 : 1];
  if (j.norm_w) {
#pragma unroll
    for (int k = 0; k < NP; ++k) {
      const int i = (lane + 32 * k) * VEC;
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        wlo[k * VEC + e] = i < half ? __ldg(j.norm_w + i + e) : 0.f;
        whi[k * VEC + e] = i < half ? __ldg(j.norm_w + i + half + e) : 0.f;
      }
    }
    if constexpr (TAIL) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int t = lane + 32 * k;
        wtl[k] = t < ntail ? make_float2(__ldg(j.norm_w + R + 2 * t), __ldg(j.norm_w + R + 2 * t + 1))
                           : make_float2(0.f, 0.f);
      }
    }
  }
  // Row indices in 32 bits where they fit (the 64-bit division is a long
  // instruction sequence, paid per row).
  const bool narrow = rows < (1L << 31);
  auto split_row = [&](long row, long& hrow, int& l) {
    if (narrow) {
      const uint32_t rr = static_cast<uint32_t>(row), L = static_cast<uint32_t>(j.L);
      const uint32_t h = rr / L;
      hrow = h;
      l = static_cast<int>(rr - h * L);
    } else {
      hrow = row / j.L;
      l = static_cast<int>(row - hrow * j.L);
    }
  };

  for (long row0 = gwarp * RPW; row0 < rows; row0 += warps * RPW) {
    float lo[RPW][NP * VEC], hi[RPW][NP * VEC];
    float2 cs[RPW][NP * VEC];
    float2 tl[RPW][TAIL ? 4 : 1], vv[RPW][APPEND ? 4 : 1];
    bool live[RPW];
    int pos[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const long row = row0 + r;
      live[r] = row < rows;
      pos[r] = 0;
      if (!live[r]) continue;
      long hrow;
      int l;
      split_row(row, hrow, l);
      const int b = static_cast<int>(narrow ? static_cast<uint32_t>(hrow) / static_cast<uint32_t>(j.NH)
                                            : hrow / j.NH);
      const int s0 = j.start ? j.start[b] : 0;
      // Device-side re-check of the positions the host could not see.
      if (s0 < 0 || (long)s0 + j.L - 1 >= (long)j.max_positions) {
        if (lane == 0 && l == 0) report(j.status, ATTN_DEV_POSITION);
        live[r] = false;
        continue;
      }
      if (append && j.window == 0 && (long)s0 + j.L > (long)j.capacity) {
        if (lane == 0 && l == 0) report(j.status, ATTN_DEV_CAPACITY);
        live[r] = false;
        continue;
      }
      pos[r] = s0 + l;
      const float* x = j.x + row * D;
#pragma unroll
      for (int k = 0; k < NP; ++k) {
        const int i = (lane + 32 * k) * VEC;
        if (i < half) {
          load_vec<VEC>(x + i, lo[r] + k * VEC);
          load_vec<VEC>(x + i + half, hi[r] + k * VEC);
        }
      }
      if (j.table) {
        const float2* tab = j.table + (long)pos[r] * half;
#pragma unroll
        for (int k = 0; k < NP; ++k) {
          const int i = (lane + 32 * k) * VEC;
          if (i < half) {
            if constexpr (VEC == 4) {                // two 16-byte loads (half % 4 == 0)
              const float4 t0 = __ldg(reinterpret_cast<const float4*>(tab + i));
              const float4 t1 = __ldg(reinterpret_cast<const float4*>(tab + i) + 1);
              cs[r][k * 4] = make_float2(t0.x, t0.y);
              cs[r][k * 4 + 1] = make_float2(t0.z, t0.w);
              cs[r][k * 4 + 2] = make_float2(t1.x, t1.y);
              cs[r][k * 4 + 3] = make_float2(t1.z, t1.w);
            } else {
#pragma unroll
              for (int e = 0; e < VEC; ++e) cs[r][k * VEC + e] = tab[i + e];
            }
          }
        }
      }
      if constexpr (TAIL) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int t = lane + 32 * k;
          if (t < ntail) tl[r][k] = *reinterpret_cast<const float2*>(x + R + 2 * t);
        }
      }
      if constexpr (APPEND) {
        const float2* vs = reinterpret_cast<const float2*>(j.v + row * D);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int t = lane + 32 * k;
          if (t < D / 2) vv[r][k] = vs[t];
        }
      }
    }

#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      if (!live[r]) continue;
      const long row = row0 + r;
      if (j.norm_w) {
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < NP; ++k)
          if ((lane + 32 * k) * VEC < half)
#pragma unroll
            for (int e = 0; e < VEC; ++e)
              ss += lo[r][k * VEC + e] * lo[r][k * VEC + e] + hi[r][k * VEC + e] * hi[r][k * VEC + e];
        if constexpr (TAIL) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (lane + 32 * k < ntail) ss += tl[r][k].x * tl[r][k].x + tl[r][k].y * tl[r][k].y;
        }
        ss = warp_sum(ss);
        const float inv_rms = 1.0f / sqrtf(ss / (float)D + j.norm_eps);
#pragma unroll
        for (int k = 0; k < NP; ++k) {
          const int i = (lane + 32 * k) * VEC;
          if (i < half) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              lo[r][k * VEC + e] = lo[r][k * VEC + e] * inv_rms * wlo[k * VEC + e];
              hi[r][k * VEC + e] = hi[r][k * VEC + e] * inv_rms * whi[k * VEC + e];
            }
          }
        }
        if constexpr (TAIL) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int t = lane + 32 * k;
            if (t < ntail) {
              tl[r][k].x = tl[r][k].x * inv_rms * wtl[k].x;
              tl[r][k].y = tl[r][k].y * inv_rms * wtl[k].y;
            }
          }
        }
      }
      if (j.table) {
#pragma unroll
        for (int k = 0; k < NP; ++k) {
          const int i = (lane + 32 * k) * VEC;
          if (i < half) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              const float2 c = cs[r][k * VEC + e];
              const float a = lo[r][k * VEC + e], bb = hi[r][k * VEC + e];
              lo[r][k * VEC + e] = fmaf(a, c.x, -bb * c.y);
              hi[r][k * VEC + e] = fmaf(a, c.y, bb * c.x);
            }
          }
        }
      }
      float* x = (j.y ? j.y : j.x) + row * D;
      // Write back the rotated row (in place or to y) ...
      if (j.table || j.norm_w || j.y) {
#pragma unroll
        for (int k = 0; k < NP; ++k) {
          const int i = (lane + 32 * k) * VEC;
          if (i < half) {
            store_vec<VEC>(x + i, lo[r] + k * VEC);
            store_vec<VEC>(x + i + half, hi[r] + k * VEC);
          }
        }
        if (TAIL && (j.norm_w || j.y)) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int t = lane + 32 * k;
            if (t < ntail) *reinterpret_cast<float2*>(x + R + 2 * t) = tl[r][k];
          }
        }
      }
      // ... and, for key rows, into the cache next to the value row.
      if constexpr (APPEND) {
        long hrow;                                        // b * NH + head
        int l;
        split_row(row, hrow, l);
        // Of a chunk longer than the ring only its last W positions survive;
        // writing the earlier ones would race on the same slots.
        if (j.window > 0 && l < j.L - j.window) continue;
        const long slot = j.window > 0 ? (long)(pos[r] % j.window) : (long)pos[r];
        const long dst = (hrow * j.capacity + slot) * D;
        float* kc = j.k_cache + dst;
#pragma unroll
        for (int k = 0; k < NP; ++k) {
          const int i = (lane + 32 * k) * VEC;
          if (i < half) {
            store_vec<VEC>(kc + i, lo[r] + k * VEC);
            store_vec<VEC>(kc + i + half, hi[r] + k * VEC);
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int t = lane + 32 * k;
          if (t < ntail) *reinterpret_cast<float2*>(kc + R + 2 * t) = tl[r][k];
        }
        float2* vd = reinterpret_cast<float2*>(j.v_cache + dst);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int t = lane + 32 * k;
          if (t < D / 2) vd[t] = vv[r][k];
        }
      }
    }
  }
}

// Rows per warp: 4 for plain rotations, 2 when value rows and tails ride along
// (register budget vs. reads in flight).
template <int VEC>
cudaError_t launch_rows(const RopeJob& j, bool append, bool tail, long blocks,
                        cudaStream_t stream) {
  const unsigned g4 = (unsigned)blocks, g2 = (unsigned)(blocks * 2 < 152L * 8 ? blocks * 2 : 152L * 8);
  if (append)
    rope_rows_kernel<VEC, 2, true, true><<<g2, 256, 0, stream>>>(j);
  else if (tail)
    rope_rows_kernel<VEC, 2, false, true><<<g2, 256, 0, stream>>>(j);
  else
    rope_rows_kernel<VEC, 4, false, false><<<g4, 256, 0, stream>>>(j);
  return cudaGetLastError();
}

cudaError_t launch_rope_rows(const RopeJob& j, cudaStream_t stream) {
  const int half = j.R / 2;
  const long rows = (long)j.B * j.NH * j.L;
  if (rows == 0) return cudaSuccess;
  const int threads = 256, wpb = threads / 32;
  long blocks = (rows + wpb * 4 - 1) / (wpb * 4);
  const long cap = 152L * 8;                    // one full wave of 8 blocks per SM
  if (blocks > cap) blocks = cap;
  const bool append = j.k_cache != nullptr;
  // dims past R read only where there are any (the norm over full rotary needs none)
  const bool tail = append || (j.R < j.D && (j.norm_w != nullptr || j.y != nullptr));
  if (half % 4 == 0 && half >= 128)
    return launch_rows<4>(j, append, tail, blocks, stream);
  if (half % 2 == 0) return launch_rows<2>(j, append, tail, blocks, stream);
  return launch_rows<1>(j, append, tail, blocks, stream);
}

}  // namespace gqa
