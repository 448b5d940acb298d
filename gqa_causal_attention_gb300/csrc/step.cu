// The memory pass of a whole prefill step ("mojolearn.transformer",
// TransformerBlock.forward from a fresh state: the chunk's keys and values
// enter the cache, then attention runs over them).
//
// One pass reads k and v once and writes everything the attention and the
// cache need: k after RMSNorm and RoPE into its cache slots (and into a
// workspace copy when the cache is a ring too short to hold every key), v into
// its cache slots, and v transposed (V^T, the K-major operand of the tensor
// core's P V product) into the workspace. k and v themselves are only read.
// The tensor-core prefill then reads the rotated keys straight from the cache.
// kv_cache_append uses the same pass with the rotated keys written back over k
// (every row of a tile is in shared memory before any is written) and no V^T.
//
// Head dims 64, 128 and 256 (append_vt_pow2_kernel): a tile is 32 consecutive
// rows of one (b, kv head). Both 32 x D tiles go through shared memory as
// 16-byte units, unit u of row r stored at position u ^ (r mod 32) of its row,
// so that a warp's 16-byte stores of a row and its 16-byte column reads (one
// unit of 32 rows) both spread over all banks. V^T: lane r reads unit u of key
// r (dims 4u..4u+3) and writes four V^T rows of 32 keys, 128 bytes each; one
// warp rotates a key row at a time. The grid is one wave of resident blocks,
// each walking tiles with a stride of the grid; the next tile's k and v are
// loaded into registers while the current one is written, so every block keeps
// its loads in flight through the whole pass.
// Other head dims (append_vt_any_kernel): one block per tile, rows padded to an
// odd number of floats, scalar transposes.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace gqa {

namespace {

constexpr int kStepRows = 32;
constexpr int kStepThreads = 256;

// Rotated (and normalised) keys of row r of the tile into the cache slot and kr.
// x(i) reads element i of the row from shared memory.
template <class X>
__device__ __forceinline__ void rotate_key_row(const AppendVtJob& j, const X& x, int D, int lane,
                                               int pos, float* kc, float* kr) {
  const int R = j.R, half = R / 2;
  float inv = 1.0f;
  if (j.norm_w) {
    float ss = 0.f;
    for (int i = lane; i < D; i += 32) ss = fmaf(x(i), x(i), ss);
    ss = warp_sum(ss);
    inv = 1.0f / sqrtf(ss / static_cast<float>(D) + j.norm_eps);
  }
  const float2* tab = j.table ? j.table + static_cast<long>(pos) * half : nullptr;
  for (int i = lane; i < half; i += 32) {
    float a = x(i), c = x(i + half);
    if (j.norm_w) {
      a = a * inv * j.norm_w[i];
      c = c * inv * j.norm_w[i + half];
    }
    const float2 cs = tab ? tab[i] : make_float2(1.f, 0.f);
    const float y0 = fmaf(a, cs.x, -c * cs.y);
    const float y1 = fmaf(a, cs.y, c * cs.x);
    if (kc) {
      kc[i] = y0;
      kc[i + half] = y1;
    }
    if (kr) {
      kr[i] = y0;
      kr[i + half] = y1;
    }
  }
  for (int i = R + lane; i < D; i += 32) {
    const float y = j.norm_w ? x(i) * inv * j.norm_w[i] : x(i);
    if (kc) kc[i] = y;
    if (kr) kr[i] = y;
  }
}

// Threads per block of the head-dim-D pass: 8 warps up to D = 128, 16 at D = 256
// (four 16-byte units of k and of v per thread and tile either way).
template <int D>
__host__ __device__ constexpr int pow2_threads() { return D > 128 ? 512 : 256; }

template <int D>
__global__ void __launch_bounds__(pow2_threads<D>(), D > 128 ? 2 : 4) append_vt_pow2_kernel(AppendVtJob j) {
  constexpr int kThreads = pow2_threads<D>();
  constexpr int D4 = D / 4;                                  // 16-byte units per row
  constexpr int NV = kStepRows * D4 / kThreads;              // units per thread per tensor
  constexpr int SW = D4 < 32 ? D4 : 32;                      // unit u of row r at u ^ (r % SW)
  static_assert(D4 % 8 == 0 && NV >= 1, "head dims 32 x 2^n");
  extern __shared__ float4 sm4[];
  if (gated_off(j.skip)) return;
  float4* ks = sm4;
  float4* vs = sm4 + kStepRows * D4;
  __shared__ float inv_row[kStepRows];                       // 1 / rms of each key row
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  // 32-bit tile indices (the host bounds the tile count below 2^31).
  const int tph = (j.L + kStepRows - 1) / kStepRows;        // tiles per (b, kv head)
  const int ntiles = tph * j.B * j.Hkv;
  auto at = [](int r, int u) { return r * D4 + (u ^ (r % SW)); };
  float4 pk[NV], pv[NV];
  auto fetch = [&](int t) {
    const int bh = t / tph;
    const int l0 = (t - bh * tph) * kStepRows;
    const int nv = min(kStepRows, j.L - l0) * D4;
    const long src0 = (static_cast<long>(bh) * j.L + l0) * D4;   // in 16-byte units
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = tid + i * kThreads;
      if (e < nv) {
        pk[i] = __ldg(reinterpret_cast<const float4*>(j.k) + src0 + e);
        pv[i] = __ldg(reinterpret_cast<const float4*>(j.v) + src0 + e);
      }
    }
  };
  // Of a chunk longer than the ring only its last W positions are stored (the
  // earlier ones would land on the same slots).
  const int first_kept = j.window > 0 ? j.L - j.window : 0;

  int t = blockIdx.x;
  if (t < ntiles) fetch(t);
  for (; t < ntiles; t += gridDim.x) {
    const int bh = t / tph;
    const int b = bh / j.Hkv;
    const int l0 = (t - bh * tph) * kStepRows;
    const int rows = min(kStepRows, j.L - l0);
    const int nv = rows * D4;
    __syncthreads();                                         // the previous tile is written out
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = tid + i * kThreads;
      if (e < nv) {
        ks[at(e / D4, e % D4)] = pk[i];
        vs[at(e / D4, e % D4)] = pv[i];
      }
    }
    __syncthreads();
    if (t + gridDim.x < ntiles) fetch(t + gridDim.x);        // in flight while this tile is written
    const int s0 = j.start ? j.start[b] : 0;
    // Device-side re-check of the positions the host could not see (block-uniform).
    if (s0 < 0 || static_cast<long>(s0) + j.L - 1 >= static_cast<long>(j.max_positions)) {
      if (tid == 0 && l0 == 0 && bh % j.Hkv == 0) report(j.status, ATTN_DEV_POSITION);
      continue;
    }
    if (j.window == 0 && static_cast<long>(s0) + j.L > static_cast<long>(j.capacity)) {
      if (tid == 0 && l0 == 0 && bh % j.Hkv == 0) report(j.status, ATTN_DEV_CAPACITY);
      continue;
    }
    auto slot_of = [&](int l) -> long {
      const long p = static_cast<long>(s0) + l;
      return j.window > 0 ? p % j.window : p;
    };
    // values: cache rows, 16-byte stores
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = tid + i * kThreads;
      const int r = e / D4, u = e % D4;
      if (e < nv && l0 + r >= first_kept)
        reinterpret_cast<float4*>(j.v_cache)[(static_cast<long>(bh) * j.capacity + slot_of(l0 + r)) *
                                                 D4 + u] = vs[at(r, u)];
    }
    // V^T: lane = key, four rows of 32 keys per unit
    if (j.vt && lane < rows) {
#pragma unroll
      for (int u = warp; u < D4; u += kThreads / 32) {
        const float4 x = vs[at(lane, u)];
        float* dst = j.vt + (static_cast<long>(bh) * D + 4 * u) * j.vt_pitch + l0 + lane;
        dst[0] = x.x;
        dst[j.vt_pitch] = x.y;
        dst[2 * j.vt_pitch] = x.z;
        dst[3 * j.vt_pitch] = x.w;
      }
    }
    // keys: RMSNorm (optional) then RoPE
    if (j.R % 8 == 0) {
      // 16-byte units: item k < hu rotates units k and k + hu (pairs 4k..4k+3),
      // item k >= hu passes unit k + hu (dims past R) through the norm only.
      const int hu = j.R / 8, ni = D4 - hu, half = j.R / 2;
      if (j.norm_w) {
        for (int r = warp; r < rows; r += kThreads / 32) {
          float ss = 0.f;
#pragma unroll
          for (int u = lane; u < D4; u += 32) {
            const float4 x = ks[at(r, u)];
            ss = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, ss))));
          }
          ss = warp_sum(ss);
          if (lane == 0) inv_row[r] = 1.0f / sqrtf(ss / static_cast<float>(D) + j.norm_eps);
        }
        __syncthreads();
      }
      const float4* w4 = reinterpret_cast<const float4*>(j.norm_w);
      for (int idx = tid; idx < rows * ni; idx += kThreads) {
        const int r = idx / ni, k = idx - r * ni;
        const int l = l0 + r;
        float4* kc = l >= first_kept ? reinterpret_cast<float4*>(
                                           j.k_cache + (static_cast<long>(bh) * j.capacity + slot_of(l)) * D)
                                     : nullptr;
        float4* kr = j.kr ? reinterpret_cast<float4*>(j.kr + (static_cast<long>(bh) * j.L + l) * D)
                          : nullptr;
        const float inv = j.norm_w ? inv_row[r] : 1.0f;
        if (k < hu) {
          float4 a = ks[at(r, k)], c = ks[at(r, k + hu)];
          if (j.norm_w) {
            const float4 wa = __ldg(w4 + k), wc = __ldg(w4 + k + hu);
            a = make_float4(a.x * inv * wa.x, a.y * inv * wa.y, a.z * inv * wa.z, a.w * inv * wa.w);
            c = make_float4(c.x * inv * wc.x, c.y * inv * wc.y, c.z * inv * wc.z, c.w * inv * wc.w);
          }
          float4 t0 = make_float4(1.f, 0.f, 1.f, 0.f), t1 = t0;   // (cos, sin) of pairs 4k..4k+3
          if (j.table) {
            const float4* tb =
                reinterpret_cast<const float4*>(j.table + static_cast<long>(s0 + l) * half + 4 * k);
            t0 = __ldg(tb);
            t1 = __ldg(tb + 1);
          }
          const float4 y0 = make_float4(fmaf(a.x, t0.x, -c.x * t0.y), fmaf(a.y, t0.z, -c.y * t0.w),
                                        fmaf(a.z, t1.x, -c.z * t1.y), fmaf(a.w, t1.z, -c.w * t1.w));
          const float4 y1 = make_float4(fmaf(a.x, t0.y, c.x * t0.x), fmaf(a.y, t0.w, c.y * t0.z),
                                        fmaf(a.z, t1.y, c.z * t1.x), fmaf(a.w, t1.w, c.w * t1.z));
          if (kc) {
            kc[k] = y0;
            kc[k + hu] = y1;
          }
          if (kr) {
            kr[k] = y0;
            kr[k + hu] = y1;
          }
        } else {
          const int u = k + hu;
          float4 x = ks[at(r, u)];
          if (j.norm_w) {
            const float4 wx = __ldg(w4 + u);
            x = make_float4(x.x * inv * wx.x, x.y * inv * wx.y, x.z * inv * wx.z, x.w * inv * wx.w);
          }
          if (kc) kc[u] = x;
          if (kr) kr[u] = x;
        }
      }
    } else {
      // one warp per row, scalar pairs
      const float* kf = reinterpret_cast<const float*>(ks);
      for (int r = warp; r < rows; r += kThreads / 32) {
        const int l = l0 + r;
        float* kc = l >= first_kept
                        ? j.k_cache + (static_cast<long>(bh) * j.capacity + slot_of(l)) * D
                        : nullptr;
        float* kr = j.kr ? j.kr + (static_cast<long>(bh) * j.L + l) * D : nullptr;
        auto x = [&](int i) { return kf[4 * at(r, i / 4) + i % 4]; };
        rotate_key_row(j, x, D, lane, s0 + l, kc, kr);
      }
    }
  }
}

__global__ void __launch_bounds__(kStepThreads) append_vt_any_kernel(AppendVtJob j) {
  extern __shared__ float sm[];
  if (gated_off(j.skip)) return;
  const int D = j.D, S = D + 1;
  float* ks = sm;
  float* vs = sm + kStepRows * S;
  const int bh = blockIdx.y;
  const int b = bh / j.Hkv;
  const int l0 = blockIdx.x * kStepRows;
  const int rows = min(kStepRows, j.L - l0);
  const int s0 = j.start ? j.start[b] : 0;
  // Device-side re-check of the positions the host could not see.
  if (s0 < 0 || static_cast<long>(s0) + j.L - 1 >= static_cast<long>(j.max_positions)) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && bh % j.Hkv == 0) report(j.status, ATTN_DEV_POSITION);
    return;
  }
  if (j.window == 0 && static_cast<long>(s0) + j.L > static_cast<long>(j.capacity)) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && bh % j.Hkv == 0) report(j.status, ATTN_DEV_CAPACITY);
    return;
  }
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const long src0 = (static_cast<long>(bh) * j.L + l0) * D;
  const int nv = rows * (D / 4);
  for (int e = tid; e < nv; e += kStepThreads) {
    const int r = e / (D / 4), c = 4 * (e % (D / 4));
    const float4 kk = __ldg(reinterpret_cast<const float4*>(j.k + src0 + static_cast<long>(r) * D + c));
    const float4 vv = __ldg(reinterpret_cast<const float4*>(j.v + src0 + static_cast<long>(r) * D + c));
    float* kd = ks + r * S + c;
    float* vd = vs + r * S + c;
    kd[0] = kk.x; kd[1] = kk.y; kd[2] = kk.z; kd[3] = kk.w;
    vd[0] = vv.x; vd[1] = vv.y; vd[2] = vv.z; vd[3] = vv.w;
  }
  __syncthreads();

  // Of a chunk longer than the ring only its last W positions are stored (the
  // earlier ones would land on the same slots).
  const int first_kept = j.window > 0 ? j.L - j.window : 0;
  auto slot_of = [&](int l) -> long {
    const long p = static_cast<long>(s0) + l;
    return j.window > 0 ? p % j.window : p;
  };

  // values: cache rows, 16-byte stores
  for (int e = tid; e < nv; e += kStepThreads) {
    const int r = e / (D / 4), c = 4 * (e % (D / 4));
    const int l = l0 + r;
    if (l < first_kept) continue;
    const float* vr = vs + r * S + c;
    *reinterpret_cast<float4*>(j.v_cache + (static_cast<long>(bh) * j.capacity + slot_of(l)) * D +
                               c) = make_float4(vr[0], vr[1], vr[2], vr[3]);
  }
  // V^T rows: 32 keys of dim d, one 128-byte store per warp
  if (j.vt) {
    for (int d = warp; d < D; d += kStepThreads / 32) {
      if (lane < rows)
        j.vt[(static_cast<long>(bh) * D + d) * j.vt_pitch + l0 + lane] = vs[lane * S + d];
    }
  }
  // keys: RMSNorm (optional) then RoPE, one warp per row
  const int R = j.R, half = R / 2;
  for (int r = warp; r < rows; r += kStepThreads / 32) {
    const int l = l0 + r;
    const int pos = s0 + l;
    const float* x = ks + r * S;
    float inv = 1.0f;
    if (j.norm_w) {
      float ss = 0.f;
      for (int i = lane; i < D; i += 32) ss = fmaf(x[i], x[i], ss);
      ss = warp_sum(ss);
      inv = 1.0f / sqrtf(ss / static_cast<float>(D) + j.norm_eps);
    }
    const bool keep = l >= first_kept;
    float* kc = keep ? j.k_cache + (static_cast<long>(bh) * j.capacity + slot_of(l)) * D : nullptr;
    float* kr = j.kr ? j.kr + (static_cast<long>(bh) * j.L + l) * D : nullptr;
    const float2* tab = j.table ? j.table + static_cast<long>(pos) * half : nullptr;
    for (int i = lane; i < half; i += 32) {
      float a = x[i], c = x[i + half];
      if (j.norm_w) {
        a = a * inv * j.norm_w[i];
        c = c * inv * j.norm_w[i + half];
      }
      const float2 cs = tab ? tab[i] : make_float2(1.f, 0.f);
      const float y0 = fmaf(a, cs.x, -c * cs.y);
      const float y1 = fmaf(a, cs.y, c * cs.x);
      if (kc) {
        kc[i] = y0;
        kc[i + half] = y1;
      }
      if (kr) {
        kr[i] = y0;
        kr[i + half] = y1;
      }
    }
    for (int i = R + lane; i < D; i += 32) {
      const float y = j.norm_w ? x[i] * inv * j.norm_w[i] : x[i];
      if (kc) kc[i] = y;
      if (kr) kr[i] = y;
    }
  }
}

}  // namespace

bool append_vt_supports(int D) { return D % 4 == 0 && D >= 4 && D <= kMaxHeadDim; }

namespace {

template <int D>
cudaError_t launch_pow2(const AppendVtJob& j, cudaStream_t stream) {
  // Per device and context: the dynamic shared memory allowed, and the grid of
  // one wave (SMs x resident blocks); a CUDA error as its negative code.
  constexpr int smem = 2 * kStepRows * D * static_cast<int>(sizeof(float));
  static PerContext<int> wave;
  int grid = wave.get(
      [] {
        if (smem > 48 * 1024) {
          if (cudaError_t e = cudaFuncSetAttribute(append_vt_pow2_kernel<D>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   smem);
              e != cudaSuccess)
            return -static_cast<int>(e);
        }
        int dev = 0, sms = 0, per_sm = 0;
        if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return -static_cast<int>(e);
        if (cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            e != cudaSuccess)
          return -static_cast<int>(e);
        if (cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &per_sm, append_vt_pow2_kernel<D>, pow2_threads<D>(), smem);
            e != cudaSuccess)
          return -static_cast<int>(e);
        return sms * (per_sm > 0 ? per_sm : 1);
      },
      -static_cast<int>(cudaErrorInvalidDevice), [](int g) { return g > 0; });
  if (grid <= 0) return static_cast<cudaError_t>(-grid);
  const long ntiles = static_cast<long>((j.L + kStepRows - 1) / kStepRows) * j.B * j.Hkv;
  if (ntiles + grid > 0x7fffffffL) return cudaErrorInvalidValue;   // 32-bit tile indices
  if (ntiles < grid) grid = static_cast<int>(ntiles);
  append_vt_pow2_kernel<D><<<grid, pow2_threads<D>(), smem, stream>>>(j);
  return cudaGetLastError();
}

cudaError_t launch_any(const AppendVtJob& j, cudaStream_t stream) {
  if (static_cast<long>(j.B) * j.Hkv > 65535) return cudaErrorInvalidValue;
  const int smem = 2 * kStepRows * (j.D + 1) * static_cast<int>(sizeof(float));
  if (smem > 48 * 1024) {
    // the larger dynamic shared memory is allowed once per device and context
    static PerContext<cudaError_t> attr;
    if (const cudaError_t e = attr.get(
            [] {
              return cudaFuncSetAttribute(append_vt_any_kernel,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          2 * kStepRows * (kMaxHeadDim + 1) * 4);
            },
            cudaErrorInvalidDevice, [](cudaError_t r) { return r == cudaSuccess; });
        e != cudaSuccess)
      return e;
  }
  const dim3 grid((j.L + kStepRows - 1) / kStepRows, j.B * j.Hkv);
  append_vt_any_kernel<<<grid, kStepThreads, smem, stream>>>(j);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append_vt(const AppendVtJob& j, cudaStream_t stream) {
  if (!append_vt_supports(j.D) || j.L < 1 || j.B < 1 || j.Hkv < 1) return cudaErrorInvalidValue;
  switch (j.D) {
    case 64: return launch_pow2<64>(j, stream);
    case 128: return launch_pow2<128>(j, stream);
    case 256: return launch_pow2<256>(j, stream);
    default: return launch_any(j, stream);
  }
}

}  // namespace gqa
