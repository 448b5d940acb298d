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
// A block takes 32 consecutive rows of one (b, kv head): both 32 x D tiles go
// through shared memory (rows padded to an odd number of floats so that the
// column reads of the transpose hit distinct banks); one warp rotates a key row
// at a time, and V^T rows of 32 keys are 128-byte stores.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace gqa {

namespace {

constexpr int kStepRows = 32;
constexpr int kStepThreads = 256;

__global__ void __launch_bounds__(kStepThreads) append_vt_kernel(AppendVtJob j) {
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

cudaError_t launch_append_vt(const AppendVtJob& j, cudaStream_t stream) {
  if (!append_vt_supports(j.D) || j.L < 1 || j.B < 1) return cudaErrorInvalidValue;
  if (static_cast<long>(j.B) * j.Hkv > 65535) return cudaErrorInvalidValue;
  const int smem = 2 * kStepRows * (j.D + 1) * static_cast<int>(sizeof(float));
  if (smem > 48 * 1024) {
    // the larger dynamic shared memory is allowed once per device
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
      if (cudaError_t e = cudaFuncSetAttribute(append_vt_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               2 * kStepRows * (kMaxHeadDim + 1) * 4);
          e != cudaSuccess)
        return e;
      done[dev] = true;
    }
  }
  const dim3 grid((j.L + kStepRows - 1) / kStepRows, j.B * j.Hkv);
  append_vt_kernel<<<grid, kStepThreads, smem, stream>>>(j);
  return cudaGetLastError();
}

}  // namespace gqa
