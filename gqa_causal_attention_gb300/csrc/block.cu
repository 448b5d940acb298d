// The decoder block around the attention ("mojolearn.transformer",
// TransformerBlock.forward with state None, computing Hugging Face's
// LlamaDecoderLayer.forward): the memory-bound pieces around the tensor-core
// projections of gemm_tc.cu -- RMSNorm of token rows and, for head dims that
// the projection kernel cannot read head-major, the token-major <-> head-major
// permute. Activations are token-major [B * L, width] as the pages' (B, L,
// d_model) input.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace gqa {

namespace {

// RMSNorm of each row of x [T, n] ("Core Layers -- Deep Reference", RMSNorm):
// y = x / sqrt(mean x^2 + eps) * (w, or 1 + w). One warp per row; 16-byte
// accesses when n % 4 == 0. With round_out the results are rounded to the
// nearest TF32 value (the projections read only those bits).
__global__ void __launch_bounds__(256) rmsnorm_rows_kernel(const float* __restrict__ x,
                                                           const float* __restrict__ w,
                                                           float* __restrict__ y, long T, int n,
                                                           float eps, int offset, int round_out,
                                                           const int32_t* skip) {
  if (gated_off(skip)) return;
  const int lane = threadIdx.x & 31;
  const long nw = static_cast<long>(gridDim.x) * 8;
  const bool vec = (n % 4) == 0;
  for (long row = static_cast<long>(blockIdx.x) * 8 + threadIdx.x / 32; row < T; row += nw) {
    const float* xr = x + row * n;
    float* yr = y + row * n;
    float ss = 0.f;
    if (vec) {
      const float4* x4 = reinterpret_cast<const float4*>(xr);
      for (int i = lane; i < n / 4; i += 32) {
        const float4 v = x4[i];
        ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
      }
    } else {
      for (int i = lane; i < n; i += 32) ss = fmaf(xr[i], xr[i], ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = 1.0f / sqrtf(ss / static_cast<float>(n) + eps);
    auto one = [&](float xv, float wv) {
      const float r = xv * inv * (offset ? 1.0f + wv : wv);
      return round_out ? tc::round_tf32(r) : r;
    };
    if (vec) {
      const float4* x4 = reinterpret_cast<const float4*>(xr);
      const float4* w4 = reinterpret_cast<const float4*>(w);
      float4* y4 = reinterpret_cast<float4*>(yr);
      for (int i = lane; i < n / 4; i += 32) {
        const float4 v = x4[i], g = w4[i];
        y4[i] = make_float4(one(v.x, g.x), one(v.y, g.y), one(v.z, g.z), one(v.w, g.w));
      }
    } else {
      for (int i = lane; i < n; i += 32) yr[i] = one(xr[i], w[i]);
    }
  }
}

// out[b, q, p, :] = in[b, p, q, :] for in [B, P, Q, D] (token-major <-> head-major).
__global__ void __launch_bounds__(256) swap_mid_kernel(const float* __restrict__ in,
                                                       float* __restrict__ out, int B, int P, int Q,
                                                       int D, const int32_t* skip) {
  if (gated_off(skip)) return;
  const long total = static_cast<long>(B) * P * Q * D;
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const int d = static_cast<int>(i % D);
    long r = i / D;
    const int q = static_cast<int>(r % Q);
    r /= Q;
    const int p = static_cast<int>(r % P);
    const long b = r / P;
    out[((b * Q + q) * P + p) * D + d] = in[i];
  }
}

unsigned grid_for(long n, int per_block) {
  long blocks = (n + per_block - 1) / per_block;
  if (blocks > 152L * 16) blocks = 152L * 16;
  return static_cast<unsigned>(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_rmsnorm_rows(const float* x, const float* w, float* y, long T, int n,
                                float eps, bool offset, bool round_out, cudaStream_t stream,
                                const int32_t* skip) {
  rmsnorm_rows_kernel<<<grid_for(T, 8), 256, 0, stream>>>(x, w, y, T, n, eps, offset ? 1 : 0,
                                                          round_out ? 1 : 0, skip);
  return cudaGetLastError();
}

cudaError_t launch_swap_mid(const float* in, float* out, int B, int P, int Q, int D,
                            cudaStream_t stream, const int32_t* skip) {
  swap_mid_kernel<<<grid_for(static_cast<long>(B) * P * Q * D, 256), 256, 0, stream>>>(in, out, B,
                                                                                       P, Q, D, skip);
  return cudaGetLastError();
}

}  // namespace gqa
