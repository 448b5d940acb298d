// The decoder block around the attention ("mojolearn.transformer",
// TransformerBlock.forward with state None, computing Hugging Face's
// LlamaDecoderLayer.forward): input RMSNorm, q/k/v projections, (q/k norm,)
// RoPE and causal GQA attention, output projection + residual,
// post-attention RMSNorm, SiLU-gated MLP + residual.
//
// The projections are plain fp32 GEMMs (cuBLAS, default math: no TF32); the
// attention is this library's prefill with q RMSNorm/RoPE fused; the rest are
// the small memory-bound kernels below. Activations are token-major
// [B * L, width] as the pages' (B, L, d_model) input; the attention's
// head-major [B, heads, L, D] views come from one permute each way.
#include <cublas_v2.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace gqa {

namespace {

// RMSNorm of each row of x [T, n] ("Core Layers -- Deep Reference", RMSNorm):
// y = x / sqrt(mean x^2 + eps) * (w, or 1 + w). One warp per row.
__global__ void __launch_bounds__(256) rmsnorm_rows_kernel(const float* __restrict__ x,
                                                           const float* __restrict__ w,
                                                           float* __restrict__ y, long T, int n,
                                                           float eps, int offset) {
  const int lane = threadIdx.x & 31;
  const long nw = static_cast<long>(gridDim.x) * 8;
  for (long row = static_cast<long>(blockIdx.x) * 8 + threadIdx.x / 32; row < T; row += nw) {
    const float* xr = x + row * n;
    float ss = 0.f;
    for (int i = lane; i < n; i += 32) ss = fmaf(xr[i], xr[i], ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = 1.0f / sqrtf(ss / static_cast<float>(n) + eps);
    float* yr = y + row * n;
    for (int i = lane; i < n; i += 32) yr[i] = xr[i] * inv * (offset ? 1.0f + w[i] : w[i]);
  }
}

// out[b, q, p, :] = in[b, p, q, :] for in [B, P, Q, D] (token-major <-> head-major).
__global__ void __launch_bounds__(256) swap_mid_kernel(const float* __restrict__ in,
                                                       float* __restrict__ out, int B, int P, int Q,
                                                       int D) {
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

// gate <- SiLU(gate) * up, elementwise.
__global__ void __launch_bounds__(256) swiglu_kernel(float* __restrict__ gate,
                                                     const float* __restrict__ up, long n) {
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const float g = gate[i];
    gate[i] = g / (1.0f + expf(-g)) * up[i];
  }
}

unsigned grid_for(long n, int per_block) {
  long blocks = (n + per_block - 1) / per_block;
  if (blocks > 152L * 16) blocks = 152L * 16;
  return static_cast<unsigned>(blocks < 1 ? 1 : blocks);
}

std::mutex g_blas_mutex;
cublasHandle_t g_blas = nullptr;

}  // namespace

cudaError_t launch_rmsnorm_rows(const float* x, const float* w, float* y, long T, int n,
                                float eps, bool offset, cudaStream_t stream) {
  rmsnorm_rows_kernel<<<grid_for(T, 8), 256, 0, stream>>>(x, w, y, T, n, eps, offset ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_swap_mid(const float* in, float* out, int B, int P, int Q, int D,
                            cudaStream_t stream) {
  swap_mid_kernel<<<grid_for(static_cast<long>(B) * P * Q * D, 256), 256, 0, stream>>>(in, out, B,
                                                                                       P, Q, D);
  return cudaGetLastError();
}

cudaError_t launch_swiglu(float* gate, const float* up, long n, cudaStream_t stream) {
  swiglu_kernel<<<grid_for(n, 256), 256, 0, stream>>>(gate, up, n);
  return cudaGetLastError();
}

// Y [T, N] = X [T, K] . W^T (W [N, K], torch's [out, in]) + beta * Y, fp32.
int gemm_xwt(const float* X, const float* W, float* Y, long T, int N, int K, float beta,
             cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_blas_mutex);
  if (!g_blas && cublasCreate(&g_blas) != CUBLAS_STATUS_SUCCESS) {
    g_blas = nullptr;
    return -1;
  }
  if (cublasSetStream(g_blas, stream) != CUBLAS_STATUS_SUCCESS) return -1;
  const float alpha = 1.0f;
  // Column-major view: Y^T [N, T] = W (as [K, N], transposed) . X^T [K, T].
  return cublasSgemm(g_blas, CUBLAS_OP_T, CUBLAS_OP_N, N, static_cast<int>(T), K, &alpha, W, K, X,
                     K, &beta, Y, N) == CUBLAS_STATUS_SUCCESS
             ? 0
             : -1;
}

}  // namespace gqa
