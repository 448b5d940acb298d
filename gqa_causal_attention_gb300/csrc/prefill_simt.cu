// Prefill attention on the CUDA cores, for head dimensions the tensor-core
// kernel does not take (D % 4 != 0).
//
// Flash-style ("Core Layers -- Deep Reference", "Flash Attention": the exact
// attention output without materialising the L x L matrix): a block holds 32
// query rows of one head, streams the visible key/value rows through shared
// memory 16 at a time and keeps a running maximum, sum and output per row.
// Four threads share a query row, each owning every fourth dimension.
#include "common.cuh"
#include "kernels.h"

namespace gqa {

namespace {
constexpr int kBQ = 32;
constexpr int kBK = 16;
constexpr int kTPR = 4;
constexpr int kThreads = kBQ * kTPR;
constexpr float kLog2e = 1.4426950408889634f;
}  // namespace

template <int NE>
__global__ void __launch_bounds__(kThreads) prefill_simt_kernel(AttnShape a) {
  __shared__ float sk[kBK][NE * kTPR];
  __shared__ float sv[kBK][NE * kTPR];
  if (gated_off(a.skip)) return;
  const int D = a.D, L = a.L;
  const int G = a.H / a.Hkv;
  const int bh = blockIdx.y;                    // b * H + h
  const int b = bh / a.H, h = bh % a.H;
  const int hk = h / G;
  const int q0 = blockIdx.x * kBQ;
  const int r = threadIdx.x / kTPR, t4 = threadIdx.x % kTPR;
  const int qi = q0 + r;
  // Ragged batch: keys and queries at or past the row's length are padding;
  // padding queries are written as +0.0.
  int Lb = L;
  if (a.lengths) {
    const int n = a.lengths[b];
    if ((n < 1 || n > L) && threadIdx.x == 0 && blockIdx.x == 0 && h == 0)
      report(a.status, ATTN_DEV_LENGTH);
    Lb = n < 0 ? 0 : (n > L ? L : n);
  }
  const bool row_ok = qi < Lb;

  float q[NE], o[NE];
#pragma unroll
  for (int e = 0; e < NE; ++e) {
    const int d = t4 + kTPR * e;
    q[e] = (row_ok && d < D) ? a.q[((long)bh * L + qi) * D + d] * a.scale : 0.f;
    o[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const bool capped = a.softcap > 0.f;
  const float cap_k = capped ? 2.0f * kLog2e / a.softcap : 0.f;

  const int qlast = min(q0 + kBQ, L) - 1;
  const int kbeg = a.window > 0 ? max(0, q0 - a.window + 1) : 0;
  const long kvoff = ((long)b * a.Hkv + hk) * L * D;
  for (int k0 = (kbeg / kBK) * kBK; k0 <= qlast; k0 += kBK) {
    __syncthreads();
    for (int t = threadIdx.x; t < kBK * D; t += kThreads) {
      const int kk = t / D, d = t % D;
      const int key = k0 + kk;
      sk[kk][d] = key < L ? a.k[kvoff + (long)key * D + d] : 0.f;
      sv[kk][d] = key < L ? a.v[kvoff + (long)key * D + d] : 0.f;
    }
    __syncthreads();
#pragma unroll 1
    for (int kk = 0; kk < kBK; ++kk) {
      const int key = k0 + kk;
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < NE; ++e) {
        const int d = t4 + kTPR * e;
        if (d < D) s = fmaf(q[e], sk[kk][d], s);
      }
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      const bool vis = row_ok && key < Lb && key <= qi && (a.window == 0 || key > qi - a.window);
      if (!vis) continue;
      if (capped) s = softcap_apply(s, a.softcap, cap_k);
      s *= kLog2e;
      const float mn = fmaxf(m, s);
      const float corr = exp2f(m - mn);
      const float p = exp2f(s - mn);
      m = mn;
      l = l * corr + p;
#pragma unroll
      for (int e = 0; e < NE; ++e) {
        const int d = t4 + kTPR * e;
        if (d < D) o[e] = fmaf(p, sv[kk][d], o[e] * corr);
      }
    }
  }
  if (qi >= L) return;
  const float inv = row_ok ? 1.0f / l : 0.f;
  if (!row_ok) {
#pragma unroll
    for (int e = 0; e < NE; ++e) o[e] = 0.f;
  }
#pragma unroll
  for (int e = 0; e < NE; ++e) {
    const int d = t4 + kTPR * e;
    if (d < D) a.out[((long)bh * L + qi) * D + d] = o[e] * inv;
  }
}

cudaError_t launch_prefill_simt(const AttnShape& a, cudaStream_t stream) {
  dim3 grid((a.L + kBQ - 1) / kBQ, a.B * a.H);
  if (a.D <= 64)
    prefill_simt_kernel<16><<<grid, kThreads, 0, stream>>>(a);
  else if (a.D <= 128)
    prefill_simt_kernel<32><<<grid, kThreads, 0, stream>>>(a);
  else
    prefill_simt_kernel<64><<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gqa
