// Keys and values for a prefill chunk that continues a cached prefix
// ("mojolearn.transformer", TransformerBlock.forward with a carried
// TransformerState: the chunk's queries attend to the cached positions and to
// the chunk itself; under a window only the last W positions count, the cache
// being a ring of W slots).
//
// Per (b, kv head) the key buffer lists, in position order, the prefix rows
// kept in the cache (start - pre .. start - 1) and then the chunk's L rows, so
// the tensor-core prefill treats them like one contiguous key sequence in which
// query row l sits at key index pre + l. K is copied as rows, V is transposed
// (the K-major B operand of P V), both through 32 x 32 tiles with 16-byte
// accesses. Rows past pre + L are zeros (their scores are masked).
#include "common.cuh"
#include "kernels.h"

namespace gqa {

namespace {

__global__ void __launch_bounds__(256) gather_kv_kernel(GatherJob j) {
  __shared__ float tile[32][33];
  if (gated_off(j.skip)) return;
  const int bh = blockIdx.z;
  const int b = bh / j.Hkv;
  const int r0 = blockIdx.x * 32, d0 = blockIdx.y * 32;
  const int r = threadIdx.x / 8, q = threadIdx.x % 8;
  const int D = j.D;

  // Prefix rows of batch row b (a bad start is reported and treated as no prefix).
  const int st = j.start[b];
  int pre = 0;
  bool bad = st < 0 || st > j.max_start || (j.window == 0 && st > j.capacity);
  if (!bad) pre = j.window > 0 ? min(st, j.window - 1) : st;
  if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0 && bh % j.Hkv == 0) {
    j.pre[b] = pre;
    if (bad) report(j.status, st < 0 || st > j.max_start ? ATTN_DEV_POSITION : ATTN_DEV_CAPACITY);
  }

  const long head_cache = static_cast<long>(bh) * j.capacity * D;
  const long head_chunk = static_cast<long>(bh) * j.L * D;
  // source row of key row x: cache slot, chunk row, or none
  auto src_of = [&](int x, bool value) -> const float* {
    if (x < pre) {
      const int pos = st - pre + x;
      const int slot = j.window > 0 ? pos % j.window : pos;
      return (value ? j.v_cache : j.k_cache) + head_cache + static_cast<long>(slot) * D;
    }
    if (x < pre + j.L) return (value ? j.v : j.k) + head_chunk + static_cast<long>(x - pre) * D;
    return nullptr;
  };
  {
    const int x = r0 + r, d = d0 + 4 * q;
    float4 kx = make_float4(0.f, 0.f, 0.f, 0.f), vx = kx;
    if (x < j.Lk && d < D) {
      const float* ks = src_of(x, false);
      const float* vs = src_of(x, true);
      if (ks) {
        kx = __ldg(reinterpret_cast<const float4*>(ks + d));
        vx = __ldg(reinterpret_cast<const float4*>(vs + d));
      }
      *reinterpret_cast<float4*>(j.kg + (static_cast<long>(bh) * j.Lk + x) * D + d) = kx;
    }
    tile[r][4 * q] = vx.x;
    tile[r][4 * q + 1] = vx.y;
    tile[r][4 * q + 2] = vx.z;
    tile[r][4 * q + 3] = vx.w;
  }
  __syncthreads();
  {
    const int d = d0 + r, x = r0 + 4 * q;
    if (d < D && x < j.Lk)
      *reinterpret_cast<float4*>(j.vtg + (static_cast<long>(bh) * D + d) * j.vt_pitch + x) =
          make_float4(tile[4 * q][r], tile[4 * q + 1][r], tile[4 * q + 2][r], tile[4 * q + 3][r]);
  }
}

}  // namespace

cudaError_t launch_gather_kv(const GatherJob& j, cudaStream_t stream) {
  const dim3 grid((j.Lk + 31) / 32, (j.D + 31) / 32, j.B * j.Hkv);
  gather_kv_kernel<<<grid, 256, 0, stream>>>(j);
  return cudaGetLastError();
}

}  // namespace gqa
