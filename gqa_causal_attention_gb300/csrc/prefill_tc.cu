// Tensor-core prefill: the V^T pre-pass and the entry points that run it
// before the persistent kernel (prefill_tq.cu).
//
// TF32 operands of tcgen05.mma must be K-major (an MN-major TF32 B operand is
// not computed on this part), so for O += P V the values arrive transposed: a
// pre-pass writes V^T [B*Hkv, D, Lp] (rows of pitch Lp = L rounded up to 4)
// into the caller's workspace, and TMA streams it like K.
#include "prefill_common.cuh"

namespace gqa {

namespace {

using namespace prefill;

// vt[bh, d, l] = v[bh, l, d] for D % 4 == 0: 32 x 32 tiles through shared
// memory, 16-byte loads along d and 16-byte stores along l (rows of vt have a
// pitch Lp that is a multiple of 4, so a store may run into the padding).
__global__ void __launch_bounds__(256) transpose_v_kernel(const float* __restrict__ v,
                                                          float* __restrict__ vt, int L, int D,
                                                          int Lp, const int32_t* lengths,
                                                          int Hkv, int32_t* status,
                                                          const int32_t* skip) {
  __shared__ float tile[32][33];
  if (gated_off(skip)) return;
  const long bh = blockIdx.z;
  const int l0 = blockIdx.x * 32, d0 = blockIdx.y * 32;
  const int r = threadIdx.x / 8, q = threadIdx.x % 8;
  const float* src = v + bh * L * D;
  float* dst = vt + bh * D * Lp;
  int Lb = L;                                   // keys past the row's length read as 0
  if (lengths) {
    const int n = lengths[bh / Hkv];
    if ((n < 1 || n > L) && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0 &&
        bh % Hkv == 0)
      report(status, ATTN_DEV_LENGTH);
    Lb = n < 0 ? 0 : (n > L ? L : n);
  }
  {
    const int l = l0 + r, d = d0 + 4 * q;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (l < Lb && d < D) x = __ldg(reinterpret_cast<const float4*>(src + static_cast<long>(l) * D + d));
    tile[r][4 * q] = x.x;
    tile[r][4 * q + 1] = x.y;
    tile[r][4 * q + 2] = x.z;
    tile[r][4 * q + 3] = x.w;
  }
  __syncthreads();
  {
    const int d = d0 + r, l = l0 + 4 * q;
    if (d < D && l < L)
      *reinterpret_cast<float4*>(dst + static_cast<long>(d) * Lp + l) =
          make_float4(tile[4 * q][r], tile[4 * q + 1][r], tile[4 * q + 2][r], tile[4 * q + 3][r]);
  }
}

}  // namespace

bool prefill_tc_supports(int D) { return D % 4 == 0 && D >= 32 && D <= kMaxHeadDim; }

int prefill_vt_pitch(int L) { return (L + 3) / 4 * 4; }

cudaError_t launch_transpose_v(const float* v, float* vt, int BHkv, int L, int D, int vt_pitch,
                               cudaStream_t stream, const int32_t* lengths, int Hkv,
                               int32_t* status, const int32_t* skip) {
  transpose_v_kernel<<<dim3((L + 31) / 32, (D + 31) / 32, BHkv), 256, 0, stream>>>(
      v, vt, L, D, vt_pitch, lengths, Hkv, status, skip);
  return cudaGetLastError();
}

cudaError_t launch_prefill_tc(const AttnShape& s, cudaStream_t stream) {
  if (!prefill_tc_supports(s.D)) return cudaErrorNotSupported;
  if (cudaError_t e = launch_transpose_v(s.v, s.vt, s.B * s.Hkv, s.L, s.D, s.vt_pitch, stream,
                                         s.lengths, s.Hkv, s.status, s.skip);
      e != cudaSuccess)
    return e;
  return launch_prefill_tc_vt(s, stream);
}

cudaError_t launch_prefill_tc_vt(const AttnShape& s, cudaStream_t stream) {
  if (!prefill_tc_supports(s.D)) return cudaErrorNotSupported;
  return launch_prefill_tq(s, stream);
}

}  // namespace gqa
