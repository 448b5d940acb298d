// Pieces shared by the tensor-core prefill kernels: launch arguments, the
// timeout-only drain wait, row-wise TMEM moves and TMA tensor maps.
#pragma once

#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace gqa {
namespace prefill {

constexpr int kBM = 128;                       // query rows per tile = MMA M = TMEM lanes
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;           // rescale O when the max grows by > 2^8
constexpr int kSmemLimit = 232448;             // 227 KB of dynamic shared memory per block
constexpr int kTmemCols = 512;

struct TcArgs {
  const float* q;                              // [B, H, L, D] (read directly when Q is in TMEM)
  float* out;
  int B, H, Hkv, L, D;
  int G, QT, ntiles, npairs;                   // per (b, kv head): tiles and tile groups
  int units;                                   // persistent kernel: B * H * QT query tiles
  // Fused q RMSNorm + RoPE (persistent kernel): rope_table == nullptr means q is rotated.
  const float2* rope_table;                    // [max_positions][R/2] (cos, sin)
  const int32_t* rope_start;                   // [B], or nullptr: every row starts at 0
  const float* qnorm_w;                        // [D] or nullptr
  float qnorm_eps;
  int rope_R, rope_max_positions;
  int window;
  int softcap_on;
  float c_score;                               // scale * log2(e)
  float c_cap_in;                              // 2 * log2(e) * scale / cap
  float c_cap_out;                             // log2(e) * cap
  int32_t* status;
  // Keys continuing a cached prefix (persistent kernel): kv_off[b] keys precede
  // query row 0 of batch row b in the key buffer, which has Lk rows per head.
  // kv_off == nullptr: keys are the chunk's own (offset 0, Lk = L).
  const int32_t* kv_off;
  int Lk;
  // Ragged batch (nullptr: every row has length L): see AttnShape::lengths.
  const int32_t* lengths;
  const int32_t* skip;                         // non-finite check: see common.cuh gated_off
};

// Real length of batch row b (lengths outside [0, L] are clamped; the V^T
// pre-pass or the SIMT kernel reports them).
__device__ __forceinline__ int row_len(const TcArgs& a, int b) {
  if (!a.lengths) return a.L;
  const int v = a.lengths[b];
  return v < 0 ? 0 : (v > a.L ? a.L : v);
}

// Position of query row 0 of batch row b (fused RoPE); no start array: 0.
__device__ __forceinline__ int start_of(const TcArgs& a, int b) {
  return a.rope_start ? a.rope_start[b] : 0;
}

// Timeout-only wait used while winding down after an abort.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = tc::globaltimer();
  while (!tc::mbar_try_wait(bar, parity)) {
    if (tc::globaltimer() - t0 > tc::kWaitLimitNs) return;
  }
}

// ---------------------------------------------------------------- softmax helpers
// The block's P is accepted against the running reference while its sum stays
// at most 2^kRescaleLog2 (no single weight can then exceed it).
constexpr float kRescaleLimit = 256.0f;
static_assert(kRescaleLog2 == 8.0f, "limit is 2^kRescaleLog2");

// Row maximum of N scores (three-input maxima, 8 chains).
template <int N>
__device__ __forceinline__ float tq_max(const float* s) {
  float mx[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) mx[j] = s[j];
  int c = 8;
#pragma unroll
  for (; c + 16 <= N; c += 16)
#pragma unroll
    for (int j = 0; j < 8; ++j) mx[j] = tc::max3(mx[j], s[c + j], s[c + 8 + j]);
#pragma unroll
  for (; c < N; c += 8)
#pragma unroll
    for (int j = 0; j < 8; ++j) mx[j] = fmaxf(mx[j], s[c + j]);
  return fmaxf(tc::max3(mx[0], mx[1], mx[2]),
               fmaxf(tc::max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])));
}

// p = 2^(score * cs - m) in place, truncated to the TF32 value the tensor core
// uses (so the row sum adds exactly the weights applied to V); returns the sum.
// Pairs of columns go through the paired fp32 FMA / add.
template <int N>
__device__ __forceinline__ float tq_exp_sum(float* s, float cs, float m) {
  const uint64_t c2 = tc::pack2(cs, cs), m2 = tc::pack2(-m, -m);
  uint64_t acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = tc::pack2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < N; c += 2) {
    float x0, x1;
    tc::unpack2(tc::fma2(tc::pack2(s[c], s[c + 1]), c2, m2), x0, x1);
    const float p0 = tc::trunc_tf32(tc::ex2(x0)), p1 = tc::trunc_tf32(tc::ex2(x1));
    s[c] = p0;
    s[c + 1] = p1;
    acc[(c / 2) % 4] = tc::add2(acc[(c / 2) % 4], tc::pack2(p0, p1));
  }
  float a0, a1;
  tc::unpack2(tc::add2(tc::add2(acc[0], acc[1]), tc::add2(acc[2], acc[3])), a0, a1);
  return a0 + a1;
}

template <int N>
__device__ __forceinline__ void tmem_ld_row(uint32_t addr, float* v) {
  if constexpr (N % 64 == 0) {
#pragma unroll
    for (int c = 0; c < N; c += 64) tc::tmem_ld64(addr + c, v + c);
  } else {
#pragma unroll
    for (int c = 0; c < N; c += 32) tc::tmem_ld32(addr + c, v + c);
  }
}

template <int N>
__device__ __forceinline__ void tmem_st_row(uint32_t addr, const float* v) {
  if constexpr (N % 64 == 0) {
#pragma unroll
    for (int c = 0; c < N; c += 64) tc::tmem_st64(addr + c, v + c);
  } else {
#pragma unroll
    for (int c = 0; c < N; c += 32) tc::tmem_st32(addr + c, v + c);
  }
}

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// [NH, L, D] fp32 rows as a 3-D tensor map; boxes of 32 columns x box_rows rows.
// Heads are head_rows rows apart (0: L, contiguous).
inline bool make_map(CUtensorMap* m, const float* base, int D, int L, int NH, int box_rows,
                     long head_rows = 0) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(NH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4,
                                 static_cast<cuuint64_t>(head_rows > 0 ? head_rows : L) * D * 4};
  const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output [NH, L, D] for TMA stores of 16 columns x 32 rows (64-byte swizzle).
inline bool make_map_out16(CUtensorMap* m, const float* base, int D, int L, int NH) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(NH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4,
                                 static_cast<cuuint64_t>(L) * D * 4};
  const cuuint32_t box[3] = {16, 32, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// V^T [B*Hkv, D, L] (rows of pitch Lp) for TMA: boxes of 32 keys x box_rows dims.
inline bool make_map_vt(CUtensorMap* m, const float* base, int D, int L, int Lp, int NH, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(D),
                              static_cast<cuuint64_t>(NH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(Lp) * 4,
                                 static_cast<cuuint64_t>(Lp) * D * 4};
  const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace prefill
}  // namespace gqa
