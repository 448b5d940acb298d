// The decoder block's projections on the tcgen05 tensor cores
// ("mojolearn.transformer", TransformerBlock: the bias-free linear maps
// q_proj, k_proj, v_proj, o_proj, gate_proj, up_proj, down_proj; y = x W^T
// with W in torch's [out, in] layout).
//
// Y[t, n] = sum_k X[t, k] W[n, k]: both operands are K-major (k contiguous),
// the layout the tensor core reads without any transpose. TF32 operands, fp32
// accumulation in tensor memory.
//
// Persistent kernel, one block per SM, 192 threads:
//   warp 0      TMA producer: per 32-wide K block, a 128-row tile of X and two
//               128-row tiles of weight rows into one ring stage (48 KB, 4 stages);
//   warp 1      MMA issuer: 4 x tcgen05.mma kind::tf32 M128 N256 K8 per stage
//               into one of two 256-column accumulators in tensor memory;
//   warps 2-5   epilogue: tensor memory -> registers (one output row per
//               thread), the segment's epilogue, global stores. Two accumulators
//               let the epilogue of one tile overlap the next tile's products.
// A launch covers up to three "segments" that share X: n-tiles are numbered
// across them, and each segment has its own weights, output and epilogue
// (q, k and v projections in one launch; gate and up in one SwiGLU segment).
//
// Epilogues:
//   STORE   out = acc, row-major [T, n] or head-major [B, heads, L, D]
//           (column h * D + d of token (b, l) -> out[b, h, l, d]);
//   ADD     out = res + acc (res may be out itself: each element is read and
//           written by the same thread);
//   SWIGLU  the stage's weight halves are gate rows and up rows of the same
//           columns: out[t, j] = SiLU(gate) * up over 128 columns per tile.
// X is token-major [T, K] (a 3-D tensor map), or head-major [B, H, L, D] with
// K = H * D (a 4-D map; m-tiles then stay inside one batch row), which lets
// o_proj read the attention output as the attention kernel writes it.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "prefill_common.cuh"
#include "tc_ptx.cuh"

namespace gqa {

namespace {

constexpr int kGBM = 128;                       // tile rows (MMA M, tensor-memory lanes)
constexpr int kGBN = 256;                       // accumulator columns (MMA N)
constexpr int kGBK = 32;                        // K per stage: 32 fp32 = one 128-byte swizzle row
constexpr int kGNS = 4;                         // ring stages
constexpr int kGAStage = kGBM * kGBK * 4;       // 16 KB
constexpr int kGBHalf = 128 * kGBK * 4;         // 16 KB: 128 weight rows
constexpr int kGStage = kGAStage + 2 * kGBHalf; // 48 KB
constexpr int kGThreads = 192;
constexpr int kGSmem = kGNS * kGStage + 1024 + 512;
constexpr int kGroupM = 16;                     // m-tiles per raster group (L2 reuse of weights)

enum { kEpiStore = 0, kEpiAdd = 1, kEpiSwiglu = 2 };

struct GSeg {
  int n;                     // output columns
  int ntiles, tile0;         // n-tiles of this segment and the first one's global index
  int map_lo, map_hi;        // weight maps of the two 128-row halves of a stage
  int hi_off, nstep;         // half 1 starts hi_off rows after half 0; columns per n-tile
  int mode;
  int round_out;             // round outputs to the nearest TF32 value (they feed a GEMM)
  float* out;
  long ldo;
  int heads;                 // > 0: head-major out [B, heads, L, D]
  const float* res;
  long ldr;
};

struct GArgs {
  int T, K, L, D;
  int batched;               // X head-major: m-tile = (b, l0)
  int mt_per_b, m_tiles, n_tiles, tiles, kblocks;
  int nseg;
  GSeg seg[3];
  int32_t* status;
  const int32_t* skip;
};

struct GBars {
  uint64_t full[kGNS];
  uint64_t empty[kGNS];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct GTile {
  int m, n;                  // m-tile, n-tile (global across segments)
  int s, n0;                 // segment, its first output column
};

__device__ __forceinline__ GTile tile_of(const GArgs& a, int x) {
  // Groups of kGroupM m-tiles walk every n-tile: the weights of a wave's tiles
  // and its X rows both stay in L2.
  const int per_group = kGroupM * a.n_tiles;
  const int g = x / per_group, r = x % per_group;
  const int m0 = g * kGroupM;
  const int gm = min(kGroupM, a.m_tiles - m0);
  GTile t;
  t.m = m0 + r % gm;
  t.n = r / gm;
  t.s = 0;
  for (int s = 1; s < a.nseg; ++s)
    if (t.n >= a.seg[s].tile0) t.s = s;
  t.n0 = (t.n - a.seg[t.s].tile0) * a.seg[t.s].nstep;
  return t;
}

__device__ void g_producer(const GArgs& a, const CUtensorMap* ta, const CUtensorMap* tb0,
                           const CUtensorMap* tb1, const CUtensorMap* tb2, uint8_t* ring,
                           GBars* bars) {
  volatile int* abort = &bars->abort;
  const CUtensorMap* tb[3] = {tb0, tb1, tb2};
  tc::tma_prefetch(ta);
  for (int s = 0; s < a.nseg; ++s) tc::tma_prefetch(tb[s]);
  int stage = 0;
  uint32_t phase = 0;
  uint32_t fill_parity[kGNS];
  bool filled[kGNS];
#pragma unroll
  for (int s = 0; s < kGNS; ++s) filled[s] = false;
  bool ok = true;
  for (int x = blockIdx.x; x < a.tiles && ok; x += gridDim.x) {
    const GTile t = tile_of(a, x);
    const GSeg& sg = a.seg[t.s];
    int b = 0, row0 = t.m * kGBM;
    if (a.batched) {
      b = t.m / a.mt_per_b;
      row0 = (t.m % a.mt_per_b) * kGBM;
    }
    for (int kb = 0; kb < a.kblocks; ++kb) {
      if (!(ok = tc::mbar_wait(&bars->empty[stage], phase ^ 1u, abort))) break;
      uint64_t* full = &bars->full[stage];
      uint8_t* dst = ring + stage * kGStage;
      tc::mbar_arrive_expect_tx(full, kGStage);
      const int k0 = kb * kGBK;
      if (a.batched)
        tc::tma_load_4d(dst, ta, full, k0 % a.D, row0, k0 / a.D, b);
      else
        tc::tma_load_3d(dst, ta, full, k0, row0, 0);
      tc::tma_load_3d(dst + kGAStage, tb[sg.map_lo], full, k0, t.n0, 0);
      tc::tma_load_3d(dst + kGAStage + kGBHalf, tb[sg.map_hi], full, k0, t.n0 + sg.hi_off, 0);
      fill_parity[stage] = phase;
      filled[stage] = true;
      if (++stage == kGNS) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (!ok) {
    // Copies still in flight land before the block exits.
    for (int s = 0; s < kGNS; ++s)
      if (filled[s]) prefill::drain_wait(&bars->full[s], fill_parity[s]);
  }
}

__device__ void g_mma(const GArgs& a, uint32_t tmem, uint8_t* ring, GBars* bars) {
  volatile int* abort = &bars->abort;
  constexpr uint32_t idesc = tc::idesc_tf32(kGBM, kGBN, false);
  const uint64_t base = tc::sdesc_sw128(tc::smem_u32(ring), 16, 1024);
  int stage = 0;
  uint32_t phase = 0;
  uint32_t it = 0;
  bool ok = true;
  for (int x = blockIdx.x; x < a.tiles && ok; x += gridDim.x, ++it) {
    const uint32_t acc = it & 1u;
    if (!(ok = tc::mbar_wait(&bars->acc_empty[acc], ((it >> 1) & 1u) ^ 1u, abort))) break;
    tc::fence_after_sync();
    const uint32_t d = tmem + acc * kGBN;
    for (int kb = 0; kb < a.kblocks; ++kb) {
      if (!(ok = tc::mbar_wait(&bars->full[stage], phase, abort))) break;
      tc::fence_after_sync();
      const uint64_t ad = base + static_cast<uint32_t>((stage * kGStage) >> 4);
      const uint64_t bd = base + static_cast<uint32_t>((stage * kGStage + kGAStage) >> 4);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        tc::mma_tf32_ss(d, ad + ((32 * j) >> 4), bd + ((32 * j) >> 4), idesc, (kb | j) != 0);
      tc::mma_commit(&bars->empty[stage]);
      if (++stage == kGNS) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (ok) tc::mma_commit(&bars->acc_full[acc]);
  }
  // Every product issued has completed before tensor memory is released.
  tc::mma_commit(&bars->drain);
  prefill::drain_wait(&bars->drain, 0);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.0f + __expf(-g)) * u;
}

// Store 32 consecutive output columns n .. n + 31 of one row (v), with the segment's
// epilogue; columns past sg.n are dropped.
__device__ __forceinline__ void g_store32(const GArgs& a, const GSeg& sg, long t, int b, int l,
                                          int n, float* v) {
  if (sg.round_out) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = tc::round_tf32(v[i]);
  }
  const bool full = n + 32 <= sg.n;
  if (sg.heads > 0) {
    if (full && a.D % 32 == 0) {
      const int h = n / a.D, d = n % a.D;
      float4* dst = reinterpret_cast<float4*>(
          sg.out + ((static_cast<long>(b) * sg.heads + h) * a.L + l) * a.D + d);
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int c = n + i;
        if (c < sg.n)
          sg.out[((static_cast<long>(b) * sg.heads + c / a.D) * a.L + l) * a.D + c % a.D] = v[i];
      }
    }
    return;
  }
  float* dst = sg.out + t * sg.ldo + n;
  if (full) {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int i = 0; i < 8; ++i) d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (n + i < sg.n) dst[i] = v[i];
  }
}

__device__ void g_epilogue(const GArgs& a, uint32_t tmem, GBars* bars, int quarter, int lane) {
  volatile int* abort = &bars->abort;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  uint32_t it = 0;
  for (int x = blockIdx.x; x < a.tiles; x += gridDim.x, ++it) {
    const uint32_t acc = it & 1u;
    if (!tc::mbar_wait(&bars->acc_full[acc], (it >> 1) & 1u, abort)) break;
    tc::fence_after_sync();
    const GTile t = tile_of(a, x);
    const GSeg& sg = a.seg[t.s];
    const int r = quarter * 32 + lane;
    int b, l;
    long row;
    bool valid;
    if (a.batched) {
      b = t.m / a.mt_per_b;
      l = (t.m % a.mt_per_b) * kGBM + r;
      valid = l < a.L;
      row = static_cast<long>(b) * a.L + l;
    } else {
      row = static_cast<long>(t.m) * kGBM + r;
      valid = row < a.T;
      b = valid ? static_cast<int>(row / a.L) : 0;
      l = valid ? static_cast<int>(row % a.L) : 0;
    }
    const uint32_t col = lane_base + acc * kGBN;
    if (sg.mode == kEpiSwiglu) {
      for (int c = 0; c < kGBN / 2; c += 32) {
        float g[32], u[32];
        __syncwarp();
        tc::tmem_ld32(col + c, g);
        tc::tmem_ld32(col + kGBN / 2 + c, u);
        if (c + 32 >= kGBN / 2) {           // last load of the tile: release the accumulator
          tc::fence_before_sync();
          tc::mbar_arrive(&bars->acc_empty[acc]);
        }
        if (valid && t.n0 + c < sg.n) {
#pragma unroll
          for (int i = 0; i < 32; ++i) g[i] = silu_mul(g[i], u[i]);
          g_store32(a, sg, row, b, l, t.n0 + c, g);
        }
      }
    } else {
      for (int c = 0; c < kGBN; c += 32) {
        float v[32];
        __syncwarp();
        tc::tmem_ld32(col + c, v);
        if (c + 32 >= kGBN) {
          tc::fence_before_sync();
          tc::mbar_arrive(&bars->acc_empty[acc]);
        }
        const int n = t.n0 + c;
        if (valid && n < sg.n) {
          if (sg.mode == kEpiAdd) {
            const float* rs = sg.res + row * sg.ldr + n;
            if (n + 32 <= sg.n) {
              const float4* r4 = reinterpret_cast<const float4*>(rs);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 q = r4[i];
                v[4 * i] += q.x;
                v[4 * i + 1] += q.y;
                v[4 * i + 2] += q.z;
                v[4 * i + 3] += q.w;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (n + i < sg.n) v[i] += rs[i];
            }
          }
          g_store32(a, sg, row, b, l, n, v);
        }
      }
    }
    __syncwarp();
  }
}

__global__ void __launch_bounds__(kGThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a,
                   const __grid_constant__ CUtensorMap tm_b0,
                   const __grid_constant__ CUtensorMap tm_b1,
                   const __grid_constant__ CUtensorMap tm_b2, const GArgs a) {
  if (gated_off(a.skip)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  GBars* bars = reinterpret_cast<GBars*>(ring + kGNS * kGStage);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGNS; ++s) {
      tc::mbar_init(&bars->full[s], 1);
      tc::mbar_init(&bars->empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&bars->acc_full[i], 1);
      tc::mbar_init(&bars->acc_empty[i], 128);
    }
    tc::mbar_init(&bars->drain, 1);
    bars->abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&bars->tmem_base, 2 * kGBN);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  if (warp == 0) {
    if (lane == 0) g_producer(a, &tm_a, &tm_b0, &tm_b1, &tm_b2, ring, bars);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) g_mma(a, tmem, ring, bars);
    __syncwarp();
  } else {
    g_epilogue(a, tmem, bars, warp % 4, lane);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && bars->abort) report(a.status, ATTN_DEV_TIMEOUT);
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 2 * kGBN);
  }
}

// ---------------------------------------------------------------- CTA-pair kernel
// Tiles of 256 rows x 256 columns on a cluster of two CTAs (one per SM). CTA r
// of the pair holds rows 128 r .. 128 r + 127 of the tile in its tensor memory
// and stages, per K block, its 128 X rows and weight rows 128 r .. 128 r + 127
// of the tile's 256 (32 KB per stage, 6 stages). The even CTA issues
// tcgen05.mma.cta_group::2 M256 N256 K8 products, which read each CTA's X rows
// and both CTAs' weight rows from their shared memory: an SM streams 32 KB from
// L2 per 512 tensor cycles instead of 48 KB. Both CTAs' copies complete on the
// even CTA's `full` barrier; its commits arrive on both CTAs' `empty`,
// `acc_full` and `drain` barriers; each epilogue warp of either CTA hands the
// accumulator back with one arrive on the even CTA's `acc_empty`.
constexpr int kG2M = 2 * kGBM;                  // tile rows
constexpr int kG2NS = 6;                        // ring stages
constexpr int kG2Stage = kGAStage + kGBHalf;    // 32 KB
constexpr int kG2Smem = kG2NS * kG2Stage + 1024 + 512;

struct G2Bars {
  uint64_t full[kG2NS];       // even CTA: both CTAs' copies of a stage have landed
  uint64_t empty[kG2NS];      // each CTA: the products reading a stage are done
  uint64_t acc_full[2];       // each CTA: an accumulator is complete
  uint64_t acc_empty[2];      // even CTA: all eight epilogue warps have read it
  uint64_t drain;             // each CTA: every product has completed
  uint32_t tmem_base;
  int abort;
};

// First row of this CTA's half of m-tile m, and its batch row (head-major X).
__device__ __forceinline__ void g2_rows(const GArgs& a, int m, uint32_t rank, int& b, int& row0) {
  const int half = kGBM * static_cast<int>(rank & 1u);
  if (a.batched) {
    b = m / a.mt_per_b;
    row0 = (m % a.mt_per_b) * kG2M + half;
  } else {
    b = 0;
    row0 = m * kG2M + half;
  }
}

__device__ void g2_producer(const GArgs& a, uint32_t rank, const CUtensorMap* ta,
                            const CUtensorMap* tb0, const CUtensorMap* tb1,
                            const CUtensorMap* tb2, uint8_t* ring, G2Bars* bars) {
  volatile int* abort = &bars->abort;
  const CUtensorMap* tb[3] = {tb0, tb1, tb2};
  tc::tma_prefetch(ta);
  for (int s = 0; s < a.nseg; ++s) tc::tma_prefetch(tb[s]);
  const bool odd = rank & 1u;
  const uint32_t lead = rank & ~1u;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t fill_parity[kG2NS];
  bool filled[kG2NS];
#pragma unroll
  for (int s = 0; s < kG2NS; ++s) filled[s] = false;
  bool ok = true;
  for (int x = blockIdx.x / 2; x < a.tiles && ok; x += gridDim.x / 2) {
    const GTile t = tile_of(a, x);
    const GSeg& sg = a.seg[t.s];
    int b, row0;
    g2_rows(a, t.m, rank, b, row0);
    const CUtensorMap* tw = tb[odd ? sg.map_hi : sg.map_lo];
    const int wrow = t.n0 + (odd ? sg.hi_off : 0);
    for (int kb = 0; kb < a.kblocks; ++kb) {
      if (!(ok = tc::mbar_wait(&bars->empty[stage], phase ^ 1u, abort))) break;
      uint8_t* dst = ring + stage * kG2Stage;
      const uint32_t full = tc::cluster_addr(tc::smem_u32(&bars->full[stage]), lead);
      if (!odd) tc::mbar_arrive_expect_tx(&bars->full[stage], 2 * kG2Stage);
      const int k0 = kb * kGBK;
      if (a.batched)
        tc::tma_load_4d_pair(dst, ta, full, k0 % a.D, row0, k0 / a.D, b);
      else
        tc::tma_load_3d_pair(dst, ta, full, k0, row0, 0);
      tc::tma_load_3d_pair(dst + kGAStage, tw, full, k0, wrow, 0);
      fill_parity[stage] = phase;
      filled[stage] = true;
      if (++stage == kG2NS) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (!ok && !odd) {
    // Copies still in flight (both CTAs') land before the pair may exit.
    for (int s = 0; s < kG2NS; ++s)
      if (filled[s]) prefill::drain_wait(&bars->full[s], fill_parity[s]);
  }
}

// The even CTA's issuing thread.
__device__ void g2_mma(const GArgs& a, uint32_t tmem, uint8_t* ring, G2Bars* bars) {
  volatile int* abort = &bars->abort;
  constexpr uint32_t idesc = tc::idesc_tf32(kG2M, kGBN, false);
  const uint64_t base = tc::sdesc_sw128(tc::smem_u32(ring), 16, 1024);
  int stage = 0;
  uint32_t phase = 0;
  uint32_t it = 0;
  bool ok = true;
  for (int x = blockIdx.x / 2; x < a.tiles && ok; x += gridDim.x / 2, ++it) {
    const uint32_t acc = it & 1u;
    if (!(ok = tc::mbar_wait_cluster(&bars->acc_empty[acc], ((it >> 1) & 1u) ^ 1u, abort)))
      break;
    tc::fence_after_sync();
    const uint32_t d = tmem + acc * kGBN;
    for (int kb = 0; kb < a.kblocks; ++kb) {
      if (!(ok = tc::mbar_wait_cluster(&bars->full[stage], phase, abort))) break;
      tc::fence_after_sync();
      const uint64_t ad = base + static_cast<uint32_t>((stage * kG2Stage) >> 4);
      const uint64_t bd = base + static_cast<uint32_t>((stage * kG2Stage + kGAStage) >> 4);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        tc::mma_tf32_ss_pair(d, ad + ((32 * j) >> 4), bd + ((32 * j) >> 4), idesc, (kb | j) != 0);
      tc::mma_commit_pair(&bars->empty[stage]);
      if (++stage == kG2NS) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (ok) tc::mma_commit_pair(&bars->acc_full[acc]);
  }
  // Every product issued has completed before either CTA releases its tensor memory.
  tc::mma_commit_pair(&bars->drain);
  prefill::drain_wait(&bars->drain, 0);
}

__device__ void g2_epilogue(const GArgs& a, uint32_t rank, uint32_t tmem, G2Bars* bars,
                            int quarter, int lane) {
  volatile int* abort = &bars->abort;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  const uint32_t lead = rank & ~1u;
  uint32_t it = 0;
  for (int x = blockIdx.x / 2; x < a.tiles; x += gridDim.x / 2, ++it) {
    const uint32_t acc = it & 1u;
    if (!tc::mbar_wait_cluster(&bars->acc_full[acc], (it >> 1) & 1u, abort)) break;
    tc::fence_after_sync();
    const GTile t = tile_of(a, x);
    const GSeg& sg = a.seg[t.s];
    int b, row0;
    g2_rows(a, t.m, rank, b, row0);
    const int r = row0 + quarter * 32 + lane;
    int l;
    long row;
    bool valid;
    if (a.batched) {
      l = r;
      valid = l < a.L;
      row = static_cast<long>(b) * a.L + l;
    } else {
      row = r;
      valid = row < a.T;
      b = valid ? static_cast<int>(row / a.L) : 0;
      l = valid ? static_cast<int>(row % a.L) : 0;
    }
    const uint32_t col = lane_base + acc * kGBN;
    // the warp's loads of this accumulator are done: one arrive for the warp
    auto release = [&]() {
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0)
        tc::mbar_arrive_cluster(tc::cluster_addr(tc::smem_u32(&bars->acc_empty[acc]), lead));
    };
    if (sg.mode == kEpiSwiglu) {
      for (int c = 0; c < kGBN / 2; c += 32) {
        float gt[32], u[32];
        __syncwarp();
        tc::tmem_ld32(col + c, gt);
        tc::tmem_ld32(col + kGBN / 2 + c, u);
        if (c + 32 >= kGBN / 2) release();
        if (valid && t.n0 + c < sg.n) {
#pragma unroll
          for (int i = 0; i < 32; ++i) gt[i] = silu_mul(gt[i], u[i]);
          g_store32(a, sg, row, b, l, t.n0 + c, gt);
        }
      }
    } else {
      for (int c = 0; c < kGBN; c += 32) {
        float v[32];
        __syncwarp();
        tc::tmem_ld32(col + c, v);
        if (c + 32 >= kGBN) release();
        const int n = t.n0 + c;
        if (valid && n < sg.n) {
          if (sg.mode == kEpiAdd) {
            const float* rs = sg.res + row * sg.ldr + n;
            if (n + 32 <= sg.n) {
              const float4* r4 = reinterpret_cast<const float4*>(rs);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 q = r4[i];
                v[4 * i] += q.x;
                v[4 * i + 1] += q.y;
                v[4 * i + 2] += q.z;
                v[4 * i + 3] += q.w;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (n + i < sg.n) v[i] += rs[i];
            }
          }
          g_store32(a, sg, row, b, l, n, v);
        }
      }
    }
    __syncwarp();
  }
}

__global__ void __launch_bounds__(kGThreads, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_b0,
                    const __grid_constant__ CUtensorMap tm_b1,
                    const __grid_constant__ CUtensorMap tm_b2, const GArgs a) {
  if (gated_off(a.skip)) return;                // both CTAs of a pair read the same word
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  G2Bars* bars = reinterpret_cast<G2Bars*>(ring + kG2NS * kG2Stage);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = tc::cluster_rank();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kG2NS; ++s) {
      tc::mbar_init(&bars->full[s], 1);
      tc::mbar_init(&bars->empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&bars->acc_full[i], 1);
      tc::mbar_init(&bars->acc_empty[i], 8);
    }
    tc::mbar_init(&bars->drain, 1);
    bars->abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc_pair(&bars->tmem_base, 2 * kGBN);
    tc::tmem_relinquish_pair();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();                           // both CTAs' barriers exist before any remote use
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  if (warp == 0) {
    if (lane == 0) g2_producer(a, rank, &tm_a, &tm_b0, &tm_b1, &tm_b2, ring, bars);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && (rank & 1u) == 0) g2_mma(a, tmem, ring, bars);
    __syncwarp();
  } else {
    g2_epilogue(a, rank, tmem, bars, warp % 4, lane);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && bars->abort) report(a.status, ATTN_DEV_TIMEOUT);
  if (warp == 1) {
    // The odd CTA's tensor memory is written by the even CTA's products.
    if ((rank & 1u) && lane == 0) prefill::drain_wait(&bars->drain, 0);
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem, 2 * kGBN);
  }
  tc::cluster_sync();                           // neither CTA leaves while the other may use its memory
}

// rows x K fp32, K contiguous, as a 3-D map {K, rows, 1} with 32 x 128 boxes.
bool map_rows(CUtensorMap* m, const float* base, int K, long rows) {
  auto enc = prefill::encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows), 1};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 4,
                                 static_cast<cuuint64_t>(rows) * K * 4};
  const cuuint32_t box[3] = {32, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Head-major [B, H, L, D] as a 4-D map {D, L, H, B} with 32 x 128 x 1 x 1 boxes.
bool map_heads(CUtensorMap* m, const float* base, int B, int H, int L, int D) {
  auto enc = prefill::encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 4,
                                 static_cast<cuuint64_t>(L) * D * 4,
                                 static_cast<cuuint64_t>(H) * L * D * 4};
  const cuuint32_t box[4] = {32, 128, 1, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of two that fit on the current device at once (per device and
// context), after setting the pair kernel's shared-memory size; -1 on a CUDA error.
int pair_clusters() {
  static PerContext<int> cache;
  return cache.get(
      [] {
        if (cudaFuncSetAttribute(gemm_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kG2Smem) != cudaSuccess) {
          cudaGetLastError();
          return -1;
        }
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(kGThreads);
        cfg.dynamicSmemBytes = kG2Smem;
        cudaLaunchAttribute attr{};
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_tc2_kernel, &cfg) != cudaSuccess) {
          cudaGetLastError();
          n = 0;
        }
        return n;
      },
      -1, [](int n) { return n >= 0; });
}

int g_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 152;
  }
  return n;
}

}  // namespace

bool gemm_tc_supports(const GemmJob& j) {
  if (j.T < 1 || j.K < 1 || j.K % 4 || j.nseg < 1 || j.nseg > 3) return false;
  if (j.x_heads > 0 && (j.D % 32 || j.x_heads * j.D != j.K || j.L < 1 || j.T % j.L)) return false;
  for (int s = 0; s < j.nseg; ++s) {
    const GemmSegment& g = j.seg[s];
    if (g.n < 1 || !g.w || !g.out) return false;
    if (g.mode == kEpiSwiglu && !g.w_up) return false;
    if (g.out_heads > 0 && (g.out_heads * j.D != g.n || g.mode != kEpiStore || j.L < 1)) return false;
    if (g.out_heads == 0 && (g.ldo % 4 || g.ldo < g.n)) return false;
    if (g.mode == kEpiAdd && (!g.res || g.ldr % 4 || g.ldr < g.n)) return false;
  }
  return true;
}

cudaError_t launch_gemm_tc(const GemmJob& j, cudaStream_t stream) {
  if (!gemm_tc_supports(j)) return cudaErrorInvalidValue;
  static PerContext<cudaError_t> attr;
  if (const cudaError_t e = attr.get(
          [] {
            return cudaFuncSetAttribute(gemm_tc_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmem);
          },
          cudaErrorInvalidDevice, [](cudaError_t r) { return r == cudaSuccess; });
      e != cudaSuccess)
    return e;
  GArgs a{};
  a.T = static_cast<int>(j.T);
  a.K = j.K;
  a.L = j.L > 0 ? j.L : 1;
  a.D = j.D > 0 ? j.D : 1;
  a.batched = j.x_heads > 0;
  if (a.batched) {
    a.mt_per_b = (j.L + kGBM - 1) / kGBM;
    a.m_tiles = static_cast<int>(j.T / j.L) * a.mt_per_b;
  } else {
    a.mt_per_b = 0;
    a.m_tiles = static_cast<int>((j.T + kGBM - 1) / kGBM);
  }
  a.kblocks = (j.K + kGBK - 1) / kGBK;
  a.nseg = j.nseg;
  a.status = j.status;
  a.skip = j.skip;
  CUtensorMap tb[3];
  int tiles_n = 0;
  for (int s = 0; s < j.nseg; ++s) {
    const GemmSegment& g = j.seg[s];
    GSeg& o = a.seg[s];
    o.n = g.n;
    o.mode = g.mode;
    o.round_out = g.round_out;
    o.out = g.out;
    o.ldo = g.ldo;
    o.heads = g.out_heads;
    o.res = g.res;
    o.ldr = g.ldr;
    o.tile0 = tiles_n;
    if (g.mode == kEpiSwiglu) {
      // one segment takes two maps: gate rows (half 0) and up rows (half 1)
      if (j.nseg != 1) return cudaErrorInvalidValue;
      if (!map_rows(&tb[0], g.w, j.K, g.n) || !map_rows(&tb[1], g.w_up, j.K, g.n))
        return cudaErrorInvalidValue;
      o.map_lo = 0;
      o.map_hi = 1;
      o.hi_off = 0;
      o.nstep = kGBN / 2;
    } else {
      if (!map_rows(&tb[s], g.w, j.K, g.n)) return cudaErrorInvalidValue;
      o.map_lo = o.map_hi = s;
      o.hi_off = kGBN / 2;
      o.nstep = kGBN;
    }
    o.ntiles = (g.n + o.nstep - 1) / o.nstep;
    tiles_n += o.ntiles;
  }
  for (int s = (j.seg[0].mode == kEpiSwiglu ? 2 : j.nseg); s < 3; ++s) tb[s] = tb[0];
  a.n_tiles = tiles_n;
  a.tiles = a.m_tiles * a.n_tiles;
  CUtensorMap ta;
  const bool ok = a.batched ? map_heads(&ta, j.x, static_cast<int>(j.T / j.L), j.x_heads, j.L, j.D)
                            : map_rows(&ta, j.x, j.K, j.T);
  if (!ok) return cudaErrorInvalidValue;
  // The pair kernel, one tile per cluster of two SMs (as many clusters as fit at
  // once, found per device); the one-SM kernel only if no such cluster can run.
  int clusters = pair_clusters();
  if (clusters < 0) return cudaErrorUnknown;
  if (clusters > 0) {
    GArgs p = a;
    if (p.batched) {
      p.mt_per_b = (j.L + kG2M - 1) / kG2M;
      p.m_tiles = static_cast<int>(j.T / j.L) * p.mt_per_b;
    } else {
      p.m_tiles = static_cast<int>((j.T + kG2M - 1) / kG2M);
    }
    p.tiles = p.m_tiles * p.n_tiles;
    if (p.tiles < clusters) clusters = p.tiles;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(kGThreads);
    cfg.dynamicSmemBytes = kG2Smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_tc2_kernel, ta, tb[0], tb[1], tb[2], p);
  }
  const int sms = g_sm_count();
  const int grid = a.tiles < sms ? a.tiles : sms;
  gemm_tc_kernel<<<grid, kGThreads, kGSmem, stream>>>(ta, tb[0], tb[1], tb[2], a);
  return cudaGetLastError();
}

}  // namespace gqa
