// Prefill attention on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// What it computes: "Core Layers -- Deep Reference", "Flash Attention" -- the
// exact softmax(Q K^T) V of the causal (or windowed, "mojolearn.transformer"
// window) mask, without materialising the score matrix -- with the query
// heads of one key/value head sharing it ("MHA and GQA": groups of
// n_heads // kv_heads query heads per key/value head).
//
// How, on GB300:
//  * One block owns NQ tiles of 128 query rows. With NQ = 2 the two tiles are
//    two query heads of the same KV group (same positions whenever the group
//    size is even), so every K/V tile brought into shared memory serves both.
//  * TMA (cp.async.bulk.tensor, 128-byte swizzle) streams Q once and K/V
//    blocks of BK keys through an NS-stage ring. Out-of-range rows and
//    columns arrive as zeros.
//  * One thread issues tcgen05.mma (kind::tf32: fp32 data, TF32 products,
//    fp32 accumulation). S = Q K^T goes to tensor memory (two buffers per
//    tile, so the next S is computed while softmax works on this one), and
//    O += P V reads P straight from tensor memory (A operand in TMEM) and
//    V^T from shared memory, accumulating O in TMEM. TF32 operands must be
//    K-major (an MN-major TF32 B operand is not computed on this part), so V
//    arrives transposed: a pre-pass writes V^T [B*Hkv, D, L] into the
//    caller's workspace and TMA streams it like K.
//  * Four softmax warps per tile own one query row per thread: they read S
//    from TMEM, apply scale, softcap and mask, keep the running maximum and
//    sum (base 2), and write P (rounded to TF32) back over S. O is rescaled
//    in TMEM only when the running maximum grows by more than 2^8.
//  * Key blocks entirely outside the causal/window band are never loaded.
//  * Every pipeline wait is bounded; a wait that runs out reports
//    ATTN_DEV_TIMEOUT, the block drains its own copies and MMAs, frees its
//    tensor memory and exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace gqa {

namespace {

constexpr int kBM = 128;                       // query rows per tile = MMA M = TMEM lanes
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;           // rescale O when the max grows by > 2^8
constexpr int kSmemLimit = 232448;             // 227 KB of dynamic shared memory per block
constexpr int kTmemCols = 512;

struct TcArgs {
  float* out;
  int B, H, Hkv, L, D;
  int G, QT, ntiles, npairs;                   // per (b, kv head): tiles and tile groups
  int window;
  int softcap_on;
  float c_score;                               // scale * log2(e)
  float c_cap_in;                              // 2 * log2(e) * scale / cap
  float c_cap_out;                             // log2(e) * cap
  int32_t* status;
};

struct alignas(8) Bars {
  uint64_t q_full;
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t s_full[2][2];
  uint64_t p_ready[2][2];
  uint64_t o_done[2];
  uint64_t o_final[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <int DP_>
struct Cfg {
  static constexpr int DP = DP_;                        // head dim padded to 32
  static constexpr int NQ = DP <= 128 ? 2 : 1;          // query tiles per block
  static constexpr int BK = DP <= 128 ? 64 : 32;        // keys per block
  static constexpr int kChunks = DP / 32;               // 128-byte column chunks
  static constexpr int kQChunk = kBM * 128;
  static constexpr int kQBytes = NQ * kChunks * kQChunk;
  static constexpr int kKVChunk = BK * 128;
  static constexpr int kStage = kChunks * kKVChunk;
  static constexpr int kVtChunk = DP * 128;             // 32 keys x DP rows of V^T
  static constexpr int kNSraw = (kSmemLimit - 2048 - kQBytes) / kStage;
  static constexpr int NS = kNSraw > 8 ? 8 : kNSraw;
  static constexpr int kThreads = 64 + NQ * 128;
  // At least half the SM's shared memory, so exactly one block (and one
  // 512-column tensor-memory allocation) is resident per SM.
  static constexpr int kSmemNeed = kQBytes + NS * kStage + 2048;
  static constexpr int kSmem = kSmemNeed > kSmemLimit / 2 + 4096 ? kSmemNeed
                                                                  : kSmemLimit / 2 + 4096;
  static __host__ __device__ constexpr int o_col(int t) { return t * DP; }
  static __host__ __device__ constexpr int s_col(int t, int b) { return NQ * DP + (2 * t + b) * BK; }
  static_assert(NS >= 2, "shared memory too small for two stages");
  static_assert(NQ * (DP + 2 * BK) <= kTmemCols, "tensor memory budget");
  static_assert(kSmem <= kSmemLimit, "shared memory budget");
};

// Timeout-only wait used while winding down after an abort.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = tc::globaltimer();
  while (!tc::mbar_try_wait(bar, parity)) {
    if (tc::globaltimer() - t0 > tc::kWaitLimitNs) return;
  }
}

struct Unit {
  int b, hk;
  int q0[2], head[2];
  bool valid[2];
  int jlo, n;
};

template <class C>
__device__ __forceinline__ Unit decode_unit(const TcArgs& a) {
  Unit u;
  const int BH = a.B * a.Hkv;
  const int bh = blockIdx.x % BH, pr = blockIdx.x / BH;
  u.b = bh / a.Hkv;
  u.hk = bh % a.Hkv;
  int jlo = 1 << 30, jhi = -1;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int ti = pr * C::NQ + t;
    u.valid[t] = t < C::NQ && ti < a.ntiles;
    const int qt = a.QT - 1 - ti / a.G;                  // heaviest tiles first
    u.q0[t] = qt * kBM;
    u.head[t] = u.hk * a.G + ti % a.G;
    if (u.valid[t]) {
      const int lo = a.window > 0 ? max(0, u.q0[t] - a.window + 1) / C::BK : 0;
      const int hi = min(u.q0[t] + kBM - 1, a.L - 1) / C::BK;
      jlo = min(jlo, lo);
      jhi = max(jhi, hi);
    }
  }
  u.jlo = jlo;
  u.n = jhi - jlo + 1;
  return u;
}

// ---------------------------------------------------------------- producer (one thread)
template <class C>
__device__ void run_producer(const Unit& u, const TcArgs& a, const CUtensorMap* tq,
                             const CUtensorMap* tk, const CUtensorMap* tv, uint8_t* sq,
                             uint8_t* skv, Bars* bars) {
  volatile int* abort = &bars->abort;
  tc::tma_prefetch(tq);
  tc::tma_prefetch(tk);
  tc::tma_prefetch(tv);
  uint32_t qbytes = 0;
#pragma unroll
  for (int t = 0; t < C::NQ; ++t)
    if (u.valid[t]) qbytes += C::kChunks * C::kQChunk;
  tc::mbar_arrive_expect_tx(&bars->q_full, qbytes);
#pragma unroll
  for (int t = 0; t < C::NQ; ++t) {
    if (!u.valid[t]) continue;
    for (int c = 0; c < C::kChunks; ++c)
      tc::tma_load_3d(sq + (t * C::kChunks + c) * C::kQChunk, tq, &bars->q_full, 32 * c, u.q0[t],
                      u.b * a.H + u.head[t]);
  }
  int stage = 0;
  uint32_t phase = 0;
  uint32_t fill_parity[8];
  bool filled[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) filled[s] = false;
  // A K block: BK rows of 32-column chunks. A V^T block: BK/32 chunks of 32
  // keys, each DP rows (one per head dimension).
  auto load = [&](bool is_v, int j) -> bool {
    if (!tc::mbar_wait(&bars->kv_empty[stage], phase ^ 1u, abort)) return false;
    tc::mbar_arrive_expect_tx(&bars->kv_full[stage], C::kStage);
    uint8_t* dst = skv + stage * C::kStage;
    if (!is_v) {
      for (int c = 0; c < C::kChunks; ++c)
        tc::tma_load_3d(dst + c * C::kKVChunk, tk, &bars->kv_full[stage], 32 * c, j * C::BK,
                        u.b * a.Hkv + u.hk);
    } else {
      for (int c = 0; c < C::BK / 32; ++c)
        tc::tma_load_3d(dst + c * C::kVtChunk, tv, &bars->kv_full[stage], j * C::BK + 32 * c, 0,
                        u.b * a.Hkv + u.hk);
    }
    filled[stage] = true;
    fill_parity[stage] = phase;
    if (++stage == C::NS) {
      stage = 0;
      phase ^= 1u;
    }
    return true;
  };
  // Order of use by the MMA issuer: K_0, then (K_{i+1}, V_i) for each block i.
  bool ok = load(false, u.jlo);
  for (int i = 0; ok && i < u.n; ++i) {
    if (i + 1 < u.n) ok = load(false, u.jlo + i + 1);
    if (ok) ok = load(true, u.jlo + i);
  }
  (void)ok;
  // Every copy this block started lands before the block may exit, whether or
  // not the consumers saw it (they may have stopped on an abort).
  drain_wait(&bars->q_full, 0);
  for (int s = 0; s < C::NS; ++s)
    if (filled[s]) drain_wait(&bars->kv_full[s], fill_parity[s]);
}

// ---------------------------------------------------------------- MMA issuer (one thread)
template <class C>
__device__ void run_mma(const Unit& u, uint32_t tmem, uint8_t* sq, uint8_t* skv, Bars* bars) {
  volatile int* abort = &bars->abort;
  constexpr uint32_t id_s = tc::idesc_tf32(kBM, C::BK, false);
  constexpr uint32_t id_pv = tc::idesc_tf32(kBM, C::DP, false);
  int stage = 0;
  uint32_t phase = 0;
  auto next = [&](int& st) -> bool {
    if (!tc::mbar_wait(&bars->kv_full[stage], phase, abort)) return false;
    st = stage;
    if (++stage == C::NS) {
      stage = 0;
      phase ^= 1u;
    }
    return true;
  };
  // S_t[buf] = Q_t K^T: K-major A (Q) and B (K), 8 columns of D per instruction.
  auto issue_s = [&](int t, int buf, int st) {
    const uint32_t d = tmem + C::s_col(t, buf);
    const uint32_t qa = tc::smem_u32(sq + t * C::kChunks * C::kQChunk);
    const uint32_t kb = tc::smem_u32(skv + st * C::kStage);
#pragma unroll
    for (int kk = 0; kk < C::DP / 8; ++kk) {
      const int c = kk / 4, off = (kk % 4) * 32;
      tc::mma_tf32_ss(d, tc::sdesc_sw128(qa + c * C::kQChunk + off, 16, 1024),
                      tc::sdesc_sw128(kb + c * C::kKVChunk + off, 16, 1024), id_s, kk > 0);
    }
  };
  // O_t += P_t[buf] V: A from tensor memory, B = V^T (K-major, keys contiguous).
  auto issue_pv = [&](int t, int buf, int st, bool acc) {
    const uint32_t d = tmem + C::o_col(t);
    const uint32_t vb = tc::smem_u32(skv + st * C::kStage);
#pragma unroll
    for (int kk = 0; kk < C::BK / 8; ++kk) {
      const int c = kk / 4, off = (kk % 4) * 32;
      tc::mma_tf32_ts(d, tmem + C::s_col(t, buf) + 8 * kk,
                      tc::sdesc_sw128(vb + c * C::kVtChunk + off, 16, 1024), id_pv,
                      (acc || kk > 0) ? 1u : 0u);
    }
  };

  bool ok = tc::mbar_wait(&bars->q_full, 0, abort);
  int st = 0;
  if (ok) ok = next(st);
  if (ok) {
    tc::fence_after_sync();
#pragma unroll
    for (int t = 0; t < C::NQ; ++t)
      if (u.valid[t]) {
        issue_s(t, 0, st);
        tc::mma_commit(&bars->s_full[t][0]);
      }
    tc::mma_commit(&bars->kv_empty[st]);
  }
  for (int i = 0; ok && i < u.n; ++i) {
    if (i + 1 < u.n) {
      if (!(ok = next(st))) break;
#pragma unroll
      for (int t = 0; t < C::NQ; ++t)
        if (u.valid[t]) {
          issue_s(t, (i + 1) & 1, st);
          tc::mma_commit(&bars->s_full[t][(i + 1) & 1]);
        }
      tc::mma_commit(&bars->kv_empty[st]);
    }
    if (!(ok = next(st))) break;
#pragma unroll
    for (int t = 0; t < C::NQ; ++t) {
      if (!u.valid[t]) continue;
      if (!(ok = tc::mbar_wait(&bars->p_ready[t][i & 1], (i >> 1) & 1, abort))) break;
      tc::fence_after_sync();
      issue_pv(t, i & 1, st, i > 0);
      tc::mma_commit(&bars->o_done[t]);
    }
    if (!ok) break;
    tc::mma_commit(&bars->kv_empty[st]);
  }
#pragma unroll
  for (int t = 0; t < C::NQ; ++t)
    if (u.valid[t]) tc::mma_commit(&bars->o_final[t]);
  // No MMA may still run when the block frees its tensor memory.
  tc::mma_commit(&bars->drain);
  drain_wait(&bars->drain, 0);
}

// ---------------------------------------------------------------- softmax (4 warps per tile)
// Thread = one query row. All tcgen05.ld/st below run on full warps.
template <class C>
__device__ void run_softmax(const Unit& u, const TcArgs& a, uint32_t tmem, Bars* bars, int t,
                            int quarter, int lane) {
  volatile int* abort = &bars->abort;
  const int row = quarter * 32 + lane;
  const int qpos = u.q0[t] + row;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  float m_ref = -INFINITY, l = 0.f;
  bool ok = true;

  for (int i = 0; i < u.n; ++i) {
    const int buf = i & 1;
    ok = tc::mbar_wait(&bars->s_full[t][buf], (i >> 1) & 1, abort);
    if (__any_sync(0xffffffffu, !ok)) {       // leave together: tcgen05.ld is warp-wide
      ok = false;
      break;
    }
    tc::fence_after_sync();
    float s[C::BK];
#pragma unroll
    for (int c = 0; c < C::BK; c += 32) tc::tmem_ld32(lane_base + C::s_col(t, buf) + c, s + c);

    // scores in log2 units, optionally softcapped: cap * tanh(score / cap)
    if (a.softcap_on) {
#pragma unroll
      for (int c = 0; c < C::BK; ++c) {
        const float e = exp2f(s[c] * a.c_cap_in);
        s[c] = a.c_cap_out - __fdividef(2.0f * a.c_cap_out, e + 1.0f);
      }
    } else {
#pragma unroll
      for (int c = 0; c < C::BK; ++c) s[c] *= a.c_score;
    }
    const int k0 = (u.jlo + i) * C::BK;
    const bool whole = (k0 + C::BK - 1 <= qpos) && (a.window == 0 || k0 > qpos - a.window);
    if (!whole) {
#pragma unroll
      for (int c = 0; c < C::BK; ++c) {
        const int kp = k0 + c;
        if (kp > qpos || (a.window > 0 && kp <= qpos - a.window)) s[c] = -INFINITY;
      }
    }
    float mb = s[0];
#pragma unroll
    for (int c = 1; c < C::BK; ++c) mb = fmaxf(mb, s[c]);
    const float m_new = fmaxf(m_ref, mb);

    // Rescale O only when the running maximum has grown a lot (warp-uniform).
    const bool grow = m_ref != -INFINITY && m_new - m_ref > kRescaleLog2;
    if (__any_sync(0xffffffffu, grow)) {
      ok = tc::mbar_wait(&bars->o_done[t], (i - 1) & 1, abort);
      if (__any_sync(0xffffffffu, !ok)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const float f = grow ? exp2f(m_ref - m_new) : 1.0f;
#pragma unroll 1
      for (int c = 0; c < C::DP; c += 32) {
        float o[32];
        tc::tmem_ld32(lane_base + C::o_col(t) + c, o);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] *= f;
        tc::tmem_st32(lane_base + C::o_col(t) + c, o);
      }
      if (grow) {
        l *= f;
        m_ref = m_new;
      }
    }
    if (m_ref == -INFINITY) m_ref = m_new;      // first visible keys of this row (O, l are 0)

    float ps = 0.f;
#pragma unroll
    for (int c = 0; c < C::BK; ++c) {
      const float p = m_ref == -INFINITY ? 0.f : tc::round_tf32(exp2f(s[c] - m_ref));
      ps += p;
      s[c] = p;
    }
    l += ps;
#pragma unroll
    for (int c = 0; c < C::BK; c += 32) tc::tmem_st32(lane_base + C::s_col(t, buf) + c, s + c);
    tc::fence_before_sync();
    tc::mbar_arrive(&bars->p_ready[t][buf]);
  }

  // Epilogue: O / l to global memory, row by row.
  if (ok) ok = tc::mbar_wait(&bars->o_final[t], 0, abort);
  if (__any_sync(0xffffffffu, !ok || *abort)) return;
  tc::fence_after_sync();
  const float inv = 1.0f / l;
  const bool live = qpos < a.L;
  float* dst = a.out + ((static_cast<long>(u.b) * a.H + u.head[t]) * a.L + qpos) * a.D;
#pragma unroll 1
  for (int c = 0; c < C::DP; c += 32) {
    float o[32];
    tc::tmem_ld32(lane_base + C::o_col(t) + c, o);
    if (live) {
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        if (c + e < a.D)
          *reinterpret_cast<float4*>(dst + c + e) =
              make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv, o[e + 3] * inv);
      }
    }
  }
}

template <int DP>
__global__ void __launch_bounds__(Cfg<DP>::kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const TcArgs a) {
  using C = Cfg<DP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sq = smem;
  uint8_t* skv = smem + C::kQBytes;
  Bars* bars = reinterpret_cast<Bars*>(skv + C::NS * C::kStage);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const Unit u = decode_unit<C>(a);

  if (threadIdx.x == 0) {
    tc::mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::NS; ++s) {
      tc::mbar_init(&bars->kv_full[s], 1);
      tc::mbar_init(&bars->kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      for (int b = 0; b < 2; ++b) {
        tc::mbar_init(&bars->s_full[t][b], 1);
        tc::mbar_init(&bars->p_ready[t][b], 128);
      }
      tc::mbar_init(&bars->o_done[t], 1);
      tc::mbar_init(&bars->o_final[t], 1);
    }
    tc::mbar_init(&bars->drain, 1);
    bars->abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&bars->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    if (lane == 0) run_producer<C>(u, a, &tm_q, &tm_k, &tm_v, sq, skv, bars);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) run_mma<C>(u, tmem, sq, skv, bars);
    __syncwarp();
  } else {
    const int t = (warp - 2) / 4;
    if (u.valid[t]) run_softmax<C>(u, a, tmem, bars, t, warp % 4, lane);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && bars->abort) report(a.status, ATTN_DEV_TIMEOUT);
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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
bool make_map(CUtensorMap* m, const float* base, int D, int L, int NH, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(NH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4,
                                 static_cast<cuuint64_t>(L) * D * 4};
  const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// V^T [B*Hkv, D, L] (rows of pitch Lp) for TMA: boxes of 32 keys x box_rows dims.
bool make_map_vt(CUtensorMap* m, const float* base, int D, int L, int Lp, int NH, int box_rows) {
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

// vt[bh, d, l] = v[bh, l, d], 32 x 32 tiles through shared memory.
__global__ void __launch_bounds__(256) transpose_v_kernel(const float* __restrict__ v,
                                                          float* __restrict__ vt, int L, int D,
                                                          int Lp) {
  __shared__ float tile[32][33];
  const long bh = blockIdx.z;
  const int l0 = blockIdx.x * 32, d0 = blockIdx.y * 32;
  const float* src = v + bh * L * D;
  float* dst = vt + bh * D * Lp;
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int l = l0 + r, d = d0 + threadIdx.x;
    tile[r][threadIdx.x] = (l < L && d < D) ? src[static_cast<long>(l) * D + d] : 0.f;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int d = d0 + r, l = l0 + threadIdx.x;
    if (d < D && l < L) dst[static_cast<long>(d) * Lp + l] = tile[threadIdx.x][r];
  }
}

template <int DP>
cudaError_t launch_dp(const AttnShape& s, cudaStream_t stream) {
  using C = Cfg<DP>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(prefill_tc_kernel<DP>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, s.q, s.D, s.L, s.B * s.H, kBM) ||
      !make_map(&tk, s.k, s.D, s.L, s.B * s.Hkv, C::BK) ||
      !make_map_vt(&tv, s.vt, s.D, s.L, s.vt_pitch, s.B * s.Hkv, C::DP))
    return cudaErrorInvalidValue;
  transpose_v_kernel<<<dim3((s.L + 31) / 32, (s.D + 31) / 32, s.B * s.Hkv), dim3(32, 8), 0,
                       stream>>>(s.v, s.vt, s.L, s.D, s.vt_pitch);
  if (cudaError_t e = cudaGetLastError(); e != cudaSuccess) return e;
  TcArgs a{};
  a.out = s.out;
  a.B = s.B; a.H = s.H; a.Hkv = s.Hkv; a.L = s.L; a.D = s.D;
  a.G = s.H / s.Hkv;
  a.QT = (s.L + kBM - 1) / kBM;
  a.ntiles = a.G * a.QT;
  a.npairs = (a.ntiles + C::NQ - 1) / C::NQ;
  a.window = s.window;
  a.softcap_on = s.softcap > 0.f;
  a.c_score = s.scale * kLog2e;
  a.c_cap_in = s.softcap > 0.f ? 2.0f * kLog2e * s.scale / s.softcap : 0.f;
  a.c_cap_out = kLog2e * s.softcap;
  a.status = s.status;
  const long grid = static_cast<long>(s.B) * s.Hkv * a.npairs;
  prefill_tc_kernel<DP><<<static_cast<unsigned>(grid), C::kThreads, C::kSmem, stream>>>(tq, tk, tv,
                                                                                        a);
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supports(int D) { return D % 4 == 0 && D >= 32 && D <= kMaxHeadDim; }

int prefill_vt_pitch(int L) { return (L + 3) / 4 * 4; }

cudaError_t launch_prefill_tc(const AttnShape& s, cudaStream_t stream) {
  if (!prefill_tc_supports(s.D)) return cudaErrorNotSupported;
  switch ((s.D + 31) / 32) {
    case 1: return launch_dp<32>(s, stream);
    case 2: return launch_dp<64>(s, stream);
    case 3: return launch_dp<96>(s, stream);
    case 4: return launch_dp<128>(s, stream);
    case 5: return launch_dp<160>(s, stream);
    case 6: return launch_dp<192>(s, stream);
    case 7: return launch_dp<224>(s, stream);
    default: return launch_dp<256>(s, stream);
  }
}

}  // namespace gqa
