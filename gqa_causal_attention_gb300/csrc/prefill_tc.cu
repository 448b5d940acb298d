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
#include "prefill_common.cuh"

namespace gqa {

namespace {

using namespace prefill;

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

// Two shapes. DP <= 128: Q lives in tensor memory (A operand of S = Q K^T
// from TMEM), 128-key blocks (N = 128 MMAs run at the full TF32 rate) and a
// double-buffered S: TMEM = Q | O | S0 | S1. DP > 128: Q stays in shared
// memory and 32-key blocks keep K/V stages within the 227 KB.
template <int DP_>
struct Cfg {
  static constexpr int DP = DP_;                        // head dim padded to 32
  static constexpr bool QTM = DP <= 128;                // Q in tensor memory
  static constexpr int NQ = 1;                          // query tiles per block
  static constexpr int BK = QTM ? 128 : 32;             // keys per block
  static constexpr int kChunks = DP / 32;               // 128-byte column chunks
  static constexpr int kQChunk = kBM * 128;
  static constexpr int kQBytes = QTM ? 0 : NQ * kChunks * kQChunk;
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
  static constexpr int kQCol = 0;                       // QTM: Q columns [0, DP)
  static constexpr int kOBase = QTM ? DP : 0;
  static __host__ __device__ constexpr int o_col(int t) { return kOBase + t * DP; }
  static __host__ __device__ constexpr int s_col(int t, int b) {
    return kOBase + NQ * DP + (2 * t + b) * BK;
  }
  static_assert(NS >= 2, "shared memory too small for two stages");
  static_assert(kOBase + NQ * (DP + 2 * BK) <= kTmemCols, "tensor memory budget");
  static_assert(kSmem <= kSmemLimit, "shared memory budget");
};

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
  if constexpr (!C::QTM) {
    uint32_t qbytes = 0;
#pragma unroll
    for (int t = 0; t < C::NQ; ++t)
      if (u.valid[t]) qbytes += C::kChunks * C::kQChunk;
    tc::mbar_arrive_expect_tx(&bars->q_full, qbytes);
#pragma unroll
    for (int t = 0; t < C::NQ; ++t) {
      if (!u.valid[t]) continue;
      for (int c = 0; c < C::kChunks; ++c)
        tc::tma_load_3d(sq + (t * C::kChunks + c) * C::kQChunk, tq, &bars->q_full, 32 * c,
                        u.q0[t], u.b * a.H + u.head[t]);
    }
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
  if constexpr (!C::QTM) drain_wait(&bars->q_full, 0);
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
  // Descriptors are built once; an operand offset is added to the start-address
  // field (address >> 4), which stays below 2^14 for any shared-memory address.
  uint64_t qdesc[2];
#pragma unroll
  for (int t = 0; t < 2; ++t)
    qdesc[t] = tc::sdesc_sw128(tc::smem_u32(sq + (t < C::NQ ? t : 0) * C::kChunks * C::kQChunk),
                               16, 1024);
  const uint64_t kvdesc = tc::sdesc_sw128(tc::smem_u32(skv), 16, 1024);
  // S_t[buf] = Q_t K^T: K-major A (Q) and B (K), 8 columns of D per instruction.
  auto issue_s = [&](int t, int buf, int st) {
    const uint32_t d = tmem + C::s_col(t, buf);
    const uint64_t qd = qdesc[t];
    const uint64_t kd = kvdesc + static_cast<uint32_t>((st * C::kStage) >> 4);
#pragma unroll
    for (int kk = 0; kk < C::DP / 8; ++kk) {
      const int c = kk / 4, off = (kk % 4) * 32;
      if constexpr (C::QTM)
        tc::mma_tf32_ts(d, tmem + C::kQCol + 8 * kk, kd + ((c * C::kKVChunk + off) >> 4), id_s,
                        kk > 0);
      else
        tc::mma_tf32_ss(d, qd + ((c * C::kQChunk + off) >> 4),
                        kd + ((c * C::kKVChunk + off) >> 4), id_s, kk > 0);
    }
  };
  // O_t += P_t[buf] V: A from tensor memory, B = V^T (K-major, keys contiguous).
  auto issue_pv = [&](int t, int buf, int st, bool acc) {
    const uint32_t d = tmem + C::o_col(t);
    const uint64_t vd = kvdesc + static_cast<uint32_t>((st * C::kStage) >> 4);
#pragma unroll
    for (int kk = 0; kk < C::BK / 8; ++kk) {
      const int c = kk / 4, off = (kk % 4) * 32;
      tc::mma_tf32_ts(d, tmem + C::s_col(t, buf) + 8 * kk, vd + ((c * C::kVtChunk + off) >> 4),
                      id_pv, (acc || kk > 0) ? 1u : 0u);
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
  constexpr int BK = C::BK;
  constexpr int NA = 8;                       // independent partial max / sum chains
  volatile int* abort = &bars->abort;
  const int row = quarter * 32 + lane;
  const int qpos = u.q0[t] + row;
  const int Lb = row_len(a, u.b);             // keys at or past the row's length: masked
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  // Running max m (log2 units, of the scaled and capped scores) and sum l.
  float m_ref = -INFINITY, l = 0.f;
  bool ok = true;

  if constexpr (C::QTM) {
    // This thread's query row goes into the Q columns of its TMEM lane (zeros
    // past the sequence end and past D), then the MMA issuer may start.
    const bool live = qpos < a.L;
    const float* src = a.q + ((static_cast<long>(u.b) * a.H + u.head[t]) * a.L + qpos) * a.D;
#pragma unroll 1
    for (int c = 0; c < C::DP; c += 32) {
      float qv[32];
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live && c + e < a.D) x = __ldg(reinterpret_cast<const float4*>(src + c + e));
        qv[e] = x.x; qv[e + 1] = x.y; qv[e + 2] = x.z; qv[e + 3] = x.w;
      }
      tc::tmem_st32(lane_base + C::kQCol + c, qv);
    }
    tc::fence_before_sync();
    tc::mbar_arrive(&bars->q_full);
  }

  for (int i = 0; i < u.n; ++i) {
    const int buf = i & 1;
    ok = tc::mbar_wait(&bars->s_full[t][buf], (i >> 1) & 1, abort);
    if (__any_sync(0xffffffffu, !ok)) {       // leave together: tcgen05.ld is warp-wide
      ok = false;
      break;
    }
    tc::fence_after_sync();
    float s[BK];
    tmem_ld_row<BK>(lane_base + C::s_col(t, buf), s);

    // Softcap turns raw scores into log2-unit capped scores:
    // log2(e) * cap * tanh(scale * s / cap) = c_out - 2 c_out / (2^(s c_in) + 1).
    if (a.softcap_on) {
#pragma unroll
      for (int c = 0; c < BK; ++c) {
        const float e = tc::ex2(s[c] * a.c_cap_in);
        s[c] = fmaf(-2.0f * a.c_cap_out, tc::rcp(e + 1.0f), a.c_cap_out);
      }
    }
    // Keys outside the causal / window band of this row (boundary blocks only).
    const int k0 = (u.jlo + i) * BK;
    const int hi = min(qpos, Lb - 1) - k0;                        // visible: c <= hi
    const int lo = a.window > 0 ? qpos - a.window + 1 - k0 : -1;  // visible: c >= lo
    // One compare and select per column (a combined condition compiles to
    // per-column branches that diverge across the rows of a warp).
    if (hi < BK - 1) {
#pragma unroll
      for (int c = 0; c < BK; ++c) s[c] = c > hi ? -INFINITY : s[c];
    }
    if (lo > 0) {
#pragma unroll
      for (int c = 0; c < BK; ++c) s[c] = c < lo ? -INFINITY : s[c];
    }
    float mx[NA];
#pragma unroll
    for (int j = 0; j < NA; ++j) mx[j] = s[j];
#pragma unroll
    for (int c = NA; c < BK; ++c) mx[c % NA] = fmaxf(mx[c % NA], s[c]);
#pragma unroll
    for (int j = NA / 2; j > 0; j /= 2)
#pragma unroll
      for (int q = 0; q < j; ++q) mx[q] = fmaxf(mx[q], mx[q + j]);
    // Scores in log2 units: capped ones already are; plain ones get scale * log2(e).
    const float cs = a.softcap_on ? 1.0f : a.c_score;
    const float m_new = fmaxf(m_ref, mx[0] * cs);

    // Rescale O only when the running maximum has grown a lot (warp-uniform).
    const bool grow = m_ref != -INFINITY && m_new - m_ref > kRescaleLog2;
    if (__any_sync(0xffffffffu, grow)) {
      ok = tc::mbar_wait(&bars->o_done[t], (i - 1) & 1, abort);
      if (__any_sync(0xffffffffu, !ok)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const float f = grow ? tc::ex2(m_ref - m_new) : 1.0f;
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
    if (m_ref == -INFINITY) m_ref = m_new;    // first visible keys of the row (O, l are 0)
    // Reference for the exponent: -inf only while every key so far was masked,
    // and then every score is -inf too, so any finite value gives p = 0.
    const float mref = m_ref == -INFINITY ? 0.f : m_ref;

    // p = 2^(score - m), truncated to the TF32 value the tensor core will use, so
    // that l sums exactly the weights applied to V.
    float ps[NA];
#pragma unroll
    for (int j = 0; j < NA; ++j) ps[j] = 0.f;
#pragma unroll
    for (int c = 0; c < BK; ++c) {
      const float p = tc::trunc_tf32(tc::ex2(fmaf(s[c], cs, -mref)));
      ps[c % NA] += p;
      s[c] = p;
    }
#pragma unroll
    for (int j = NA / 2; j > 0; j /= 2)
#pragma unroll
      for (int q = 0; q < j; ++q) ps[q] += ps[q + j];
    l += ps[0];
    tmem_st_row<BK>(lane_base + C::s_col(t, buf), s);
    tc::fence_before_sync();
    tc::mbar_arrive(&bars->p_ready[t][buf]);
  }

  // Epilogue: O / l to global memory, row by row.
  if (ok) ok = tc::mbar_wait(&bars->o_final[t], 0, abort);
  if (__any_sync(0xffffffffu, !ok || *abort)) return;
  tc::fence_after_sync();
  // Padding rows of a ragged batch (qpos >= Lb) are written as +0.0.
  const float inv = qpos < Lb ? 1.0f / l : 0.f;
  const bool live = qpos < a.L;
  float* dst = a.out + ((static_cast<long>(u.b) * a.H + u.head[t]) * a.L + qpos) * a.D;
#pragma unroll 1
  for (int c = 0; c < C::DP; c += 32) {
    float o[32];
    tc::tmem_ld32(lane_base + C::o_col(t) + c, o);
    if (qpos >= Lb) {
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = 0.f;
    }
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
    tc::mbar_init(&bars->q_full, C::QTM ? 128 : 1);
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

// vt[bh, d, l] = v[bh, l, d] for D % 4 == 0: 32 x 32 tiles through shared
// memory, 16-byte loads along d and 16-byte stores along l (rows of vt have a
// pitch Lp that is a multiple of 4, so a store may run into the padding).
__global__ void __launch_bounds__(256) transpose_v_kernel(const float* __restrict__ v,
                                                          float* __restrict__ vt, int L, int D,
                                                          int Lp, const int32_t* lengths,
                                                          int Hkv, int32_t* status) {
  __shared__ float tile[32][33];
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
  TcArgs a{};
  a.q = s.q;
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
  a.lengths = s.lengths;
  const long grid = static_cast<long>(s.B) * s.Hkv * a.npairs;
  prefill_tc_kernel<DP><<<static_cast<unsigned>(grid), C::kThreads, C::kSmem, stream>>>(tq, tk, tv,
                                                                                        a);
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supports(int D) { return D % 4 == 0 && D >= 32 && D <= kMaxHeadDim; }

int prefill_vt_pitch(int L) { return (L + 3) / 4 * 4; }

cudaError_t launch_transpose_v(const float* v, float* vt, int BHkv, int L, int D, int vt_pitch,
                               cudaStream_t stream, const int32_t* lengths, int Hkv,
                               int32_t* status) {
  transpose_v_kernel<<<dim3((L + 31) / 32, (D + 31) / 32, BHkv), 256, 0, stream>>>(
      v, vt, L, D, vt_pitch, lengths, Hkv, status);
  return cudaGetLastError();
}

cudaError_t launch_prefill_tc(const AttnShape& s, cudaStream_t stream) {
  if (!prefill_tc_supports(s.D)) return cudaErrorNotSupported;
  if (cudaError_t e = launch_transpose_v(s.v, s.vt, s.B * s.Hkv, s.L, s.D, s.vt_pitch, stream,
                                         s.lengths, s.Hkv, s.status);
      e != cudaSuccess)
    return e;
  return launch_prefill_tc_vt(s, stream);
}

cudaError_t launch_prefill_tc_vt(const AttnShape& s, cudaStream_t stream) {
  if (!prefill_tc_supports(s.D)) return cudaErrorNotSupported;
  if (s.D <= 128) return launch_prefill_tq(s, stream);
  switch ((s.D + 31) / 32) {
    case 5: return launch_dp<160>(s, stream);
    case 6: return launch_dp<192>(s, stream);
    case 7: return launch_dp<224>(s, stream);
    default: return launch_dp<256>(s, stream);
  }
}

}  // namespace gqa
