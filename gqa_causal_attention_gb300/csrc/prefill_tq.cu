// Persistent tensor-core prefill for head dimensions up to 128.
//
// Same computation as prefill_tc.cu ("Core Layers -- Deep Reference", "Flash
// Attention"; causal or windowed mask of "mojolearn.transformer"), organised
// for GB300 throughput:
//  * One block per SM walks a list of work units (one 128-row query tile of
//    one head each), heaviest tiles first, in snake order across blocks.
//  * Q sits in tensor memory as the A operand of S = Q K^T, so the MMA reads
//    only K (and later V^T) from shared memory; blocks of 128 keys give
//    M128 N128 K8 TF32 instructions, which run at the full tensor rate.
//    TMEM = Q | O | S0 | S1 (S double-buffered: S of the next key block is
//    computed while softmax turns this one into P).
//  * TMA streams Q tiles, K blocks and V^T blocks of successive units through
//    one ring of stages. The MMA issuer moves each Q tile from shared to
//    tensor memory with tcgen05.cp, in order with its MMAs, so the next
//    unit's first S products overlap the previous unit's last softmax and its
//    epilogue; only the first P V of a unit waits for O to be read out.
//  * With q RoPE fused (gqa_attn_prefill_rope), the softmax warps rotate each
//    Q tile in tensor memory after tcgen05.cp and before its first S MMA (the
//    tile enters the ring right after the previous unit's last K block, so
//    this overlaps that unit's last P V products).
//  * Softmax, masking, softcap, rescaling and the epilogue are those of the
//    non-persistent kernel (one query row per thread, base-2 online softmax,
//    P truncated to TF32 in place of S).
//  * Every pipeline wait is bounded; a wait that runs out reports
//    ATTN_DEV_TIMEOUT and the block winds down (drains its copies and MMAs,
//    frees its tensor memory).
#include "prefill_common.cuh"

namespace gqa {

namespace {

using namespace prefill;

template <int DP_>
struct PCfg {
  static constexpr int DP = DP_;
  static constexpr int BK = 128;                        // keys per block
  static constexpr int kChunks = DP / 32;
  static constexpr int kKChunk = BK * 128;              // 128 rows x 128 B (K block or Q tile)
  static constexpr int kVtChunk = DP * 128;             // DP rows x 128 B (32 keys of V^T)
  static constexpr int kStage = kChunks * kKChunk;      // one K block, V^T block or Q tile
  static constexpr int kEpi = 4 * 4096;                 // per-warp 32 x 32 output staging
  static constexpr int kNSraw = (kSmemLimit - 2048 - kEpi) / kStage;
  static constexpr int NS = kNSraw > 8 ? 8 : kNSraw;
  static constexpr int kThreads = 64 + 128;          // producer, MMA, 4 softmax
  static constexpr int kSmemNeed = NS * kStage + kEpi + 2048;
  static constexpr int kSmem =
      kSmemNeed > kSmemLimit / 2 + 4096 ? kSmemNeed : kSmemLimit / 2 + 4096;
  static constexpr int kQCol = 0, kOCol = DP, kSCol = 2 * DP;
  static_assert(NS >= 3, "ring too short");
  static_assert(kSCol + 2 * BK <= kTmemCols, "tensor memory budget");
  static_assert(kSmem <= kSmemLimit, "shared memory budget");
};

struct PBars {
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t s_full[2];
  uint64_t p_ready[2];
  uint64_t o_done;
  uint64_t o_final;
  uint64_t o_free;
  uint64_t q_copied;                           // a Q tile is in tensor memory (one phase per unit)
  uint64_t q_ready;                            // fused RoPE: that Q tile is rotated
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct PUnit {
  int b, h, q0, jlo, n;
  int qk0;                                    // key index of query row q0 (q0 + kv_off[b])
};

// Unit x of round r for block c: snake order evens out the heavy-first list.
__device__ __forceinline__ int unit_of(int c, int r, int nblocks) {
  return r * nblocks + ((r & 1) ? nblocks - 1 - c : c);
}

template <class C>
__device__ __forceinline__ PUnit get_unit(const TcArgs& a, int x) {
  PUnit u;
  const int BH = a.B * a.H;
  const int rank = x / BH, bh = x % BH;
  u.b = bh / a.H;
  u.h = bh % a.H;
  u.q0 = (a.QT - 1 - rank) * kBM;
  const int off = a.kv_off ? a.kv_off[u.b] : 0;
  u.qk0 = u.q0 + off;
  const int lo = a.window > 0 ? max(0, u.qk0 - a.window + 1) / C::BK : 0;
  const int hi = min(u.qk0 + kBM - 1, off + a.L - 1) / C::BK;
  u.jlo = lo;
  u.n = hi - lo + 1;
  return u;
}

// ---------------------------------------------------------------- producer (one thread)
// Ring order: the first unit's Q tile; then per unit K_0 .. K_{n-1} interleaved
// with V^T_0 .. V^T_{n-1} as K_0, (K_{i+1}, V^T_i)..., and the next unit's Q
// tile. With fused RoPE that Q tile comes right after this unit's last K block,
// so it lands while this unit's last P V products are pending and the softmax
// warps can rotate it in tensor memory before the next unit's first S = Q K^T;
// otherwise it comes after the last V^T block.
template <class C>
__device__ void tq_producer(const TcArgs& a, const CUtensorMap* tq, const CUtensorMap* tk,
                            const CUtensorMap* tv, uint8_t* skv, PBars* bars) {
  volatile int* abort = &bars->abort;
  tc::tma_prefetch(tq);
  tc::tma_prefetch(tk);
  tc::tma_prefetch(tv);
  int stage = 0;
  uint32_t phase = 0;
  uint32_t fill_parity[8];
  bool filled[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) filled[s] = false;
  // kind: 0 = Q tile, 1 = K block, 2 = V^T block
  auto load = [&](int kind, const PUnit& u, int j) -> bool {
    if (!tc::mbar_wait(&bars->kv_empty[stage], phase ^ 1u, abort)) return false;
    uint64_t* full = &bars->kv_full[stage];
    tc::mbar_arrive_expect_tx(full, C::kStage);
    uint8_t* dst = skv + stage * C::kStage;
    if (kind == 0) {
      for (int c = 0; c < C::kChunks; ++c)
        tc::tma_load_3d(dst + c * C::kKChunk, tq, full, 32 * c, u.q0, u.b * a.H + u.h);
    } else if (kind == 1) {
      for (int c = 0; c < C::kChunks; ++c)
        tc::tma_load_3d(dst + c * C::kKChunk, tk, full, 32 * c, j * C::BK,
                        u.b * a.Hkv + u.h / a.G);
    } else {
      for (int c = 0; c < C::BK / 32; ++c)
        tc::tma_load_3d(dst + c * C::kVtChunk, tv, full, j * C::BK + 32 * c, 0,
                        u.b * a.Hkv + u.h / a.G);
    }
    filled[stage] = true;
    fill_parity[stage] = phase;
    if (++stage == C::NS) {
      stage = 0;
      phase ^= 1u;
    }
    return true;
  };
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int x = unit_of(blockIdx.x, r, gridDim.x);
    if (x >= a.units) break;
    const PUnit u = get_unit<C>(a, x);
    const int xn = unit_of(blockIdx.x, r + 1, gridDim.x);
    const bool has_next = xn < a.units;
    const PUnit un = get_unit<C>(a, has_next ? xn : x);
    // Warm the next Q tile into L2 now: its load comes within a few blocks.
    if (has_next)
      for (int c = 0; c < C::kChunks; ++c)
        tc::tma_prefetch_l2_3d(tq, 32 * c, un.q0, un.b * a.H + un.h);
    const bool early = a.rope_table && has_next;  // next Q after the last K, else after the last V
    if (r == 0) ok = load(0, u, 0);
    if (ok) ok = load(1, u, u.jlo);
    if (ok && u.n == 1 && early) ok = load(0, un, 0);
    for (int i = 0; ok && i < u.n; ++i) {
      if (i + 1 < u.n) {
        ok = load(1, u, u.jlo + i + 1);
        if (ok && i + 2 == u.n && early) ok = load(0, un, 0);
      }
      if (ok) ok = load(2, u, u.jlo + i);
    }
    if (ok && has_next && !early) ok = load(0, un, 0);
  }
  // Every copy this block started lands before the block may exit.
  for (int s = 0; s < C::NS; ++s)
    if (filled[s]) drain_wait(&bars->kv_full[s], fill_parity[s]);
}

// ---------------------------------------------------------------- MMA issuer (one thread)
template <class C>
__device__ void tq_mma(const TcArgs& a, uint32_t tmem, uint8_t* skv, PBars* bars) {
  volatile int* abort = &bars->abort;
  constexpr uint32_t id_s = tc::idesc_tf32(kBM, C::BK, false);
  constexpr uint32_t id_pv = tc::idesc_tf32(kBM, C::DP, false);
  // Descriptors are built once; an operand offset is added to the start-address
  // field (address >> 4), which stays below 2^14 for any shared-memory address.
  const uint64_t base_desc = tc::sdesc_sw128(tc::smem_u32(skv), 16, 1024);
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
  auto stage_desc = [&](int st) { return base_desc + static_cast<uint32_t>((st * C::kStage) >> 4); };
  // S[buf] = Q K^T: A = Q from TMEM, B = K block (K-major).
  auto issue_s = [&](int buf, int st) {
    const uint32_t d = tmem + C::kSCol + buf * C::BK;
    const uint64_t kd = stage_desc(st);
#pragma unroll
    for (int kk = 0; kk < C::DP / 8; ++kk) {
      const int c = kk / 4, off = (kk % 4) * 32;
      tc::mma_tf32_ts(d, tmem + C::kQCol + 8 * kk, kd + ((c * C::kKChunk + off) >> 4), id_s,
                      kk > 0);
    }
  };
  // O += P V: A = P from TMEM (in place of S), B = V^T block (K-major).
  auto issue_pv = [&](int buf, int st, bool acc) {
    const uint32_t d = tmem + C::kOCol;
    const uint64_t vd = stage_desc(st);
#pragma unroll
    for (int kk = 0; kk < C::BK / 8; ++kk) {
      const int c = kk / 4, off = (kk % 4) * 32;
      tc::mma_tf32_ts(d, tmem + C::kSCol + buf * C::BK + 8 * kk,
                      vd + ((c * C::kVtChunk + off) >> 4), id_pv, (acc || kk > 0) ? 1u : 0u);
    }
  };

  // Q tile: shared -> tensor memory, in order behind every earlier MMA that
  // read the previous Q; q_copied tells the softmax warps it is there.
  auto copy_q = [&]() -> bool {
    int st = 0;
    if (!next(st)) return false;
    const uint64_t qd = stage_desc(st);
#pragma unroll
    for (int kk = 0; kk < C::DP / 8; ++kk) {
      const int c = kk / 4, j = kk % 4;
      tc::tmem_cp_128x256b(tmem + C::kQCol + 8 * kk, qd + ((c * C::kKChunk + 32 * j) >> 4));
    }
    tc::mma_commit(&bars->q_copied);
    tc::mma_commit(&bars->kv_empty[st]);
    return true;
  };

  uint32_t g = 0, uc = 0;       // key blocks and units done so far by this block
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int x = unit_of(blockIdx.x, r, gridDim.x);
    if (x >= a.units) break;
    const PUnit u = get_unit<C>(a, x);
    const bool has_next = unit_of(blockIdx.x, r + 1, gridDim.x) < a.units;
    const bool early = a.rope_table && has_next;    // ring order as in the producer
    int st = 0;
    if (r == 0 && !(ok = copy_q())) break;
    // With fused RoPE the softmax warps rotate Q in tensor memory first.
    if (a.rope_table && !(ok = tc::mbar_wait(&bars->q_ready, uc & 1, abort))) break;
    tc::fence_after_sync();
    if (!(ok = next(st))) break;
    issue_s(g & 1, st);
    tc::mma_commit(&bars->s_full[g & 1]);
    tc::mma_commit(&bars->kv_empty[st]);
    if (u.n == 1 && early && !(ok = copy_q())) break;
    for (int i = 0; i < u.n; ++i) {
      const uint32_t G = g + i;
      if (i + 1 < u.n) {
        if (!(ok = next(st))) break;
        issue_s((G + 1) & 1, st);
        tc::mma_commit(&bars->s_full[(G + 1) & 1]);
        tc::mma_commit(&bars->kv_empty[st]);
        if (i + 2 == u.n && early && !(ok = copy_q())) break;
      }
      if (!(ok = next(st))) break;
      if (!(ok = tc::mbar_wait(&bars->p_ready[G & 1], (G >> 1) & 1, abort))) break;
      if (i == 0 && uc > 0 && !(ok = tc::mbar_wait(&bars->o_free, (uc - 1) & 1, abort))) break;
      tc::fence_after_sync();
      issue_pv(G & 1, st, i > 0);
      tc::mma_commit(&bars->o_done);
      tc::mma_commit(&bars->kv_empty[st]);
    }
    if (!ok) break;
    tc::mma_commit(&bars->o_final);
    if (has_next && !early && !(ok = copy_q())) break;
    g += u.n;
    ++uc;
  }
  // No MMA or copy may still run when the block frees its tensor memory.
  tc::mma_commit(&bars->drain);
  drain_wait(&bars->drain, 0);
}

// ---------------------------------------------------------------- fused q RoPE (softmax warps)
// Rotates the unit's Q tile where the MMA reads it, in tensor memory: thread =
// query row, as in the softmax. RMSNorm (if q_norm_w) over the row first, then
// RoPE at the row's absolute position start[b] + q0 + row, pairs (i, i + R/2)
// taken 32 at a time with tcgen05.ld / tcgen05.st, (cos, sin) from the row's
// table line. Rows past L hold zeros (TMA fill) and are left alone. Requires
// D % 32 == 0, D <= 128 and R % 64 == 0.
template <class C>
__device__ bool tq_rotate_q(const TcArgs& a, uint32_t lane_base, PBars* bars, const PUnit& u,
                            int row, uint32_t ucx) {
  volatile int* abort = &bars->abort;
  const int qpos = u.q0 + row;
  const bool live = qpos < a.L;
  const long p = static_cast<long>(a.rope_start[u.b]) + qpos;
  const bool inrange = p >= 0 && p < a.rope_max_positions;
  if (live && !inrange) report(a.status, ATTN_DEV_POSITION);
  const bool rot = live && inrange;
  const int half = a.rope_R / 2;
  const float4* trow = reinterpret_cast<const float4*>(a.rope_table + (rot ? p : 0) * half);
  // The row's whole table line (R/2 <= 64 pairs, two per 16-byte load) is
  // requested before the wait, so its latency overlaps it.
  float4 t0[16], t1[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    t0[e] = rot ? __ldg(trow + e) : make_float4(1.f, 0.f, 1.f, 0.f);
    t1[e] = rot && half > 32 ? __ldg(trow + 16 + e) : make_float4(1.f, 0.f, 1.f, 0.f);
  }
  const bool ok = tc::mbar_wait(&bars->q_copied, ucx & 1, abort);
  if (__any_sync(0xffffffffu, !ok)) return false;   // tcgen05.ld is warp-wide
  tc::fence_after_sync();
  const uint32_t qa = lane_base + C::kQCol;
  float inv = 1.0f;
  if (a.qnorm_w) {
    float ss = 0.f;
#pragma unroll 1
    for (int c = 0; c < a.D; c += 32) {
      float x[32];
      tc::tmem_ld32(qa + c, x);
#pragma unroll
      for (int e = 0; e < 32; ++e) ss = fmaf(x[e], x[e], ss);
    }
    // rows past L stay zero (with eps = 0 their 1/rms would be infinite)
    inv = live ? 1.0f / sqrtf(ss / static_cast<float>(a.D) + a.qnorm_eps) : 1.0f;
  }
  auto scale = [&](float* x, int c) {
    const float4* w = reinterpret_cast<const float4*>(a.qnorm_w + c);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float4 we = __ldg(w + e);
      x[4 * e] *= inv * we.x; x[4 * e + 1] *= inv * we.y;
      x[4 * e + 2] *= inv * we.z; x[4 * e + 3] *= inv * we.w;
    }
  };
  // pairs c0 .. c0 + 31 with (cos, sin) in t
  auto rotate32 = [&](int c0, const float4* t) {
    float x0[32], x1[32];
    tc::tmem_ld32(qa + c0, x0);
    tc::tmem_ld32(qa + c0 + half, x1);
    if (a.qnorm_w) {
      scale(x0, c0);
      scale(x1, c0 + half);
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float4 cs = t[e];
      const float a0 = x0[2 * e], b0 = x1[2 * e], a1 = x0[2 * e + 1], b1 = x1[2 * e + 1];
      x0[2 * e] = fmaf(a0, cs.x, -b0 * cs.y);
      x1[2 * e] = fmaf(a0, cs.y, b0 * cs.x);
      x0[2 * e + 1] = fmaf(a1, cs.z, -b1 * cs.w);
      x1[2 * e + 1] = fmaf(a1, cs.w, b1 * cs.z);
    }
    tc::tmem_st32(qa + c0, x0);
    tc::tmem_st32(qa + c0 + half, x1);
  };
  rotate32(0, t0);
  if (half > 32) rotate32(32, t1);
  if (a.qnorm_w) {                            // columns past R: normalised, not rotated
#pragma unroll 1
    for (int c = a.rope_R; c < a.D; c += 32) {
      float x[32];
      tc::tmem_ld32(qa + c, x);
      scale(x, c);
      tc::tmem_st32(qa + c, x);
    }
  }
  tc::fence_before_sync();
  tc::mbar_arrive(&bars->q_ready);
  return true;
}

// ---------------------------------------------------------------- softmax (4 warps)
// Thread = one query row of the current unit; tcgen05.ld/st run on full warps.
template <class C, bool ROPE>
__device__ void tq_softmax(const TcArgs& a, uint32_t tmem, PBars* bars, int quarter, int lane,
                           const CUtensorMap* tout, uint8_t* stage_out) {
  constexpr int BK = C::BK;
  volatile int* abort = &bars->abort;
  const int row = quarter * 32 + lane;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  const float cs = a.softcap_on ? 1.0f : a.c_score;   // raw score -> log2 units
  uint32_t g = 0, uc = 0;
  bool ok = true;
  // Fused RoPE: the first unit's Q is rotated up front, every later one right
  // after the previous unit's last P (before its epilogue), while the tensor
  // core still runs that unit's last P V products.
  if (ROPE && blockIdx.x < a.units)
    ok = tq_rotate_q<C>(a, lane_base, bars, get_unit<C>(a, unit_of(blockIdx.x, 0, gridDim.x)),
                        row, 0);
  for (int r = 0; ok; ++r) {
    const int x = unit_of(blockIdx.x, r, gridDim.x);
    if (x >= a.units) break;
    const PUnit u = get_unit<C>(a, x);
    const int qpos = u.qk0 + row;               // the query's own key index
    float m_ref = -INFINITY, l = 0.f;         // running max (log2 units) and sum

    for (int i = 0; i < u.n; ++i) {
      const uint32_t G = g + i;
      const int buf = G & 1;
      ok = tc::mbar_wait(&bars->s_full[buf], (G >> 1) & 1, abort);
      if (__any_sync(0xffffffffu, !ok)) {     // leave together: tcgen05.ld is warp-wide
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t scol = lane_base + C::kSCol + buf * BK;
      float s[BK];
      // Softcap: log2(e) * cap * tanh(scale * s / cap) = c_out - 2 c_out / (2^(s c_in) + 1);
      // then the keys outside this row's causal / window band (boundary blocks only).
      const int k0 = (u.jlo + i) * BK;
      const int hi = qpos - k0;                                     // visible: c <= hi
      const int lo = a.window > 0 ? qpos - a.window + 1 - k0 : -1;  // visible: c >= lo
      auto load_scores = [&]() {
        tmem_ld_row<BK>(scol, s);
        if (a.softcap_on) {
#pragma unroll
          for (int c = 0; c < BK; ++c) {
            const float e = tc::ex2(s[c] * a.c_cap_in);
            s[c] = fmaf(-2.0f * a.c_cap_out, tc::rcp(e + 1.0f), a.c_cap_out);
          }
        }
        if (hi < BK - 1 || lo > 0) {
#pragma unroll
          for (int c = 0; c < BK; ++c) s[c] = (c > hi || c < lo) ? -INFINITY : s[c];
        }
      };
      load_scores();

      // Common case: P against the running reference m_ref. It stands unless a
      // score exceeds m_ref by more than 2^8 (where the reference is moved);
      // then the block's sum of P exceeds 2^8 as well, and the block is done
      // again below with its maximum (S is still in tensor memory).
      bool slow = m_ref == -INFINITY;
      float lsum = 0.f;
      if (!__any_sync(0xffffffffu, slow)) {
        lsum = tq_exp_sum<BK>(s, cs, m_ref);
        slow = !(lsum <= kRescaleLimit);
        if (__any_sync(0xffffffffu, slow)) load_scores();
      }
      if (__any_sync(0xffffffffu, slow)) {
        const float m_new = fmaxf(m_ref, tq_max<BK>(s) * cs);
        // Rescale O only when the running maximum has grown a lot (warp-uniform).
        const bool grow = m_ref != -INFINITY && m_new - m_ref > kRescaleLog2;
        if (__any_sync(0xffffffffu, grow)) {
          ok = tc::mbar_wait(&bars->o_done, (G - 1) & 1, abort);
          if (__any_sync(0xffffffffu, !ok)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const float f = grow ? tc::ex2(m_ref - m_new) : 1.0f;
#pragma unroll 1
          for (int c = 0; c < C::DP; c += 32) {
            float o[32];
            tc::tmem_ld32(lane_base + C::kOCol + c, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= f;
            tc::tmem_st32(lane_base + C::kOCol + c, o);
          }
          if (grow) {
            l *= f;
            m_ref = m_new;
          }
        }
        if (m_ref == -INFINITY) m_ref = m_new;  // first visible keys of the row (O, l are 0)
        // -inf only while every key so far was masked; then every score is -inf.
        lsum = tq_exp_sum<BK>(s, cs, m_ref == -INFINITY ? 0.f : m_ref);
      }
      l += lsum;
      tmem_st_row<BK>(scol, s);
      tc::fence_before_sync();
      tc::mbar_arrive(&bars->p_ready[buf]);
    }
    if (!ok) break;
    const int xn = unit_of(blockIdx.x, r + 1, gridDim.x);
    if (ROPE && xn < a.units &&
        !(ok = tq_rotate_q<C>(a, lane_base, bars, get_unit<C>(a, xn), row, uc + 1)))
      break;

    // Epilogue: read O out of TMEM (then O is free for the next unit), scale by
    // 1/l, and write it with TMA: each warp stages 32 rows x 32 columns in a
    // 128-byte-swizzled tile and stores that box (rows past L are clipped).
    ok = tc::mbar_wait(&bars->o_final, uc & 1, abort);
    if (__any_sync(0xffffffffu, !ok || *abort)) {
      ok = false;
      break;
    }
    tc::fence_after_sync();
    float o[C::DP];
    tmem_ld_row<C::DP>(lane_base + C::kOCol, o);
    tc::fence_before_sync();
    tc::mbar_arrive(&bars->o_free);
    const float inv = 1.0f / l;
#pragma unroll
    for (int c = 0; c < C::DP; c += 32) {
      if (lane == 0) tc::bulk_wait_read();      // the previous box has left the staging tile
      __syncwarp();
      float4* row_out = reinterpret_cast<float4*>(stage_out + lane * 128);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        row_out[q ^ (lane & 7)] = make_float4(o[c + 4 * q] * inv, o[c + 4 * q + 1] * inv,
                                              o[c + 4 * q + 2] * inv, o[c + 4 * q + 3] * inv);
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        tc::tma_store_3d(tout, stage_out, c, u.q0 + quarter * 32, u.b * a.H + u.h);
        tc::bulk_commit();
      }
    }
    g += u.n;
    ++uc;
  }
  if (lane == 0) tc::bulk_wait_all();           // output boxes written before the block exits
  __syncwarp();
}

template <int DP, bool ROPE>
__global__ void __launch_bounds__(PCfg<DP>::kThreads, 1)
    prefill_tq_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o, const TcArgs a) {
  using C = PCfg<DP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* skv = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sepi = skv + C::NS * C::kStage;      // 4 x 4 KB output staging tiles
  PBars* bars = reinterpret_cast<PBars*>(sepi + C::kEpi);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NS; ++s) {
      tc::mbar_init(&bars->kv_full[s], 1);
      tc::mbar_init(&bars->kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bars->s_full[b], 1);
      tc::mbar_init(&bars->p_ready[b], 128);
    }
    tc::mbar_init(&bars->o_done, 1);
    tc::mbar_init(&bars->o_final, 1);
    tc::mbar_init(&bars->o_free, 128);
    tc::mbar_init(&bars->q_copied, 1);
    tc::mbar_init(&bars->q_ready, 128);
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
    if (lane == 0) tq_producer<C>(a, &tm_q, &tm_k, &tm_v, skv, bars);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) tq_mma<C>(a, tmem, skv, bars);
    __syncwarp();
  } else {
    tq_softmax<C, ROPE>(a, tmem, bars, warp % 4, lane, &tm_o, sepi + (warp % 4) * 4096);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && bars->abort) report(a.status, ATTN_DEV_TIMEOUT);
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 152;
  }
  return n;
}

template <int DP, bool ROPE>
cudaError_t launch_tq(const AttnShape& s, cudaStream_t stream) {
  using C = PCfg<DP>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(prefill_tq_kernel<DP, ROPE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int Lk = s.Lk > 0 ? s.Lk : s.L;
  CUtensorMap tq, tk, tv, to;
  if (!make_map(&tq, s.q, s.D, s.L, s.B * s.H, kBM) ||
      !make_map(&tk, s.k, s.D, Lk, s.B * s.Hkv, C::BK) ||
      !make_map_vt(&tv, s.vt, s.D, Lk, s.vt_pitch, s.B * s.Hkv, C::DP) ||
      !make_map(&to, s.out, s.D, s.L, s.B * s.H, 32))
    return cudaErrorInvalidValue;
  TcArgs a{};
  a.q = s.q;
  a.out = s.out;
  a.B = s.B; a.H = s.H; a.Hkv = s.Hkv; a.L = s.L; a.D = s.D;
  a.G = s.H / s.Hkv;
  a.QT = (s.L + kBM - 1) / kBM;
  a.units = s.B * s.H * a.QT;
  a.window = s.window;
  a.softcap_on = s.softcap > 0.f;
  a.c_score = s.scale * kLog2e;
  a.c_cap_in = s.softcap > 0.f ? 2.0f * kLog2e * s.scale / s.softcap : 0.f;
  a.c_cap_out = kLog2e * s.softcap;
  a.status = s.status;
  a.rope_table = ROPE ? s.rope.table : nullptr;
  a.rope_start = s.rope.start;
  a.qnorm_w = s.rope.norm_w;
  a.qnorm_eps = s.rope.norm_eps;
  a.rope_R = s.rope.R;
  a.rope_max_positions = s.rope.max_positions;
  a.kv_off = s.kv_off;
  a.Lk = Lk;
  const int grid = a.units < sm_count() ? a.units : sm_count();
  prefill_tq_kernel<DP, ROPE><<<grid, C::kThreads, C::kSmem, stream>>>(tq, tk, tv, to, a);
  return cudaGetLastError();
}

}  // namespace

bool prefill_fuses_rope(int D) { return D % 32 == 0 && D <= 128; }

bool prefill_tq_supports_kv_off(int D) { return D % 4 == 0 && D >= 32 && D <= 128; }

// D <= 128; V^T must already be in s.vt (launch_prefill_tc runs the transpose first).
cudaError_t launch_prefill_tq(const AttnShape& s, cudaStream_t stream) {
  switch ((s.D + 31) / 32) {
    // with q RoPE fused (R % 64 == 0, so D >= 64) or without
    case 1: return s.rope.table ? cudaErrorNotSupported : launch_tq<32, false>(s, stream);
    case 2: return s.rope.table ? launch_tq<64, true>(s, stream) : launch_tq<64, false>(s, stream);
    case 3: return s.rope.table ? launch_tq<96, true>(s, stream) : launch_tq<96, false>(s, stream);
    case 4: return s.rope.table ? launch_tq<128, true>(s, stream) : launch_tq<128, false>(s, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace gqa
