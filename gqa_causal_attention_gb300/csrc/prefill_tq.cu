// Persistent tensor-core prefill for head dimensions 32..256 (multiples of 4).
//
// What it computes: "Core Layers -- Deep Reference", "Flash Attention" -- the
// exact softmax(Q K^T) V of the causal (or windowed, "mojolearn.transformer"
// window) mask without materialising the score matrix, the query heads of one
// key/value head reading the same K and V ("MHA and GQA").
//
// How, on GB300:
//  * One block per SM walks a list of work units (one 128-row query tile of
//    one head each), heaviest tiles first, in snake order across blocks.
//  * Q sits in tensor memory as the A operand of S = Q K^T, so the MMA reads
//    only K (and later V^T) from shared memory; blocks of 128 keys give
//    M128 N128 K8 TF32 instructions (kind::tf32: fp32 data, TF32 products,
//    fp32 accumulation), which run at the full tensor rate.
//    TMEM = Q | O | S0 | S1 (S double-buffered: S of the next key block is
//    computed while softmax turns this one into P). Head dims past 128 keep
//    only Q's first 128 dims in tensor memory and the rest in shared memory
//    (see PCfg), with 64-key blocks.
//  * TMA streams Q tiles, K blocks and V^T blocks of successive units through
//    one ring of stages; a unit's Q tile enters right after the previous
//    unit's last K block. The S issuer moves it to tensor memory with
//    tcgen05.cp, in pipe order right after that unit's last S, which frees its
//    stage early; the next unit's first S products then overlap the previous
//    unit's last softmax and its epilogue. With q RoPE fused
//    (gqa_attn_prefill_rope) the softmax warps normalise and rotate the tile in
//    tensor memory after the previous unit's last P. Out-of-range rows and
//    columns arrive as zeros; key blocks outside the causal/window band are
//    never loaded.
//  * S = Q K^T and O += P V^T come from two issuing threads on different SM
//    sub-partitions, each sharing its sub-partition with one softmax warp.
//  * Four softmax warps own one query row per thread: they read S from tensor
//    memory, apply scale, softcap and mask, keep the running maximum and sum
//    (base 2), and write P (truncated to TF32) back over S. O is rescaled in
//    tensor memory only when the running maximum grows by more than 2^8.
//  * Every pipeline wait is bounded; a wait that runs out reports
//    ATTN_DEV_TIMEOUT and the block winds down (drains its copies and MMAs,
//    frees its tensor memory).
#include "prefill_common.cuh"

namespace gqa {

namespace {

using namespace prefill;

// RAGGED_: per-row lengths (gqa_attn_prefill_ragged); a separate instantiation,
// so the other calls keep the code (and instruction-cache footprint) without it.
// WIDE (head dims 160..256): Q and O of a whole head cannot both sit in the 512
// TMEM columns, so Q is split: dims 0..127 (Q_a) in tensor memory and the rest
// (Q_b) in a shared-memory buffer outside the ring, read as the A operand of the
// second half of S = Q K^T. TMEM = Q_a 128 | O DP | S 2 x 64 columns (64-key
// blocks). Ring stages are 32 KB: Q_a crosses as two 64-column parts, a K block
// as two 128-column parts, V^T as one item per 32 keys.
template <int DP_, bool RAGGED_ = false>
struct PCfg {
  static constexpr int DP = DP_;                        // head dim padded to 32: Q, K, O width
  static constexpr bool RAGGED = RAGGED_;
  static constexpr bool WIDE = DP > 128;
  static constexpr int BK = WIDE ? 64 : 128;            // keys per block
  static constexpr int kChunks = DP / 32;               // 32-column chunks of Q and K
  static constexpr int kQaChunks = WIDE ? 4 : kChunks;  // Q chunks in tensor memory
  static constexpr int kQPC = WIDE ? 2 : kChunks;       // Q chunks per ring item
  static constexpr int kKPC = WIDE ? 4 : kChunks;       // K chunks per ring item
  static constexpr int kVPC = WIDE ? 1 : BK / 32;       // 32-key V^T chunks per ring item
  static constexpr int QP = kQaChunks / kQPC;           // ring items per Q tile
  static constexpr int KP = (kChunks + kKPC - 1) / kKPC;  // ring items per K block
  static constexpr int VI = BK / 32 / kVPC;             // ring items per V^T block
  static constexpr int kQChunk = kBM * 128;             // 128 rows x 128 B of Q
  static constexpr int kKChunk = BK * 128;              // BK rows x 128 B of K
  static constexpr int kVtChunk = DP * 128;             // DP rows x 128 B (32 keys of V^T)
  static constexpr int kQBytes = kQPC * kQChunk;
  static constexpr int kKBytes = kKPC * kKChunk;
  static constexpr int kVBytes = kVPC * kVtChunk;
  static constexpr int kStage =                         // one Q part, K part or V^T item
      kQBytes > kKBytes ? (kQBytes > kVBytes ? kQBytes : kVBytes)
                        : (kKBytes > kVBytes ? kKBytes : kVBytes);
  static constexpr int kQb = (kChunks - kQaChunks) * kQChunk;   // Q_b buffer (WIDE)
  static constexpr int kEpi = 4 * 4096;                 // per-warp 32 x 32 output staging
  static constexpr int kTab = WIDE ? 0 : 32 * 64 * 8;   // RoPE table rows 0..31, up to 64 pairs
  static constexpr int kNSraw = (kSmemLimit - 2048 - kEpi - kTab - kQb) / kStage;
  static constexpr int NS = kNSraw > 8 ? 8 : kNSraw;
  static constexpr int kThreads = 64 + 128 + 32;     // producer, S issuer, 4 softmax, P V issuer
  static constexpr int kSmemNeed = NS * kStage + kQb + kEpi + kTab + 2048;
  static constexpr int kSmem =
      kSmemNeed > kSmemLimit / 2 + 4096 ? kSmemNeed : kSmemLimit / 2 + 4096;
  static constexpr int kQCol = 0, kOCol = kQaChunks * 32, kSCol = kOCol + DP;
  // The issuers' ring waits stay alias-free (see the producer's ring order)
  // from 3 stages with one-item Q tiles, K and V^T blocks, and from 4 with the
  // WIDE parts.
  static_assert(NS >= (WIDE ? 4 : 3), "ring too short");
  static_assert(VI == 1 || VI == 2, "V^T items per block: one, or one per half of P");
  static_assert(DP % 32 == 0 && DP <= 256, "head dim: 32-column chunks, an even number of output boxes");
  static_assert(kSCol + 2 * BK <= kTmemCols, "tensor memory budget");
  static_assert(kSmem <= kSmemLimit, "shared memory budget");
};

struct PBars {
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t s_full[2];
  uint64_t p_ready[2][2];                      // [S buffer][half]: P of those columns written
  uint64_t o_done[2];                          // P V of block X done (X % 2)
  uint64_t o_half[2];                          // P V of block X's first half done (X % 2)
  uint64_t o_final;
  uint64_t o_free;
  uint64_t q_copied;                           // a Q tile is in tensor memory (one phase per unit)
  uint64_t q_ready;                            // fused RoPE: that Q tile is rotated
  uint64_t qb_full;                            // WIDE: a Q_b tile landed (one phase per tile)
  uint64_t qb_empty;                           // WIDE: the S products reading Q_b are done
  uint64_t drain[2];                           // each issuer's MMAs and copies done
  uint32_t tmem_base;
  int abort;
};

struct PUnit {
  int b, h, q0, jlo, n;                       // n = 0: every row is padding (ragged batch)
  int qk0;                                    // key index of query row q0 (q0 + kv_off[b])
  int klast;                                  // the row's last real key index
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
  const int Lb = C::RAGGED ? row_len(a, u.b) : a.L;
  u.qk0 = u.q0 + off;
  u.klast = off + Lb - 1;
  const int lo = a.window > 0 ? max(0, u.qk0 - a.window + 1) / C::BK : 0;
  const int hi = min(u.qk0 + kBM - 1, u.klast) / C::BK;
  u.jlo = lo;
  u.n = u.q0 < Lb ? hi - lo + 1 : 0;
  return u;
}

// The first round at or after r whose unit has key blocks (or the first round
// past the end); every role walks the same sequence.
template <class C>
__device__ __forceinline__ int next_live(const TcArgs& a, int r) {
  if (!C::RAGGED) return r;                     // without lengths no unit is empty
  for (;; ++r) {
    const int x = unit_of(blockIdx.x, r, gridDim.x);
    if (x >= a.units || get_unit<C>(a, x).n > 0) return r;
  }
}

// ---------------------------------------------------------------- producer (one thread)
// Ring order: the first unit's Q tile; then per unit K_0 .. K_{n-1} interleaved
// with V^T_0 .. V^T_{n-1} as K_0, (K_{i+1}, V^T_i)..., with the next unit's Q
// tile right after the last K block (WIDE: its Q_a parts right before the last
// V^T block), so it lands while this unit's last P V products are pending and
// moves to tensor memory before the next unit's first S = Q K^T. WIDE: a Q_a
// tile, K block or V^T block is several items, and the next Q_b tile is loaded
// into its own buffer after the last V^T block, once the S products that read
// the current one are done. These orders keep every issuer's ring wait
// alias-free: when an issuer waits for the k-th fill of a stage, the (k-1)-th
// has landed, either as one of its own items or as shown by the cross-role
// barrier it waited on first (checked for all unit sequences of up to 4 units
// of 1..5 blocks, 3..8 stages one-item, 4..6 stages WIDE).
template <class C>
__device__ void tq_producer(const TcArgs& a, const CUtensorMap* tq, const CUtensorMap* tk,
                            const CUtensorMap* tv, uint8_t* skv, uint8_t* sqb, PBars* bars) {
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
  // kind: 0 = Q part, 1 = K part, 2 = V^T item
  auto load = [&](int kind, const PUnit& u, int j, int part) -> bool {
    if (!tc::mbar_wait(&bars->kv_empty[stage], phase ^ 1u, abort)) return false;
    uint64_t* full = &bars->kv_full[stage];
    uint8_t* dst = skv + stage * C::kStage;
    if (kind == 0) {
      const int c0 = part * C::kQPC;
      tc::mbar_arrive_expect_tx(full, C::kQBytes);
      for (int c = c0; c < c0 + C::kQPC; ++c)
        tc::tma_load_3d(dst + (c - c0) * C::kQChunk, tq, full, 32 * c, u.q0, u.b * a.H + u.h);
    } else if (kind == 1) {
      const int c0 = part * C::kKPC, c1 = min(c0 + C::kKPC, C::kChunks);
      tc::mbar_arrive_expect_tx(full, (c1 - c0) * C::kKChunk);
      for (int c = c0; c < c1; ++c)
        tc::tma_load_3d(dst + (c - c0) * C::kKChunk, tk, full, 32 * c, j * C::BK,
                        u.b * a.Hkv + u.h / a.G);
    } else {
      tc::mbar_arrive_expect_tx(full, C::kVBytes);
      for (int c = 0; c < C::kVPC; ++c)
        tc::tma_load_3d(dst + c * C::kVtChunk, tv, full, j * C::BK + 32 * (part * C::kVPC + c),
                        0, u.b * a.Hkv + u.h / a.G);
    }
    filled[stage] = true;
    fill_parity[stage] = phase;
    if (++stage == C::NS) {
      stage = 0;
      phase ^= 1u;
    }
    return true;
  };
  auto load_items = [&](int kind, int items, const PUnit& u, int j) -> bool {
    for (int p = 0; p < items; ++p)
      if (!load(kind, u, j, p)) return false;
    return true;
  };
  // WIDE: Q_b of the t-th tile, once the S products of tile t - 1 released the buffer.
  uint32_t qb_loads = 0;
  auto load_qb = [&](const PUnit& u) -> bool {
    if (qb_loads > 0 && !tc::mbar_wait(&bars->qb_empty, (qb_loads - 1) & 1, abort)) return false;
    tc::mbar_arrive_expect_tx(&bars->qb_full, C::kQb);
    for (int c = C::kQaChunks; c < C::kChunks; ++c)
      tc::tma_load_3d(sqb + (c - C::kQaChunks) * C::kQChunk, tq, &bars->qb_full, 32 * c, u.q0,
                      u.b * a.H + u.h);
    ++qb_loads;
    return true;
  };
  bool ok = true;
  for (int r = next_live<C>(a, 0), first = 1; ok; first = 0) {
    const int x = unit_of(blockIdx.x, r, gridDim.x);
    if (x >= a.units) break;
    const PUnit u = get_unit<C>(a, x);
    const int rn = next_live<C>(a, r + 1);
    const int xn = unit_of(blockIdx.x, rn, gridDim.x);
    const bool has_next = xn < a.units;
    const PUnit un = get_unit<C>(a, has_next ? xn : x);
    // Warm the next Q tile (and its RoPE table lines) into L2 now: they are
    // read within a few blocks.
    if (has_next) {
      for (int c = 0; c < C::kChunks; ++c)
        tc::tma_prefetch_l2_3d(tq, 32 * c, un.q0, un.b * a.H + un.h);
      if (a.rope_table) {
        const long half = a.rope_R / 2;
        const long p0 = min(max(static_cast<long>(start_of(a, un.b)) + un.q0, 0L),
                            static_cast<long>(a.rope_max_positions - 1));
        const long p1 = min(p0 + kBM, static_cast<long>(a.rope_max_positions));
        tc::bulk_prefetch_l2(a.rope_table + p0 * half, static_cast<uint32_t>((p1 - p0) * half * 8));
      }
    }
    if (first) {
      ok = load_items(0, C::QP, u, 0);
      if (ok && C::WIDE) ok = load_qb(u);
    }
    if (ok) ok = load_items(1, C::KP, u, u.jlo);
    if (ok && !C::WIDE && u.n == 1 && has_next) ok = load_items(0, C::QP, un, 0);
    for (int i = 0; ok && i < u.n; ++i) {
      if (i + 1 < u.n) {
        ok = load_items(1, C::KP, u, u.jlo + i + 1);
        if (ok && !C::WIDE && i + 2 == u.n && has_next) ok = load_items(0, C::QP, un, 0);
      }
      if (ok && C::WIDE && i + 1 == u.n && has_next) ok = load_items(0, C::QP, un, 0);
      if (ok) ok = load_items(2, C::VI, u, u.jlo + i);
    }
    if (ok && C::WIDE && has_next) ok = load_qb(un);
    r = rn;
  }
  // Every copy this block started lands before the block may exit.
  for (int s = 0; s < C::NS; ++s)
    if (filled[s]) drain_wait(&bars->kv_full[s], fill_parity[s]);
  if (qb_loads > 0) drain_wait(&bars->qb_full, (qb_loads - 1) & 1);
}

// ---------------------------------------------------------------- MMA issuers (two threads)
// S = Q K^T and O += P V^T are issued by two threads on different SM
// sub-partitions (warps 1 and 6), so that neither stream's waits (for a free S
// buffer, for the softmax's P) hold back the other's products; measured, this
// kept the tensor pipe busier than one issuing thread. Both walk the producer's ring order, each taking its own items and stepping
// over the other's; P V of block X signals o_done[X % 2], so every wait on it
// (S of block X + 2 overwrites X's P; a rescale of O in block X + 1) names a
// phase that cannot be two behind.
template <class C>
struct RingCursor {
  int stage = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void skip() {
    if (++stage == C::NS) {
      stage = 0;
      phase ^= 1u;
    }
  }
  __device__ __forceinline__ bool take(PBars* bars, volatile int* abort, int& st) {
    if (!tc::mbar_wait(&bars->kv_full[stage], phase, abort)) return false;
    st = stage;
    skip();
    return true;
  }
};

template <class C>
__device__ __forceinline__ uint64_t stage_desc(uint64_t base_desc, int st) {
  return base_desc + static_cast<uint32_t>((st * C::kStage) >> 4);
}

// The S issuer: Q tiles to tensor memory (tcgen05.cp) and S = Q K^T.
template <class C>
__device__ void tq_mma_s(const TcArgs& a, uint32_t tmem, uint8_t* skv, uint8_t* sqb,
                         PBars* bars) {
  volatile int* abort = &bars->abort;
  constexpr uint32_t id_s = tc::idesc_tf32(kBM, C::BK, false);
  // Descriptors are built once; an operand offset is added to the start-address
  // field (address >> 4), which stays below 2^14 for any shared-memory address.
  const uint64_t base_desc = tc::sdesc_sw128(tc::smem_u32(skv), 16, 1024);
  const uint64_t qb_desc = tc::sdesc_sw128(tc::smem_u32(sqb), 16, 1024);
  RingCursor<C> ring;
  // Q tile (WIDE: Q_a): shared -> tensor memory, in pipe order behind the last S
  // that read the previous Q (so the next unit's S products follow without a
  // wait); its stages are free once the copies are done.
  auto copy_q = [&]() -> bool {
#pragma unroll
    for (int p = 0; p < C::QP; ++p) {
      int st = 0;
      if (!ring.take(bars, abort, st)) return false;
      const uint64_t qd = stage_desc<C>(base_desc, st);
#pragma unroll
      for (int c = 0; c < C::kQPC; ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          tc::tmem_cp_128x256b(tmem + C::kQCol + 32 * (p * C::kQPC + c) + 8 * j,
                               qd + ((c * C::kQChunk + 32 * j) >> 4));
      tc::mma_commit(&bars->kv_empty[st]);
    }
    tc::mma_commit(&bars->q_copied);
    return true;
  };
  // S[G % 2] = Q K^T for global block G, once P V of block G - 2 has read that buffer.
  // The o_done wait comes before the ring wait: it also shows that the stage's
  // previous item (possibly a V^T this thread skipped) has landed, so the
  // parity of the ring wait cannot alias an older fill. Q chunks past Q_a
  // (WIDE) are read from the Q_b buffer.
  auto issue_s = [&](uint32_t G) -> bool {
    if (G >= 2 && !tc::mbar_wait(&bars->o_done[G & 1], ((G - 2) >> 1) & 1, abort)) return false;
    const uint32_t d = tmem + C::kSCol + (G & 1) * C::BK;
#pragma unroll
    for (int p = 0; p < C::KP; ++p) {
      int st = 0;
      if (!ring.take(bars, abort, st)) return false;
      tc::fence_after_sync();
      const uint64_t kd = stage_desc<C>(base_desc, st);
      const int c0 = p * C::kKPC, c1 = min(c0 + C::kKPC, C::kChunks);
#pragma unroll
      for (int c = c0; c < c1; ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint64_t b = kd + (((c - c0) * C::kKChunk + 32 * j) >> 4);
          if (c < C::kQaChunks)
            tc::mma_tf32_ts(d, tmem + C::kQCol + 32 * c + 8 * j, b, id_s, (c | j) != 0);
          else
            tc::mma_tf32_ss(d, qb_desc + (((c - C::kQaChunks) * C::kQChunk + 32 * j) >> 4), b,
                            id_s, 1u);
        }
      tc::mma_commit(&bars->kv_empty[st]);
    }
    tc::mma_commit(&bars->s_full[G & 1]);
    return true;
  };
  auto skip = [&](int items) {
    for (int e = 0; e < items; ++e) ring.skip();
  };

  uint32_t g = 0, tcnt = 0;     // key blocks and live units done so far by this block
  bool ok = true;
  for (int r = next_live<C>(a, 0); ok;) {
    const int x = unit_of(blockIdx.x, r, gridDim.x);
    if (x >= a.units) break;
    const PUnit u = get_unit<C>(a, x);
    const int rn = next_live<C>(a, r + 1);
    const bool has_next = unit_of(blockIdx.x, rn, gridDim.x) < a.units;
    if (tcnt == 0 && !(ok = copy_q())) break;
    // With fused RoPE the softmax warps rotate Q in tensor memory first.
    if (a.rope_table) {
      if (!(ok = tc::mbar_wait(&bars->q_ready, tcnt & 1, abort))) break;
      tc::fence_after_sync();
    }
    if (C::WIDE) {
      if (!(ok = tc::mbar_wait(&bars->qb_full, tcnt & 1, abort))) break;
      tc::fence_after_sync();
    }
    if (!(ok = issue_s(g))) break;
    if (!C::WIDE && u.n == 1 && has_next && !(ok = copy_q())) break;
    for (int i = 0; i < u.n; ++i) {
      if (i + 1 < u.n) {
        if (!(ok = issue_s(g + i + 1))) break;
        if (!C::WIDE && i + 2 == u.n && has_next && !(ok = copy_q())) break;
      }
      if (C::WIDE && i + 1 == u.n) {
        // Q_b is free once this unit's S products are done.
        tc::mma_commit(&bars->qb_empty);
        if (has_next) {
          // The stages the Q_a parts refill last held V^T items up to block
          // g + i - 1: its P V (which the next S waits for anyway) shows they landed.
          const uint32_t G = g + i - 1;
          if (g + i >= 1 && !(ok = tc::mbar_wait(&bars->o_done[G & 1], (G >> 1) & 1, abort)))
            break;
          if (!(ok = copy_q())) break;
        }
      }
      skip(C::VI);                                  // V^T_i: the P V issuer's
    }
    if (!ok) break;
    g += u.n;
    ++tcnt;
    r = rn;
  }
  // No MMA or copy of this thread may still run when the block frees its TMEM.
  tc::mma_commit(&bars->drain[0]);
  drain_wait(&bars->drain[0], 0);
}

// The P V issuer: O += P V^T once the softmax has written P of the block.
template <class C>
__device__ void tq_mma_pv(const TcArgs& a, uint32_t tmem, uint8_t* skv, PBars* bars) {
  volatile int* abort = &bars->abort;
  constexpr uint32_t id_pv = tc::idesc_tf32(kBM, C::DP, false);
  const uint64_t base_desc = tc::sdesc_sw128(tc::smem_u32(skv), 16, 1024);
  RingCursor<C> ring;
  auto skip = [&](int items) {
    for (int e = 0; e < items; ++e) ring.skip();
  };
  uint32_t g = 0, uc = 0;
  bool ok = true;
  for (int r = next_live<C>(a, 0); ok;) {
    const int x = unit_of(blockIdx.x, r, gridDim.x);
    if (x >= a.units) break;
    const PUnit u = get_unit<C>(a, x);
    const int rn = next_live<C>(a, r + 1);
    const bool has_next = unit_of(blockIdx.x, rn, gridDim.x) < a.units;
    if (uc == 0) skip(C::QP);                       // the first Q tile
    skip(C::KP);                                    // K_0
    if (!C::WIDE && u.n == 1 && has_next) skip(C::QP);       // next Q
    for (int i = 0; i < u.n; ++i) {
      const uint32_t G = g + i;
      if (i + 1 < u.n) {
        skip(C::KP);                                // K_{i+1}
        if (!C::WIDE && i + 2 == u.n && has_next) skip(C::QP);   // next Q
      }
      if (C::WIDE && i + 1 == u.n && has_next) skip(C::QP);      // next Q_a
      // P of block G arrives in two halves of BK / 2 keys; the products of the
      // first half run while the softmax computes the second. P's first half
      // comes before the ring wait: S of block G has then read K_G, so the
      // stage's previous item has landed and the wait cannot alias.
      constexpr int KH = C::BK / 16;              // 8-key steps per half
      int st_item[2] = {0, 0};
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        if (!(ok = tc::mbar_wait(&bars->p_ready[G & 1][hh], (G >> 1) & 1, abort))) break;
        if (C::VI == 2 || hh == 0) {              // this half's V^T item
          if (!(ok = ring.take(bars, abort, st_item[hh]))) break;
          if (hh == 0 && i == 0 && uc > 0 &&
              !(ok = tc::mbar_wait(&bars->o_free, (uc - 1) & 1, abort)))
            break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + C::kOCol;
        const uint64_t vd = stage_desc<C>(base_desc, st_item[C::VI == 2 ? hh : 0]);
#pragma unroll
        for (int kk = hh * KH; kk < (hh + 1) * KH; ++kk) {
          const int kl = C::VI == 2 ? kk - hh * KH : kk;   // 8-key step within the item
          const int c = kl / 4, off = (kl % 4) * 32;
          tc::mma_tf32_ts(d, tmem + C::kSCol + (G & 1) * C::BK + 8 * kk,
                          vd + ((c * C::kVtChunk + off) >> 4), id_pv, (i > 0 || kk > 0) ? 1u : 0u);
        }
        if (C::VI == 2) tc::mma_commit(&bars->kv_empty[st_item[hh]]);
        if (hh == 0) tc::mma_commit(&bars->o_half[G & 1]);
      }
      if (!ok) break;
      if (C::VI == 1) tc::mma_commit(&bars->kv_empty[st_item[0]]);
      tc::mma_commit(&bars->o_done[G & 1]);
    }
    if (!ok) break;
    tc::mma_commit(&bars->o_final);
    g += u.n;
    ++uc;
    r = rn;
  }
  tc::mma_commit(&bars->drain[1]);
  drain_wait(&bars->drain[1], 0);
}

// ---------------------------------------------------------------- fused q RoPE (softmax warps)
// Rotates the next unit's Q tile where the MMA reads it, in tensor memory:
// thread = query row, as in the softmax. RMSNorm (if q_norm_w) over the row
// first, then RoPE at the row's absolute position p = start[b] + q0 + row,
// pairs (i, i + R/2) taken 32 at a time with tcgen05.ld / tcgen05.st; requires
// D % 32 == 0, D <= 128 and R % 64 == 0. Rows past L hold zeros (TMA fill).
// The angle of row 32 w + l of warp w is split as (B + l) theta_i with
// B = start[b] + q0 + 32 w, and its cosine and sine are formed by the
// angle-addition identities from table row B (one line per warp, prefetched
// into L1 and read with broadcast loads) and table row l < 32, which stays in
// shared memory for the whole kernel; the fp32 products differ from table row
// p by a few ulp. (Reading table row p per thread would scatter each load
// instruction over 32 cache lines and stall the SM's load/store path, mbarrier
// operations included, for thousands of cycles.)
template <class C>
__device__ bool tq_rotate_q(const TcArgs& a, uint32_t lane_base, PBars* bars,
                            const uint8_t* stage_tab, const PUnit& u, int start_b, int quarter,
                            int lane, uint32_t ucx) {
  volatile int* abort = &bars->abort;
  const int row = quarter * 32 + lane;
  const bool live = u.q0 + row < a.L;
  const int half = a.rope_R / 2;                 // 32 or 64 pairs
  // Row B; a position outside the table is reported (the host bounds start[b]
  // too) and clamped, so the loads stay in bounds.
  const long p0 = static_cast<long>(start_b) + u.q0 + quarter * 32;
  if (live && !(p0 + lane >= 0 && p0 + lane < a.rope_max_positions))
    report(a.status, ATTN_DEV_POSITION);
  const long pb = min(max(p0, 0L), static_cast<long>(a.rope_max_positions - 1));
  const float4* brow = reinterpret_cast<const float4*>(a.rope_table + pb * half);
  if (lane < half / 16) tc::prefetch_l1(brow + 8 * lane);   // its 128-byte lines
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
  auto scale = [&](float* x, int c, int n) {
    const float4* w = reinterpret_cast<const float4*>(a.qnorm_w + c);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (4 * e >= n) break;
      const float4 we = __ldg(w + e);
      x[4 * e] *= inv * we.x; x[4 * e + 1] *= inv * we.y;
      x[4 * e + 2] *= inv * we.z; x[4 * e + 3] *= inv * we.w;
    }
  };
  if (a.qnorm_w) {                               // columns past R: normalised, not rotated
#pragma unroll 1
    for (int c = a.rope_R; c < C::DP; c += 32) {
      float x[32];
      tc::tmem_ld32(qa + c, x);
      scale(x, c, 32);
      tc::tmem_st32(qa + c, x);
    }
  }
  const float4* lrow = reinterpret_cast<const float4*>(stage_tab) + lane * 32;
  // 32 pairs per round (one paired TMEM load and store, one wait each)
#pragma unroll 1
  for (int j = 0; j < half / 32; ++j) {
    float x0[32], x1[32];
    tc::tmem_ld32x2(qa + 32 * j, qa + 32 * j + half, x0, x1);
    if (a.qnorm_w) {
      scale(x0, 32 * j, 32);
      scale(x1, 32 * j + half, 32);
    }
#pragma unroll
    for (int g = 0; g < 16; ++g) {
      // (cos, sin) of (B + l) theta for pairs 32 j + 2 g, + 1
      const int src = 16 * j + g;
      const float4 cb = __ldg(brow + src);                 // row B (the same for every lane)
      const float4 cl = lrow[src ^ lane];                  // row l (swizzled granules)
      const float4 cs = make_float4(fmaf(cb.x, cl.x, -cb.y * cl.y), fmaf(cb.y, cl.x, cb.x * cl.y),
                                    fmaf(cb.z, cl.z, -cb.w * cl.w), fmaf(cb.w, cl.z, cb.z * cl.w));
      const float a0 = x0[2 * g], b0 = x1[2 * g], a1 = x0[2 * g + 1], b1 = x1[2 * g + 1];
      x0[2 * g] = fmaf(a0, cs.x, -b0 * cs.y);
      x1[2 * g] = fmaf(a0, cs.y, b0 * cs.x);
      x0[2 * g + 1] = fmaf(a1, cs.z, -b1 * cs.w);
      x1[2 * g + 1] = fmaf(a1, cs.w, b1 * cs.z);
    }
    tc::tmem_st32x2(qa + 32 * j, qa + 32 * j + half, x0, x1);
  }
  tc::fence_before_sync();
  tc::mbar_arrive(&bars->q_ready);
  return true;
}

// ---------------------------------------------------------------- softmax (4 warps)
// Thread = one query row of the current unit; tcgen05.ld/st run on full warps.
template <class C, bool ROPE>
__device__ void tq_softmax(const TcArgs& a, uint32_t tmem, PBars* bars, int quarter, int lane,
                           const CUtensorMap* tout, uint8_t* stage_out, const uint8_t* stage_tab) {
  constexpr int BK = C::BK;
  static_assert(!(ROPE && C::WIDE), "q RoPE is fused for head dims up to 128");
  volatile int* abort = &bars->abort;
  const int row = quarter * 32 + lane;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  const float cs = a.softcap_on ? 1.0f : a.c_score;   // raw score -> log2 units
  uint32_t g = 0, uc = 0;       // key blocks and live units done so far
  bool ok = true;
  // Fused RoPE: the first unit's Q is rotated up front, every later one right
  // after the previous unit's last P (before its epilogue), while the tensor
  // core runs that unit's last P V products.
  const int r0 = next_live<C>(a, 0);
  if (ROPE && unit_of(blockIdx.x, r0, gridDim.x) < a.units) {
    const PUnit u0 = get_unit<C>(a, unit_of(blockIdx.x, r0, gridDim.x));
    ok = tq_rotate_q<C>(a, lane_base, bars, stage_tab, u0, start_of(a, u0.b), quarter, lane, 0);
  }
  // The warp's 32 rows x 16 columns from column c0 to the output, through two
  // alternating 2 KB staging tiles (64-byte swizzle: 16-byte granule g of row r
  // at g ^ ((r / 2) % 4)); a tile is rewritten once the store issued two boxes
  // earlier has read it: box c0 / 16 uses tile (c0 / 16) % 2, and a unit stores
  // an even number of boxes. value(q) gives columns c0 + 4 q .. c0 + 4 q + 3 of
  // this thread's row; rows past L and columns past D are clipped.
  auto store_box = [&](const PUnit& uu, int c0, auto value) {
    uint8_t* tile = stage_out + ((c0 / 16) & 1) * 2048;
    if (lane == 0) tc::bulk_wait_read_all_but_one();
    __syncwarp();
    float4* row_out = reinterpret_cast<float4*>(tile + lane * 64);
#pragma unroll
    for (int q = 0; q < 4; ++q) row_out[q ^ ((lane >> 1) & 3)] = value(q);
    tc::fence_proxy_async();
    __syncwarp();
    if (lane == 0) {
      tc::tma_store_3d(tout, tile, c0, uu.q0 + quarter * 32, uu.b * a.H + uu.h);
      tc::bulk_commit();
    }
  };
  for (int r = r0; ok;) {
    const int x = unit_of(blockIdx.x, r, gridDim.x);
    if (x >= a.units) break;
    const PUnit u = get_unit<C>(a, x);
    const int rn = next_live<C>(a, r + 1);
    const int xn = unit_of(blockIdx.x, rn, gridDim.x);
    // start[b] of the next unit, read now so that its latency is not on the
    // path of that unit's rotation.
    const int next_start = ROPE && xn < a.units ? start_of(a, get_unit<C>(a, xn).b) : 0;
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
      const int k0 = (u.jlo + i) * BK;
      const int hi = (C::RAGGED ? min(qpos, u.klast) : qpos) - k0;  // visible: c <= hi
      const int lo = a.window > 0 ? qpos - a.window + 1 - k0 : -1;  // visible: c >= lo
      // Boundary blocks (the causal diagonal, a window's edge): softcap and the
      // band mask are applied in tensor memory first, 32 columns at a time in a
      // rolled loop, so the unrolled 128-column code below stays lean. Chunks
      // that no row of the warp sees are written as -inf without a load;
      // chunks every row sees are left alone unless softcap needs applying.
      const bool edge = __any_sync(0xffffffffu, hi < BK - 1 || lo > 0);
      if (edge) {
#pragma unroll 1
        for (int c0 = 0; c0 < BK; c0 += 32) {
          float x[32];
          const bool none = __all_sync(0xffffffffu, hi < c0 || lo > c0 + 31);
          const bool all = __all_sync(0xffffffffu, hi >= c0 + 31 && lo <= c0);
          if (none) {
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] = -INFINITY;
          } else {
            if (all && !a.softcap_on) continue;
            tc::tmem_ld32(scol + c0, x);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              if (a.softcap_on) {
                const float t = tc::ex2(x[e] * a.c_cap_in);
                x[e] = fmaf(-2.0f * a.c_cap_out, tc::rcp(t + 1.0f), a.c_cap_out);
              }
              const int c = c0 + e;
              x[e] = c > hi ? -INFINITY : x[e];
              x[e] = c < lo ? -INFINITY : x[e];
            }
          }
          tc::tmem_st32(scol + c0, x);
        }
      }
      // P in two halves of H2 columns, each released to the P V issuer as soon
      // as it is written (its products then overlap the second half's softmax).
      // Per half, pass 0, the common case: P against the running reference
      // m_ref. It stands unless a score exceeds m_ref by more than 2^8 (where
      // the reference is moved); then the half's sum of P exceeds 2^8 as well.
      // Pass 1 (a row's first visible keys, or pass 0 rejected): S read again,
      // P against the new maximum, after O is rescaled once every product that
      // wrote it is done: P V of block G - 1 for the first half, and P V of
      // this block's first half for the second. One rolled copy of the code
      // serves both halves and passes: this kernel's code far exceeds the
      // instruction caches, so every copy of an unrolled loop costs fetch stalls.
      constexpr int H2 = BK / 2;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t hcol = scol + hh * H2;
        float s[H2];
        float lsum = 0.f;
        const bool fast = !__any_sync(0xffffffffu, m_ref == -INFINITY);
#pragma unroll 1
        for (int pass = fast ? 0 : 1; pass < 2; ++pass) {
          tmem_ld_row<H2>(hcol, s);
          // Softcap: log2(e) * cap * tanh(scale * s / cap) = c_out - 2 c_out / (2^(s c_in) + 1)
          // (boundary blocks have it already).
          if (a.softcap_on && !edge) {
#pragma unroll
            for (int c = 0; c < H2; ++c) {
              const float e = tc::ex2(s[c] * a.c_cap_in);
              s[c] = fmaf(-2.0f * a.c_cap_out, tc::rcp(e + 1.0f), a.c_cap_out);
            }
          }
          float m_use = m_ref;
          if (pass == 1) {
            const float m_new = fmaxf(m_ref, tq_max<H2>(s) * cs);
            // Rescale O only when the running maximum has grown a lot (warp-uniform).
            const bool grow = m_ref != -INFINITY && m_new - m_ref > kRescaleLog2;
            if (__any_sync(0xffffffffu, grow)) {
              ok = hh == 0 ? tc::mbar_wait(&bars->o_done[(G - 1) & 1], ((G - 1) >> 1) & 1, abort)
                           : tc::mbar_wait(&bars->o_half[G & 1], (G >> 1) & 1, abort);
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
            m_use = m_ref == -INFINITY ? 0.f : m_ref;
          }
          lsum = tq_exp_sum<H2>(s, cs, m_use);
          if (pass == 1 || !__any_sync(0xffffffffu, !(lsum <= kRescaleLimit))) break;
        }
        if (!ok) break;
        l += lsum;
        tmem_st_row<H2>(hcol, s);
        tc::fence_before_sync();
        tc::mbar_arrive(&bars->p_ready[buf][hh]);
      }
      if (!ok) break;
    }
    if (!ok) break;
    if (ROPE && xn < a.units &&
        !(ok = tq_rotate_q<C>(a, lane_base, bars, stage_tab, get_unit<C>(a, xn), next_start,
                              quarter, lane, uc + 1)))
      break;

    // Epilogue: read O out of TMEM (then O is free for the next unit), scale by
    // 1/l and store it; padding rows of a ragged batch are written as +0.0.
    ok = tc::mbar_wait(&bars->o_final, uc & 1, abort);
    if (__any_sync(0xffffffffu, !ok || *abort)) {
      ok = false;
      break;
    }
    tc::fence_after_sync();
    const bool real = !C::RAGGED || qpos <= u.klast;
    const float inv = real ? 1.0f / l : 0.f;
    if constexpr (!C::WIDE) {
      float o[C::DP];
      tmem_ld_row<C::DP>(lane_base + C::kOCol, o);
      tc::fence_before_sync();
      tc::mbar_arrive(&bars->o_free);
#pragma unroll
      for (int c = 0; c < C::DP; c += 16)
        store_box(u, c, [&](int q) {
          const float* e = o + c + 4 * q;
          return real ? make_float4(e[0] * inv, e[1] * inv, e[2] * inv, e[3] * inv)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        });
    } else {
      // 32 columns at a time: the whole row would not fit in registers.
#pragma unroll 1
      for (int c = 0; c < C::DP; c += 32) {
        float o[32];
        tc::tmem_ld32(lane_base + C::kOCol + c, o);
#pragma unroll
        for (int h = 0; h < 32; h += 16)
          store_box(u, c + h, [&](int q) {
            const float* e = o + h + 4 * q;
            return real ? make_float4(e[0] * inv, e[1] * inv, e[2] * inv, e[3] * inv)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
          });
      }
      tc::fence_before_sync();
      tc::mbar_arrive(&bars->o_free);
    }
    g += u.n;
    ++uc;
    r = rn;
  }
  // Units with no real row (ragged batch): zeros.
  if (C::RAGGED && ok) {
    for (int r = 0;; ++r) {
      const int x = unit_of(blockIdx.x, r, gridDim.x);
      if (x >= a.units) break;
      const PUnit u = get_unit<C>(a, x);
      if (u.n > 0) continue;
#pragma unroll 1
      for (int c = 0; c < C::DP; c += 16)
        store_box(u, c, [](int) { return make_float4(0.f, 0.f, 0.f, 0.f); });
    }
  }
  if (lane == 0) tc::bulk_wait_all();           // output boxes written before the block exits
  __syncwarp();
}

template <int DP, bool ROPE, bool RAGGED>
__global__ void __launch_bounds__(PCfg<DP>::kThreads, 1)
    prefill_tq_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o, const TcArgs a) {
  using C = PCfg<DP, RAGGED>;
  if (gated_off(a.skip)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* skv = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sqb = skv + C::NS * C::kStage;       // Q_b (WIDE; 1024-byte aligned)
  uint8_t* sepi = sqb + C::kQb;                 // 4 x 4 KB output staging tiles
  uint8_t* stab = sepi + C::kEpi;               // RoPE table rows 0..31 (ROPE)
  PBars* bars = reinterpret_cast<PBars*>(stab + C::kTab);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NS; ++s) {
      tc::mbar_init(&bars->kv_full[s], 1);
      tc::mbar_init(&bars->kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bars->s_full[b], 1);
      tc::mbar_init(&bars->p_ready[b][0], 128);
      tc::mbar_init(&bars->p_ready[b][1], 128);
      tc::mbar_init(&bars->o_half[b], 1);
    }
    tc::mbar_init(&bars->o_done[0], 1);
    tc::mbar_init(&bars->o_done[1], 1);
    tc::mbar_init(&bars->o_final, 1);
    tc::mbar_init(&bars->o_free, 128);
    tc::mbar_init(&bars->q_copied, 1);
    tc::mbar_init(&bars->q_ready, 128);
    tc::mbar_init(&bars->qb_full, 1);
    tc::mbar_init(&bars->qb_empty, 1);
    tc::mbar_init(&bars->drain[0], 1);
    tc::mbar_init(&bars->drain[1], 1);
    bars->abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&bars->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  if (ROPE) {
    // Table rows l < 32 ((cos, sin) of l theta_i, pairs i < R/2) stay here; row
    // l's 16-byte granule g (pairs 2 g, 2 g + 1) sits at g ^ l, so that a warp
    // whose lane l reads granule g of row l hits distinct banks. Rows past the
    // table (max_positions < 32) are never used for a valid position.
    const int half = a.rope_R / 2, gran = half / 2;
    float4* t = reinterpret_cast<float4*>(stab);
    for (int e = threadIdx.x; e < 32 * gran; e += C::kThreads) {
      const int l = e / gran, gidx = e % gran;
      const float4* src = reinterpret_cast<const float4*>(a.rope_table + static_cast<long>(l) * half);
      t[l * 32 + (gidx ^ l)] = l < a.rope_max_positions ? __ldg(src + gidx)
                                                          : make_float4(1.f, 0.f, 1.f, 0.f);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    if (lane == 0) tq_producer<C>(a, &tm_q, &tm_k, &tm_v, skv, sqb, bars);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) tq_mma_s<C>(a, tmem, skv, sqb, bars);
    __syncwarp();
  } else if (warp == 6) {
    if (lane == 0) tq_mma_pv<C>(a, tmem, skv, bars);
    __syncwarp();
  } else {
    tq_softmax<C, ROPE>(a, tmem, bars, warp % 4, lane, &tm_o, sepi + (warp % 4) * 4096, stab);
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

template <int DP, bool ROPE, bool RAGGED>
cudaError_t launch_tq(const AttnShape& s, cudaStream_t stream) {
  using C = PCfg<DP, RAGGED>;
  // The shared-memory allowance is a function attribute of each device's context.
  static PerContext<cudaError_t> attr;
  const cudaError_t attr_err = attr.get(
      [] {
        return cudaFuncSetAttribute(prefill_tq_kernel<DP, ROPE, RAGGED>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
      },
      cudaErrorInvalidDevice, [](cudaError_t e) { return e == cudaSuccess; });
  if (attr_err != cudaSuccess) return attr_err;
  const int Lk = s.Lk > 0 ? s.Lk : s.L;
  CUtensorMap tq, tk, tv, to;
  if (!make_map(&tq, s.q, s.D, s.L, s.B * s.H, kBM) ||
      !make_map(&tk, s.k, s.D, Lk, s.B * s.Hkv, C::BK, s.k_head_rows) ||
      !make_map_vt(&tv, s.vt, s.D, Lk, s.vt_pitch, s.B * s.Hkv, C::DP) ||
      !make_map_out16(&to, s.out, s.D, s.L, s.B * s.H))
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
  a.lengths = s.lengths;
  a.skip = s.skip;
  const int grid = a.units < sm_count() ? a.units : sm_count();
  prefill_tq_kernel<DP, ROPE, RAGGED><<<grid, C::kThreads, C::kSmem, stream>>>(tq, tk, tv, to, a);
  return cudaGetLastError();
}

// The ragged instantiation only when the call has lengths.
template <int DP, bool ROPE>
cudaError_t launch_tq_r(const AttnShape& s, cudaStream_t stream) {
  return s.lengths ? launch_tq<DP, ROPE, true>(s, stream) : launch_tq<DP, ROPE, false>(s, stream);
}

}  // namespace

bool prefill_fuses_rope(int D) { return D % 32 == 0 && D <= 128; }

bool prefill_tq_supports_kv_off(int D) { return D % 4 == 0 && D >= 32 && D <= 256; }

// 32 <= D <= 256, D % 4 == 0; V^T must already be in s.vt (launch_prefill_tc runs
// the transpose first). q RoPE is fused only for D <= 128.
cudaError_t launch_prefill_tq(const AttnShape& s, cudaStream_t stream) {
  switch ((s.D + 31) / 32) {
    // with q RoPE fused (R % 64 == 0, so D >= 64) or without
    case 1: return s.rope.table ? cudaErrorNotSupported : launch_tq_r<32, false>(s, stream);
    case 2: return s.rope.table ? launch_tq_r<64, true>(s, stream) : launch_tq_r<64, false>(s, stream);
    case 3: return s.rope.table ? launch_tq_r<96, true>(s, stream) : launch_tq_r<96, false>(s, stream);
    case 4: return s.rope.table ? launch_tq_r<128, true>(s, stream)
                                : launch_tq_r<128, false>(s, stream);
    // two sub-units (output halves) per query tile, no fused RoPE
    case 5: return s.rope.table ? cudaErrorNotSupported : launch_tq_r<160, false>(s, stream);
    case 6: return s.rope.table ? cudaErrorNotSupported : launch_tq_r<192, false>(s, stream);
    case 7: return s.rope.table ? cudaErrorNotSupported : launch_tq_r<224, false>(s, stream);
    case 8: return s.rope.table ? cudaErrorNotSupported : launch_tq_r<256, false>(s, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace gqa
