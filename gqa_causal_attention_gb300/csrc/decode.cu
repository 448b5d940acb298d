// Single-token decode over a caller-owned cache, split over the key axis.
//
// "mojolearn.transformer", TransformerBlock.step: one new token per row at
// position cached_tokens, attending every cached position (or the last W of
// them under a window; the cache is then a ring of W slots, TransformerState).
// Softmax attention is invariant to the order of its keys, so the live slots
// of a ring are read in slot order.
//
// Split-KV: block (split, kv-head group, b) reduces `chunk` cache slots for
// the GT query heads that share one KV head, so every K/V byte is read once
// for the whole group. Each block leaves (m, l, o) partial results -- row
// maximum and sum in base 2, unnormalised output -- and the combine kernel
// merges them with the usual log-sum-exp rescaling. A row that fits in one
// split is finished by its split block directly.
//
// The work is HBM-bound: 2 * D * 4 bytes per cached position and KV head.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

#include <mutex>

namespace gqa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kDecodeThreads = 128;
constexpr int kDecodeWarps = kDecodeThreads / 32;
constexpr int kUnroll = 4;          // keys per warp per step

// Lane-to-dimension map. V4: lane owns dims 4*lane + 128*k .. +3 (D % 128 == 0);
// otherwise lane owns dims lane + 32*k (any D <= 256).
template <bool V4, int NV>
struct Dims {
  static __device__ __forceinline__ int dim(int lane, int e) {
    return V4 ? (4 * lane + 128 * (e / 4) + (e % 4)) : (lane + 32 * e);
  }
  static __device__ __forceinline__ void load(const float* __restrict__ row, int lane, int D,
                                              float* r) {
    if (V4) {
#pragma unroll
      for (int k = 0; k < NV / 4; ++k) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(row + 4 * lane + 128 * k));
        r[4 * k] = t.x; r[4 * k + 1] = t.y; r[4 * k + 2] = t.z; r[4 * k + 3] = t.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        const int d = lane + 32 * e;
        r[e] = d < D ? __ldg(row + d) : 0.f;
      }
    }
  }
};

}  // namespace

template <int GT, int NV, bool V4>
__global__ void __launch_bounds__(kDecodeThreads) decode_split_kernel(DecodeJob j) {
  using DM = Dims<V4, NV>;
  __shared__ float sm_m[kDecodeWarps][GT];
  __shared__ float sm_l[kDecodeWarps][GT];
  __shared__ float sm_o[kDecodeWarps][GT][kMaxHeadDim];
  if (gated_off(j.skip)) return;

  const int split = blockIdx.x, b = blockIdx.z;
  const int G = j.H / j.Hkv;
  const int ngroups = (G + GT - 1) / GT;
  const int hkv = blockIdx.y / ngroups;
  const int g0 = (blockIdx.y % ngroups) * GT;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int D = j.D;

  const int n = j.cache_len[b];
  if (n < 1 || n > j.max_cache_len || (j.window == 0 && n > j.capacity)) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) report(j.status, ATTN_DEV_LENGTH);
    return;
  }
  const int nlive = j.window > 0 ? min(n, j.window) : n;
  const int nsplit_b = (nlive + j.chunk - 1) / j.chunk;
  const int k0 = split * j.chunk;
  if (k0 >= nlive) return;
  const int k1 = min(k0 + j.chunk, nlive);

  // Queries of the GT heads, pre-multiplied by the softmax scale.
  float q[GT][NV];
#pragma unroll
  for (int g = 0; g < GT; ++g) {
    const int h = hkv * G + g0 + g;
    if (g0 + g < G) {
      DM::load(j.q + ((long)b * j.H + h) * D, lane, D, q[g]);
#pragma unroll
      for (int e = 0; e < NV; ++e) q[g][e] *= j.scale;
    } else {
#pragma unroll
      for (int e = 0; e < NV; ++e) q[g][e] = 0.f;
    }
  }

  const long head_off = ((long)b * j.Hkv + hkv) * j.capacity * D;
  const float* kbase = j.k_cache + head_off;
  const float* vbase = j.v_cache + head_off;
  const bool capped = j.softcap > 0.f;
  const float cap_k = capped ? 2.0f * kLog2e / j.softcap : 0.f;

  float m[GT], l[GT], o[GT][NV];
#pragma unroll
  for (int g = 0; g < GT; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < NV; ++e) o[g][e] = 0.f;
  }

  for (int base = k0 + warp * kUnroll; base < k1; base += kDecodeWarps * kUnroll) {
    float kr[kUnroll][NV], vr[kUnroll][NV];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (base + u < k1) {
        DM::load(kbase + (long)(base + u) * D, lane, D, kr[u]);
        DM::load(vbase + (long)(base + u) * D, lane, D, vr[u]);
      }
    }
    float s[kUnroll][GT];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
      for (int g = 0; g < GT; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < NV; ++e) acc = fmaf(q[g][e], kr[u][e], acc);
        acc = warp_sum(acc);
        if (capped) acc = softcap_apply(acc, j.softcap, cap_k);
        s[u][g] = (base + u < k1) ? acc * kLog2e : -INFINITY;
      }
    }
#pragma unroll
    for (int g = 0; g < GT; ++g) {
      float mx = s[0][g];
#pragma unroll
      for (int u = 1; u < kUnroll; ++u) mx = fmaxf(mx, s[u][g]);
      const float mn = fmaxf(m[g], mx);
      const float corr = exp2f(m[g] - mn);
      m[g] = mn;
      float p[kUnroll];
      float ps = 0.f;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        p[u] = exp2f(s[u][g] - mn);
        ps += p[u];
      }
      l[g] = l[g] * corr + ps;
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        float acc = o[g][e] * corr;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (base + u < k1) acc = fmaf(p[u], vr[u][e], acc);
        o[g][e] = acc;
      }
    }
  }

  // Merge the warps of this block.
#pragma unroll
  for (int g = 0; g < GT; ++g) {
    if (lane == 0) {
      sm_m[warp][g] = m[g];
      sm_l[warp][g] = l[g];
    }
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      const int d = DM::dim(lane, e);
      if (d < D) sm_o[warp][g][d] = o[g][e];
    }
  }
  __syncthreads();

  const bool single = nsplit_b == 1;
  for (int t = threadIdx.x; t < GT * D; t += kDecodeThreads) {
    const int g = t / D, d = t % D;
    if (g0 + g >= G) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, sm_m[w][g]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) {
      const float c = sm_m[w][g] == -INFINITY ? 0.f : exp2f(sm_m[w][g] - M);
      num = fmaf(c, sm_o[w][g][d], num);
      den = fmaf(c, sm_l[w][g], den);
    }
    const long hrow = (long)b * j.H + hkv * G + g0 + g;
    if (single) {
      j.out[hrow * D + d] = num / den;
    } else {
      const long pi = hrow * j.nsplit + split;
      j.partial[pi * D + d] = num;
      if (d == 0) {
        float* ml = j.partial + (long)j.B * j.H * j.nsplit * D;
        ml[2 * pi] = M;
        ml[2 * pi + 1] = den;
      }
    }
  }
}

// ---------------------------------------------------------------- bulk-copy split kernel
// D % 4 == 0: the same split-KV reduction with the cache rows streamed by the
// copy engine. One warp per block; a ring of `nst` stages, each holding KW
// consecutive cache slots of K and of V (each one contiguous run of bytes,
// fetched by cp.async.bulk onto the stage's mbarrier), so the bytes in flight
// are bounded by shared memory rather than registers. Lane l owns dimensions
// 4l + 128c .. +3 of every row.
//
// Scores of a batch: each lane forms its partial dot products for the KW keys
// x GT heads (KW * GT = 32 values), and a butterfly reduce-scatter over the
// warp (5 shuffle steps, 31 shuffles) leaves lane l holding the full score of
// key l / GT and head l % GT. Running maximum and sum then reduce over the
// lanes of one head; P V needs each p broadcast once.
constexpr int kBulkMaxStages = 4;

// A fused step's RMSNorm (optional) and RoPE at position p of one 128-dim row in
// the bulk lane map (lane l holds dims 4l .. 4l + 3): the partner of a rotated dim
// i < R/2 is i + R/2, R/8 lanes away (R % 8 == 0). Every lane must call it.
__device__ __forceinline__ void bulk_rotate_row(const DecodeStepArgs& st, const float* row,
                                                const float* nw, int p, int lane, float* x) {
  const float4 t = __ldg(reinterpret_cast<const float4*>(row) + lane);
  x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
  if (nw) {
    float ss = fmaf(x[0], x[0], fmaf(x[1], x[1], fmaf(x[2], x[2], x[3] * x[3])));
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss / 128.0f + st.norm_eps);
    const float4 w = __ldg(reinterpret_cast<const float4*>(nw) + lane);
    x[0] = x[0] * inv * w.x; x[1] = x[1] * inv * w.y; x[2] = x[2] * inv * w.z; x[3] = x[3] * inv * w.w;
  }
  const int hl = st.R / 8;                    // lanes per half of the rotated dims
  const bool low = lane < hl;
  float o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) o[e] = __shfl_sync(0xffffffffu, x[e], low ? lane + hl : lane - hl);
  if (lane < 2 * hl) {
    const int i = 4 * (low ? lane : lane - hl);       // pairs i .. i + 3
    const float4* tab = reinterpret_cast<const float4*>(st.table + static_cast<long>(p) * (st.R / 2) + i);
    const float4 t0 = __ldg(tab), t1 = __ldg(tab + 1);
    const float cs[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)                      // low: a = x, c = o; high: a = o, c = x
      x[e] = low ? fmaf(x[e], cs[2 * e], -o[e] * cs[2 * e + 1])
                 : fmaf(o[e], cs[2 * e + 1], x[e] * cs[2 * e]);
  }
}

// FUSED (NC == 1, D == 128): the whole decode step (st), a separate instantiation.
template <int GT, int NC, int KW, bool FUSED = false>
__global__ void __launch_bounds__(32) decode_bulk_kernel(DecodeJob j, int nst, DecodeStepArgs st) {
  constexpr int NVAL = KW * GT;               // scores per batch
  constexpr int RL = 32 / NVAL;               // lanes holding each reduced score
  static_assert(NVAL <= 32 && 32 % NVAL == 0, "batch shape");
  constexpr int NV = 4 * NC;                  // dims per lane
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kBulkMaxStages];
  __shared__ int abort_flag;
  if (gated_off(j.skip)) return;

  const int lane = threadIdx.x;
  const int split = blockIdx.x, b = blockIdx.z;
  const int G = j.H / j.Hkv;
  const int ngroups = (G + GT - 1) / GT;
  const int hkv = blockIdx.y / ngroups;
  const int g0 = (blockIdx.y % ngroups) * GT;
  const int D = FUSED ? 128 : j.D;

  int n;
  if (FUSED) {
    const int p = st.pos[b];
    const bool in_table = p >= 0 && p < st.max_positions;
    const bool has_slot = j.window > 0 || p < j.capacity;
    n = in_table && has_slot ? p + 1 : 0;
    if (lane == 0 && split == 0 && blockIdx.y == 0) {       // one block per batch row
      if (!in_table) report(j.status, ATTN_DEV_POSITION);
      else if (!has_slot) report(j.status, ATTN_DEV_CAPACITY);
      st.cache_len[b] = n;                                   // for the combine pass
    }
  } else {
    n = j.cache_len[b];
  }
  if (n < 1 || n > j.max_cache_len || (j.window == 0 && n > j.capacity)) {
    if (lane == 0 && split == 0 && blockIdx.y == 0) report(j.status, ATTN_DEV_LENGTH);
    return;
  }
  const int nlive = j.window > 0 ? min(n, j.window) : n;
  const int nsplit_b = (nlive + j.chunk - 1) / j.chunk;
  const int k0 = split * j.chunk;
  if (k0 >= nlive) return;
  const int k1 = min(k0 + j.chunk, nlive);
  const int nb = (k1 - k0 + KW - 1) / KW;    // batches of this block
  if (FUSED) {
    // The split holding the new position's slot writes its rotated k and its v
    // there first (every head group of the KV head writes the same values); the
    // proxy fence orders those writes before this block's bulk copies read them.
    const int p = n - 1;
    const int slot = j.window > 0 ? p % j.window : p;
    if (slot >= k0 && slot < k1) {
      const long src = (long)b * j.Hkv + hkv;
      float x[4];
      bulk_rotate_row(st, st.k_new + src * 128, st.k_norm_w, p, lane, x);
      // a step's cache is the caller's writable cache (DecodeJob holds it read-only)
      float4* kd = reinterpret_cast<float4*>(const_cast<float*>(j.k_cache) + (src * j.capacity + slot) * 128);
      float4* vd = reinterpret_cast<float4*>(const_cast<float*>(j.v_cache) + (src * j.capacity + slot) * 128);
      kd[lane] = make_float4(x[0], x[1], x[2], x[3]);
      vd[lane] = __ldg(reinterpret_cast<const float4*>(st.v_new + src * 128) + lane);
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    __syncwarp();
  }

  const long head_off = ((long)b * j.Hkv + hkv) * j.capacity * D;
  const float* kbase = j.k_cache + head_off;
  const float* vbase = j.v_cache + head_off;
  const uint32_t part_bytes = KW * D * 4;     // K (then V) rows of one stage
  auto stage_k = [&](int s) { return reinterpret_cast<const float*>(ring + 2 * s * part_bytes); };
  auto stage_v = [&](int s) {
    return reinterpret_cast<const float*>(ring + (2 * s + 1) * part_bytes);
  };
  auto issue = [&](int t) {                   // lane 0: batch t into stage t % nst
    const int s = t % nst;
    const int kb = k0 + t * KW;
    const uint32_t bytes = static_cast<uint32_t>(min(KW, k1 - kb)) * D * 4;
    tc::mbar_arrive_expect_tx(&full[s], 2 * bytes);
    tc::bulk_load(ring + 2 * s * part_bytes, kbase + (long)kb * D, bytes, &full[s]);
    tc::bulk_load(ring + (2 * s + 1) * part_bytes, vbase + (long)kb * D, bytes, &full[s]);
  };
  if (lane == 0) {
    for (int s = 0; s < nst; ++s) tc::mbar_init(&full[s], 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncwarp();
  const int first = min(nst, nb);
  if (lane == 0)
    for (int t = 0; t < first; ++t) issue(t);

  // Queries of the GT heads (scaled), this lane's dimensions.
  float q[GT][NV];
#pragma unroll
  for (int g = 0; g < GT; ++g) {
    if (FUSED) {
      float x[4] = {0.f, 0.f, 0.f, 0.f};
      if (g0 + g < G)                          // warp-uniform
        bulk_rotate_row(st, st.q_raw + ((long)b * j.H + hkv * G + g0 + g) * 128, st.q_norm_w,
                        n - 1, lane, x);
#pragma unroll
      for (int e = 0; e < 4; ++e) q[g][e] = x[e] * j.scale;
      continue;
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int d = 4 * lane + 128 * c;
      float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
      if (g0 + g < G && d < D)
        t = __ldg(reinterpret_cast<const float4*>(j.q + ((long)b * j.H + hkv * G + g0 + g) * D + d));
      q[g][4 * c] = t.x * j.scale; q[g][4 * c + 1] = t.y * j.scale;
      q[g][4 * c + 2] = t.z * j.scale; q[g][4 * c + 3] = t.w * j.scale;
    }
  }
  const bool capped = j.softcap > 0.f;
  const float cap_k = capped ? 2.0f * kLog2e / j.softcap : 0.f;
  auto load_row = [&](const float* row, float* r) {
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int d = 4 * lane + 128 * c;
      float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
      if (d < D) t = *reinterpret_cast<const float4*>(row + d);
      r[4 * c] = t.x; r[4 * c + 1] = t.y; r[4 * c + 2] = t.z; r[4 * c + 3] = t.w;
    }
  };

  const int my_u = lane / RL / GT;            // key (within the batch) and head of this
  float m_run = -INFINITY, l_run = 0.f;       // lane's score; running max / sum of that head
  float o[GT][NV];
#pragma unroll
  for (int g = 0; g < GT; ++g)
#pragma unroll
    for (int e = 0; e < NV; ++e) o[g][e] = 0.f;

  int t = 0;
  for (; t < nb; ++t) {
    const int s = t % nst;
    const bool ok = tc::mbar_wait(&full[s], (t / nst) & 1, &abort_flag);
    if (__any_sync(0xffffffffu, !ok)) break;
    const int valid = min(KW, k1 - (k0 + t * KW));
    const float* sk = stage_k(s);
    const float* sv = stage_v(s);

    // partial dot products, index u * GT + g
    float v[NVAL];
#pragma unroll
    for (int u = 0; u < KW; ++u) {
      float kr[NV];
      load_row(sk + u * D, kr);
#pragma unroll
      for (int g = 0; g < GT; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < NV; ++e) acc = fmaf(q[g][e], kr[e], acc);
        v[u * GT + g] = acc;
      }
    }
    // reduce-scatter: the step over lane bit `off` halves the values a lane
    // keeps (upper half where that bit is set); once one value is left the
    // remaining bits are summed outright. Lane l ends with the full score of
    // index l / RL.
#pragma unroll
    for (int half = NVAL / 2, off = 16; half >= 1; half >>= 1, off >>= 1) {
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float send = upper ? v[i] : v[i + half];
        const float keep = upper ? v[i + half] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
#pragma unroll
    for (int off = RL / 2; off >= 1; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    float sc = v[0];
    if (capped) sc = softcap_apply(sc, j.softcap, cap_k);
    sc = my_u < valid ? sc * kLog2e : -INFINITY;
    // over the keys of one head: lanes that differ above bit log2(RL * GT)
    float mx = sc;
#pragma unroll
    for (int off = RL * GT; off < 32; off <<= 1)
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float m_new = fmaxf(m_run, mx);
    const float corr = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);
    const float p = m_new == -INFINITY ? 0.f : exp2f(sc - m_new);
    float ps = p;
#pragma unroll
    for (int off = RL * GT; off < 32; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l_run = l_run * corr + ps;
    m_run = m_new;

#pragma unroll
    for (int g = 0; g < GT; ++g) {
      const float cg = __shfl_sync(0xffffffffu, corr, g * RL);
#pragma unroll
      for (int e = 0; e < NV; ++e) o[g][e] *= cg;
    }
#pragma unroll
    for (int u = 0; u < KW; ++u) {
      if (u < valid) {                        // slots past the copied rows hold stale bytes
        float vr[NV];
        load_row(sv + u * D, vr);
#pragma unroll
        for (int g = 0; g < GT; ++g) {
          const float pg = __shfl_sync(0xffffffffu, p, (u * GT + g) * RL);
#pragma unroll
          for (int e = 0; e < NV; ++e) o[g][e] = fmaf(pg, vr[e], o[g][e]);
        }
      }
    }
    __syncwarp();                             // every lane is done reading stage s
    if (lane == 0 && t + nst < nb) issue(t + nst);
  }
  if (t < nb) {
    // A wait ran out: let the copies already issued land, then report.
    if (lane == 0) {
      for (int u = t; u < min(nb, t + nst); ++u) {
        const uint64_t t0 = tc::globaltimer();
        while (!tc::mbar_try_wait(&full[u % nst], (u / nst) & 1))
          if (tc::globaltimer() - t0 > tc::kWaitLimitNs) break;
      }
      report(j.status, ATTN_DEV_TIMEOUT);
    }
    return;
  }

  const bool single = nsplit_b == 1;
#pragma unroll
  for (int g = 0; g < GT; ++g) {
    const float M = __shfl_sync(0xffffffffu, m_run, g * RL);
    const float L = __shfl_sync(0xffffffffu, l_run, g * RL);
    if (g0 + g >= G) continue;
    const long hrow = (long)b * j.H + hkv * G + g0 + g;
    const float inv = 1.0f / L;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int d = 4 * lane + 128 * c;
      if (d >= D) continue;
      if (single) {
        *reinterpret_cast<float4*>(j.out + hrow * D + d) =
            make_float4(o[g][4 * c] * inv, o[g][4 * c + 1] * inv, o[g][4 * c + 2] * inv,
                        o[g][4 * c + 3] * inv);
      } else {
        const long pi = hrow * j.nsplit + split;
        *reinterpret_cast<float4*>(j.partial + pi * D + d) =
            make_float4(o[g][4 * c], o[g][4 * c + 1], o[g][4 * c + 2], o[g][4 * c + 3]);
      }
    }
    if (!single && lane == 0) {
      const long pi = hrow * j.nsplit + split;
      float* ml = j.partial + (long)j.B * j.H * j.nsplit * D;
      ml[2 * pi] = M;
      ml[2 * pi + 1] = L;
    }
  }
}

// out[b, h, :] = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s over the splits of row b.
__global__ void __launch_bounds__(128) decode_combine_kernel(DecodeJob j) {
  if (gated_off(j.skip)) return;
  const int h = blockIdx.x, b = blockIdx.y;
  const int n = j.cache_len[b];
  if (n < 1 || n > j.max_cache_len || (j.window == 0 && n > j.capacity)) return;
  const int nlive = j.window > 0 ? min(n, j.window) : n;
  const int ns = (nlive + j.chunk - 1) / j.chunk;
  if (ns <= 1) return;                       // finished by the split block
  const long hrow = (long)b * j.H + h;
  const float* ml = j.partial + (long)j.B * j.H * j.nsplit * j.D + 2 * hrow * j.nsplit;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, ml[2 * s]);
  float den = 0.f;
  for (int s = 0; s < ns; ++s) den = fmaf(exp2f(ml[2 * s] - M), ml[2 * s + 1], den);
  const float inv = 1.0f / den;
  const float* op = j.partial + hrow * j.nsplit * j.D;
  for (int d = threadIdx.x; d < j.D; d += blockDim.x) {
    float num = 0.f;
    for (int s = 0; s < ns; ++s) num = fmaf(exp2f(ml[2 * s] - M), op[(long)s * j.D + d], num);
    j.out[hrow * j.D + d] = num * inv;
  }
}

void decode_split_plan(int B, int Hkv, int max_cache_len, int window, int* nsplit, int* chunk) {
  const int eff = window > 0 ? (max_cache_len < window ? max_cache_len : window) : max_cache_len;
  const int units = B * Hkv;
  // Many short splits: the blocks' lengths then even out across the SMs (at
  // the batched-decode size 256-slot splits beat 512 by 5 %, 1024 lost 11 %);
  // the partial results cost 2 (D + 2) floats per split and head.
  const int per_row = (4096 + units - 1) / units;
  int c = (eff + per_row - 1) / per_row;
  c = ((c + 63) / 64) * 64;
  if (c < 64) c = 64;                            // few rows: more, shorter splits fill the GPU
  if (c > 256) c = 256;
  *chunk = c;
  *nsplit = (eff + c - 1) / c;
}

// The plan's split count is not monotone in the length: it peaks at per_row at
// the end of each chunk band (64 per_row, 128 per_row, ... positions) and drops
// when the chunk grows. The largest count over every length up to
// max_cache_len is therefore per_row once the first band is passed.
int decode_split_bound(int B, int Hkv, int max_cache_len, int window) {
  int nsplit, chunk;
  decode_split_plan(B, Hkv, max_cache_len, window, &nsplit, &chunk);
  const int eff = window > 0 ? (max_cache_len < window ? max_cache_len : window) : max_cache_len;
  const int units = B * Hkv;
  const int per_row = (4096 + units - 1) / units;
  if (eff > 64 * per_row && nsplit < per_row) nsplit = per_row;
  return nsplit;
}

size_t decode_partial_bytes(int B, int H, int Hkv, int D, int max_cache_len, int window,
                            bool bound) {
  int nsplit, chunk;
  if (bound)
    nsplit = decode_split_bound(B, Hkv, max_cache_len, window);
  else
    decode_split_plan(B, Hkv, max_cache_len, window, &nsplit, &chunk);
  if (nsplit <= 1) return 16;      // never read; a non-empty buffer keeps the rule simple
  return (size_t)B * H * nsplit * (D + 2) * sizeof(float);
}

// ---------------------------------------------------------------- head-pair split kernel
// Groups of 8 query heads per key/value head (G % 8 == 0), D % 4 == 0, D <= 128:
// the same split-KV reduction and the same bulk-copy ring, with a lane map that
// spends fewer instructions per key. The bulk kernel above holds 4 dims of all
// 8 heads per lane, so each score needs a 32-lane reduction and P V a shuffle
// per weight; here lane l = (pair l / 8, group l % 8) holds heads 2 pair,
// 2 pair + 1 and dims 32 c + 4 group .. + 3 (c < 4; 16-byte shared loads of one
// row by the 8 groups fall on distinct banks). A score is summed over the 8
// lanes of its pair (3 shuffles), which then all hold it, so the running
// maximum, the sum and P V need no further exchange.
// Shared memory per warp: its ring, at least the 36 floats per lane it hands to
// warp 0 at the end (which also covers warp 0's 8 D + 17 floats for a cluster
// merge).
constexpr float kPairRescaleLog2 = 8.0f;   // O is rescaled when the max grows by > 2^8

// A fused step's RMSNorm (optional) and RoPE at position p of one 128-dim row, in
// the head-pair lane map: lane group grp holds dims 32 c + 4 grp .. + 3 (c < 4);
// the 8 lanes of a group reduce the sum of squares together. With R = 128 or 64
// the partner dim i + R/2 of every rotated dim i sits in the same lane (c + 2 or
// c + 1). Every lane must call it (the reduction shuffles over the whole warp).
__device__ __forceinline__ void pair_rotate_row(const DecodeStepArgs& j, const float* row,
                                                const float* nw, int p, int grp, float* x) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float4 t = __ldg(reinterpret_cast<const float4*>(row + 32 * c + 4 * grp));
    x[4 * c] = t.x; x[4 * c + 1] = t.y; x[4 * c + 2] = t.z; x[4 * c + 3] = t.w;
  }
  if (nw) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = 1.0f / sqrtf(ss / 128.0f + j.norm_eps);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 w = __ldg(reinterpret_cast<const float4*>(nw + 32 * c + 4 * grp));
      x[4 * c] = x[4 * c] * inv * w.x; x[4 * c + 1] = x[4 * c + 1] * inv * w.y;
      x[4 * c + 2] = x[4 * c + 2] * inv * w.z; x[4 * c + 3] = x[4 * c + 3] * inv * w.w;
    }
  }
  const int half = j.R / 2;
  const float4* tab = reinterpret_cast<const float4*>(j.table + static_cast<long>(p) * half);
  // dims of chunk c pair with those of chunk c2 (c2 = c + R / 64); both compile-time
  auto rot = [&](auto cc, auto cc2) {
    constexpr int c = decltype(cc)::value, c2 = decltype(cc2)::value;
    const float4 t0 = __ldg(tab + (32 * c + 4 * grp) / 2), t1 = __ldg(tab + (32 * c + 4 * grp) / 2 + 1);
    const float cs[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = x[4 * c + e], o = x[4 * c2 + e];
      x[4 * c + e] = fmaf(a, cs[2 * e], -o * cs[2 * e + 1]);
      x[4 * c2 + e] = fmaf(a, cs[2 * e + 1], o * cs[2 * e]);
    }
  };
  using I0 = std::integral_constant<int, 0>;
  using I1 = std::integral_constant<int, 1>;
  using I2 = std::integral_constant<int, 2>;
  using I3 = std::integral_constant<int, 3>;
  if (half == 64) {
    rot(I0{}, I2{});
    rot(I1{}, I3{});
  } else {
    rot(I0{}, I1{});
  }
}

__host__ __device__ inline uint32_t pair_ring_stride(int nst, uint32_t part_bytes) {
  const uint32_t ring = static_cast<uint32_t>(nst) * 2 * part_bytes, merge = 36u * 32 * 4;
  return ((ring > merge ? ring : merge) + 127) / 128 * 128;
}

// NW warps per block share one split: warp w takes batches w, w + NW, ... of
// it through its own ring, and the warps' running (max, sum, O) are merged in
// shared memory at the end, so a split costs one partial result whatever NW is.
// FUSED (D128 only): the whole decode step (st), a separate instantiation so
// that the plain kernel's code is not touched by the step's prologue.
// CL > 1: the grid's x is one cluster of CL blocks per (row, group of 8 heads);
// block r takes the r-th of CL equal runs of whole batches of the row's cached
// keys, and the blocks merge their (max, sum, O) through distributed shared
// memory and write the output themselves (no partials, no combine pass).
// Clustered blocks: registers for 16 warps per SM (no bound otherwise).
template <int NW, int KP, bool D128, bool FUSED = false, int CL = 1>
__global__ void __launch_bounds__(32 * NW, CL > 1 ? 16 / NW : 0) decode_pair_kernel(DecodeJob j, int nst,
                                                              DecodeStepArgs st) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full_all[NW][kBulkMaxStages];
  __shared__ int abort_flag;
  if (gated_off(j.skip)) return;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int pair = lane >> 3, grp = lane & 7;
  const int split = blockIdx.x, b = blockIdx.z;
  const int G = j.H / j.Hkv;
  const int ngroups = G / 8;
  const int hkv = blockIdx.y / ngroups;
  const int g0 = (blockIdx.y % ngroups) * 8;
  const int D = D128 ? 128 : j.D;            // D128: every lane's 16 dims are real

  int n;
  if (FUSED) {
    const int p = st.pos[b];
    const bool in_table = p >= 0 && p < st.max_positions;
    const bool has_slot = j.window > 0 || p < j.capacity;
    n = in_table && has_slot ? p + 1 : 0;
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) {   // one block per batch row
      if (!in_table) report(j.status, ATTN_DEV_POSITION);
      else if (!has_slot) report(j.status, ATTN_DEV_CAPACITY);
      st.cache_len[b] = n;                                    // for the combine pass
    }
  } else {
    n = j.cache_len[b];
  }
  if (n < 1 || n > j.max_cache_len || (j.window == 0 && n > j.capacity)) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) report(j.status, ATTN_DEV_LENGTH);
    return;                                   // the whole block leaves together
  }
  const int nlive = j.window > 0 ? min(n, j.window) : n;
  const int nsplit_b = (nlive + j.chunk - 1) / j.chunk;
  int k0, k1;
  if constexpr (CL > 1) {
    // Every block of the cluster stays to the end (the merge's barriers), also
    // one whose run is empty.
    const int per = (nlive + CL * KP - 1) / (CL * KP) * KP;
    k0 = min(split * per, nlive);
    k1 = min(k0 + per, nlive);
  } else {
    k0 = split * j.chunk;
    if (k0 >= nlive) return;
    k1 = min(k0 + j.chunk, nlive);
  }
  const int nb = (k1 - k0 + KP - 1) / KP;                 // batches of the split
  if (FUSED && warp == 0) {
    // The split holding the new position's slot writes its rotated k and its v
    // there first (every group of a KV head writes the same values); the proxy
    // fence orders those writes before this block's bulk copies read them.
    const int p = n - 1;
    const int slot = j.window > 0 ? p % j.window : p;
    if (slot >= k0 && slot < k1) {
      const long src = (long)b * j.Hkv + hkv;
      float x[16];
      pair_rotate_row(st, st.k_new + src * 128, st.k_norm_w, p, grp, x);
      // a step's cache is the caller's writable cache (DecodeJob holds it read-only)
      float* kd = const_cast<float*>(j.k_cache) + (src * j.capacity + slot) * 128;
      float* vd = const_cast<float*>(j.v_cache) + (src * j.capacity + slot) * 128;
      const float* vs = st.v_new + src * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int d = 32 * c + 4 * grp;
        if (pair == 0)
          *reinterpret_cast<float4*>(kd + d) = make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
        else if (pair == 1)
          *reinterpret_cast<float4*>(vd + d) = __ldg(reinterpret_cast<const float4*>(vs + d));
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
  }
  const int nbw = nb > warp ? (nb - warp + NW - 1) / NW : 0;   // this warp's: warp + NW i

  const long head_off = ((long)b * j.Hkv + hkv) * j.capacity * D;
  const float* kbase = j.k_cache + head_off;
  const float* vbase = j.v_cache + head_off;
  const uint32_t part_bytes = KP * D * 4;
  const uint32_t stride = pair_ring_stride(nst, part_bytes);
  uint8_t* ring = smem + warp * stride;
  uint64_t* full = full_all[warp];
  auto issue = [&](int i) {                   // lane 0: this warp's batch i into stage i % nst
    const int s = i % nst;
    const int kb = k0 + (warp + NW * i) * KP;
    const uint32_t bytes = static_cast<uint32_t>(min(KP, k1 - kb)) * D * 4;
    tc::mbar_arrive_expect_tx(&full[s], 2 * bytes);
    tc::bulk_load(ring + 2 * s * part_bytes, kbase + (long)kb * D, bytes, &full[s]);
    tc::bulk_load(ring + (2 * s + 1) * part_bytes, vbase + (long)kb * D, bytes, &full[s]);
  };
  if (threadIdx.x == 0) abort_flag = 0;
  if (lane == 0) {
    for (int s = 0; s < nst; ++s) tc::mbar_init(&full[s], 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (lane == 0)
    for (int i = 0; i < min(nst, nbw); ++i) issue(i);

  // this lane's 16 dims of a row (zeros past D)
  auto load16 = [&](const float* row, float* r) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int d = 32 * c + 4 * grp;
      float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
      if (D128 || d < D) t = *reinterpret_cast<const float4*>(row + d);
      r[4 * c] = t.x; r[4 * c + 1] = t.y; r[4 * c + 2] = t.z; r[4 * c + 3] = t.w;
    }
  };
  // q (pre-scaled) and O as pairs of adjacent dims: one paired FMA serves two.
  // Scores come out in log2 units: q carries scale * log2(e), and the softcap
  // runs on the scaled score with the cap scaled alike (L c tanh(s / c) =
  // (L c) tanh(L s / (L c)), L = log2 e).
  const float qscale = j.scale * kLog2e;
  uint64_t q2[2][8], o2[2][8];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const long qrow = (long)b * j.H + hkv * G + g0 + 2 * pair + h;
    if (FUSED) {
      float x[16];
      pair_rotate_row(st, st.q_raw + qrow * 128, st.q_norm_w, n - 1, grp, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) q2[h][e] = tc::pack2(x[2 * e] * qscale, x[2 * e + 1] * qscale);
    } else {
      const float* qr = j.q + qrow * D;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int d = 32 * c + 4 * grp;
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
        if (D128 || d < D) t = __ldg(reinterpret_cast<const float4*>(qr + d));
        q2[h][2 * c] = tc::pack2(t.x * qscale, t.y * qscale);
        q2[h][2 * c + 1] = tc::pack2(t.z * qscale, t.w * qscale);
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) o2[h][e] = tc::pack2(0.f, 0.f);
  }
  const bool capped = j.softcap > 0.f;
  const float cap_l2 = j.softcap * kLog2e;                  // the cap in log2 units
  const float cap_k = capped ? 2.0f / j.softcap : 0.f;      // 2 log2(e) / cap_l2
  // Weights are taken against a reference maximum m_run (log2 units) that moves
  // only when a score exceeds it by more than 2^kPairRescaleLog2; O and l are
  // rescaled then. A weight is therefore at most 2^kPairRescaleLog2, and most
  // batches need no rescale.
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

  int i = 0;
  for (; i < nbw; ++i) {
    const int s = i % nst;
    const bool ok = tc::mbar_wait(&full[s], (i / nst) & 1, &abort_flag);
    if (__any_sync(0xffffffffu, !ok)) break;
    const int valid = min(KP, k1 - (k0 + (warp + NW * i) * KP));
    const float* sk = reinterpret_cast<const float*>(ring + 2 * s * part_bytes);
    const float* sv = reinterpret_cast<const float*>(ring + (2 * s + 1) * part_bytes);
    // Only a split's last batch can be partial: the full ones skip the key checks.
    auto batch = [&](auto full_c) {
      constexpr bool FULL = decltype(full_c)::value;
      float sc[2][KP];
#pragma unroll
      for (int u = 0; u < KP; ++u) {
        float kr[16];
        load16(sk + u * D, kr);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint64_t acc = tc::pack2(0.f, 0.f);   // even and odd dims: two FMA chains
#pragma unroll
          for (int e = 0; e < 8; ++e)
            acc = tc::fma2(q2[h][e], tc::pack2(kr[2 * e], kr[2 * e + 1]), acc);
          float a0, a1;
          tc::unpack2(acc, a0, a1);
          float sum = a0 + a1;
#pragma unroll
          for (int off = 1; off < 8; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
          sc[h][u] = sum;
        }
      }
      if (capped) {                           // one branch per batch
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int u = 0; u < KP; ++u) sc[h][u] = softcap_apply(sc[h][u], cap_l2, cap_k);
      }
      if (!FULL) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int u = 0; u < KP; ++u)
            if (u >= valid) sc[h][u] = -INFINITY;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float mx = sc[h][0];
#pragma unroll
        for (int u = 1; u < KP; ++u) mx = fmaxf(mx, sc[h][u]);
        const bool grow = mx > m_run[h] + kPairRescaleLog2;   // also the row's first finite score
        if (__any_sync(0xffffffffu, grow)) {
          const float corr = grow ? tc::ex2(m_run[h] - mx) : 1.f;   // 0 while O and l are 0
          const uint64_t c2 = tc::pack2(corr, corr);
#pragma unroll
          for (int e = 0; e < 8; ++e) o2[h][e] = tc::mul2(o2[h][e], c2);
          l_run[h] *= corr;
          if (grow) m_run[h] = mx;
        }
        const float mu = m_run[h] == -INFINITY ? 0.f : m_run[h];   // all keys so far masked
        float ls = 0.f;
#pragma unroll
        for (int u = 0; u < KP; ++u) {
          sc[h][u] = tc::ex2(sc[h][u] - mu);
          ls += sc[h][u];
        }
        l_run[h] += ls;
      }
#pragma unroll
      for (int u = 0; u < KP; ++u) {
        if (FULL || u < valid) {              // slots past the copied rows hold stale bytes
          float vr[16];
          load16(sv + u * D, vr);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint64_t p2 = tc::pack2(sc[h][u], sc[h][u]);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              o2[h][e] = tc::fma2(p2, tc::pack2(vr[2 * e], vr[2 * e + 1]), o2[h][e]);
          }
        }
      }
    };
    if (valid == KP)
      batch(std::true_type{});
    else
      batch(std::false_type{});
    __syncwarp();                             // every lane is done reading stage s
    if (lane == 0 && i + nst < nbw) issue(i + nst);
  }
  float o[2][16];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int e = 0; e < 8; ++e) tc::unpack2(o2[h][e], o[h][2 * e], o[h][2 * e + 1]);
  const bool timed_out = i < nbw;
  if (timed_out && lane == 0) {
    // A wait ran out: let the copies already issued land, then report.
    for (int u = i; u < min(nbw, i + nst); ++u) {
      const uint64_t t0 = tc::globaltimer();
      while (!tc::mbar_try_wait(&full[u % nst], (u / nst) & 1))
        if (tc::globaltimer() - t0 > tc::kWaitLimitNs) break;
    }
    report(j.status, ATTN_DEV_TIMEOUT);
  }

  if (NW > 1) {
    // Merge: warps 1.. leave (m, l, O) in their (now idle) ring, warp 0 folds them in.
    // Every warp reaches the barrier, also after a timeout.
    __syncthreads();                          // all rings idle
    float* xs = reinterpret_cast<float*>(ring) + lane * 36;
    if (warp > 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        xs[h] = m_run[h];
        xs[2 + h] = l_run[h];
#pragma unroll
        for (int e = 0; e < 16; ++e) xs[4 + 16 * h + e] = o[h][e];
      }
    }
    __syncthreads();
    if (CL == 1 && warp > 0) return;
    for (int w = 1; warp == 0 && w < NW; ++w) {
      const float* ys = reinterpret_cast<const float*>(smem + w * stride) + lane * 36;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float m2 = ys[h];
        const float M = fmaxf(m_run[h], m2);
        if (M == -INFINITY) continue;         // neither warp saw a key
        const float f1 = exp2f(m_run[h] - M), f2 = exp2f(m2 - M);
        l_run[h] = l_run[h] * f1 + ys[2 + h] * f2;
#pragma unroll
        for (int e = 0; e < 16; ++e) o[h][e] = o[h][e] * f1 + ys[4 + 16 * h + e] * f2;
        m_run[h] = M;
      }
    }
  }
  if constexpr (CL > 1) {
    // Warp 0 leaves the block's (m, l, O) and its abort flag in its own ring
    // (idle now; 8 D + 17 floats, within pair_ring_stride's merge area): O of
    // head hh at [hh D, hh D + D), m at 8 D + hh, l at 8 D + 8 + hh, the flag at
    // 8 D + 16. After the cluster barrier, thread t of block r merges output
    // elements e = r 32 NW + t (+ multiples of CL 32 NW) over the CL blocks.
    float* ex = reinterpret_cast<float*>(smem);
    if (warp == 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int hh = 2 * pair + h;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int d = 32 * c + 4 * grp;
          if (D128 || d < D)
            *reinterpret_cast<float4*>(ex + hh * D + d) =
                make_float4(o[h][4 * c], o[h][4 * c + 1], o[h][4 * c + 2], o[h][4 * c + 3]);
        }
        if (grp == 0) {
          ex[8 * D + hh] = m_run[h];
          ex[8 * D + 8 + hh] = l_run[h];
        }
      }
      if (lane == 0) ex[8 * D + 16] = abort_flag ? 1.f : 0.f;
    }
    tc::cluster_sync();                       // every block's export is written
    const uint32_t ex_a = tc::smem_u32(ex);
    const long orow = (long)b * j.H + hkv * G + g0;
    for (int e = split * NW * 32 + threadIdx.x; e < 8 * D; e += CL * NW * 32) {
      const int hh = e / D, d = e - hh * D;
      float mv[CL], lv[CL], ov[CL];
      float bad = 0.f;
#pragma unroll
      for (int r = 0; r < CL; ++r) {
        const uint32_t base = tc::cluster_addr(ex_a, r);
        mv[r] = tc::ld_cluster_f32(base + 4u * (8 * D + hh));
        lv[r] = tc::ld_cluster_f32(base + 4u * (8 * D + 8 + hh));
        ov[r] = tc::ld_cluster_f32(base + 4u * e);
        bad += tc::ld_cluster_f32(base + 4u * (8 * D + 16));
      }
      float M = mv[0];
#pragma unroll
      for (int r = 1; r < CL; ++r) M = fmaxf(M, mv[r]);
      float L = 0.f, O = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int r = 0; r < CL; ++r) {
          const float f = exp2f(mv[r] - M);   // 0 for a block without keys
          L = fmaf(lv[r], f, L);
          O = fmaf(ov[r], f, O);
        }
      }
      if (bad == 0.f) j.out[(orow + hh) * D + d] = L > 0.f ? O / L : 0.f;
    }
    tc::cluster_sync();                       // no block leaves while its export is read
    return;
  }
  if (__any_sync(0xffffffffu, timed_out) || abort_flag) return;

  const bool single = nsplit_b == 1;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const long hrow = (long)b * j.H + hkv * G + g0 + 2 * pair + h;
    const float inv = 1.0f / l_run[h];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int d = 32 * c + 4 * grp;
      if (!D128 && d >= D) continue;
      if (single) {
        *reinterpret_cast<float4*>(j.out + hrow * D + d) =
            make_float4(o[h][4 * c] * inv, o[h][4 * c + 1] * inv, o[h][4 * c + 2] * inv,
                        o[h][4 * c + 3] * inv);
      } else {
        const long pi = hrow * j.nsplit + split;
        *reinterpret_cast<float4*>(j.partial + pi * D + d) =
            make_float4(o[h][4 * c], o[h][4 * c + 1], o[h][4 * c + 2], o[h][4 * c + 3]);
      }
    }
    if (!single && grp == 0) {
      const long pi = hrow * j.nsplit + split;
      float* ml = j.partial + (long)j.B * j.H * j.nsplit * D;
      ml[2 * pi] = m_run[h];
      ml[2 * pi + 1] = l_run[h];
    }
  }
}

// Batches of KW = 8 keys (32 / GT when that is smaller) and about 16 KB of
// ring per block: 13 one-warp blocks per SM at D = 128. Measured on the
// batched-decode workload, wider rings (fewer blocks) and narrower batches
// (more per-batch overhead) were both slower.
constexpr int kBulkKeys = 8;
constexpr int kBulkStageBudget = 16 * 1024;   // ring bytes per block (at least 2 stages)
constexpr int kPairWarps = 1, kPairKeys = 8;   // head-pair kernel: warps per split, keys per batch

template <int GT, int NC>
static cudaError_t launch_bulk(const DecodeJob& j, dim3 grid, cudaStream_t stream,
                               const DecodeStepArgs* step) {
  constexpr int KW = GT * kBulkKeys > 32 ? 32 / GT : kBulkKeys;
  const int stage = 2 * KW * j.D * 4;
  int nst = kBulkStageBudget / stage;
  nst = nst < 2 ? 2 : (nst > kBulkMaxStages ? kBulkMaxStages : nst);
  if constexpr (NC == 1) {                    // a fused step has D = 128
    if (step) {
      decode_bulk_kernel<GT, NC, KW, true><<<grid, 32, nst * stage, stream>>>(j, nst, *step);
      return cudaSuccess;
    }
  }
  decode_bulk_kernel<GT, NC, KW><<<grid, 32, nst * stage, stream>>>(j, nst, DecodeStepArgs{});
  return cudaSuccess;
}

template <int GT>
static cudaError_t launch_gt(const DecodeJob& j, cudaStream_t stream, const DecodeStepArgs* step) {
  const int G = j.H / j.Hkv;
  const int ngroups = (G + GT - 1) / GT;
  dim3 grid(j.nsplit, j.Hkv * ngroups, j.B);
  if (j.D % 4 == 0) {
    cudaError_t e = j.D <= 128 ? launch_bulk<GT, 1>(j, grid, stream, step)
                               : launch_bulk<GT, 2>(j, grid, stream, step);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess || j.nsplit <= 1) return e;
    decode_combine_kernel<<<dim3(j.H, j.B), 128, 0, stream>>>(j);
    return cudaGetLastError();
  }
  if (j.D % 128 == 0) {
    if (j.D == 128)
      decode_split_kernel<GT, 4, true><<<grid, kDecodeThreads, 0, stream>>>(j);
    else
      decode_split_kernel<GT, 8, true><<<grid, kDecodeThreads, 0, stream>>>(j);
  } else {
    decode_split_kernel<GT, kMaxHeadDim / 32, false><<<grid, kDecodeThreads, 0, stream>>>(j);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || j.nsplit <= 1) return e;
  decode_combine_kernel<<<dim3(j.H, j.B), 128, 0, stream>>>(j);
  return cudaGetLastError();
}

// One decode step's prep pass: a warp per q or k row (RMSNorm, RoPE at the row's
// position), v rows copied beside their k rows, cache lengths set.
__global__ void __launch_bounds__(256) decode_prep_kernel(DecodePrepJob j) {
  if (gated_off(j.skip)) return;
  const int lane = threadIdx.x & 31;
  const long nwarps = gridDim.x * 8L, gw = blockIdx.x * 8L + threadIdx.x / 32;
  const long qrows = (long)j.B * j.H, rows = qrows + (long)j.B * j.Hkv;
  const int D = j.D, R = j.R, half = R / 2;
  for (long row = gw; row < rows; row += nwarps) {
    const bool isq = row < qrows;
    const long r = isq ? row : row - qrows;
    const int nh = isq ? j.H : j.Hkv;
    const int b = static_cast<int>(r / nh);
    const int p = j.pos[b];
    const bool in_table = p >= 0 && p < j.max_positions;
    const bool has_slot = j.window > 0 || p < j.capacity;
    const bool lead = isq && r % nh == 0 && lane == 0;     // one report per batch row
    if (lead) {
      if (!in_table) report(j.status, ATTN_DEV_POSITION);
      else if (!has_slot) report(j.status, ATTN_DEV_CAPACITY);
      j.cache_len[b] = in_table && has_slot ? p + 1 : 0;
    }
    if (!in_table || !has_slot) continue;
    const float* x = (isq ? j.q : j.k) + r * D;
    const float* nw = isq ? j.q_norm_w : j.k_norm_w;
    const long slot = j.window > 0 ? p % j.window : p;
    float* y = isq ? j.qrot + r * D : j.k_cache + (r * j.capacity + slot) * D;
    float inv = 1.0f;
    if (nw) {
      float ss = 0.f;
      for (int i = lane; i < D; i += 32) ss = fmaf(x[i], x[i], ss);
      ss = warp_sum(ss);
      inv = 1.0f / sqrtf(ss / static_cast<float>(D) + j.norm_eps);
    }
    const float2* tab = j.table + static_cast<long>(p) * half;
    for (int i = lane; i < half; i += 32) {
      float a = x[i], c = x[i + half];
      if (nw) {
        a = a * inv * nw[i];
        c = c * inv * nw[i + half];
      }
      const float2 cs = tab[i];
      y[i] = fmaf(a, cs.x, -c * cs.y);
      y[i + half] = fmaf(a, cs.y, c * cs.x);
    }
    for (int i = R + lane; i < D; i += 32) y[i] = nw ? x[i] * inv * nw[i] : x[i];
    if (!isq) {
      const float* vr = j.v + r * D;
      float* vd = j.v_cache + (r * j.capacity + slot) * D;
      for (int i = lane; i < D; i += 32) vd[i] = vr[i];
    }
  }
}

cudaError_t launch_decode_prep(const DecodePrepJob& j, cudaStream_t stream) {
  const long rows = (long)j.B * (j.H + j.Hkv);
  long blocks = (rows + 7) / 8;
  if (blocks > 152L * 8) blocks = 152L * 8;
  if (blocks < 1) blocks = 1;
  decode_prep_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(j);
  return cudaGetLastError();
}

bool decode_step_fuses(int H, int Hkv, int D, int R) {
  if (Hkv < 1 || D != 128 || R < 8 || R > 128 || R % 8 != 0) return false;
  // the head-pair kernel (8 heads per group) holds dims 32 c + 4 g: R = 64 or 128;
  // the bulk kernel (other groups) holds dims 4 l .. 4 l + 3: any R % 8 == 0
  return (H / Hkv) % 8 == 0 ? (R == 64 || R == 128) : true;
}

// The clustered head-pair kernel: one cluster per (row, group of 8 heads), in
// one of two shapes, both 16 warps per SM with 2-stage rings: up to
// kPairShortKeys live positions 8 blocks x 4 warps with 4-key batches (8 KB of
// ring per warp; half the blocks to merge, so a shorter fixed cost), beyond that
// 16 blocks x 2 warps with 6-key batches (12 KB per warp). With a cluster per
// group a row's splits merge through distributed shared memory instead of
// partial results and a combine launch; it is used when every group fits on the
// GPU at once. Measured on the carried-decode shape (B = 8, 64 query heads over
// 8 KV heads, graph-timed steps) at 64 / 512 / 1024 / 1536 / 2048 / 8192 cached
// positions: 8 x 4 x 4 keys 7.8 / 12.9 / 19.0 / 26.7 / 33.3 / 106.2 us, 16 x 2 x
// 6 keys 10.4 / 14.5 / 20.3 / 26.2 / 32.7 / 101.5 us; a third ring stage was
// 1-2 % slower, 8 x 4 with 6-key batches did not fit one wave.
template <int CL_, int NW_, int KP_>
struct PairCluster {
  static constexpr int CL = CL_, NW = NW_, KP = KP_, NST = 2;
};
using PairShort = PairCluster<8, 4, 4>;
using PairLong = PairCluster<16, 2, 6>;
constexpr int kPairShortKeys = 1280;

template <class P, bool FUSED>
static cudaLaunchConfig_t pair_cluster_config(const DecodeJob& j, cudaStream_t stream,
                                              cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(P::CL, j.Hkv * (j.H / j.Hkv / 8), j.B);
  cfg.blockDim = dim3(32 * P::NW);
  cfg.dynamicSmemBytes = P::NW * pair_ring_stride(P::NST, P::KP * 128 * 4);
  cfg.stream = stream;
  attr->id = cudaLaunchAttributeClusterDimension;
  attr->val.clusterDim.x = P::CL;
  attr->val.clusterDim.y = 1;
  attr->val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Clusters of this shape that fit on the current device at once (cached per
// device; 0 when clusters of that size cannot be launched).
template <class P, bool FUSED>
static int pair_cluster_capacity(const DecodeJob& j) {
  static PerContext<int> cache;           // the cluster-size permission is per context
  return cache.get(
      [&j] {
        auto kern = decode_pair_kernel<P::NW, P::KP, true, FUSED, P::CL>;
        int n = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess) {
          cudaLaunchAttribute attr{};
          const cudaLaunchConfig_t cfg = pair_cluster_config<P, FUSED>(j, nullptr, &attr);
          if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
        }
        cudaGetLastError();
        return n;
      },
      0);
}

template <class P, bool FUSED>
static cudaError_t launch_pair_cluster(const DecodeJob& j, const DecodeStepArgs& st,
                                       cudaStream_t stream) {
  cudaLaunchAttribute attr{};
  const cudaLaunchConfig_t cfg = pair_cluster_config<P, FUSED>(j, stream, &attr);
  return cudaLaunchKernelEx(&cfg, decode_pair_kernel<P::NW, P::KP, true, FUSED, P::CL>, j,
                            P::NST, st);
}

// 8 heads per group at D = 128 and every group fitting at once: 1 for the short
// shape, 2 for the long one; 0 otherwise.
static int pair_cluster_kind(const DecodeJob& j, bool step) {
  const int G = j.H / j.Hkv;
  if (G % 8 != 0 || j.D != 128) return 0;
  const long groups = (long)j.B * j.Hkv * (G / 8);
  const int eff = j.window > 0 ? min(j.max_cache_len, j.window) : j.max_cache_len;
  if (eff <= kPairShortKeys &&
      groups <= (step ? pair_cluster_capacity<PairShort, true>(j)
                      : pair_cluster_capacity<PairShort, false>(j)))
    return 1;
  if (groups <= (step ? pair_cluster_capacity<PairLong, true>(j)
                      : pair_cluster_capacity<PairLong, false>(j)))
    return 2;
  return 0;
}

int decode_launches(const DecodeJob& j, bool step) {
  return pair_cluster_kind(j, step) ? 1 : (j.nsplit > 1 ? 2 : 1);
}

cudaError_t launch_decode(const DecodeJob& j, cudaStream_t stream, const DecodeStepArgs* step) {
  const int G = j.H / j.Hkv;
  switch (pair_cluster_kind(j, step != nullptr)) {
    case 1:
      return step ? launch_pair_cluster<PairShort, true>(j, *step, stream)
                  : launch_pair_cluster<PairShort, false>(j, DecodeStepArgs{}, stream);
    case 2:
      return step ? launch_pair_cluster<PairLong, true>(j, *step, stream)
                  : launch_pair_cluster<PairLong, false>(j, DecodeStepArgs{}, stream);
    default:
      break;
  }
  if (G % 8 == 0 && j.D % 4 == 0 && j.D <= 128) {
    // One warp per split with a 2-stage ring of 8-key batches (16 KB at D = 128).
    // Measured on the long carried decode (B = 8, 64 query heads over 8 KV heads,
    // 1-2 k cached positions): 2 or 4 warps per split and 4-key batches were no
    // faster; every setting stays near 3 TB/s there.
    constexpr int NW = kPairWarps, KP = kPairKeys;
    const int nst = 2;
    const uint32_t smem = NW * pair_ring_stride(nst, KP * j.D * 4);
    const dim3 grid(j.nsplit, j.Hkv * (G / 8), j.B);
    const DecodeStepArgs none{};
    if (step)
      decode_pair_kernel<NW, KP, true, true><<<grid, 32 * NW, smem, stream>>>(j, nst, *step);
    else if (j.D == 128)
      decode_pair_kernel<NW, KP, true><<<grid, 32 * NW, smem, stream>>>(j, nst, none);
    else
      decode_pair_kernel<NW, KP, false><<<grid, 32 * NW, smem, stream>>>(j, nst, none);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || j.nsplit <= 1) return e;
    decode_combine_kernel<<<dim3(j.H, j.B), 128, 0, stream>>>(j);
    return cudaGetLastError();
  }
  if (G == 1) return launch_gt<1>(j, stream, step);
  if (G == 2) return launch_gt<2>(j, stream, step);
  if (G <= 4) return launch_gt<4>(j, stream, step);
  return launch_gt<8>(j, stream, step);
}

}  // namespace gqa
