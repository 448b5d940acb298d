// The opt-in check for non-finite inputs ("mojolearn.transformer",
// TransformerBlock: non-finite weights, inputs or cache values are an error
// raised before any computation).
//
// When the check is on, an entry point first launches finite_check_kernel over
// the values its computation will read -- the call's tensors, and of a cache
// only the slots the call reads -- and every kernel of the call then starts by
// reading the caller's status word: if the check has OR-ed ATTN_DEV_NONFINITE
// into it, the kernel returns before touching anything, so no output of the
// call is written. Nothing is synchronised; the check is one extra read pass
// over the inputs, which is why it is off unless asked for.
#include <stdlib.h>
#include <string.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace gqa {

namespace {

std::atomic<int> g_check{-1};   // -1: not read from the environment yet

__device__ __forceinline__ bool not_finite(float x) {
  return (__float_as_uint(x) & 0x7f800000u) == 0x7f800000u;   // inf or NaN
}

// Rows [lo, hi) of outer index o (= b * NH + head) that the call reads, as
// row-membership: in_rows(r) for r < R.
struct RowSet {
  long lo, hi;          // plain range
  long ring_lo, W;      // ring prefix: rows r with (r - ring_lo) mod W < hi (W > 0)
};

__device__ __forceinline__ RowSet rows_of(const FiniteRegion& g, int b) {
  RowSet s{0, g.R, 0, 0};
  if (g.mode == kFiniteLen || g.mode == kFiniteCache) {
    const long n = g.info[b];
    s.hi = n < 0 ? 0 : (n > g.R ? g.R : n);
  } else if (g.mode == kFinitePrefix) {
    const long st = g.info[b];
    if (st <= 0) {
      s.hi = 0;
    } else if (g.window == 0) {
      s.hi = st > g.R ? g.R : st;
    } else {
      // positions st - pre .. st - 1 with pre = min(st, W - 1), at slot position mod W
      const long pre = st < g.window - 1 ? st : g.window - 1;
      s.W = g.window;
      s.ring_lo = (st - pre) % g.window;
      s.hi = pre;
    }
  }
  return s;
}

__global__ void __launch_bounds__(256) finite_check_kernel(FiniteJob j) {
  __shared__ int bad_block;
  if (threadIdx.x == 0) bad_block = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long nwarps = static_cast<long>(gridDim.x) * 8;
  const long gwarp = static_cast<long>(blockIdx.x) * 8 + threadIdx.x / 32;
  bool bad = false;
  for (int ri = 0; ri < j.n; ++ri) {
    const FiniteRegion& g = j.r[ri];
    const long outer = static_cast<long>(g.B) * g.NH;
    const long total = outer * g.R;
    const bool vec = g.C % 4 == 0 && g.ld % 4 == 0 &&
                     (reinterpret_cast<uintptr_t>(g.p) & 15u) == 0;
    for (long x = gwarp; x < total; x += nwarps) {
      const long o = x / g.R, r = x % g.R;
      const RowSet s = rows_of(g, static_cast<int>(o / g.NH));
      const bool in = s.W > 0 ? ((r - s.ring_lo) % s.W + s.W) % s.W < s.hi
                              : (r >= s.lo && r < s.hi);
      if (!in) continue;
      const float* row = g.p + (o * g.R + r) * g.ld;
      if (vec) {
        const float4* r4 = reinterpret_cast<const float4*>(row);
        for (long c = lane; c < g.C / 4; c += 32) {
          const float4 v = r4[c];
          bad |= not_finite(v.x) | not_finite(v.y) | not_finite(v.z) | not_finite(v.w);
        }
      } else {
        for (long c = lane; c < g.C; c += 32) bad |= not_finite(row[c]);
      }
    }
  }
  if (bad) bad_block = 1;
  __syncthreads();
  if (threadIdx.x == 0 && bad_block) report(j.status, ATTN_DEV_NONFINITE);
}

}  // namespace

int check_finite_enabled() {
  int v = g_check.load();
  if (v < 0) {
    const char* e = getenv("ATTN_CHECK_FINITE");
    int want = (e && *e && strcmp(e, "0") != 0) ? 1 : 0;
    int expect = -1;
    g_check.compare_exchange_strong(expect, want);
    v = g_check.load();
  }
  return v;
}

int set_check_finite(int on) {
  const int prev = check_finite_enabled();
  if (on >= 0) g_check.store(on ? 1 : 0);
  return prev;
}

cudaError_t launch_finite_check(const FiniteJob& j, cudaStream_t stream) {
  long rows = 0;
  for (int i = 0; i < j.n; ++i) rows += static_cast<long>(j.r[i].B) * j.r[i].NH * j.r[i].R;
  long blocks = (rows + 7) / 8;
  if (blocks > 152L * 8) blocks = 152L * 8;
  if (blocks < 1) blocks = 1;
  finite_check_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(j);
  return cudaGetLastError();
}

}  // namespace gqa
