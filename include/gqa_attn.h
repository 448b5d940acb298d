/*
 * gqa_attn.h -- C ABI of the grouped-query causal attention library
 * (libgqa_attn.so, CUDA kernels for sm_103a).
 *
 * The operation is the self-attention of one Llama-shaped decoder layer as
 * the "mojolearn.transformer" page states it (TransformerBlock: grouped-query
 * attention with RoPE and a KV cache; options window, rope_theta,
 * rope_scaling, rope_dim, max_positions, qk_norm, attn_softcap, norm_eps;
 * TransformerState: the caller-owned cache; step: one token at position
 * cached_tokens). The formulas are those of "Core Layers -- Deep Reference"
 * (sections "RMSNorm", "RoPE", "MHA and GQA", "Sliding window attention").
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensors are fp32, contiguous, row-major, in DEVICE memory owned by the
 *   caller, except the host buffers of gqa_attn_prefill_from_host. No call
 *   allocates or frees device memory; the only device memory the library keeps
 *   is the fixed scratch array of gqa_attn_decode_static, and the only other
 *   state is the pair of copy streams per device of gqa_attn_prefill_from_host
 *   and, per device and context, the kernels' function attributes (shared
 *   memory sizes, cluster sizes) set on first use with the occupancy figures
 *   worked out then; a new context (after cudaDeviceReset) sets them again.
 *   Tensor pointers must be 16-byte aligned (ATTN_ERR_ALIGN otherwise).
 * - Shapes: Q and outputs [B, H, L, D]; K and V [B, Hkv, L, D]; caches
 *   [B, Hkv, capacity, D]. H % Hkv == 0; query head h reads key/value head
 *   h / (H / Hkv) (contiguous groups). D is even, 2 <= D <= 256.
 * - Positions are absolute: row b's token l sits at start[b] + l.
 * - stream is a cudaStream_t (NULL: the legacy default stream). Every call
 *   only enqueues work on it (and, for gqa_attn_prefill_from_host, on its copy
 *   streams, joined back into it) and returns; nothing is synchronised.
 * - Errors: arguments are checked on the host before anything is launched,
 *   and a negative ATTN_ERR_* is returned with nothing enqueued. Values that
 *   live on the device (start, cache_len) are checked again by the kernels:
 *   a row that breaks a rule is skipped (its outputs are left untouched) and
 *   an ATTN_DEV_* bit is OR-ed into *status (a caller-owned device int32,
 *   which may be NULL to skip the report, except with the non-finite check
 *   on: see attn_set_check_finite). Kernels never trap.
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host-side return codes. */
#define ATTN_OK             0
#define ATTN_ERR_NULL      -1  /* a required pointer is NULL */
#define ATTN_ERR_SHAPE     -2  /* sizes break the shape rules above */
#define ATTN_ERR_POSITION  -3  /* a position would reach max_positions */
#define ATTN_ERR_CAPACITY  -4  /* a position has no cache slot (no window) */
#define ATTN_ERR_WORKSPACE -5  /* workspace missing or too small */
#define ATTN_ERR_ALIGN     -6  /* a tensor pointer is not 16-byte aligned */
#define ATTN_ERR_PARAM     -7  /* RoPE parameters or a rope table are invalid */
#define ATTN_ERR_CUDA      -8  /* a CUDA launch or query failed */

/* Device status bits, OR-ed into *status by the kernels. */
#define ATTN_DEV_POSITION  1   /* start[b] < 0 or start[b] + L - 1 >= max_positions */
#define ATTN_DEV_CAPACITY  2   /* start[b] + L > capacity without a window */
#define ATTN_DEV_LENGTH    4   /* cache_len[b] outside [1, max_cache_len] or > capacity,
                                  or a ragged prefill's lengths[b] outside [1, L] */
#define ATTN_DEV_TIMEOUT   8   /* a pipeline wait ran past its limit; outputs invalid */
#define ATTN_DEV_NONFINITE 16  /* the opt-in check found an inf or NaN input; the call
                                  (and every later checked call on this status word)
                                  computed nothing, see attn_set_check_finite */

/* RoPE frequency scaling ("mojolearn.transformer", rope_scaling). */
#define ATTN_ROPE_SCALING_NONE   0
#define ATTN_ROPE_SCALING_LINEAR 1  /* every frequency divided by factor */
#define ATTN_ROPE_SCALING_LLAMA3 2  /* Llama 3 frequency ramp */

/*
 * Rotary position parameters ("mojolearn.transformer": rope_theta,
 * rope_scaling, rope_dim, max_positions). Frequencies are
 * theta_i = theta^(-2i/R) for i < R/2 ("Core Layers -- Deep Reference",
 * "RoPE", with the rotary width R as d_h), then scaled:
 *   LINEAR: theta_i / factor;
 *   LLAMA3: with wavelength w = 2*pi/theta_i, kept when
 *           w < original_max_positions / high_freq_factor, divided by factor
 *           when w > original_max_positions / low_freq_factor, and in between
 *           (1-s)*theta_i/factor + s*theta_i with
 *           s = (original_max_positions / w - low) / (high - low).
 * Pairs are rotate-half, (i, i + R/2), and dims R..D-1 pass through.
 */
typedef struct attn_rope_params {
    double theta;                    /* RoPE base, > 0 */
    int32_t rope_dim;                /* R: even, <= D; 0 means D */
    int32_t max_positions;           /* positions must stay below; 0 means 8192 */
    int32_t scaling_type;            /* ATTN_ROPE_SCALING_* */
    int32_t original_max_positions;  /* LLAMA3 only */
    double factor;                   /* LINEAR and LLAMA3, > 0 */
    double low_freq_factor;          /* LLAMA3 only */
    double high_freq_factor;         /* LLAMA3 only, > low_freq_factor */
} attn_rope_params;

/*
 * Bytes of the cos/sin table for these parameters at head dimension D:
 * max_positions * (R/2) * 2 floats. Returns 0 if the parameters are invalid.
 */
size_t attn_rope_table_bytes(const attn_rope_params* rp, int D);

/*
 * Fill a caller-owned device table [max_positions][R/2][2] with
 * (cos, sin) of position * theta_i. Angles and their cosines and sines are
 * computed in fp64 on the device and rounded once to fp32 ("Core Layers --
 * Deep Reference", "RoPE": frequencies precomputed once into an angle table).
 * Build it once per parameter set and pass it to the calls below.
 */
int attn_rope_table_init(const attn_rope_params* rp, int D, float* table, size_t table_bytes,
                         void* stream);

/*
 * In place on x [B, Hx, L, D] (queries, or any per-head rows): optional
 * RMSNorm over D, y = x / sqrt(mean(x^2) + norm_eps) * norm_w ("mojolearn
 * .transformer", qk_norm: before RoPE; "Core Layers -- Deep Reference",
 * "RMSNorm"), then RoPE at position start[b] + l using table (built by
 * attn_rope_table_init with the same rp and D).
 *   start      device int32 [B]
 *   max_start  host bound on every start[b], checked against max_positions
 *   norm_w     device [D] or NULL (no norm)
 */
int attn_rope_apply(float* x, int B, int Hx, int L, int D, const int32_t* start,
                    int32_t max_start, const attn_rope_params* rp, const float* table,
                    const float* norm_w, float norm_eps, int32_t* status, void* stream);

/*
 * Cache append ("mojolearn.transformer", TransformerState; "Core Layers --
 * Deep Reference", "Static KV-Cache": new rows written at the cache index).
 * For each row b, kv head, token l at position p = start[b] + l:
 *   k[b,hkv,l,:] <- RoPE(RMSNorm(k)) in place (norm if k_norm_w, RoPE if rp);
 *   k_cache[b,hkv,slot(p),:] <- that rotated k;  v_cache[...] <- v (exact copy).
 * slot(p) = p without a window (capacity >= every p + 1), p mod W with one
 * (window = W > 0: the caches are rings with capacity == W; of a chunk longer
 * than W only its last W positions are stored). rp == NULL (then table and
 * k_norm_w must be NULL too) stores k as given.
 */
int kv_cache_append(float* k, const float* v, int B, int Hkv, int L, int D,
                    const int32_t* start, int32_t max_start, const attn_rope_params* rp,
                    const float* table, const float* k_norm_w, float norm_eps, float* k_cache,
                    float* v_cache, int capacity, int window, int32_t* status, void* stream);

/*
 * Multi-token prefill attention over the chunk's own keys (a prefill from an
 * empty cache; "mojolearn.transformer", forward with a zero state):
 *   out[b,h,l,:] = sum_m softmax_m(cap(scale * q[b,h,l,:] . k[b,h/G,m,:])) v[b,h/G,m,:]
 * over keys m <= l with l - m < window (window = 0: all m <= l). cap(s) =
 * softcap * tanh(s / softcap) when softcap > 0 ("mojolearn.transformer",
 * attn_softcap). scale <= 0 means 1/sqrt(D). q and k are already rotated.
 * For D % 4 == 0 and D >= 32 the work runs on the tcgen05 tensor cores (TF32
 * operands, fp32 accumulation and softmax); other even D run on the CUDA cores
 * in fp32.
 *   workspace  device scratch of gqa_attn_prefill_workspace_size bytes
 *              (holds a transposed copy of v; contents clobbered)
 */
size_t gqa_attn_prefill_workspace_size(int B, int Hkv, int L, int D);
int gqa_attn_prefill(const float* q, const float* k, const float* v, float* out, int B, int H,
                     int Hkv, int L, int D, int window, float softcap, float scale,
                     void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Prefill attention with the queries' RMSNorm and RoPE fused in: the same
 * result as attn_rope_apply(q, start, rp, table, q_norm_w) followed by
 * gqa_attn_prefill, but q is the raw query and is left unmodified. k must
 * already be rotated (kv_cache_append does that). For D % 32 == 0, D <= 128 and
 * rope_dim % 64 == 0 the rotation happens inside the tensor-core kernel, in
 * tensor memory after the Q tile's copy there; other shapes rotate q into the
 * workspace first. Positions are start[b] + l; max_start bounds every start[b].
 * rp == NULL (then table and q_norm_w must be NULL; start is not read): q is
 * already rotated and the call is gqa_attn_prefill.
 */
size_t gqa_attn_prefill_rope_workspace_size(int B, int H, int Hkv, int L, int D,
                                            const attn_rope_params* rp);
int gqa_attn_prefill_rope(const float* q, const float* k, const float* v, float* out, int B,
                          int H, int Hkv, int L, int D, const int32_t* start, int32_t max_start,
                          const attn_rope_params* rp, const float* table, const float* q_norm_w,
                          float norm_eps, int window, float softcap, float scale,
                          void* workspace, size_t workspace_bytes, int32_t* status,
                          void* stream);

/*
 * v transposed for the tensor-core prefill: vt[b, hkv, d, m] = v[b, hkv, m, d],
 * each (b, hkv, d) row holding gqa_attn_vt_pitch(L) floats (the first L used).
 * gqa_attn_prefill and gqa_attn_prefill_rope build it in their workspace on
 * every call; a caller can build it once with gqa_attn_v_transpose and hand it
 * to gqa_attn_prefill_rope_vt. Tensor-core head dims only (D % 4 == 0,
 * 32 <= D <= 256; ATTN_ERR_SHAPE otherwise).
 *   v   [B, Hkv, L, D]                          fp32, 16-byte aligned, read
 *   vt  B * Hkv * D * gqa_attn_vt_pitch(L) floats, 16-byte aligned, written
 */
int gqa_attn_vt_pitch(int L);
int gqa_attn_v_transpose(const float* v, float* vt, int B, int Hkv, int L, int D, void* stream);

/*
 * gqa_attn_prefill_rope with v given transposed (vt as gqa_attn_v_transpose
 * writes it, read only): the attention kernel alone, no pre-pass. Same
 * arguments and results otherwise; tensor-core head dims only. The workspace
 * (gqa_attn_prefill_rope_vt_workspace_size bytes) holds rotated q for the
 * shapes that do not rotate inside the kernel; for the others it may be NULL.
 */
size_t gqa_attn_prefill_rope_vt_workspace_size(int B, int H, int L, int D,
                                               const attn_rope_params* rp);
int gqa_attn_prefill_rope_vt(const float* q, const float* k, const float* vt, float* out, int B,
                             int H, int Hkv, int L, int D, const int32_t* start,
                             int32_t max_start, const attn_rope_params* rp, const float* table,
                             const float* q_norm_w, float norm_eps, int window, float softcap,
                             float scale, void* workspace, size_t workspace_bytes,
                             int32_t* status, void* stream);

/*
 * One whole prefill step from a fresh cache ("mojolearn.transformer",
 * TransformerBlock.forward with an empty TransformerState): for positions
 * 0 .. L-1 the keys and values enter the cache and attention runs over them,
 *   k_cache, v_cache  <- as kv_cache_append with start 0 would write them;
 *   out               <- as gqa_attn_prefill_rope with start 0 computes it.
 * Unlike kv_cache_append, k and v are only read (k is not rotated in place).
 *   q [B, H, L, D] raw; k, v [B, Hkv, L, D] raw; out [B, H, L, D];
 *   caches [B, Hkv, capacity, D]: capacity >= L without a window, a ring of
 *   capacity == window slots with one (of a chunk longer than the ring only
 *   its last window positions are stored).
 * For D % 4 == 0 and D >= 32 one memory pass reads k and v once and writes the
 * rotated keys into the cache, v into the cache and v transposed into the
 * workspace; the tensor-core kernel then reads the keys from the cache (from a
 * rotated copy in the workspace when a ring is shorter than L), with q's RMSNorm
 * and RoPE fused as in gqa_attn_prefill_rope. Other even D run on the CUDA
 * cores. B * Hkv <= 65535.
 *   workspace  gqa_attn_prefill_step_workspace_size bytes
 */
size_t gqa_attn_prefill_step_workspace_size(int B, int H, int Hkv, int L, int D, int window,
                                            const attn_rope_params* rp);
int gqa_attn_prefill_step(const float* q, const float* k, const float* v, float* out, int B,
                          int H, int Hkv, int L, int D, const attn_rope_params* rp,
                          const float* table, const float* q_norm_w, const float* k_norm_w,
                          float norm_eps, float* k_cache, float* v_cache, int capacity,
                          int window, float softcap, float scale, void* workspace,
                          size_t workspace_bytes, int32_t* status, void* stream);

/*
 * One whole prefill step with q, k, v and the output in host memory
 * ("mojolearn.transformer", TransformerBlock.forward: the caller hands in the
 * step's tensors and reads the result back). q, k, v are copied to the
 * caller's device buffers, kv_cache_append rotates k in place and
 * stores k and v at their cache slots, gqa_attn_prefill_rope writes out, and out
 * is copied back to out_host. Results equal those two calls over the whole batch.
 *   q_host, out_host        host [B, H, L, D]; k_host, v_host  host [B, Hkv, L, D].
 *                           Page-locked (cudaHostAlloc / cudaHostRegister) memory
 *                           lets the copies overlap the kernels; pageable memory
 *                           works but serialises them. Not read or written after
 *                           the caller's stream has passed this call.
 *   q, k, v, out            device buffers of the same shapes (overwritten; k ends
 *                           up rotated, as kv_cache_append leaves it)
 *   k_cache, v_cache, capacity, window, k_norm_w: as kv_cache_append;
 *   start, max_start, rp, table, q_norm_w, norm_eps, softcap, scale: as
 *   gqa_attn_prefill_rope; workspace: gqa_attn_prefill_from_host_workspace_size bytes.
 * The step is cut into at most 16 chunks: groups of whole batch rows, or, with
 * fewer than 16 rows, slices of a row's kv heads together with their query heads
 * (one chunk when L * D or capacity * D is not a multiple of 4). Each chunk's
 * host-to-device copies run on one library-owned stream, its kernels on `stream`
 * and its device-to-host copy on another library-owned stream, so copies and
 * kernels of different chunks overlap. The two copy streams of a device are created by the
 * first call on it (with that device current) and kept for that device's context (made
 * again after cudaDeviceReset). The call
 * returns once everything is enqueued; `stream` passes the call only after the
 * last copy to out_host. All checks run before anything is enqueued.
 */
size_t gqa_attn_prefill_from_host_workspace_size(int B, int H, int Hkv, int L, int D,
                                                 int capacity, const attn_rope_params* rp);
int gqa_attn_prefill_from_host(const float* q_host, const float* k_host, const float* v_host,
                               float* out_host, float* q, float* k, float* v, float* out, int B,
                               int H, int Hkv, int L, int D, const int32_t* start,
                               int32_t max_start, const attn_rope_params* rp, const float* table,
                               const float* q_norm_w, const float* k_norm_w, float norm_eps,
                               float* k_cache, float* v_cache, int capacity, int window,
                               float softcap, float scale, void* workspace,
                               size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Prefill of a chunk that continues a carried cache ("mojolearn.transformer",
 * TransformerBlock.forward with a TransformerState): the chunk's L queries at
 * positions start[b] + l attend, causally, to the positions kept in the cache
 * before the chunk and to the chunk itself:
 *   out[b,h,l,:] = sum over positions m <= p = start[b] + l (and p - m < window
 *   when window > 0) of softmax_m(cap(scale * q . key_m)) value_m,
 * with key_m, value_m read from the cache for m < start[b] and from k, v (the
 * chunk, row m - start[b]) for m >= start[b].
 *   q        [B, H, L, D]   raw if rp != NULL (RMSNorm + RoPE applied here, at
 *                           positions start[b] + l, as in gqa_attn_prefill_rope;
 *                           q is not modified), else already rotated
 *   k, v     [B, Hkv, L, D] the chunk's keys (rotated, e.g. by attn_rope_apply
 *                           or kv_cache_append) and values
 *   k_cache, v_cache [B, Hkv, capacity, D] the carried cache, rotated keys, as
 *                           kv_cache_append fills it: slot = position (window 0,
 *                           capacity >= every start[b]) or position mod window
 *                           (a ring, capacity == window). With a ring, call this
 *                           before appending the chunk, whose rows may overwrite
 *                           the prefix the chunk's first queries need.
 *   start    [B] device int32, positions already cached; max_start bounds them
 *   workspace gqa_attn_prefill_cached_workspace_size bytes (the gathered keys,
 *            transposed values and, for some rope shapes, rotated q)
 * Head dims D % 4 == 0, 32 <= D <= 256 (ATTN_ERR_SHAPE otherwise). A start[b]
 * outside [0, max_start] (or above capacity without a window) sets
 * ATTN_DEV_POSITION (ATTN_DEV_CAPACITY) and that row attends only to the chunk.
 * Cost: the gather reads the kept prefix of every (b, kv head) once per call.
 */
size_t gqa_attn_prefill_cached_workspace_size(int B, int H, int Hkv, int L, int D,
                                              int32_t max_start, int window,
                                              const attn_rope_params* rp);
int gqa_attn_prefill_cached(const float* q, const float* k, const float* v, const float* k_cache,
                            const float* v_cache, int capacity, float* out, int B, int H,
                            int Hkv, int L, int D, const int32_t* start, int32_t max_start,
                            const attn_rope_params* rp, const float* table,
                            const float* q_norm_w, float norm_eps, int window, float softcap,
                            float scale, void* workspace, size_t workspace_bytes,
                            int32_t* status, void* stream);

/*
 * Prefill of a ragged batch ("mojolearn.transformer", TransformerBlock.forward
 * with lengths, a fresh sequence per row: start 0): row b is real at positions
 * [0, lengths[b]) and padding after. Every real query's output equals that row
 * run alone at its own length,
 *   out[b,h,l,:] = sum over m <= l (and l - m < window when window > 0) of
 *                  softmax_m(cap(scale * q . k_m)) v_m        for l < lengths[b],
 * and padding outputs are exactly +0.0 (l >= lengths[b]). Padding rows of q, k
 * and v are never read into a real output, whatever they hold (inf and NaN
 * included): padding values meet no zero weight in P V.
 *   q        [B, H, L, D]   raw if rp != NULL (RMSNorm + RoPE at position l, as
 *                           in gqa_attn_prefill_rope with start 0; q is not
 *                           modified), else already rotated
 *   k, v     [B, Hkv, L, D] rotated keys and values
 *   lengths  [B] device int32 in [1, L]; a value outside sets ATTN_DEV_LENGTH
 *            and is clamped to [0, L]
 *   workspace gqa_attn_prefill_ragged_workspace_size bytes
 * Other arguments as for gqa_attn_prefill_rope (rp, table, q_norm_w may be NULL
 * when rp is NULL). In the persistent kernel (D % 4 == 0, D >= 32) query tiles with no
 * real row cost no attention work.
 */
size_t gqa_attn_prefill_ragged_workspace_size(int B, int H, int Hkv, int L, int D,
                                              const attn_rope_params* rp);
int gqa_attn_prefill_ragged(const float* q, const float* k, const float* v, float* out, int B,
                            int H, int Hkv, int L, int D, const int32_t* lengths,
                            const attn_rope_params* rp, const float* table,
                            const float* q_norm_w, float norm_eps, int window, float softcap,
                            float scale, void* workspace, size_t workspace_bytes,
                            int32_t* status, void* stream);

/*
 * One decoder block around the attention ("mojolearn.transformer",
 * TransformerBlock.forward with state None, i.e. a fresh sequence at positions
 * 0 .. L-1, computing Hugging Face's LlamaDecoderLayer.forward):
 *   h   = x + o_proj(attention(RMSNorm_in(x)))
 *   out = h + down_proj(SiLU(gate_proj(n)) * up_proj(n)),  n = RMSNorm_post(h)
 * with the attention of gqa_attn_prefill_rope (q/k RMSNorm when q_norm / k_norm
 * are given, RoPE per rp, causal or window, softcap). RMSNorm scales by w, or by
 * 1 + w when norm_offset != 0 (Gemma). No biases.
 *   x, out   [B, L, d_model] with d_model = H * D (distinct buffers)
 *   weights  torch's [out, in] layout: q_proj [H*D, d_model], k_proj and v_proj
 *            [Hkv*D, d_model], o_proj [d_model, H*D], gate_proj and up_proj
 *            [IT, d_model], down_proj [d_model, IT]; norms [d_model]; q_norm,
 *            k_norm [D] or NULL
 *   workspace gqa_block_forward_workspace_size bytes
 * The seven projections run as attn_linear does (tcgen05 tensor cores, TF32
 * operands, fp32 accumulation): q, k and v in one launch writing head-major,
 * o_proj reading the attention's head-major output (D % 32 == 0) and adding x,
 * gate and up in one launch whose epilogue forms SiLU(gate) * up, down_proj
 * adding h in place. d_model and IT must be multiples of 4 and x != out
 * (ATTN_ERR_SHAPE otherwise).
 */
typedef struct attn_block_weights {
    const float* input_norm;         /* input_layernorm.weight [d_model] */
    const float* post_norm;          /* post_attention_layernorm.weight [d_model] */
    const float* wq;                 /* q_proj.weight */
    const float* wk;                 /* k_proj.weight */
    const float* wv;                 /* v_proj.weight */
    const float* wo;                 /* o_proj.weight */
    const float* w_gate;             /* gate_proj.weight */
    const float* w_up;               /* up_proj.weight */
    const float* w_down;             /* down_proj.weight */
    const float* q_norm;             /* q_norm.weight [D] or NULL */
    const float* k_norm;             /* k_norm.weight [D] or NULL */
} attn_block_weights;

size_t gqa_block_forward_workspace_size(int B, int L, int H, int Hkv, int D, int IT,
                                        const attn_rope_params* rp);
int gqa_block_forward(const float* x, float* out, int B, int L, int H, int Hkv, int D, int IT,
                      const attn_block_weights* w, int norm_offset, float norm_eps,
                      const attn_rope_params* rp, const float* table, int window, float softcap,
                      float scale, void* workspace, size_t workspace_bytes, int32_t* status,
                      void* stream);

/*
 * One bias-free linear map on the tcgen05 tensor cores ("mojolearn.transformer",
 * TransformerBlock: q_proj ... down_proj are linear maps without bias, weights
 * in torch's [out, in] layout):
 *   y[t, n] = sum_k x[t, k] * w[n, k]  (+ residual[t, n] when residual != NULL)
 *   x [T, K], w [N, K], y and residual [T, N]; fp32 in memory, TF32 operands
 *   (the tensor core reads the top 19 bits of each value), fp32 accumulation.
 *   residual may equal y (in-place add); x and w must not overlap y.
 * K and N multiples of 4 (16-byte rows; ATTN_ERR_SHAPE otherwise). T == 0 is a
 * no-op.
 */
int attn_linear(const float* x, const float* w, const float* residual, float* y, long T, int N,
                int K, int32_t* status, void* stream);

/*
 * The identical numeric mode ("mojolearn.transformer", TransformerBlock
 * numeric_mode 'identical': decoding token by token, or a prefill continued
 * from a carried cache, gives the same bits as one prefill over the whole
 * sequence). Both calls below run one kernel whose per-query arithmetic
 * depends only on the query's position and the visible key positions: the
 * score of key m is a fixed-order dot product, the maximum is exact, and the
 * softmax sum and P V run over keys in ascending position order. So, with
 * keys and values appended by kv_cache_append (the cache holds the same bits
 * as the appended rows) and queries rotated by attn_rope_apply:
 *   gqa_attn_decode_identical at cache_len[b] = p + 1 ==
 *   gqa_attn_prefill_identical row p (start 0)  ==
 *   gqa_attn_prefill_identical of any chunk holding position p, continued
 *   from the cache of the positions before it,
 * bit for bit. Results equal the other prefill/decode calls within the usual
 * tolerance, not bitwise. CUDA cores, scores computed twice: for
 * reproducibility, not speed.
 *
 * Prefill: q [B, H, L, D] rotated, k, v [B, Hkv, L, D] rotated keys / values of
 * the chunk at positions start[b] + l (start NULL: 0, then max_start must be
 * 0). With k_cache, v_cache ([B, Hkv, capacity, D], slot = position, or
 * position mod window with capacity == window) positions below start[b] are
 * read from the cache; without, only the chunk's own keys are seen (as in
 * gqa_attn_prefill). A start[b] outside [0, max_start] (or above capacity
 * without a window) sets ATTN_DEV_POSITION (ATTN_DEV_CAPACITY) and the row's
 * outputs are left untouched.
 * Decode: as gqa_attn_decode, without a workspace.
 */
int gqa_attn_prefill_identical(const float* q, const float* k, const float* v,
                               const float* k_cache, const float* v_cache, int capacity,
                               float* out, int B, int H, int Hkv, int L, int D,
                               const int32_t* start, int32_t max_start, int window,
                               float softcap, float scale, int32_t* status, void* stream);
int gqa_attn_decode_identical(const float* q, const float* k_cache, const float* v_cache,
                              const int32_t* cache_len, int32_t max_cache_len, float* out, int B,
                              int H, int Hkv, int D, int capacity, int window, float softcap,
                              float scale, int32_t* status, void* stream);

/*
 * Bytes of scratch gqa_attn_decode needs for these sizes (split-KV partial
 * results). max_cache_len bounds every cache_len[b]. The size never shrinks as
 * max_cache_len grows, so a buffer sized for the largest length serves every
 * call with a smaller one (a call itself needs only the bytes its own split
 * plan uses, which can be fewer).
 */
size_t gqa_attn_decode_workspace_size(int B, int H, int Hkv, int D, int max_cache_len,
                                      int window);

/*
 * Single-token decode ("mojolearn.transformer", step: forward with L = 1 at
 * position cached_tokens). Row b's query q[b,:,0,:] (rotated) sits at
 * p = cache_len[b] - 1 (cache_len counts the token just appended) and reads
 * cache positions max(0, p - W + 1) .. p: slots 0 .. p without a window, or
 * the min(cache_len[b], W) live slots of the ring with one.
 *   q [B, H, 1, D], out [B, H, 1, D]; caches [B, Hkv, capacity, D].
 *   cache_len       device int32 [B], each in [1, max_cache_len]
 *   workspace       device scratch of gqa_attn_decode_workspace_size bytes
 * Output rows are overwritten; the workspace contents are clobbered.
 */
int gqa_attn_decode(const float* q, const float* k_cache, const float* v_cache,
                    const int32_t* cache_len, int32_t max_cache_len, float* out, int B, int H,
                    int Hkv, int D, int capacity, int window, float softcap, float scale,
                    void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/*
 * One whole decode step ("mojolearn.transformer", TransformerBlock.step: the new
 * token of each row at position cached_tokens): for row b the token sits at
 * p = pos[b] (the number of positions already cached), and
 *   k_cache, v_cache slot(p) <- RoPE(RMSNorm(k)), v    (as kv_cache_append at p)
 *   out[b,h,0,:] <- attention of RoPE(RMSNorm(q)) over positions max(0, p-W+1) .. p
 *                   (as gqa_attn_decode with cache_len[b] = p + 1).
 * q, k and v are only read. q [B, H, 1, D], k, v [B, Hkv, 1, D] raw; out [B, H, 1, D];
 * caches as gqa_attn_decode (capacity > every p without a window).
 *   pos      device int32 [B]; max_pos bounds every pos[b] (host), < max_positions
 *   workspace gqa_attn_decode_step_workspace_size bytes (never shrinking as max_pos
 *            grows: one buffer sized for the largest position serves every step)
 * One pass rotates q and k and stores k and v at their slots; then the
 * split-KV decode of gqa_attn_decode. At D = 128 (rotary dims a multiple of 8;
 * 64 or 128 with 8 query heads per KV head) that pass is folded into the decode
 * kernel. A pos[b] outside
 * the table (or the capacity, without a window) sets ATTN_DEV_POSITION
 * (ATTN_DEV_CAPACITY) and ATTN_DEV_LENGTH, and the row is skipped.
 */
size_t gqa_attn_decode_step_workspace_size(int B, int H, int Hkv, int D, int32_t max_pos,
                                           int window);
int gqa_attn_decode_step(const float* q, const float* k, const float* v, float* out, int B,
                         int H, int Hkv, int D, const int32_t* pos, int32_t max_pos,
                         const attn_rope_params* rp, const float* table, const float* q_norm_w,
                         const float* k_norm_w, float norm_eps, float* k_cache, float* v_cache,
                         int capacity, int window, float softcap, float scale, void* workspace,
                         size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Kernels that one call with these sizes launches, with the non-finite check
 * off: gqa_attn_decode (step_rope_dim < 0; max_cache_len as passed to it) or
 * gqa_attn_decode_step (step_rope_dim = its rope_dim, 0 meaning D; max_cache_len
 * = max_pos + 1). Between one and three: the decode kernel (split-KV, or with
 * 8 query heads per KV head at D = 128 one cluster of blocks per head group
 * when all groups fit on the current device at once), the combine of a row's
 * splits, and the step's separate RoPE/append pass. Reads the current device's
 * properties; ATTN_ERR_SHAPE for sizes no call accepts.
 */
int gqa_attn_decode_launches(int B, int H, int Hkv, int D, int32_t max_cache_len, int window,
                             int step_rope_dim);

/*
 * gqa_attn_decode without a caller workspace, for callers that cannot
 * allocate device memory: code running where cudaMalloc is not allowed (a
 * plug-in inside a host framework that owns all device memory, a serving path
 * that must not allocate after start-up) or a plain C caller with no device
 * allocator. The pages this library follows have no counterpart to it.
 *
 * The split-KV scratch comes from a fixed array in this library's device
 * memory, GQA_ATTN_STATIC_SCRATCH_BYTES (32 MiB), which every GPU that loads
 * the library holds until the process exits. Arguments and results are those
 * of gqa_attn_decode. Sizes whose scratch (gqa_attn_decode_workspace_size)
 * exceeds the array are refused with ATTN_ERR_WORKSPACE before anything runs.
 * The call allocates nothing.
 *
 * - The first call on a device, with that device current, looks up the
 *   array's device address (cudaGetSymbolAddress) and keeps it for that
 *   device's current context; after cudaDeviceReset (a new context) the next
 *   call looks it up again. Make the first call on a device, and the first
 *   after a reset, before any stream capture.
 * - Host checks are those of gqa_attn_decode and come first, with its return
 *   codes; only then is the scratch size compared with the array.
 * - All calls share the one array and it keeps the last call's contents;
 *   nothing in it has to start at zero. Calls whose work overlaps on the GPU
 *   (other streams, other host threads) race on it: order them on one stream.
 */
#define GQA_ATTN_STATIC_SCRATCH_BYTES (32u << 20)
int gqa_attn_decode_static(const float* q, const float* k_cache, const float* v_cache,
                           const int32_t* cache_len, int32_t max_cache_len, float* out, int B,
                           int H, int Hkv, int D, int capacity, int window, float softcap,
                           float scale, int32_t* status, void* stream);

/*
 * Self-test of the failure path that every tensor-core kernel carries: one
 * block waits on pipeline barriers that nothing signals. Its first wait gives
 * up after the kernels' wait limit (2 s), raises the block's abort flag, the
 * second wait returns on seeing it, and the block ORs ATTN_DEV_TIMEOUT into
 * *status (device int32) -- the same code and the same report as a real stall,
 * with no fault and the context left usable. Enqueued on `stream`; the pages
 * have no counterpart to it.
 */
int attn_selftest_wait_timeout(int32_t* status, void* stream);

/*
 * The non-finite input check ("mojolearn.transformer", TransformerBlock:
 * non-finite weights, inputs or cache values raise an error before any
 * computation). Off by default; on when the environment variable
 * ATTN_CHECK_FINITE is set to anything but "" or "0" at the library's first
 * use, or after attn_set_check_finite(1). Process-wide.
 *
 * With the check on, every computing call (all of the above but the table
 * calls, v_transpose and the self-test) first enqueues one read pass over the
 * values it will read: its input tensors and weights, and of a cache only the
 * slots it reads (decode: the live slots at cache_len[b]; a continued or
 * identical prefill: the prefix its first query sees); of a ragged batch only
 * the real rows. An inf or NaN ORs ATTN_DEV_NONFINITE into *status, and every
 * kernel of the call -- and of any later checked call given the same status
 * word while that bit stays set -- returns before writing anything: outputs,
 * k rotated in place and caches are left as they were. The check needs a
 * status word: such calls return ATTN_ERR_NULL for status == NULL.
 * gqa_attn_prefill_from_host checks each chunk on its own: chunks before the
 * one with the bad value are computed, the others are not, and the copies back
 * to out_host still run.
 * on: 1 turns the check on, 0 off, < 0 leaves it; returns the previous setting.
 */
int attn_set_check_finite(int on);

/* A static string naming a return code (ATTN_OK / ATTN_ERR_*). */
const char* attn_status_string(int code);

/* Library version, e.g. "0.1.0". */
const char* attn_version(void);

/* The CUDA runtime's description of the error behind the last ATTN_ERR_CUDA
 * returned to this host thread ("no CUDA error" if there was none). A static
 * string; not cleared by later successful calls. */
const char* attn_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
