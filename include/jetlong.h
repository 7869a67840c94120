/*
 * jetlong.h -- C ABI of the B300 (sm_103a) Dynamic Bifocal RoPE attention library.
 *
 * The method is the one of "Jet-Long: Efficient Long-Context Extension with
 * Dynamic Bifocal RoPE" (arXiv 2607.07740).  The pages that describe it print
 * no formulas; the statement below is the library's reading of their prose,
 * cited per entry point by page title and section.
 *
 * Notation.  Positions p are 0-based token indices.  D is the head dimension,
 * tau = 1/sqrt(D).  theta_d = theta^(-2d/D) for d in [0, D/2).  R_p rotates
 * every pair (x_d, x_{d+D/2}) of a head vector by the angle p*theta_d
 * (half-split pair layout, the Qwen3 / Hugging Face "rotate_half" convention).
 *
 *   g(s, L)   the group factor: the smallest integer g >= 1 such that every
 *             aliased position floor(p/g), p < s, lies inside the pretrained
 *             window [0, L); equal to max(1, ceil(s/L)), so g = 1 whenever
 *             s <= L ("ResearchPod Summary", paragraph 2: smallest integer
 *             grouping that keeps remote rotation angles within the pretrained
 *             distribution; abstract on the engineersofai.com page: the factor
 *             adapts to the current length s and the base model is recovered
 *             exactly at short inputs).
 *   delta_p   floor(p/g) - p <= 0, the correction offset (position aliasing,
 *             ResearchPod transcript).
 *
 * Bifocal score of query i against key j <= i, with exact-RoPE inputs
 * q_i = R_i(raw q), k_j = R_j(raw k):
 *   i - j <  w :  tau * <q_i, k_j>                              (local, exact RoPE)
 *   i - j >= w :  tau * <R_{delta_i} q_i, R_{delta_j} k_j>      (remote, aliased)
 * followed by one softmax over all keys j <= i.  This equals the pages'
 * inclusion-exclusion merge local(window) + remote(all) - remote(window) on
 * log-sum-exp statistics ("How bifocal attention sidesteps the fixed-scaling
 * trap", seventnews.com; "How Jet-Long works", transform-ai page).  The remote
 * vectors come from an on-the-fly correction rotation of the exact-RoPE q/k;
 * no second rotated copy is stored (abstract; ResearchPod transcript on the
 * cache keeping original positions).
 *
 * Conventions shared by every entry point
 *   - Tensors are contiguous, row-major.  q / out: [B, S, Hq, D] bf16;
 *     k / v: [B, S, Hkv, D] bf16 ("BSHD"); lse: fp32 [B, Hq, S].
 *     GQA: query head h reads kv head h / (Hq / Hkv).
 *   - Every device pointer must be 16-byte aligned (TMA and 128-bit loads).
 *   - The caller owns every buffer.  No entry point allocates or frees device
 *     memory, copies between host and device, or synchronises; compute calls
 *     are asynchronous on `stream` (a cudaStream_t; NULL = legacy stream).
 *   - Argument checks run on the host before any launch and return an error
 *     code without touching memory.  A launch failure returns JL_ERR_CUDA.
 *     Device code never traps: a bounded wait that expires or a guard that
 *     fires records a code in the device status word (jl_debug_status) and the
 *     kernel returns early.
 *   - No C++ exception crosses this interface.
 *   - Bifocal off: pass L_pre >= S (prefill) or L_pre >= n (decode); g is then
 *     1, no key is corrected, and the same kernel computes plain causal RoPE
 *     attention.
 */
#ifndef JETLONG_H
#define JETLONG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes of every entry point. */
typedef enum {
    JL_OK = 0,
    JL_ERR_ARG = -1,         /* a size or parameter out of its domain            */
    JL_ERR_ALIGN = -2,       /* a pointer not 16-byte aligned                    */
    JL_ERR_UNSUPPORTED = -3, /* a valid shape this build has no kernel for (D)   */
    JL_ERR_OVERFLOW = -4,    /* an element count or byte size overflows int64    */
    JL_ERR_CUDA = -5,        /* a CUDA runtime call or launch failed             */
    JL_ERR_TIMEOUT = -6,     /* device status only: a bounded wait expired       */
    JL_ERR_WORKSPACE = -7,   /* workspace pointer NULL or smaller than required  */
    JL_ERR_GUARD = -8        /* device status only: an in-kernel guard fired (a
                                non-finite score, a length or page id out of
                                range); see the entry points                   */
} jl_status;

/* Human-readable name of a jl_status value (static string, never NULL). */
const char *jl_status_string(int status);

/* Library version as "major.minor.patch" (static string). */
const char *jl_version(void);

/*
 * Group factor g(s, L_pre) = max(1, ceil(s / L_pre)) -- host, pure.
 * Reading of the ResearchPod summary (paragraph 2, "smallest integer grouping")
 * and of the abstract (factor set by the current length s).
 *   s      current sequence length (prefill: S; decode: n), >= 1
 *   L_pre  pretrained context window, >= 1
 *   g_out  host pointer receiving g (>= 1); untouched on error
 * Returns JL_OK, JL_ERR_ARG (s < 1, L_pre < 1, g_out NULL) or JL_ERR_OVERFLOW
 * (g would not fit in int32).
 */
int jl_group_factor(int64_t s, int64_t L_pre, int32_t *g_out);

/*
 * Variant flags of the _ex entry points (the method's optional forms).
 *   JL_VARIANT_PER_QUERY_G  query i uses its own current length s = i + 1, so
 *       g = g(i + 1, L_pre) grows inside one prefill (abstract: the factor
 *       adapts to the current length s; a causal model at token i has seen
 *       i + 1 tokens).  A decode's single query already has s = n.
 *   JL_VARIANT_SLIDING  a sliding-window layer of a hybrid model: keys with
 *       i - j >= w are not attended and nothing is aliased (seventnews.com,
 *       "Generalization to hybrid attention architectures": local-window
 *       layers keep their own window); L_pre plays no part.  Must come alone.
 *   JL_VARIANT_QUERY_SHIFT  Self-Extend-style grouping (the ResearchPod
 *       summary names Self-Extend as a baseline): the aliased query position
 *       is floor(i/g) + w - floor(w/g), which makes aliased distances continue
 *       the exact ones at i - j = w, and g = g_shift(s, L_pre, w) is the
 *       smallest integer with floor((s-1)/g) + w - floor(w/g) <= L_pre - 1
 *       (see jl_group_factor_ex).  For s > L_pre it needs w < L_pre.
 * Prefill accepts PER_QUERY_G and QUERY_SHIFT one at a time
 * (JL_ERR_UNSUPPORTED for both together).
 */
#define JL_VARIANT_PER_QUERY_G 1u
#define JL_VARIANT_SLIDING 2u
#define JL_VARIANT_QUERY_SHIFT 4u

/*
 * Kernel choice of jl_bifocal_prefill_ex (combines with the variant flags).
 * Two tile kernels compute the same result (both parity-tested):
 *   - the one-CTA kernel: a CTA per 128-row query tile of two heads that share
 *     a kv head, every K tile it visits corrected by that CTA;
 *   - the two-SM kernel, where it applies (D = 128 and Hq / Hkv a multiple of
 *     4): a cluster of two CTAs per query tile of four heads, tcgen05 MMAs of
 *     M = 256 across both SMs (cta_group::2), each CTA loading and correcting
 *     half of every K tile -- half the correction work per SM.
 * By default a launch takes the two-SM kernel where it applies and the launch
 * has remote keys (g > 1, not a sliding-window layer, s - 1 >= w), the one-CTA
 * kernel otherwise: at the 128K Qwen3-8B-shaped layer on B300 the two-SM
 * kernel measured ~134 ms bifocal against ~137 ms, and ~116 ms plain against
 * ~114 ms.  JL_PREFILL_CTA_PAIR forces the two-SM kernel wherever it applies
 * (ignored elsewhere); JL_PREFILL_ONE_CTA forces the one-CTA kernel; both
 * together are JL_ERR_ARG.
 */
#define JL_PREFILL_CTA_PAIR 8u
#define JL_PREFILL_ONE_CTA 16u

/*
 * Group factor under variant flags -- host, pure.  Without JL_VARIANT_QUERY_SHIFT
 * it is jl_group_factor(s, L_pre) (w unused); with it, g_shift(s, L_pre, w) as
 * defined above.  JL_VARIANT_SLIDING gives 1 (nothing is aliased).
 * Returns JL_OK, JL_ERR_ARG (s, L_pre or w < 1, an unknown flag, g_out NULL, or
 * no g for the shifted rule) or JL_ERR_OVERFLOW.
 */
int jl_group_factor_ex(int64_t s, int64_t L_pre, int64_t w, unsigned flags, int32_t *g_out);

/*
 * Exact RoPE, in place: x[b, s, h, :] <- R_{pos0 + s}(x[b, s, h, :]).
 * The "local RoPE-faithful window" of the abstract uses the original, unscaled
 * frequencies ("How bifocal attention sidesteps the fixed-scaling trap"); this
 * call produces the exact-RoPE q, k and cache rows the attention calls consume.
 *   x      device, bf16 [B, S, H, D], 16-byte aligned, rewritten in place
 *   pos0   position of row s = 0 (>= 0; pos0 + S - 1 < 2^62)
 *   theta  RoPE base (> 0)
 * Angles are formed from an exact 64-bit fixed-point phase (turns) and
 * evaluated in fp32; the result is rounded to bf16 (nearest even).
 * Returns JL_OK, JL_ERR_ARG, JL_ERR_ALIGN, JL_ERR_UNSUPPORTED (D not even or
 * D > 256), JL_ERR_OVERFLOW or JL_ERR_CUDA.
 */
int jl_rope_apply(void *x, int B, int S, int H, int D, int64_t pos0, double theta,
                  void *stream);

/*
 * Exact RoPE fused into the KV-cache write (the step before the attention
 * path): the S_new new tokens' raw keys and their values go to cache rows
 * n_past .. n_past+S_new-1, each key rotated at its position on the way --
 * one read and one write of each byte.  The rotated keys are bit-identical to
 * jl_rope_apply at pos0 = n_past.
 *   k_raw, v   device bf16 [B, S_new, H, D]; k_raw before RoPE
 *   k_cache, v_cache  device bf16 [B, n_cap, H, D]; only rows
 *              n_past..n_past+S_new-1 are written
 *   D a multiple of 16 (<= 256), n_past >= 0, n_past + S_new <= n_cap
 * Returns JL_OK, JL_ERR_ARG, JL_ERR_ALIGN, JL_ERR_UNSUPPORTED,
 * JL_ERR_OVERFLOW or JL_ERR_CUDA.
 */
int jl_rope_cache_write(const void *k_raw, const void *v, void *k_cache, void *v_cache, int B,
                        int S_new, int H, int D, int n_past, int n_cap, double theta, void *stream);

/*
 * Bifocal causal GQA prefill attention (a TMA + tcgen05 tile kernel).
 * Numerics: the exact view multiplies the bf16 inputs as they are; the remote
 * view multiplies the corrected q and k rounded to fp16 (11-bit significand,
 * so one remote score carries a rounding error of about 4e-4 that the softmax
 * averages over the row's keys).  The rotation keeps each pair's norm, so
 * inputs whose elements all lie below 46000 in magnitude give finite fp16
 * operands; a score that is not finite is reported as JL_ERR_GUARD in the
 * device status word.  Rows at positions below 256 that have remote keys
 * (g > 1 and w < 256) see too few keys for that averaging: a second, CUDA-core
 * kernel recomputes exactly those rows in fp32 after the tile kernel.
 * out is normalised by the sum of P as rounded to bf16 for P.V (so it is a
 * weighted mean of V rows); lse uses the fp32 sum.
 * The three attention passes of the pages -- local(window, exact RoPE),
 * remote(all, aliased) and remote(window, aliased), merged by
 * inclusion-exclusion on log-sum-exp statistics (ResearchPod transcript on
 * the prefill phase; "How Jet-Long works", transform-ai page) -- are computed
 * as the single masked pass they equal: a per-tile classifier sends every
 * 128x128 tile that lies inside the window to exact scores, every tile that
 * lies outside it to corrected-rotation scores, and computes both only on the
 * tiles the window boundary crosses.  g = g(S, L_pre).
 *   q      device bf16 [B, S, Hq, D], exact RoPE at positions 0..S-1
 *   k, v   device bf16 [B, S, Hkv, D], same positions
 *   out    device bf16 [B, S, Hq, D], written
 *   lse    device fp32 [B, Hq, S], written: natural-log sum of exp(scores)
 *   B >= 1, Hq >= 1, Hkv >= 1 with Hq % Hkv == 0, S >= 1, D in {64, 128},
 *   L_pre >= 1 (pretrained window), w >= 1 (local window: key j is local
 *   for query i when 0 <= i - j < w), theta > 0.
 * Returns JL_OK, JL_ERR_ARG, JL_ERR_ALIGN, JL_ERR_UNSUPPORTED, JL_ERR_OVERFLOW
 * or JL_ERR_CUDA.  out/lse are undefined if the device status word reports a
 * timeout afterwards.
 */
int jl_bifocal_prefill(const void *q, const void *k, const void *v, void *out, float *lse,
                       int B, int Hq, int Hkv, int S, int D, int L_pre, int w,
                       double theta, void *stream);

/*
 * Bifocal prefill of a chunk over an existing cache: S_new new tokens at
 * positions n_past..n_past+S_new-1 attend to every key at positions
 * 0..n_past+S_new-1 (the cached tokens and themselves, causally).  This is
 * the prefill step the pages place before generation, run in pieces; s =
 * n_past + S_new sets g = g(s, L_pre), so a chunk scores exactly the rows a
 * full prefill of length s would give those positions.  The caller has
 * already written the chunk's exact-RoPE K/V into cache rows n_past..n_past+
 * S_new-1; the cache keeps original positions and is never rewritten.
 *   q        device bf16 [B, S_new, Hq, D], exact RoPE at n_past..n_past+S_new-1
 *   k_cache, v_cache  device bf16 [B, n_cap, Hkv, D]; rows 0..n_past+S_new-1
 *            are read, the rest of the capacity never (it may hold anything)
 *   out      device bf16 [B, S_new, Hq, D];  lse device fp32 [B, Hq, S_new]
 *   S_new >= 1, n_past >= 0, n_past + S_new <= n_cap, other arguments as in
 *   jl_bifocal_prefill (which is this call with n_past = 0, n_cap = S).
 * Returns JL_OK, JL_ERR_ARG, JL_ERR_ALIGN, JL_ERR_UNSUPPORTED, JL_ERR_OVERFLOW
 * or JL_ERR_CUDA.
 */
int jl_bifocal_prefill_chunk(const void *q, const void *k_cache, const void *v_cache, void *out,
                             float *lse, int B, int Hq, int Hkv, int S_new, int n_past, int n_cap,
                             int D, int L_pre, int w, double theta, void *stream);

/*
 * jl_bifocal_prefill_chunk with variant flags (JL_VARIANT_*; 0 gives exactly
 * jl_bifocal_prefill_chunk, and n_past = 0, n_cap = S_new a full prefill).
 * PER_QUERY_G runs one launch per range of rows that share g -- the rows
 * [(g-1) L_pre, g L_pre) -- each scored as the chunk of a prefill of length
 * g L_pre.  SLIDING visits only the key tiles the window reaches.
 * QUERY_SHIFT shifts the query's correction offset by w - floor(w/g).
 * JL_PREFILL_CTA_PAIR / JL_PREFILL_ONE_CTA choose the tile kernel (see above).
 * Returns what jl_bifocal_prefill_chunk returns; JL_ERR_ARG also for an unknown
 * flag, SLIDING with another variant flag, or a QUERY_SHIFT with no valid g;
 * JL_ERR_UNSUPPORTED for PER_QUERY_G with QUERY_SHIFT.
 */
int jl_bifocal_prefill_ex(const void *q, const void *k_cache, const void *v_cache, void *out,
                          float *lse, int B, int Hq, int Hkv, int S_new, int n_past, int n_cap,
                          int D, int L_pre, int w, double theta, unsigned flags, void *stream);

/*
 * Workspace bytes jl_bifocal_decode needs for these sizes (split-KV partial
 * statistics and one arrival counter per (batch, kv head)).  The value does
 * not grow with n: a workspace sized once serves every cache length for the
 * same (B, Hq, Hkv, D).  0 on bad sizes.
 */
size_t jl_bifocal_decode_workspace_size(int B, int Hq, int Hkv, int n, int D);

/*
 * Bifocal single-token decode over an exact-RoPE bf16 KV cache (split-KV; a
 * non-finite score is reported as JL_ERR_GUARD in the device status word).
 * Numerics: at D = 128 and n >= 256 the scores and P.V run on the tensor
 * cores (bf16 operands for exact keys, fp16 for corrected ones as in the
 * prefill, fp32 accumulation, P rounded to bf16 for P.V with out normalised
 * by the sum of the rounded P and lse by the fp32 sum); shorter caches and
 * D = 64 use fp32 arithmetic on CUDA cores throughout.  The paged decode at
 * D = 128 runs on the tensor cores for every length, its sequences shorter
 * than 256 keys with P split into a high and a low bf16 part for P.V.
 * Kernels exist for GQA group sizes Hq / Hkv in {1, 2, 4, 8}; any other group
 * size returns JL_ERR_UNSUPPORTED (this also holds for the paged and the
 * no-allocation variants).
 * The cache keeps original positions and is never rewritten; remote keys are
 * corrected at lookup time (ResearchPod transcript on the cache; abstract:
 * at most ~4% generation overhead).  The query is the token at position n-1
 * and the cache holds positions 0..n-1 including it; g = g(n, L_pre); key j
 * is exact when n-1-j < w, aliased otherwise.
 *   q        device bf16 [B, Hq, D], exact RoPE at position n-1
 *   k_cache, v_cache  device bf16 [B, n_cap, Hkv, D]; rows 0..n-1 are read,
 *            the rest of the capacity never (it may hold anything)
 *   out      device bf16 [B, Hq, D];  lse device fp32 [B, Hq]
 *   n        1 <= n <= n_cap (current length), n_cap the cache capacity
 *   workspace  device, >= jl_bifocal_decode_workspace_size() bytes, 16-byte
 *            aligned.  Its counters must be zero before the first call (e.g.
 *            allocate it zero-filled); every completed call leaves them zero.
 *            Two calls that share a workspace must not overlap on the GPU.
 * Returns JL_OK, JL_ERR_ARG, JL_ERR_ALIGN, JL_ERR_UNSUPPORTED, JL_ERR_OVERFLOW,
 * JL_ERR_WORKSPACE or JL_ERR_CUDA.
 */
int jl_bifocal_decode(const void *q, const void *k_cache, const void *v_cache, void *out,
                      float *lse, int B, int Hq, int Hkv, int n, int n_cap, int D, int L_pre,
                      int w, double theta, void *workspace, size_t ws_bytes, void *stream);

/*
 * jl_bifocal_decode with variant flags (JL_VARIANT_*; 0 gives exactly
 * jl_bifocal_decode).  PER_QUERY_G changes nothing for the single query at
 * n - 1 (its length is n).  SLIDING attends to the last min(n, w) keys only,
 * all exact.  QUERY_SHIFT uses g_shift(n, L_pre, w) and shifts the query's
 * correction offset by w - floor(w/g).  Same workspace as jl_bifocal_decode.
 * Returns what jl_bifocal_decode returns; JL_ERR_ARG also for an unknown flag,
 * SLIDING with another flag, or a QUERY_SHIFT with no valid g.
 */
int jl_bifocal_decode_ex(const void *q, const void *k_cache, const void *v_cache, void *out,
                         float *lse, int B, int Hq, int Hkv, int n, int n_cap, int D, int L_pre,
                         int w, double theta, unsigned flags, void *workspace, size_t ws_bytes,
                         void *stream);

/*
 * Bifocal decode of a batch of sequences of different lengths over a paged
 * KV cache: sequence b has n_b = seq_lens[b] tokens, its query is the token at
 * position n_b - 1, and it sets its own g = g(n_b, L_pre) -- the group factor
 * follows each sequence's current length (ResearchPod summary: "every
 * length").  Its keys live in fixed-size pages of one pool: page p of
 * sequence b (positions p*page_size .. p*page_size + page_size - 1) is pool
 * page block_table[b][p].
 *   q        device bf16 [B, Hq, D], exact RoPE at each sequence's position n_b - 1
 *   k_pages, v_pages  device bf16 [num_pages, page_size, Hkv, D], exact RoPE
 *   block_table  device int32 [B, max_pages]; entries past a sequence's last
 *            page are never read; an id that a sequence uses but that lies
 *            outside [0, num_pages) reads zeros (never faults) and is reported
 *            as JL_ERR_GUARD in the device status word
 *   seq_lens device int32 [B], 1 <= n_b <= max_n; a length outside that range
 *            is clamped into it and reported as JL_ERR_GUARD in the device
 *            status word (the call never reads past the table or the plan)
 *   out      device bf16 [B, Hq, D];  lse device fp32 [B, Hq]
 *   page_size  a multiple of 64 (the kernel's key block); max_pages * page_size
 *            >= max_n (host: a bound on every length; longer ones are clamped)
 *   workspace  as for jl_bifocal_decode, at least
 *            jl_bifocal_decode_paged_workspace_size(B, Hq, Hkv, max_n, D) bytes
 * Rows of a sequence's last page past n_b are never used, whatever they hold.
 * Returns JL_OK, JL_ERR_ARG, JL_ERR_ALIGN, JL_ERR_UNSUPPORTED, JL_ERR_OVERFLOW,
 * JL_ERR_WORKSPACE or JL_ERR_CUDA.
 */
/*
 * Workspace bytes jl_bifocal_decode_paged needs.  The kernel shares a fixed
 * number of CTAs per kv head (about two per SM) among the sequences in
 * proportion to their lengths, which it reads on the device, so a batch of one
 * long and many short sequences keeps every CTA equally busy; the workspace
 * holds that many partial results per (sequence, head) and does not depend on
 * the lengths.  0 on bad sizes.
 */
size_t jl_bifocal_decode_paged_workspace_size(int B, int Hq, int Hkv, int max_n, int D);

int jl_bifocal_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                            const int32_t *block_table, const int32_t *seq_lens, void *out,
                            float *lse, int B, int Hq, int Hkv, int D, int page_size, int num_pages,
                            int max_pages, int max_n, int L_pre, int w, double theta,
                            void *workspace, size_t ws_bytes, void *stream);

/*
 * Size of the fixed device scratch behind jl_bifocal_decode_noalloc: 8 MiB,
 * enough for B * Hq * splits * (D + 2) * 4 bytes of split partials plus the
 * arrival counters (for example B = 1, Hq = 32, D = 128 at any cache length).
 */
#define JL_DECODE_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * jl_bifocal_decode without a workspace argument.  The paper has no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory -- for instance code that runs inside another
 * runtime's fixed, pre-planned memory pool, or a plug-in that has no access
 * to an allocator -- and so cannot provide the scratch jl_bifocal_decode
 * asks for.  It computes exactly what jl_bifocal_decode computes, with the
 * same arguments (minus workspace / ws_bytes) and the same return codes.
 *
 * Scratch: a file-scope device array of JL_DECODE_NOALLOC_SCRATCH_BYTES that
 * every GPU loading this library holds until the process exits.  Shapes
 * whose split partials do not fit (jl_bifocal_decode_workspace_size() above
 * that size) are rejected with JL_ERR_WORKSPACE before anything runs.  The
 * call allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.  It clears the array's arrival counters (cudaMemsetAsync on
 * `stream`) and then launches on `stream`.
 *
 * The first call made with a given device current looks up the array's
 * device address on that device (cudaGetSymbolAddress) and caches it; make
 * that first call before any stream capture.  Every call shares the one
 * array, so two calls whose executions overlap on the GPU (different
 * streams, no ordering between them) race on it and give undefined results.
 */
int jl_bifocal_decode_noalloc(const void *q, const void *k_cache, const void *v_cache, void *out,
                              float *lse, int B, int Hq, int Hkv, int n, int n_cap, int D,
                              int L_pre, int w, double theta, void *stream);

/*
 * Debug: aliased positions floor(p/g) for p in [0, S), g = g(S, L_pre),
 * written as int32 to out_dev[0..S).  Computed on the device by the same
 * integer code the kernels use.
 */
int jl_debug_grouped_positions(int64_t S, int64_t L_pre, int32_t *out_dev, void *stream);

/*
 * Debug: the prefill tile classifier for one (S, L_pre, w), written to
 * out_dev as int8 [ceil(S/128), ceil(S/128)] (row = query tile, column = key
 * tile): 0 masked (every key after every query), 1 exact (every pair inside
 * the window), 2 remote (every pair outside it), 3 band (both), and every
 * unmasked tile is 1 when g = 1.
 */
int jl_debug_tile_classes(int S, int L_pre, int w, int8_t *out_dev, void *stream);

/*
 * Debug: exercises the failure path of every bounded device wait.  One warp
 * waits on an mbarrier that nothing arrives on, with a limit of limit_ns
 * (1 ns .. 100 ms) instead of the kernels' 2 s; the wait gives up, records
 * JL_ERR_TIMEOUT in the device status word and the kernel returns normally
 * (no trap, no hang).  gave_up_dev (device int) receives 1 when the wait gave
 * up.  Returns JL_OK, JL_ERR_ARG or JL_ERR_CUDA.
 */
int jl_debug_wait_timeout(int64_t limit_ns, int *gave_up_dev, void *stream);

/*
 * Debug: read and clear the device status word of the current device
 * (JL_OK, JL_ERR_TIMEOUT or JL_ERR_GUARD).  Synchronises the device; meant
 * for tests, not for the hot path.
 */
int jl_debug_status(int *status_out);

#ifdef __cplusplus
}
#endif

#endif /* JETLONG_H */
