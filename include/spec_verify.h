/*
 * spec_verify.h -- C ABI of the speculative-decoding verify step on GB300.
 *
 * The verify step of speculative decoding (draft model proposes gamma tokens
 * or a tree of them; the target model checks them all in one forward) has
 * three data-parallel parts, and this library does exactly those:
 *
 *   spec_verify_attn    append the new rows' K/V to a paged cache and run the
 *                       masked attention of the gamma+1 (or tree) queries;
 *   spec_reject_sample  temperature softmax of target and draft logits,
 *                       accept/reject of each draft token, and the
 *                       replacement or bonus draw;
 *   kv_commit           roll the cache back to the accepted prefix, or
 *                       compact the accepted tree path.
 *
 * Conventions shared by every call
 *   - Every tensor pointer is caller-owned DEVICE memory, dense and
 *     row-major in the stated shape.  The library never allocates, never
 *     frees and never synchronises (except spec_get_device_status).  All work
 *     is enqueued on `stream` (a cudaStream_t passed as void*; NULL = the
 *     legacy default stream).  Calls are re-entrant; the state kept between
 *     calls is a per-thread count of launches (spec_last_launch_count),
 *     cached driver entry points, and the scratch array of
 *     spec_reject_sample_noalloc with its device address per CUDA context.
 *   - Every device-side wait is bounded (spec_dims.wait_limit_kcycles); one
 *     that gives up raises SPEC_ERR_TIMEOUT.  After that bit is seen, clear
 *     the status word and zero the workspace again (spec_workspace_init)
 *     before the next call: counters inside it may be left mid-way.
 *   - B requests, M query rows per request (row 0 = the pending root token
 *     whose K/V is not cached yet, rows 1.. = drafts or tree nodes), Hq query
 *     heads, Hkv KV heads (Hq % Hkv == 0), head size D, vocabulary V.
 *   - Tree topology: parent[B][M] int32 with parent[b][0] = -1 and
 *     0 <= parent[b][n] < n for n >= 1 (BFS or any topological numbering).
 *     parent == NULL means the chain parent[n] = n - 1.
 *   - Errors the host can see (bad sizes, NULL pointers, short workspace)
 *     return at once and launch nothing.  Errors only the device can see
 *     (a block id out of range, a context that does not fit the block table,
 *     a bad temperature, a row with no distribution) set a bit in the status
 *     word kept in the workspace and make the affected request a no-op with
 *     defined outputs; read them with spec_get_device_status.
 *
 * Sources: three practitioner pages on speculative decoding -- page 1
 * "投机推理..." (kwkr.cn) §2.1, §2.3, §4.1, §4.3, §5.1, §5.3; page 2
 * "推测解码..." (cf-1.com) §2.1-§2.3, §3.3, §4.3, §5.4; page 3
 * "推测解码的工程真相 2026" (blog.lonae.com), formal-definition and
 * tree-attention sections.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum spec_status {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1,   /* bad size, NULL pointer, bad temperature/topology */
  SPEC_ERR_CAPACITY = 2,      /* ctx + M exceeds the request's block-table capacity */
  SPEC_ERR_UNSUPPORTED = 3,   /* shape or dtype this build has no kernel for */
  SPEC_ERR_CUDA = 4,          /* a CUDA runtime call failed */
  SPEC_ERR_NONFINITE = 5,     /* a logits row holds NaN/+inf or only -inf */
  SPEC_ERR_DEVICE_BOUNDS = 6, /* a block id or token id out of range */
  SPEC_ERR_TIMEOUT = 7        /* a device-side wait gave up (bounded, never hangs) */
} spec_status;

typedef enum spec_dtype { SPEC_BF16 = 0, SPEC_F32 = 1 } spec_dtype;

/* Attention kernel selection (spec_dims.attn_impl). */
typedef enum spec_attn_impl {
  SPEC_ATTN_AUTO = 0,          /* tensor cores when the shape allows, else CUDA cores */
  SPEC_ATTN_CUDA_CORES = 1,    /* split-KV on CUDA cores: group*M <= 128, D 64/128, bf16/f32 */
  SPEC_ATTN_TENSOR_CORES = 2   /* tcgen05 + TMA: bf16, D = 128, group*M <= 128 */
} spec_attn_impl;

/* Reject-sample kernel selection (spec_dims.reject_impl). */
typedef enum spec_reject_impl {
  SPEC_REJECT_AUTO = 0,        /* the staged kernels (the faster choice measured on
                                  GB300 at every shape tried) */
  SPEC_REJECT_STAGED = 1,      /* logit statistics, then for a chain with 16-byte
                                  aligned rows and no filter one tail kernel
                                  (decisions, residual masses and draw, several CTAs
                                  per request); for a tree with such rows and no
                                  filter the walk by a cluster of 8 CTAs per request
                                  beside the statistics (which still decide which
                                  requests fail); else three kernels (decisions,
                                  residual masses, residual draws); any alignment,
                                  V up to 2^20 */
  SPEC_REJECT_FUSED = 2        /* one kernel for a chain: every warp streams logit
                                  statistics and decides each request as soon as its
                                  rows are done; chains with 16-byte aligned rows
                                  (V * element size a multiple of 16, aligned row
                                  pointers), V up to 2^20, no filter;
                                  SPEC_ERR_UNSUPPORTED otherwise */
} spec_reject_impl;

typedef struct spec_dims {
  int32_t B;            /* requests in the batch */
  int32_t M;            /* query rows per request: gamma+1, or tree nodes incl. root;
                           1..128 (SPEC_ERR_UNSUPPORTED above) */
  int32_t Hq;           /* query heads */
  int32_t Hkv;          /* KV heads; query head h reads KV head h / (Hq/Hkv) */
  int32_t D;            /* head size (64 or 128) */
  int32_t block;        /* tokens per KV block; must be 16 */
  int32_t max_blocks;   /* entries per block-table row */
  int32_t num_blocks;   /* physical blocks in each cache */
  int32_t V;            /* vocabulary size */
  int32_t kv_dtype;     /* spec_dtype of q, k_new, v_new, caches and out */
  int32_t logits_dtype; /* spec_dtype of target and draft logits */
  float softmax_scale;  /* attention score scale; 0 selects 1/sqrt(D) */
  int32_t attn_impl;    /* spec_attn_impl; 0 = automatic choice */
  int32_t reject_impl;  /* spec_reject_impl; 0 = automatic choice */
  int32_t wait_limit_kcycles; /* every bounded device wait gives up after this
                                 many thousand SM clocks and raises
                                 SPEC_ERR_TIMEOUT; 0 = the default, 4e6
                                 (about 2 s at 2 GHz).  Work already issued
                                 (copies, MMAs) is always waited for before a
                                 CTA exits, whatever this limit. */
} spec_dims;

/* Bytes of caller-owned device workspace every call with these dims needs
 * (status word, split-KV partials, row statistics, per-request state).
 * Returns 0 if the dims are invalid. */
size_t spec_workspace_size(const spec_dims* dims);

/* Zero the workspace (status word included).  Call once after allocating it;
 * afterwards every call leaves it ready for the next.  An async memset on
 * `stream`. */
spec_status spec_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Synchronise `stream` and read the device status word: bit (1 << code) is
 * set for every spec_status code a device-side check raised since the last
 * clear.  clear != 0 resets the word afterwards. */
spec_status spec_get_device_status(void* ws, void* stream, int32_t* flags,
                                   int32_t clear);

/*
 * spec_verify_attn -- KV append and verify attention (one layer).
 *
 * Page 1 §2.1: feed all candidate positions at once; under the causal mask
 * each position sees only what precedes it, so the parallel pass equals
 * token-by-token decoding, provided the KV cache is extended in the right
 * order.  Page 2 §3.3: reuse the cached prefix and compute K/V only for the
 * new positions.  Page 3 (tree-attention section) and page 2 §5.4: a draft
 * tree is verified in one pass under a mask that follows the tree.
 *
 *   q        [B, M, Hq, D]   kv_dtype   queries (position encoding applied)
 *   k_new    [B, M, Hkv, D]  kv_dtype   K of the M new rows
 *   v_new    [B, M, Hkv, D]  kv_dtype   V of the M new rows
 *   k_cache  [num_blocks, Hkv, 16, D]   paged K cache (in/out)
 *   v_cache  [num_blocks, Hkv, 16, D]   paged V cache (in/out)
 *   block_table [B, max_blocks] int32   position t of request b lives in
 *                                       block block_table[b][t/16], slot t%16
 *   ctx_lens [B] int32      cached tokens of request b before this step
 *   parent   [B, M] int32 or NULL (chain)
 *   out      [B, M, Hq, D]   kv_dtype   attention output
 *   lse      [B, M, Hq] float or NULL   natural-log log-sum-exp of the
 *                                       scaled scores of each row
 *
 * Effect: rows i = 0..M-1 of k_new/v_new are written to positions
 * ctx+i; the remaining slots of the last block touched are set to zero.
 * Then row i attends to positions 0..ctx-1 and to the new positions
 * ctx+k for every k that is i or an ancestor of i (k <= i for a chain),
 * with scores scaled by softmax_scale.
 * A request whose ctx + M exceeds max_blocks*16 (SPEC_ERR_CAPACITY, the
 * pages' cue to fall back to plain decoding) or whose needed block ids are
 * out of range (SPEC_ERR_DEVICE_BOUNDS) leaves the caches untouched and
 * gets out = 0, lse = -inf.
 */
spec_status spec_verify_attn(const void* q, const void* k_new,
                             const void* v_new, void* k_cache, void* v_cache,
                             const int32_t* block_table,
                             const int32_t* ctx_lens, const int32_t* parent,
                             void* out, float* lse, const spec_dims* dims,
                             void* ws, size_t ws_bytes, void* stream);

/*
 * spec_reject_sample -- accept / reject / resample of the drafts.
 *
 * p = softmax(target/T), q = softmax(draft/T) with the request's temperature
 * (page 1 §3.3).  Draft token x of node c is accepted iff
 * u_acc(c) * q(x) < p(x), i.e. with probability min(1, p/q) (page 1 §2.3,
 * §4.1; page 2 §2.1); the walk stops at the first rejection (page 1 §4.3).
 * After a rejection the token is drawn from normalize(max(0, p - q)); if the
 * walk reaches a node without children the bonus token is drawn from p
 * (page 3, formal definition).  In a tree the children of a node are tried
 * in ascending order and each rejection replaces the working target P by
 * normalize(max(0, P - q)); the first accepted child is entered.  Draws use
 * the inverse CDF in vocabulary order: the smallest k with C_k > u*Z.
 *
 * Uniforms: Philox4x64-10 (Salmon et al., SC'11), key (seed, 0), counter
 * (n+1, b_base+b, offset, 0) for node n of request b; u_acc = (w0>>40)*2^-24,
 * u_smp = (w1>>40)*2^-24.
 *
 *   target_logits [B, M, V] logits_dtype   row n: law of n's children
 *   draft_logits  [B, M, V] logits_dtype   row n: q that drafted n's children
 *                                          (rows of leaves are not read)
 *   tokens        [B, M] int32   drafted token of node n (tokens[b][0] unused)
 *   parent        [B, M] int32 or NULL (chain)
 *   temperature   [B] float      a positive normal finite value, or 0:
 *                                greedy (page 1 §4.3, first point) -- each
 *                                row's law is the point mass on its largest
 *                                logit (smallest index among equal ones), so
 *                                a draft is accepted iff it is that token
 *                                and every draw returns it
 *   out_tokens    [B, M] int32   emitted tokens: the a accepted drafts, then
 *                                the drawn token; -1 after that
 *   path          [B, M] int32   accepted node indices, starting with 0; -1 after
 *   accepted_len  [B] int32      a (number of accepted drafts), -1 if failed
 *   probe         [B, M, 4] float or NULL: for every tested node n, p(x_n)
 *                 and q(x_n) as used in its test (cols 0, 1); at the node
 *                 where the draw happened, the mass Z of the residual that
 *                 was drawn from (1 for a bonus draw) and the probability of
 *                 the drawn token (cols 2, 3); -1 elsewhere.
 * A failed request (bad temperature, token, topology, or a needed row with
 * no distribution) gets accepted_len = -1 and -1 rows.  If a wait gave up
 * (SPEC_ERR_TIMEOUT in the status word, from this call or an earlier one not
 * yet cleared), every request of the call gets accepted_len = -1: no
 * decision is made on statistics that may be incomplete.
 */
spec_status spec_reject_sample(const void* target_logits,
                               const void* draft_logits,
                               const int32_t* tokens, const int32_t* parent,
                               const float* temperature, uint64_t seed,
                               uint64_t offset, uint64_t b_base,
                               int32_t* out_tokens, int32_t* path,
                               int32_t* accepted_len, float* probe,
                               const spec_dims* dims, void* ws,
                               size_t ws_bytes, void* stream);

/*
 * spec_reject_sample_filtered -- spec_reject_sample with top-k / top-p
 * restricted laws.
 *
 * Page 2 §5.1: target and draft must sample by one rule (its example: a
 * nucleus-sampling target against a differently sampling draft).  For a
 * request with top_k[b] = k and top_p[b] = t, the law of every row it uses,
 * target and draft alike, is restricted to a prefix of the row's tokens in
 * the order of their logits, largest first, the smaller index first among
 * equal logits: the first k tokens (k = 0: all), then the shortest prefix of
 * those whose mass reaches t times their mass (t = 1: all of them); the
 * restricted law is renormalised and the walk above runs on it, so the
 * emitted tokens follow the restricted target law.  At temperature 0 the
 * filters change nothing.
 *
 *   top_k  [B] int32 or NULL   >= 0 (0: no top-k)
 *   top_p  [B] float or NULL   in (0, 1] (1: no top-p)
 * Other arguments as in spec_reject_sample.  A request with k < 0 or t
 * outside (0, 1] fails (SPEC_ERR_INVALID_ARG, accepted_len = -1).  The probe
 * reports the restricted laws.  Filters run on the staged kernels: with
 * dims->reject_impl = SPEC_REJECT_FUSED and a filter given the call returns
 * SPEC_ERR_UNSUPPORTED and launches nothing.  Each needed row of a filtered
 * request costs a few extra passes over the row (its kept prefix is found by
 * a radix select over the logits' order keys).
 */
spec_status spec_reject_sample_filtered(const void* target_logits,
                                        const void* draft_logits,
                                        const int32_t* tokens, const int32_t* parent,
                                        const float* temperature,
                                        const int32_t* top_k, const float* top_p,
                                        uint64_t seed, uint64_t offset, uint64_t b_base,
                                        int32_t* out_tokens, int32_t* path,
                                        int32_t* accepted_len, float* probe,
                                        const spec_dims* dims, void* ws,
                                        size_t ws_bytes, void* stream);

/*
 * spec_lm_head -- logits of an LM head: logits[r, v] = sum_k hidden[r, k] *
 * weight[v, k] (bf16 inputs, fp32 accumulation on the tensor cores, bf16
 * output rounded to nearest even).
 *
 * Page 2 §1.2: decoding is bound by weight and logit reads; this is the
 * product the verify step's logits come from.
 *   hidden  [rows, H] bf16   row-major, 16-byte aligned
 *   weight  [V, H]    bf16   row-major (one vocabulary row of H weights)
 *   logits  [rows, V] bf16   output
 *   ws, ws_bytes             at least 16 bytes (its first word is the status
 *                            word of spec_get_device_status)
 * H must be a multiple of 64 and V of 256 (else SPEC_ERR_UNSUPPORTED).
 */
spec_status spec_lm_head(const void* hidden, const void* weight, int32_t rows, int32_t H,
                         int32_t V, void* logits, void* ws, size_t ws_bytes, void* stream);

/*
 * spec_reject_sample_lm_head -- the LM heads and the verify decisions in one
 * call, without a second pass over the logit rows.
 *
 * The target and draft logits of the B*M new rows are computed as in
 * spec_lm_head (target: hidden_target [B, M, Ht] x weight_target [V, Ht];
 * draft: hidden_draft [B, M, Hd] x weight_draft [V, Hd]) into target_logits
 * and draft_logits ([B, M, V] bf16, written); their epilogue also forms the
 * per-chunk statistics the decisions need (page 2 §1.2: the logit rows are
 * read once less), and spec_reject_sample's decisions and draws follow on
 * them.  Arguments after draft_logits and the outputs are those of
 * spec_reject_sample; dims->logits_dtype must be bf16, Ht and Hd multiples
 * of 64, dims->V a multiple of 256; SPEC_REJECT_FUSED is refused.
 */
spec_status spec_reject_sample_lm_head(const void* hidden_target, const void* weight_target,
                                       int32_t Ht, const void* hidden_draft,
                                       const void* weight_draft, int32_t Hd,
                                       void* target_logits, void* draft_logits,
                                       const int32_t* tokens, const int32_t* parent,
                                       const float* temperature, uint64_t seed, uint64_t offset,
                                       uint64_t b_base, int32_t* out_tokens, int32_t* path,
                                       int32_t* accepted_len, float* probe,
                                       const spec_dims* dims, void* ws, size_t ws_bytes,
                                       void* stream);

/*
 * kv_commit -- roll back / compact the cache to the accepted path.
 *
 * Page 2 §3.3: after a partial acceptance the cache past the accepted
 * position is dropped; page 2 §5.4 and page 3 (tree section): a tree verify
 * rolls back along the accepted path.  The K/V of the root and of the a
 * accepted nodes are kept; for j = 1..a (increasing), the slot ctx+path[j]
 * is moved to slot ctx+j.  new_ctx_lens[b] = ctx_lens[b] + a + 1 (the drawn
 * token's K/V comes with the next step).  For a chain nothing moves.
 *
 *   k_cache, v_cache, block_table, ctx_lens  as in spec_verify_attn
 *   new_ctx_lens [B] int32   output; may alias ctx_lens
 *   path [B, M], accepted_len [B]  as produced by spec_reject_sample
 * Requests with accepted_len < 0, a bad path, or out-of-range block ids are
 * left unchanged (new length = old length) and flagged in the status word.
 */
spec_status kv_commit(void* k_cache, void* v_cache, const int32_t* block_table,
                      const int32_t* ctx_lens, int32_t* new_ctx_lens,
                      const int32_t* path, const int32_t* accepted_len,
                      const spec_dims* dims, void* ws, size_t ws_bytes,
                      void* stream);

/*
 * spec_reject_sample_noalloc -- spec_reject_sample for callers that cannot
 * allocate device memory.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot provide a workspace: cudaMalloc may synchronise the whole device,
 * is not allowed while a stream is being captured, and engines that hand all
 * of HBM to a fixed KV-cache pool at start-up often have no allocator to call.
 * Arguments, outputs and semantics are those of spec_reject_sample without
 * ws / ws_bytes.  The scratch (a status word; 16 bytes of row statistics per
 * request, row and 2048-logit chunk -- 1024 for fp32 logits; 8 bytes of
 * residual mass per request and chunk; an 816-byte draw state per
 * request) lives in a 1 MiB array inside the library that every GPU loading
 * the library holds until exit.
 *   - Sizes whose scratch exceeds that array (for bf16 logits, roughly
 *     B * ((32 * M + 8) * ceil(V / 2048) + 816) > 1 MiB)
 *     return SPEC_ERR_UNSUPPORTED and launch nothing; use
 *     spec_reject_sample there.
 *   - The first call in a CUDA context looks up the array's device address
 *     in that context (cudaGetSymbolAddress, once per context, with the
 *     context current) and keeps it; make that first call before any stream
 *     capture.  A new context on the same device (after cudaDeviceReset, or
 *     another context made current) gets its own lookup.
 *   - No memory is allocated or freed, by the library or any routine it
 *     calls.  The status word is cleared at the start of each call with an
 *     async memset on `stream`; device-side failures show as
 *     accepted_len = -1 for the request, and the status word is not readable
 *     through this call.
 *   - Every call shares the one array: calls whose work overlaps on the GPU
 *     (different streams, or different host threads on one device) race and
 *     must be serialised by the caller.
 *   - It does not update spec_last_launch_count.
 */
spec_status spec_reject_sample_noalloc(const void* target_logits,
                                       const void* draft_logits,
                                       const int32_t* tokens,
                                       const int32_t* parent,
                                       const float* temperature, uint64_t seed,
                                       uint64_t offset, uint64_t b_base,
                                       int32_t* out_tokens, int32_t* path,
                                       int32_t* accepted_len, float* probe,
                                       const spec_dims* dims, void* stream);

/*
 * Host-side controller and metrics (no GPU work; plain host memory).
 *
 * Page 3 ("推测解码的工程真相 2026"), dynamic scheduling and observability:
 * the acceptance rate of a request's last `window` verify steps sets its
 * next draft length (above high_acceptance: gamma_high; from
 * low_acceptance to high_acceptance: gamma_mid; below: gamma_low); a
 * temperature above hot_temperature sets gamma_hot at once; a request whose
 * speculation does not pay over a full window falls back to plain decoding
 * (gamma 0) and stays there.  Page 2 §5.1: log drafted and accepted counts
 * and where the rejections fall.
 *
 * Speculative efficiency is read as page 2 §2.3's speedup of a verify step:
 * emitted tokens per step (accepted + 1) / (1 + gamma * draft_cost); a
 * request below min_efficiency falls back.  Requests the device failed
 * (accepted_len = -1, e.g. SPEC_ERR_CAPACITY, the pages' fallback trigger)
 * fall back too.
 */
#define SPEC_CTRL_MAX_WINDOW 64
#define SPEC_CTRL_HIST_BINS 10
#define SPEC_STEP_MAX_POS 129

typedef struct spec_ctrl_config {
  int32_t window;          /* steps the acceptance rate is taken over (<= 64); 16 */
  float high_acceptance;   /* 0.6 */
  float low_acceptance;    /* 0.3 */
  int32_t gamma_high;      /* 8 */
  int32_t gamma_mid;       /* 4 */
  int32_t gamma_low;       /* 2 */
  float hot_temperature;   /* 0.8 */
  int32_t gamma_hot;       /* 1 */
  float draft_cost;        /* draft forward / target forward, 0.02 */
  float min_efficiency;    /* 1.0 */
  int32_t max_gamma;       /* cap on any draft length (<= 63) */
} spec_ctrl_config;

/* Per-request state, caller-owned (zeroed by spec_ctrl_init). */
typedef struct spec_ctrl_request {
  int16_t drafted[SPEC_CTRL_MAX_WINDOW];  /* ring of the last steps */
  int16_t accepted[SPEC_CTRL_MAX_WINDOW];
  int32_t head, steps;
  int32_t gamma;           /* draft length of the next step; 0 = plain decoding */
  int32_t fallback;        /* 1 once the request fell back */
  int32_t failed_steps;
} spec_ctrl_request;

typedef struct spec_ctrl_metrics_out {
  int32_t requests;
  int32_t acceptance_hist[SPEC_CTRL_HIST_BINS]; /* per-request window rates, 0.1-wide bins */
  float acceptance_mean, acceptance_p50, acceptance_p95, acceptance_p99;
  float emitted_per_step;
  float speculative_efficiency;
  float fallback_rate;
} spec_ctrl_metrics_out;

typedef struct spec_step_stats_out {
  int32_t requests, failed;
  int64_t accepted, emitted;
  int32_t rejection_pos[SPEC_STEP_MAX_POS];  /* 1-based draft position of the first
                                                rejection; index M: none rejected */
  float tree_width_effective;  /* mean share of the tree's root-to-leaf paths through
                                  the first accepted node (-1 for chains) */
} spec_step_stats_out;

void spec_ctrl_default_config(spec_ctrl_config* cfg);
spec_status spec_ctrl_init(spec_ctrl_request* reqs, int32_t n, int32_t gamma0);
/* Feed one verify step's accepted lengths (host copy of spec_reject_sample's
 * output; temperature may be NULL) and get each request's next draft length. */
spec_status spec_ctrl_update(const spec_ctrl_config* cfg, spec_ctrl_request* reqs, int32_t n,
                             const int32_t* accepted_len, const float* temperature,
                             int32_t* next_gamma);
spec_status spec_ctrl_metrics(const spec_ctrl_config* cfg, const spec_ctrl_request* reqs,
                              int32_t n, spec_ctrl_metrics_out* out);
/* Statistics of one verify step from host copies of its outputs: accepted
 * and emitted counts, the rejection-position histogram, and, for a tree
 * (parent != NULL), the tree width effective. */
spec_status spec_step_stats(const int32_t* accepted_len, const int32_t* path,
                            const int32_t* parent, int32_t B, int32_t M,
                            spec_step_stats_out* out);

/* Host-side Philox4x64-10 block (the generator the kernels use), for
 * known-answer tests: out = Philox4x64-10(counter, key). */
void spec_philox_block(const uint64_t key[2], const uint64_t counter[4],
                       uint64_t out[4]);

/* Human-readable name of a status code. */
const char* spec_status_string(int32_t status);

/* Number of kernel launches the last call on this thread enqueued. */
int32_t spec_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
