/*
 * la.h -- C ABI of the GB300 lookahead-decoding library (libla.so).
 *
 * The method: lookahead decoding ("Break the Sequential Dependency of LLM
 * Inference Using Lookahead Decoding", arXiv 2402.02057; paper-graph-ui
 * summary, section 3.4).  One step runs a single forward pass of a
 * LLaMA-style decoder over the cached prefix plus
 *   - the lookahead branch: a window of W columns x (N-1) past Jacobi levels
 *     ("The Lookahead Branch"),
 *   - the verification branch: up to G candidate (N-1)-token suffixes taken
 *     from the n-gram pool by first token ("The Verification Branch"),
 * under the lookahead attention mask ("Integrated Forward Pass", Figure 2b),
 * then verifies the candidates (Algorithm 3 greedy, Algorithm 4 sampling),
 * accepts the longest matching prefix, harvests the window's new n-grams into
 * the pool, slides the window and commits the accepted tokens' KV.
 *
 * Conventions (all entry points):
 *   - Return LA_OK (0) or a negative LA_ERR_* code; no exception or abort
 *     crosses the ABI.  la_strerror() names a code; la_last_error() gives the
 *     message of the last failure on the calling thread.
 *   - Device pointers are CUDA device addresses on the current device; host
 *     pointers are ordinary host memory.  Each argument says which it is.
 *   - All work runs on the stream given in la_opts.cuda_stream (NULL: the
 *     legacy default stream).  Calls that return host results synchronise
 *     that stream before they return.
 *   - A handle is not thread-safe: one thread at a time per handle.
 *   - Matrices are row-major [out][in]; a token id is int32 in [0, vocab).
 */
#ifndef LA_H
#define LA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Error codes. */
#define LA_OK                   0
#define LA_ERR_INVALID_ARG     -1  /* bad pointer, size, alignment or option */
#define LA_ERR_OOM             -2  /* device or pinned host allocation failed */
#define LA_ERR_CAPACITY        -3  /* max_seq (or a caller buffer) too small for the request */
#define LA_ERR_CUDA            -4  /* a CUDA runtime or driver call failed */
#define LA_ERR_DEVICE_TIMEOUT  -5  /* a kernel's bounded wait gave up; the step's results are void */
#define LA_ERR_STATE           -6  /* call out of order (e.g. la_step before la_prefill) */
#define LA_ERR_UNSUPPORTED     -7  /* valid request this build does not handle (e.g. head_dim 96) */

/* Weight / activation element types. */
#define LA_F32   0   /* fp32 weights, fp32 activations and KV cache (SIMT GEMMs) */
#define LA_BF16  1   /* bf16 weights; GEMM inputs, KV cache, q and attention probabilities
                        as (hi, lo) bf16 pairs (about 16 mantissa bits), fp32 accumulation
                        and fp32 residual stream (tcgen05 tensor-core GEMMs and attention) */

/* n-gram pool eviction policies (la_opts.pool_policy).  The pages keep the
 * pool's management open (paper-graph-ui page, section 7, "Follow-Up
 * Research This Work Enables": LRU, FIFO or frequency-based eviction). */
#define LA_POOL_FIFO 0   /* each key's suffixes in insertion order; a full list drops the oldest;
                            candidates are the oldest G */
#define LA_POOL_LRU  1   /* least recently used first; a use (the step's winning candidate, when it
                            contributed an accepted token, or a suffix harvested again) moves an
                            entry to the most recent end; a full list drops the least recently used;
                            candidates are the G most recently used, most recent first */
#define LA_POOL_LFU  2   /* fewest uses first: every entry counts its uses (the same events as LRU) and
                            each list is ordered by (uses, time of the last use or entry); a full list
                            drops its head, the fewest-used and oldest among equals, before a new
                            suffix enters with 0 uses; candidates are the G entries with the most
                            uses, the most recent first among equals */

/* Model shape of a LLaMA-style decoder (the pages run LLaMA-2 / CodeLlama,
 * paper-graph-ui page, section 5 "Experimental setup"). */
typedef struct la_model_dims {
    int32_t n_layers;
    int32_t d_model;
    int32_t n_heads;      /* query heads */
    int32_t n_kv_heads;   /* key/value heads; n_heads % n_kv_heads == 0 (GQA) */
    int32_t head_dim;     /* 64 or 128 */
    int32_t ffn;          /* SwiGLU hidden width */
    int32_t vocab;
    float   rms_eps;      /* RMSNorm epsilon */
    float   rope_base;    /* rotary base; rotate-half pairing (i, i + head_dim/2) */
    int32_t dtype;        /* LA_F32 or LA_BF16, for every weight tensor */
} la_model_dims;

/* Device pointers to the weights, owned by the caller, which must keep them
 * alive and unchanged until la_destroy.  Each is 16-byte aligned.
 * Per-layer entries are host arrays of n_layers device pointers; the library
 * copies those arrays at la_create.
 *   embed      [vocab][d_model]          lm_head  [vocab][d_model]
 *   final_norm, attn_norm[l], ffn_norm[l]  [d_model]
 *   wq [n_heads*head_dim][d_model]       wk, wv [n_kv_heads*head_dim][d_model]
 *   wo [d_model][n_heads*head_dim]
 *   w_gate, w_up [ffn][d_model]          w_down [d_model][ffn]              */
typedef struct la_weights {
    const void *embed;
    const void *final_norm;
    const void *lm_head;
    const void *const *attn_norm;
    const void *const *wq;
    const void *const *wk;
    const void *const *wv;
    const void *const *wo;
    const void *const *ffn_norm;
    const void *const *w_gate;
    const void *const *w_up;
    const void *const *w_down;
} la_weights;

/* Decoding options (section 3.4: W lookahead width, N n-gram size / window
 * depth N-1, G verification cap; Table 3 prompt-as-reference; Table 2
 * temperature-1 sampling). */
typedef struct la_opts {
    int32_t N;                    /* n-gram length, 2..8 */
    int32_t W;                    /* window columns, >= 1 */
    int32_t G;                    /* candidates per step, 0..32 */
    int32_t max_seq;              /* KV capacity in tokens: prompt + generated + step rows */
    int32_t prompt_as_reference;  /* 1: seed the pool with the prompt's n-grams after prefill */
    int32_t pool_cap;             /* suffixes kept per first token; 0 -> G (min 1); <= 32 */
    float   temperature;          /* 0: greedy (Algorithm 3); > 0: sampling (Algorithm 4) */
    uint64_t seed;                /* window initialisation and sampling draws */
    void   *cuda_stream;          /* cudaStream_t or NULL */
    int32_t profile;              /* 1: bracket every GEMM and attention launch of la_step with CUDA
                                     events and accumulate their device time in la_stats (adds two
                                     event records per launch) */
    int32_t top_k;                /* temperature > 0: keep only the top_k most probable tokens of every
                                     sampling distribution (ties to the lower id); 0: off */
    float   top_p;                /* temperature > 0: then keep the shortest most-probable prefix whose
                                     renormalised mass reaches top_p (the crossing token included);
                                     <= 0 or >= 1: off.  Order: temperature, top_k, top_p */
    int32_t pool_policy;          /* LA_POOL_FIFO (0), LA_POOL_LRU (1) or LA_POOL_LFU (2) */
} la_opts;

typedef struct la_handle la_handle;

typedef struct la_stats_t {
    int64_t steps;            /* la_step calls since la_prefill */
    int64_t generated;        /* tokens produced: the prefill's first token + every accepted token */
    int32_t last_accept;      /* A of the last step, 1..N */
    int32_t last_candidates;  /* g of the last step, 0..G */
    int32_t prefix_len;       /* P: tokens whose KV is committed */
    int32_t rows;             /* M = 1 + (W + G)(N - 1) rows per step */
    /* With la_opts.profile = 1, summed over la_step calls since la_prefill:
     * device time (CUDA events on the handle's stream), launch count and
     * algorithmic bytes of the projection GEMMs (their weights, read once)
     * and of attention (prefix and step K/V at the weights' element size). */
    double  gemm_ms;
    double  gemm_bytes;
    int64_t gemm_launches;
    double  attn_ms;
    double  attn_bytes;
    int64_t attn_launches;
    int64_t kernel_launches;  /* kernels launched by la_step calls since la_prefill */
    double  elem_ms;          /* profile: row-wise kernels (embedding, norms, rotary/KV write, SwiGLU) */
    double  spec_ms;          /* profile: lookup, argmax, verification/pool/window, KV commit */
    int64_t h2d_bytes;        /* host-to-device bytes copied by la_prefill and la_step since la_prefill
                                 (the prompt, the initial window) */
    int64_t d2h_bytes;        /* device-to-host bytes copied back (the step state with the accepted
                                 tokens, once per la_prefill and per la_step) */
} la_stats_t;

/* Host-side snapshot of the decoding state, for resume and for checking a
 * step against an independent implementation.  The caller allocates the
 * arrays; *_cap fields give their capacities (elements). */
typedef struct la_state_t {
    int32_t  n_tokens;      /* committed tokens: prompt, then outputs; the last one (o) has no KV yet */
    int32_t  tokens_cap;
    int32_t *tokens;        /* [tokens_cap] */
    int32_t *window;        /* [(N-1) * W], level-major: window[k*W + j] = level k, column j (level 0 oldest) */
    int32_t  n_records;     /* pool entries */
    int32_t  records_cap;
    int32_t *records;       /* [records_cap][N]: first token, then the N-1 suffix tokens;
                               keys ascending, each key's suffixes in eviction order (the next
                               to be dropped first: oldest under FIFO, least recently used
                               under LRU, fewest uses then oldest under LFU); la_import_state
                               rebuilds the same order */
    int32_t *uses;          /* [records_cap] or NULL: each record's use count (LFU; 0 under FIFO
                               and LRU).  On import, NULL means 0 uses for every record */
} la_state_t;

/* Create a decoder for the given weights.  Allocates the KV cache (fp32
 * [n_layers][K, V][n_kv_heads][max_seq][head_dim]; bf16 models: K and V as
 * (hi, lo) bf16 plane pairs, V transposed), activations, the n-gram pool
 * and the window on the current device; no weight is copied.
 * Errors: INVALID_ARG (shapes, alignment, options), UNSUPPORTED, OOM, CUDA. */
int la_create(const la_model_dims *dims, const la_weights *weights, const la_opts *opts,
              la_handle **out);

/* Prefill: run the prompt (host int32[n], n >= N and n + generated + M <= max_seq)
 * causally, commit its KV, produce the first token (argmax, or a draw at
 * temperature > 0) into *first_token (host), initialise the window from the
 * prompt and, if asked, seed the pool.  Resets any previous state.
 * Passages: the prompt's forward pass and first output of the autoregressive
 * system (paper-graph-ui page, section 3.4, "The autoregressive system"); the
 * window's random initialisation from the prompt ("The Lookahead Branch");
 * prompt-as-reference seeding (section 5, "Ablation Studies (Table 3)",
 * configurations 2 and 9).
 * Errors: INVALID_ARG, CAPACITY, CUDA, DEVICE_TIMEOUT. */
int la_prefill(la_handle *h, const int32_t *prompt, int32_t n, int32_t *first_token);

/* One lookahead step.  Writes the A accepted tokens (1 <= A <= N) to host
 * out_tokens (capacity >= N) and A to *out_n.  Synchronous.
 * bf16 models without la_opts.profile: the first step of a handle launches
 * its kernels directly and captures them, with the state read-back, into a
 * CUDA graph on the handle's stream; later steps replay that graph (one
 * launch per step; results equal to direct launches bit for bit).  If the
 * capture fails the handle keeps launching directly.
 * Errors: STATE (no prefill), CAPACITY (max_seq reached), CUDA, DEVICE_TIMEOUT. */
int la_step(la_handle *h, int32_t *out_tokens, int32_t *out_n);

/* One plain autoregressive decoding step (the baseline lookahead decoding is
 * measured against; paper-graph-ui page, section 3.4 "The autoregressive
 * system"): one forward row for the last committed token, which commits its
 * KV, then argmax (or a draw at temperature > 0, keyed like the first token)
 * over the vocabulary.  Writes the new token to *token (host).  Uses the same
 * kernels as la_prefill; leaves the window and the pool untouched, so it can
 * be interleaved with la_step on one handle.
 * Errors: STATE (no prefill), CAPACITY (max_seq reached), CUDA, DEVICE_TIMEOUT. */
int la_ar_step(la_handle *h, int32_t *token);

/* Prefill, then steps until max_new tokens are produced (the prefill's first
 * token counts; the last step is truncated).  Host out[max_new]; *out_n =
 * tokens written; *n_steps = la_step calls.  Any of out_n / n_steps may be NULL.
 * Passage: the generation loop of the autoregressive system that lookahead
 * decoding replaces (paper-graph-ui page, section 3.4, "The autoregressive
 * system"), with one lookahead step per iteration. */
int la_generate(la_handle *h, const int32_t *prompt, int32_t n, int32_t max_new,
                int32_t *out, int32_t *out_n, int32_t *n_steps);

/* Counters since the last prefill (host struct).  generated / steps is the
 * step compression ratio S the pages report (paper-graph-ui page, section 5,
 * "Ablation Studies (Table 3)": tokens per decoding step); the timing fields
 * are this library's own instrumentation, with no passage. */
int la_stats(const la_handle *h, la_stats_t *out);

/* Test and resume utility; the pages have no counterpart.
 * Copy the committed tokens, window and pool to host buffers in *st.
 * Errors: STATE, CAPACITY (a cap too small; n_tokens / n_records still report
 * the sizes needed), CUDA. */
int la_export_state(la_handle *h, la_state_t *st);

/* Test and resume utility; the pages have no counterpart.
 * Replace the state with *st (same N, W): recomputes the prefix KV from the
 * tokens, loads window and pool.  Errors: INVALID_ARG, CAPACITY, CUDA. */
int la_import_state(la_handle *h, const la_state_t *st);

/* Debug utility (no passage): the rows are those the verification and the
 * lookahead branch read (paper-graph-ui page, section 3.4).
 * Logits of the last step's used rows, fp32, to host[rows * vocab]: row 0,
 * then the top lookahead level's W rows, then G*(N-1) candidate rows
 * (candidate c, depth m at 1 + W + c*(N-1) + m-1).  After la_prefill it
 * holds the prompt's last row only (rows = 1).  *rows, *vocab receive the
 * sizes; host may be NULL to query them. */
int la_debug_logits(la_handle *h, float *host, int32_t *rows, int32_t *vocab);

/* Plain bf16 GEMM on the library's tcgen05 kernel:
 *   y[r][f] = sum_k x[r][k] * w[f][k]   (fp32 accumulation, fp32 out)
 * x device bf16 [rows][k], w device bf16 [out][k], y device fp32 [rows][out];
 * all 16-byte aligned, k % 8 == 0, 1 <= rows <= 256.  splits > 1 splits k
 * across CTAs: partial sums go to `workspace` (device fp32, at least
 * splits*rows*out elements, owned by the caller) and are added in a fixed
 * order, so results are deterministic.  splits == 1 needs no workspace
 * (NULL allowed).  stream: cudaStream_t or NULL.  Asynchronous: a bounded
 * wait that gives up inside the kernel is reported by la_gemm_status.
 * Errors: INVALID_ARG, CUDA. */
int la_gemm_bf16(const void *x, const void *w, float *y, int32_t rows, int32_t out, int32_t k,
                 int32_t splits, float *workspace, void *stream);

/* Same GEMM as la_gemm_bf16, for callers that cannot allocate device memory
 * at call time (for example a plugin inside a host framework that owns every
 * device allocation, or a latency-critical loop that must not call cudaMalloc
 * and its implied synchronisation), and so cannot pass a split-K workspace.
 * The paper has no counterpart; this is a library convenience.
 *
 * The partial sums live in a fixed device array inside the library of
 * LA_NOALLOC_SCRATCH_FLOATS floats (16 MiB), which every GPU that loads the
 * library holds until the process exits.  The call allocates nothing.
 * Requires splits * rows * out <= LA_NOALLOC_SCRATCH_FLOATS, else it returns
 * LA_ERR_CAPACITY with nothing launched; other limits as la_gemm_bf16.
 * The first call on each device looks up that array's device address (with
 * the device current); make that first call before any stream capture.
 * The cached address does not survive a cudaDeviceReset in the same process.
 * All calls share the array: calls whose kernels overlap on the GPU (other
 * streams, other threads on the same device) race and must be serialised by
 * the caller.  Asynchronous on `stream`; a bounded wait that gives up inside
 * the kernel is reported by la_gemm_status.
 * Errors: INVALID_ARG, CAPACITY, CUDA. */
#define LA_NOALLOC_SCRATCH_FLOATS (4 * 1024 * 1024)
int la_gemm_bf16_noalloc(const void *x, const void *w, float *y, int32_t rows, int32_t out, int32_t k,
                         int32_t splits, void *stream);

/* Error status of the standalone GEMMs (la_gemm_bf16, la_gemm_bf16_noalloc)
 * on the current device.  Their kernels wait on TMA loads and tensor-core
 * commits with a bounded wait; one that gives up sets a bit in a per-device
 * error word and leaves that call's output incomplete.  This call
 * synchronises `stream` (cudaStream_t or NULL), reads and clears both words,
 * and returns LA_ERR_DEVICE_TIMEOUT if any bit was set since the last status
 * call, else LA_OK.  It allocates nothing.  No passage: library plumbing.
 * Errors: DEVICE_TIMEOUT, CUDA. */
int la_gemm_status(void *stream);

/* Test support for the failure path (no passage).  Launches one CTA that
 * waits, through the same bounded mbarrier wait every kernel here uses, on a
 * barrier that nothing arrives at, with a limit of limit_ns nanoseconds
 * (1e3 .. 2e9) instead of the usual 2 s.  The wait gives up, sets its
 * timeout bit and the kernel returns: nothing faults, traps or hangs.
 *   h != NULL: the bit goes to the handle's error word, on the handle's
 *     stream; the next la_step / la_ar_step then returns
 *     LA_ERR_DEVICE_TIMEOUT and the handle needs la_prefill again.
 *   h == NULL: the bit goes to the error words of la_gemm_bf16 and (once
 *     this device has called it) la_gemm_bf16_noalloc, on `stream`; the next
 *     la_gemm_status reports it.
 * Asynchronous.  Errors: INVALID_ARG (limit), CUDA. */
int la_selftest_timeout(la_handle *h, int64_t limit_ns, void *stream);

/* Test support: the static tables of a step's rows for (N, W, G), as the
 * library builds them at la_create (the mask of section 3.4 "Integrated
 * Forward Pass", Figure 2b, with row 0 the last committed token, window row
 * 1 + k W + j for level k and column j, candidate row 1 + (N-1) W + c (N-1)
 * + m - 1 for candidate c and depth m).  Host only; no GPU is touched.
 * Writes, with M = 1 + (W + G)(N - 1) and U = 1 + W + G (N - 1):
 *   depth[M]     position offset of each row from the prefix length
 *   vis[M][8]    bit s % 32 of word s / 32: row r attends to step row s
 *   used[U]      the rows whose logits the step reads (row 0, the top
 *                window level, every candidate row)
 * and *m_out = M, *u_out = U.  Errors: INVALID_ARG (N < 2, W < 1, G < 0, a
 * null pointer), CAPACITY (M > 256 or M > max_rows; nothing written). */
int la_step_tables(int32_t N, int32_t W, int32_t G, int32_t *depth, uint32_t *vis, int32_t *used, int32_t max_rows,
                   int32_t *m_out, int32_t *u_out);

/* Test support (no passage): the work split of the projection GEMMs,
 * computed on the host; no GPU is touched.  `tiles` output tiles of n_kb
 * k-units each over `ctas` persistent CTAs (CTA pairs on the GPU).
 * whole_first = 0: stream-K (the flattened tile x k-unit work cut into equal
 * contiguous runs); 1: the step gate/up GEMM's split (each CTA first takes
 * an even share of the k-units of the last tiles % ctas tiles, then
 * tiles / ctas whole tiles).  Writes up to max_segs segments as int32
 * (tile, kb0, kb1, plane) quadruples to segs, cta_first[0 .. *ctas_used]
 * (CTA c runs segments cta_first[c] .. cta_first[c + 1] - 1; cta_first must
 * hold ctas + 1 entries) and planes[0 .. tiles) (partial planes per tile;
 * plane p of a tile is its p-th segment in CTA order), and the number of
 * segments to *nseg.  Errors: INVALID_ARG (a size < 1 or a null pointer),
 * CAPACITY (more than max_segs segments; nothing written to segs). */
int la_gemm_schedule(int32_t tiles, int32_t n_kb, int32_t ctas, int32_t whole_first, int32_t *segs,
                     int32_t max_segs, int32_t *nseg, int32_t *cta_first, int32_t *ctas_used, int32_t *planes);

void la_destroy(la_handle *h);
const char *la_strerror(int code);
const char *la_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* LA_H */
