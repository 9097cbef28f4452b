// Host-side interface between the runtime (la_api.cu) and the kernel
// translation units.  Plain C++ structs and launch functions; no torch types.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "la_common.cuh"

namespace la {

// ------------------------------------------------------------------ GEMMs
// y_partial[split][r][col0 + f] = sum over this split's k range of x[r][k] * w_seg[f][k]
// for up to kMaxSeg weight matrices that share the same input rows x.
struct TcGemmParams {
    CUtensorMap a[kMaxSeg];   // weights, bf16 [out][K], box 64 x 128, 128B swizzle
    CUtensorMap b;            // input rows, bf16 [rows][K], box 64 x bn, 128B swizzle
    int nseg;
    int seg_tile0[kMaxSeg + 1];  // first 128-row tile of each segment; [nseg] = total tiles
    int seg_out[kMaxSeg];        // output features of each segment
    int seg_col0[kMaxSeg];       // column of the segment's first feature in the output row
    int n_kb;                    // K / 64 rounded up
    int splits;                  // k-splits (CTAs per tile)
    int nrows;                   // rows stored (<= bn, <= bh when bh > 0)
    int bn;                      // UMMA N: padded rows, multiple of 16, <= 256
    int bh;                      // > 0: B holds hi rows [0, bh) and lo rows [bh, 2bh) = bn; the
                                 //      epilogue adds columns c and c + bh.  0: plain bf16 rows
    int ldo;                     // output row stride (floats)
    int stages;                  // shared-memory pipeline depth
    int nrt;                     // 2-SM kernel: row tiles of 128 rows (1 or 2) multiplied with each weight
                                 //   stage; tile t of the hi (lo) rows starts at row t * 128 (bh + t * 128)
    int sub;                     // 2-SM kernel: 64-column k-blocks per stage (1, or 2 with nrt == 1); the
                                 //   schedule's k units (kb0, kb1, n_kb) are sub * 64 columns wide
    int bnh;                     // 2-SM kernel with nrt == 1: input rows per CTA (hi rows from row 0, lo rows
                                 //   from row bh; UMMA N = 2 bnh, a multiple of 16 rows); 0: gemm2_nhalf(nrt, bh)
    long long split_stride;      // floats between partial planes
    float *out;
    unsigned *err;
    const int4 *segs;            // stream-K segments (tile, kb0, kb1, plane) or nullptr (one split per CTA)
    const int *cta_first;        // [ctas + 1]: CTA c runs segs[cta_first[c] .. cta_first[c+1])
    // Gate/up GEMM with SwiGLU (2-SM kernel, fuse_out set).  a[0] = gate and
    // a[1] = up weights, boxes of 64 rows: CTA rank r of pair tile t holds
    // gate rows f0 .. f0 + 63 in its TMEM lanes 0..63 and the up rows of the
    // same features in lanes 64..127, f0 = 128 t + 64 r.  A tile one segment
    // covers (fuse_np[tile] == 1) goes from TMEM straight to silu(gate) * up,
    // written as (hi, lo) bf16 rows fuse_out[row][f] (+ fuse_lo_off) for f <
    // fuse_F.  A split tile's pieces go to output column 128 (2 t + r) + lane
    // of their partial planes and add 1 to fuse_cnt[tile]; once the count
    // reaches the next multiple of fuse_np[tile] (it is never reset), every
    // contributing CTA adds the planes, in plane order, for its share of the
    // rows (share = its plane) and writes them the same way.
    int *fuse_cnt;
    const int *fuse_np;
    __nv_bfloat16 *fuse_out;
    long long fuse_lo_off;
    int fuse_F;
};

struct TcGemm {
    TcGemmParams p;
    int grid = 0;
    int ctas = 0;                // CTAs (CTA pairs for the 2-SM kernel) of a stream-K schedule
    size_t smem = 0;
    bool pair = false;           // run k_gemm_tc2 (2-SM UMMA, 256-feature tiles, hi/lo rows, bh = 128)
};

struct SimtGemmParams {
    const float *a[kMaxSeg];
    int nseg;
    int seg_f0[kMaxSeg + 1];     // cumulative features
    int seg_col0[kMaxSeg];
    const float *x;
    int ldx;
    int K;
    int nrows;
    int ldo;
    float *out;
};

// Record `msg` as the calling thread's last error (la_last_error) and return `code`.
int set_last_error(int code, const char *msg);

// Tensor-map construction (driver entry point fetched through the runtime).
int make_tmap_bf16(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                   uint32_t box_inner, uint32_t box_outer);

// Number of CTAs of the tcgen05 GEMM that fit on one SM with `stages` at `bn`.
size_t tc_gemm_smem_bytes(int bn, int stages);
int tc_gemm_stages_for(int bn);
int tc_gemm_ctas_per_sm(int bn, int stages);
int choose_splits(int tiles, int n_kb, int slots);
// Stream-K schedule over `ctas` CTAs: segs holds 4 ints per segment.
void stream_k_schedule(int tiles, int n_kb, int ctas, std::vector<int> &segs, std::vector<int> &cta_first,
                       std::vector<int> &tile_planes);
void hybrid_schedule(int tiles, int n_kb, int ctas, std::vector<int> &segs, std::vector<int> &cta_first,
                       std::vector<int> &tile_planes);

// Fill grid/smem of a plan whose params are set.
void tc_gemm_finalize(TcGemm &g);
cudaError_t tc_gemm_launch(const TcGemm &g, cudaStream_t s);
// 2-SM kernel: shared memory, ring depth, and CTA pairs that fit at once.
// Input rows per CTA and row tile of the 2-SM kernel: bh when one row tile
// holds all rows (bh <= 128: a step, the lm_head), else 128-row tiles.
__host__ __device__ inline int gemm2_nhalf(int nrt, int bh) { return nrt == 1 && bh <= kTileM ? bh : kTileM; }
// nhalf: as gemm2_nhalf
size_t tc_gemm2_smem_bytes(int stages, int nrt = 1, int sub = 1, int nhalf = kTileM);
int tc_gemm2_stages(int nrt = 1, int sub = 1, int nhalf = kTileM);   // ring depth (at most 8)
int tc_gemm2_max_pairs();
cudaError_t tc_gemm2_launch(const TcGemm &g, cudaStream_t s);
cudaError_t simt_gemm_launch(const SimtGemmParams &p, int total_f, cudaStream_t s);
// Sum `splits` fp32 partials [split][rows][cols] into y [rows][cols] (fixed order).
cudaError_t reduce_splits_launch(const float *part, int splits, long long stride, int rows, int cols, float *y,
                                 cudaStream_t s);

// One CTA whose bounded mbarrier wait (on a barrier nothing arrives at) gives
// up after limit_ns and ORs ERR_TIMEOUT_SELFTEST into *err (and *err2 if set).
cudaError_t wait_selftest_launch(unsigned *err, unsigned *err2, unsigned long long limit_ns, cudaStream_t s);
// Error word of la_gemm_bf16_noalloc on the current device: its address
// (nullptr while the device has made no call), or read-and-clear on stream s.
cudaError_t noalloc_err_word(unsigned **out);
cudaError_t noalloc_err_take(cudaStream_t s, unsigned *bits);

// ------------------------------------------------------------------ elementwise
// T is the weight type; activations written as T go through store_act
// (fp32, or a bf16 hi/lo pair whose lo plane is lo_off elements later).
template <typename T>
cudaError_t embed_norm_launch(const T *embed, const int *tok, int nrows, int d, const T *gain, float eps, float *h,
                              T *xn, long long lo_off, cudaStream_t s);
// GEMM outputs arrive as fp32 partial planes part[plane][row][col] (plane
// stride sstride, row stride ldp); column col belongs to 128-wide tile
// col >> 7, which has planes[tile] planes (all 1 when planes is null).
// Consumers add them in plane order.
//
// Rotated q (fp32) and the rows' K/V into the fp32 cache at slots P + r;
// q, k, v columns start at 0, k_off, v_off.
cudaError_t qkv_rope_launch(const float *part, const int *planes, long long sstride, int ldp, int nrows, int nh,
                            int nkv, int hd, int k_off, int v_off, const float2 *rope, int P, const int *depth,
                            float *q, float *kc, float *vc, int max_seq, cudaStream_t s);
template <typename T>
cudaError_t resid_norm_launch(float *h, const float *part, const int *planes, long long sstride, int ldp, int d,
                              const T *gain, float eps, const int *row_map, int nrows, T *xout, long long lo_off,
                              cudaStream_t s);
// gate columns [0, F), up columns [up_off, up_off + F).
template <typename T>
cudaError_t swiglu_launch(const float *part, const int *planes, long long sstride, int ldp, int nrows, int F,
                          int up_off, T *out, long long lo_off, cudaStream_t s);
// Sums the lm_head planes into logits[rows][V], then per row the argmax
// (lowest id among equals), the max, and sum exp((l - max) * invT) if invT > 0.
cudaError_t argmax_launch(const float *part, const int *planes, long long sstride, int ldp, float *logits, int rows,
                          int V, float invT, int *amax, float *lmax, float *lsum, int top_k, float top_p,
                          unsigned *thr_key, int *thr_cut, cudaStream_t s);

// ------------------------------------------------------------------ attention
// Keys of row r: the cached prefix [0, P) plus in-step rows.  In tree mode the
// in-step keys of row r are anc[r][0..anc_cnt[r]) (slots P + a, self included);
// in causal mode (anc == nullptr) they are rows 0..r.
struct AttnArgs {
    const float *q;        // [nrows][nh][hd] fp32 (rotated)
    const float *kc;       // this layer's K cache [nkv][max_seq][hd], fp32
    const float *vc;       // V cache, same layout
    int max_seq, P, nrows, nh, nkv, hd;
    float *ws;             // prefix partials [nch][nrows][nh][hd + 4] (out, max, sum, pad)
    int nch;               // prefix chunks = ceil(P / kAttnChunk)
    const int *anc;        // [nrows][anc_stride] or nullptr
    const int *anc_cnt;
    int anc_stride;
    const uint32_t *vis_bits;  // [nrows][8] in-step visibility bits (tree mode) or nullptr (causal)
    void *out;             // [nrows][nh * hd] activations (store_act form)
    long long out_lo_off;  // lo plane offset of `out` (bf16 models)
};
constexpr int kAttnChunk = 64;
// fp32 models: SIMT split-KV (64-key chunks) + per-row in-step pass.
cudaError_t attention_launch(const AttnArgs &a, cudaStream_t s);

// bf16 models: tcgen05 attention that first sums, rotates and splits the
// QKV projection of its own KV head (see the prologue fields below).  One thread-block cluster per (KV head, tile of 128 query
// vectors); its CTAs split the keys [0, P + nrows) in 128-key chunks and
// merge their partial softmax sums through distributed shared memory.
struct AttnUmmaParams {
    CUtensorMap tq;        // q planes as [2 * nkv * qv_pad][hd], box 64 x 128
    CUtensorMap tk;        // K cache as [L * 2 * nkv * seq][hd], box 64 x 128
    CUtensorMap tv;        // V^T cache as [L * 2 * nkv * hd][seq], box 64 x hd
    int layer, nh, nkv, gq, hd, qv_pad, seq;
    int P, nrows, mtiles;
    const int *P_dev;           // if set, P is read from here (device step state) instead
    int prefix_early;           // cache slots < P were written before this launch began (a step,
                                // not a prefill chunk): their K/V loads may start before the wait
    const uint32_t *vis_bits;   // [nrows][8] in-step visibility bits, or nullptr (causal)
    __nv_bfloat16 *out;         // [nrows][nh * hd] hi plane; lo plane out_lo_off later
    long long out_lo_off;
    unsigned *err;
    // Prologue inputs: the QKV GEMM's partial planes ([plane][rows][ldp], q |
    // k | v columns, planes[tile] planes per 128-column tile), the rotary
    // table [pos][hd/2] of (cos, sin) and the step rows' depths (nullptr:
    // row r sits at P + r).  Outputs, all (hi, lo) plane pairs:
    //   q  [2][nkv][qv_pad][hd]   query vector v = row * gq + j of KV head g
    //                             is q head g * gq + j, scaled by 1/sqrt(hd)
    //   kc [L][2][nkv][seq][hd]   rows P + r of layer `layer`
    //   vc [L][2][nkv][hd][seq]   V transposed: columns P + r
    const float *part;
    const int *planes;
    long long sstride;
    int ldp, k_off, v_off, qkv_tiles;   // qkv_tiles: entries of `planes`
    const float2 *rope;
    const int *depth;
    __nv_bfloat16 *q, *kc, *vc;
};
// Fills the tensor maps; false if the driver rejects one.
bool attention_umma_maps(AttnUmmaParams &p, const void *q, const void *kc, const void *vc, int L);
// Launch for nrows rows (fields P or P_dev, nrows, layer, vis_bits set by
// the caller).  The cluster size is picked from the SM count and the largest
// prefix the launch may see (P_max), so one launch configuration serves
// every step of a captured graph.
cudaError_t attention_umma_launch(AttnUmmaParams p, int nsm, int P_max, cudaStream_t s);

// ------------------------------------------------------------------ speculation state
struct SpecState {
    int P;          // committed KV length; o sits at position P
    int o;          // last committed token
    int g;          // candidates found this step
    int A;          // tokens accepted this step
    int cstar;      // winning candidate, -1 if none
    int P_old;      // P at the start of the step
    int n_tokens;   // committed tokens = P + 1
    int acc[8];     // accepted tokens
    unsigned err;   // device error bits
};

enum PoolPolicy { kPoolFifo = 0, kPoolLru = 1, kPoolLfu = 2 };   // la_opts.pool_policy values

struct SpecDev {
    SpecState *st;
    int *tokens_log;      // [max_seq] committed tokens
    int max_seq;
    int *window;          // [N-1][W]
    int *cands;           // [G][N-1]
    int *tok;             // [M] step-row tokens
    const int *amax;      // [U] argmax of used rows
    const float *logits;  // [U][V]
    const float *lmax;    // [U] row max
    const float *lsum;    // [U] sum of exp((l - max) / T) over the tokens kept by top-k / top-p
    const unsigned *thr_key;  // [U] keep rule of each row's sampling distribution (keep_token)
    const int *thr_cut;
    int V;
    int *pkeys, *pcnt, *phead, *pent;  // pool: open-addressed table keyed by first token
    int *puse;            // [slots][cap] use count of each ring entry (LFU order)
    int nslots_log2;
    int cap;
    int policy;           // kPoolFifo, kPoolLru (uses move entries to the most recent end) or kPoolLfu
    int N, W, G, M, U;
    float T;
    unsigned long long seed;
    int *step_zero;       // [n_step_zero] counts the step's kernels start from 0 (gate/up arrivals), or nullptr
    int n_step_zero;
};

cudaError_t build_rows_launch(const SpecDev &d, cudaStream_t s);
cudaError_t finish_step_launch(const SpecDev &d, cudaStream_t s);
cudaError_t kv_commit_launch(const SpecDev &d, float *cache, int L, int nkv, int hd, cudaStream_t s);
// Same for the bf16 plane layouts (K rows, V^T columns).
cudaError_t kv_commit_split_launch(const SpecDev &d, __nv_bfloat16 *kc, __nv_bfloat16 *vc, int L, int nkv, int hd,
                                   int seq, cudaStream_t s);
// Insert n records [n][N] (key, suffix) in order, one warp, sequential
// semantics; uses (or nullptr: 0) gives each record's LFU use count.
cudaError_t pool_insert_launch(const SpecDev &d, const int *records, const int *uses, int n, cudaStream_t s);
// Insert the prompt's n-grams (tokens_log[0..n)) in ascending start position.
cudaError_t pool_seed_prompt_launch(const SpecDev &d, int n, cudaStream_t s);
// Prefill's first token: argmax or a draw at (position n, draw 0); appends to the log.
cudaError_t first_token_launch(const SpecDev &d, int n, cudaStream_t s);

}  // namespace la
