// Host-side interface between the runtime (la_api.cu) and the kernel
// translation units.  Plain C++ structs and launch functions; no torch types.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

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
    int nrows;                   // rows stored (<= bn)
    int bn;                      // UMMA N: padded rows, multiple of 16, <= 256
    int ldo;                     // output row stride (floats)
    int stages;                  // shared-memory pipeline depth
    long long split_stride;      // floats between split partials
    float *out;
    unsigned *err;
};

struct TcGemm {
    TcGemmParams p;
    int grid = 0;
    size_t smem = 0;
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

// Fill grid/smem of a plan whose params are set.
void tc_gemm_finalize(TcGemm &g);
cudaError_t tc_gemm_launch(const TcGemm &g, cudaStream_t s);
cudaError_t simt_gemm_launch(const SimtGemmParams &p, int total_f, cudaStream_t s);
// Sum `splits` fp32 partials [split][rows][cols] into y [rows][cols] (fixed order).
cudaError_t reduce_splits_launch(const float *part, int splits, long long stride, int rows, int cols, float *y,
                                 cudaStream_t s);

// ------------------------------------------------------------------ elementwise
template <typename T>
cudaError_t embed_norm_launch(const T *embed, const int *tok, int nrows, int d, const T *gain, float eps, float *h,
                              T *xn, cudaStream_t s);
template <typename T>
cudaError_t qkv_rope_launch(const float *part, int S, long long sstride, int ldp, int nrows, int nh, int nkv, int hd,
                            const float2 *rope, int P, const int *depth, float *q, T *kc, T *vc, int max_seq,
                            cudaStream_t s);
template <typename T>
cudaError_t resid_norm_launch(float *h, const float *part, int S, long long sstride, int ldp, int d, const T *gain,
                              float eps, const int *row_map, int nrows, T *xout, cudaStream_t s);
template <typename T>
cudaError_t swiglu_launch(const float *part, int S, long long sstride, int ldp, int nrows, int F, T *out,
                          cudaStream_t s);
cudaError_t argmax_launch(const float *logits, int rows, int V, float invT, int *amax, float *lmax, float *lsum,
                          cudaStream_t s);

// ------------------------------------------------------------------ attention
// Keys of row r: the cached prefix [0, P) plus in-step rows.  In tree mode the
// in-step keys of row r are anc[r][0..anc_cnt[r]) (slots P + a, self included);
// in causal mode (anc == nullptr) they are rows 0..r.
struct AttnArgs {
    const float *q;        // [nrows][nh][hd] fp32 (rotated)
    const void *kc;        // this layer's K cache [nkv][max_seq][hd]
    const void *vc;        // V cache, same layout
    int max_seq, P, nrows, nh, nkv, hd;
    float *ws;             // prefix partials [nch][nrows][nh][hd + 4] (out, max, sum, pad)
    int nch;               // prefix chunks = ceil(P / kAttnChunk)
    const int *anc;        // [nrows][anc_stride] or nullptr
    const int *anc_cnt;
    int anc_stride;
    void *out;             // [nrows][nh * hd] activations
};
constexpr int kAttnChunk = 64;
template <typename T>
cudaError_t attention_launch(const AttnArgs &a, cudaStream_t s);

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
    const float *lsum;    // [U] sum of exp((l - max) / T)
    int V;
    int *pkeys, *pcnt, *phead, *pent;  // pool: open-addressed table keyed by first token
    int nslots_log2;
    int cap;
    int N, W, G, M, U;
    float T;
    unsigned long long seed;
};

cudaError_t build_rows_launch(const SpecDev &d, cudaStream_t s);
cudaError_t finish_step_launch(const SpecDev &d, cudaStream_t s);
template <typename T>
cudaError_t kv_commit_launch(const SpecDev &d, T *cache, int L, int nkv, int hd, cudaStream_t s);
// Insert n records [n][N] (key, suffix) in order, one warp, sequential semantics.
cudaError_t pool_insert_launch(const SpecDev &d, const int *records, int n, cudaStream_t s);
// Insert the prompt's n-grams (tokens_log[0..n)) in ascending start position.
cudaError_t pool_seed_prompt_launch(const SpecDev &d, int n, cudaStream_t s);
// Prefill's first token: argmax or a draw at (position n, draw 0); appends to the log.
cudaError_t first_token_launch(const SpecDev &d, int n, cudaStream_t s);

}  // namespace la
