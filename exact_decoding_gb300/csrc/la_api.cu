// Host runtime behind include/la.h: the handle, its device buffers, the GEMM
// launch plans and the orchestration of prefill and of one lookahead step
// (paper-graph-ui page, section 3.4: lookahead branch + verification branch
// + pool update in one forward pass).  Everything that touches step data
// runs in the kernels of this library on the caller's stream; the host only
// sequences launches (after the first step: replays one captured CUDA graph
// per step) and copies the step's accepted tokens back.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/la.h"
#include "abi_guard.h"
#include "la_kernels.h"

using namespace la;

namespace {

thread_local std::string g_last_error;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

#define CK(call)                                                                                          \
    do {                                                                                                  \
        cudaError_t e_ = (call);                                                                          \
        if (e_ != cudaSuccess) return fail(LA_ERR_CUDA, "%s: %s (%s:%d)", #call, cudaGetErrorString(e_), \
                                           __FILE__, __LINE__);                                           \
    } while (0)

// Prompt rows per prefill pass.  Each pass streams every weight once; the
// 2-SM GEMM multiplies each weight stage with two 128-row tiles of them.
constexpr int kArRows = 16;      // rows of a one-row forward's GEMM input boxes
constexpr int kPrefillRows = 256;
// 64-column k-blocks per ring stage of a step's GEMMs (2: each weight row is
// read 256 contiguous bytes at a time).  Prefill passes use one.
constexpr int kStepSub = 2;

enum Mode { STEP = 0, PREFILL = 1 };
enum Kind { QKV = 0, OPROJ = 1, GATEUP = 2, DOWN = 3 };

int round_up(int x, int m) { return (x + m - 1) / m * m; }

}  // namespace

int la::set_last_error(int code, const char *msg) { return fail(code, "%s", msg); }

struct la_handle {
    la_model_dims dims{};
    la_opts opts{};
    cudaStream_t stream = nullptr;
    bool bf16 = true;
    int L = 0, d = 0, nh = 0, nkv = 0, hd = 0, F = 0, V = 0, qd = 0, kvd = 0, qkv_out = 0;
    int N = 0, W = 0, G = 0, M = 0, U = 0, cap = 0, max_seq = 0, R = 0;
    int Rp[2] = {0, 0};   // rows per GEMM partial plane: a step's rows, a prefill pass's rows
    int bn_step = 0, bn_pf = 0, bn_u = 0;
    // bf16 models: GEMM inputs are bf16 hi/lo planes, hi rows [0, bh), lo rows [bh, 2 bh)
    int bh_step = 0, bh_pf = 0, bh_u = 0;
    int act_rows = 0;   // rows of each activation buffer
    size_t act = 4;     // bytes per activation element

    // caller's weights
    const void *embed = nullptr, *final_norm = nullptr, *lm_head = nullptr;
    std::vector<const void *> attn_norm, wq, wk, wv, wo, ffn_norm, wg, wu, wd;

    // device buffers (owned)
    std::vector<void *> allocs;
    float *h = nullptr, *part = nullptr, *q = nullptr, *logits = nullptr, *lmax = nullptr, *lsum = nullptr;
    float *attn_ws = nullptr;
    void *xn = nullptr, *ao = nullptr, *fa = nullptr, *xu = nullptr, *cache = nullptr;
    // bf16 models: q planes [2][nkv][qv_pad][hd], K planes [L][2][nkv][seq][hd]
    // and V^T planes [L][2][nkv][hd][seq] (cache = K then V^T); seq =
    // max_seq rounded up to 64 slots.
    __nv_bfloat16 *qs = nullptr, *kcs = nullptr, *vcs = nullptr;
    int qv_pad = 0, seq = 0, nsm = 0;
    AttnUmmaParams attn_proto{};
    float2 *rope = nullptr;
    int *amax = nullptr, *tok = nullptr, *depth = nullptr, *anc = nullptr, *anc_cnt = nullptr, *used = nullptr;
    unsigned *thr_key = nullptr;   // [U] sampling keep rule of each used row (top-k / top-p)
    int *thr_cut = nullptr;
    int *iota = nullptr;
    uint32_t *vis_bits = nullptr;   // [M][8] in-step visibility bits
    int anc_stride = 0;
    SpecState *st = nullptr;
    SpecState *st_host = nullptr;   // pinned
    int *tokens_log = nullptr, *window = nullptr, *cands = nullptr;
    int *pkeys = nullptr, *pcnt = nullptr, *phead = nullptr, *pent = nullptr, *puse = nullptr;
    int nslots_log2 = 0;
    int *records_dev = nullptr, *uses_dev = nullptr;
    size_t records_dev_cap = 0, uses_dev_cap = 0;

    // GEMM plans (bf16): [mode][kind][layer]
    std::vector<TcGemm> plan[2][4];
    // One-row forwards (la_ar_step): the prefill plans with 16-row input
    // boxes (UMMA N = 32); same schedules, so the same partial planes.
    std::vector<TcGemm> plan_ar[4];
    TcGemm plan_lm;
    // Column layout of the GEMM partials: every matrix starts on a 128-column
    // tile boundary, so column c belongs to tile c >> 7.
    int tq = 0, tk = 0, tg = 0, td = 0, tv = 0;       // tiles of q, k (= v), gate (= up), d, vocab
    int ldo[4] = {0, 0, 0, 0}, ldo_lm = 0;
    int k_off = 0, v_off = 0, up_off = 0;
    // Per-tile partial-plane counts of each stream-K schedule ([mode][kind]);
    // null on the fp32 path (one plane).
    int *planes[2][4] = {{nullptr, nullptr, nullptr, nullptr}, {nullptr, nullptr, nullptr, nullptr}};
    // Step gate/up GEMM with SwiGLU in its epilogue: arrival count per
    // 128-column tile (zero between launches).
    bool fuse_swiglu = false;
    int *fuse_cnt = nullptr;
    int fuse_tiles = 0;
    int *planes_lm = nullptr;
    float *lm_part = nullptr;
    long long lm_stride = 0;
    size_t part_elems = 0, lm_part_elems = 0;

    // profiling (la_opts.profile): event pairs around GEMM / attention launches
    bool prof_on = false;
    std::vector<cudaEvent_t> ev;
    std::vector<int> ev_cls;
    std::vector<double> ev_bytes;
    int ev_used = 0;
    // classes: 0 GEMM, 1 attention, 2 row-wise kernels, 3 speculation kernels
    double prof_ms[4] = {0, 0, 0, 0}, prof_bytes[4] = {0, 0, 0, 0};
    int64_t prof_launches[4] = {0, 0, 0, 0};
    int64_t launches = 0;

    // Captured step (non-profiled steps after the first): every launch of
    // la_step plus the state read-back, replayed with one cudaGraphLaunch.
    cudaGraphExec_t step_graph = nullptr;
    bool graph_off = false;      // capture failed once: launch directly
    int64_t graph_launches = 0;  // kernels per replay

    // host-side bookkeeping
    bool prefilled = false;
    int P = 0;
    int64_t steps = 0, generated = 0;
    int64_t h2d_bytes = 0, d2h_bytes = 0;   // host <-> device copies since la_prefill
    int last_A = 0, last_g = 0, logits_rows = 0;

    ~la_handle() {
        if (step_graph) cudaGraphExecDestroy(step_graph);
        for (cudaEvent_t e : ev) cudaEventDestroy(e);
        for (void *p : allocs) cudaFree(p);
        if (st_host) cudaFreeHost(st_host);
    }

    template <typename T>
    int alloc(T **p, size_t n) {
        void *v = nullptr;
        if (n == 0) n = 1;
        cudaError_t e = cudaMalloc(&v, n * sizeof(T));
        if (e != cudaSuccess) return fail(LA_ERR_OOM, "cudaMalloc(%zu bytes): %s", n * sizeof(T), cudaGetErrorString(e));
        allocs.push_back(v);
        *p = static_cast<T *>(v);
        return LA_OK;
    }
    int alloc_bytes(void **p, size_t bytes) {
        void *v = nullptr;
        cudaError_t e = cudaMalloc(&v, bytes ? bytes : 1);
        if (e != cudaSuccess) return fail(LA_ERR_OOM, "cudaMalloc(%zu bytes): %s", bytes, cudaGetErrorString(e));
        allocs.push_back(v);
        *p = v;
        return LA_OK;
    }

    SpecDev spec() const {
        SpecDev s{};
        s.st = st;
        s.tokens_log = tokens_log;
        s.max_seq = max_seq;
        s.window = window;
        s.cands = cands;
        s.tok = tok;
        s.amax = amax;
        s.logits = logits;
        s.lmax = lmax;
        s.lsum = lsum;
        s.thr_key = thr_key;
        s.thr_cut = thr_cut;
        s.V = V;
        s.pkeys = pkeys;
        s.pcnt = pcnt;
        s.phead = phead;
        s.pent = pent;
        s.nslots_log2 = nslots_log2;
        s.cap = cap;
        s.puse = puse;
        s.policy = opts.pool_policy == LA_POOL_LRU ? kPoolLru : opts.pool_policy == LA_POOL_LFU ? kPoolLfu : kPoolFifo;
        s.N = N;
        s.W = W;
        s.G = G;
        s.M = M;
        s.U = U;
        s.T = opts.temperature;
        s.seed = opts.seed;
        s.step_zero = fuse_cnt;
        s.n_step_zero = fuse_cnt ? fuse_tiles : 0;
        return s;
    }

    // Start a profiled launch: returns the event-pair slot, or -1 when off.
    int prof_begin() {
        if (!prof_on) return -1;
        if (ev_used * 2 + 2 > static_cast<int>(ev.size())) {
            for (int i = 0; i < 64; ++i) {
                cudaEvent_t e;
                if (cudaEventCreate(&e) != cudaSuccess) return -1;
                ev.push_back(e);
            }
            ev_cls.resize(ev.size() / 2);
            ev_bytes.resize(ev.size() / 2);
        }
        const int i = ev_used++;
        cudaEventRecord(ev[2 * i], stream);
        return i;
    }
    void prof_end(int i, int cls, double bytes) {
        if (i < 0) return;
        cudaEventRecord(ev[2 * i + 1], stream);
        ev_cls[i] = cls;
        ev_bytes[i] = bytes;
    }
    // After the stream is synchronised: fold the recorded pairs into the totals.
    void prof_collect() {
        for (int i = 0; i < ev_used; ++i) {
            float ms = 0.f;
            if (cudaEventElapsedTime(&ms, ev[2 * i], ev[2 * i + 1]) == cudaSuccess) {
                prof_ms[ev_cls[i]] += ms;
                prof_bytes[ev_cls[i]] += ev_bytes[i];
                prof_launches[ev_cls[i]] += 1;
            }
        }
        ev_used = 0;
    }

    // K (which = 0) or V (1) cache of layer l: fp32 [nkv][max_seq][hd].
    float *kv_layer(int l, int which) const {
        const size_t plane = static_cast<size_t>(nkv) * max_seq * hd;
        return static_cast<float *>(cache) + (static_cast<size_t>(l) * 2 + which) * plane;
    }
    int bh(int mode) const { return mode == 0 ? bh_step : bh_pf; }
};

namespace {

// ------------------------------------------------------------------ step-row structure
// Parent of each step row (reading of Figure 2b): (0,0) -> row 0, (0,j) ->
// (0,j-1), (k>=1,j) -> (k-1,j), (c,1) -> row 0, (c,m) -> (c,m-1).
void step_structure(int N, int W, int G, std::vector<int> &parent, std::vector<int> &depth) {
    const int L = N - 1, M = 1 + (W + G) * L;
    parent.assign(M, -1);
    depth.assign(M, 0);
    for (int k = 0; k < L; ++k)
        for (int j = 0; j < W; ++j) {
            const int r = 1 + k * W + j;
            parent[r] = k == 0 ? (j == 0 ? 0 : r - 1) : r - W;
            depth[r] = 1 + j + k;
        }
    for (int c = 0; c < G; ++c)
        for (int m = 1; m <= L; ++m) {
            const int r = 1 + L * W + c * L + (m - 1);
            parent[r] = m == 1 ? 0 : r - 1;
            depth[r] = m;
        }
}

// Static tables of a step's rows: depth (position offset from the prefix
// length), the 256-bit visibility word of each row (bit s of word s / 32: the
// row attends to step row s, i.e. s is the row itself or one of its
// ancestors) and the rows whose logits the step reads (row 0, the top window
// level, every candidate row).
void step_tables(int N, int W, int G, std::vector<int> &depth, std::vector<uint32_t> &bits, std::vector<int> &used) {
    std::vector<int> parent;
    step_structure(N, W, G, parent, depth);
    const int M = static_cast<int>(parent.size());
    bits.assign(static_cast<size_t>(M) * 8, 0u);
    for (int r = 0; r < M; ++r)
        for (int x = r; x >= 0; x = parent[x]) bits[static_cast<size_t>(r) * 8 + x / 32] |= 1u << (x % 32);
    used.assign(1, 0);
    for (int j = 0; j < W; ++j) used.push_back(1 + (N - 2) * W + j);
    for (int c = 0; c < G; ++c)
        for (int m = 1; m < N; ++m) used.push_back(1 + (N - 1) * W + c * (N - 1) + (m - 1));
}

uint64_t splitmix64(uint64_t x) {
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

// ------------------------------------------------------------------ GEMM dispatch
// Algorithmic bytes of one projection launch: its weights, read once.  The
// input rows and outputs (about 2% of the weight bytes at M = 121) and the
// extra precision planes are not counted.
double gemm_bytes(const la_handle *h, Kind kind, int nrows) {
    (void)nrows;
    const int K = kind == OPROJ ? h->qd : kind == DOWN ? h->F : h->d;
    const int out = kind == QKV ? h->qkv_out : kind == GATEUP ? 2 * h->F : h->d;
    return static_cast<double>(out) * K * h->act;
}

int run_gemm(la_handle *h, Mode mode, Kind kind, int l, int nrows) {
    const int ldo = h->ldo[kind];
    h->launches += 1;
    const int pe = mode == STEP ? h->prof_begin() : -1;
    if (h->bf16) {
        const bool one_row = mode == PREFILL && nrows <= kArRows;
        TcGemm g = one_row ? h->plan_ar[kind][l] : h->plan[mode][kind][l];
        g.p.nrows = nrows;
        if (mode == PREFILL && !one_row) {   // one or two 128-row tiles per weight stage
            g.p.nrt = nrows > kTileM ? 2 : 1;
            tc_gemm_finalize(g);
        }
        CK(tc_gemm_launch(g, h->stream));
        h->prof_end(pe, 0, gemm_bytes(h, kind, nrows));
        return LA_OK;
    }
    SimtGemmParams p{};
    int K = h->d;
    const void *x = h->xn;
    if (kind == QKV) {
        p.nseg = 3;
        p.a[0] = static_cast<const float *>(h->wq[l]);
        p.a[1] = static_cast<const float *>(h->wk[l]);
        p.a[2] = static_cast<const float *>(h->wv[l]);
        const int outs[3] = {h->qd, h->kvd, h->kvd};
        const int col0[3] = {0, h->k_off, h->v_off};
        int acc = 0;
        for (int i = 0; i < 3; ++i) {
            p.seg_f0[i] = acc;
            p.seg_col0[i] = col0[i];
            acc += outs[i];
        }
        p.seg_f0[3] = acc;
    } else if (kind == GATEUP) {
        p.nseg = 2;
        p.a[0] = static_cast<const float *>(h->wg[l]);
        p.a[1] = static_cast<const float *>(h->wu[l]);
        p.seg_f0[0] = 0;
        p.seg_col0[0] = 0;
        p.seg_f0[1] = h->F;
        p.seg_col0[1] = h->up_off;
        p.seg_f0[2] = 2 * h->F;
    } else {
        p.nseg = 1;
        p.a[0] = static_cast<const float *>(kind == OPROJ ? h->wo[l] : h->wd[l]);
        p.seg_f0[0] = 0;
        p.seg_col0[0] = 0;
        p.seg_f0[1] = h->d;
        K = kind == OPROJ ? h->qd : h->F;
        x = kind == OPROJ ? h->ao : h->fa;
    }
    p.x = static_cast<const float *>(x);
    p.ldx = K;
    p.K = K;
    p.nrows = nrows;
    p.ldo = ldo;
    p.out = h->part;
    CK(simt_gemm_launch(p, p.seg_f0[p.nseg], h->stream));
    h->prof_end(pe, 0, gemm_bytes(h, kind, nrows));
    return LA_OK;
}

int run_lm_head(la_handle *h, int nrows, bool step) {
    h->launches += 1;
    const int pe = step ? h->prof_begin() : -1;
    const double bytes = static_cast<double>(h->V) * h->d * h->act;   // the lm_head, read once
    if (h->bf16) {
        TcGemm g = h->plan_lm;
        g.p.nrows = nrows;
        CK(tc_gemm_launch(g, h->stream));
        h->prof_end(pe, 0, bytes);
        return LA_OK;
    }
    SimtGemmParams p{};
    p.nseg = 1;
    p.a[0] = static_cast<const float *>(h->lm_head);
    p.seg_f0[0] = 0;
    p.seg_f0[1] = h->V;
    p.seg_col0[0] = 0;
    p.x = static_cast<const float *>(h->xu);
    p.ldx = h->d;
    p.K = h->d;
    p.nrows = nrows;
    p.ldo = h->ldo_lm;
    p.out = h->lm_part;
    CK(simt_gemm_launch(p, h->V, h->stream));
    h->prof_end(pe, 0, bytes);
    return LA_OK;
}

// ------------------------------------------------------------------ decoder forward
// Runs nrows rows (tokens at `tok`) through all layers with prefix length P.
// Step mode: positions P + depth[r], in-step keys from the ancestor table,
// final norm of the used rows into xu.  Prefill mode: positions P + r,
// causal in-step keys, final norm of the last row into xu row 0 when
// `final_rows` > 0.
template <typename T>
int forward(la_handle *h, Mode mode, const int *tok, int nrows, int P, bool want_logits) {
    cudaStream_t s = h->stream;
    const float eps = h->dims.rms_eps;
    h->launches += 1;
    const long long bh = h->bh(mode);
    int pe = mode == STEP ? h->prof_begin() : -1;
    CK(embed_norm_launch<T>(static_cast<const T *>(h->embed), tok, nrows, h->d,
                            static_cast<const T *>(h->attn_norm[0]), eps, h->h, static_cast<T *>(h->xn), bh * h->d,
                            s));
    h->prof_end(pe, 2, 0.0);
    const int nch = (P + kAttnChunk - 1) / kAttnChunk;
    for (int l = 0; l < h->L; ++l) {
        int rc;
        if ((rc = run_gemm(h, mode, QKV, l, nrows)) != LA_OK) return rc;
        const long long ss_qkv = static_cast<long long>(h->Rp[mode]) * h->ldo[QKV];
        // Algorithmic bytes of one attention launch: the prefix and step K/V
        // once at the weights' element size (the hi/lo planes double that).
        const double attn_bytes = (2.0 * P * h->kvd + 2.0 * nrows * h->kvd) * h->act;
        if (h->bf16) {
            AttnUmmaParams ap = h->attn_proto;
            ap.part = h->part;
            ap.planes = h->planes[mode][QKV];
            ap.sstride = ss_qkv;
            ap.ldp = h->ldo[QKV];
            ap.depth = mode == STEP ? h->depth : nullptr;
            ap.P_dev = mode == STEP ? &h->st->P : nullptr;   // steps may replay from a captured graph
            ap.prefix_early = mode == STEP ? 1 : 0;
            ap.layer = l;
            ap.P = P;
            ap.nrows = nrows;
            ap.vis_bits = mode == STEP ? h->vis_bits : nullptr;
            ap.out_lo_off = bh * h->qd;
            pe = mode == STEP ? h->prof_begin() : -1;
            CK(attention_umma_launch(ap, h->nsm, mode == STEP ? h->max_seq : P, s));
            h->prof_end(pe, 1, attn_bytes);
            h->launches += 1;   // attention (rotary prologue included)
        } else {
        pe = mode == STEP ? h->prof_begin() : -1;
        CK(qkv_rope_launch(h->part, h->planes[mode][QKV], ss_qkv, h->ldo[QKV], nrows, h->nh, h->nkv, h->hd,
                           h->k_off, h->v_off, h->rope, P, mode == STEP ? h->depth : nullptr, h->q,
                           h->kv_layer(l, 0), h->kv_layer(l, 1), h->max_seq, s));
        h->prof_end(pe, 2, 0.0);
        AttnArgs a{};
        a.q = h->q;
        a.kc = h->kv_layer(l, 0);
        a.vc = h->kv_layer(l, 1);
        a.max_seq = h->max_seq;
        a.P = P;
        a.nrows = nrows;
        a.nh = h->nh;
        a.nkv = h->nkv;
        a.hd = h->hd;
        a.ws = h->attn_ws;
        a.nch = nch;
        a.anc = mode == STEP ? h->anc : nullptr;
        a.anc_cnt = mode == STEP ? h->anc_cnt : nullptr;
        a.anc_stride = h->anc_stride;
        a.vis_bits = mode == STEP ? h->vis_bits : nullptr;
        a.out = h->ao;
        a.out_lo_off = bh * h->qd;
        pe = mode == STEP ? h->prof_begin() : -1;
        CK(attention_launch(a, s));
        h->prof_end(pe, 1, attn_bytes);
        h->launches += 2 + (nch > 0 ? 1 : 0);   // qkv_rope, attention passes
        }
        if ((rc = run_gemm(h, mode, OPROJ, l, nrows)) != LA_OK) return rc;
        const long long ss_d = static_cast<long long>(h->Rp[mode]) * h->ldo[OPROJ];
        pe = mode == STEP ? h->prof_begin() : -1;
        CK(resid_norm_launch<T>(h->h, h->part, h->planes[mode][OPROJ], ss_d, h->ldo[OPROJ], h->d,
                                static_cast<const T *>(h->ffn_norm[l]), eps, nullptr, nrows,
                                static_cast<T *>(h->xn), bh * h->d, s));
        h->prof_end(pe, 2, 0.0);
        if ((rc = run_gemm(h, mode, GATEUP, l, nrows)) != LA_OK) return rc;
        const long long ss_gu = static_cast<long long>(h->Rp[mode]) * h->ldo[GATEUP];
        if (!(mode == STEP && h->fuse_swiglu)) {   // else the gate/up GEMM wrote fa
            pe = mode == STEP ? h->prof_begin() : -1;
            CK(swiglu_launch<T>(h->part, h->planes[mode][GATEUP], ss_gu, h->ldo[GATEUP], nrows, h->F, h->up_off,
                                static_cast<T *>(h->fa), bh * h->F, s));
            h->prof_end(pe, 2, 0.0);
            h->launches += 1;   // swiglu
        }
        h->launches += 2;   // resid_norm after O, resid_norm after down
        if ((rc = run_gemm(h, mode, DOWN, l, nrows)) != LA_OK) return rc;
        const long long ss_dn = static_cast<long long>(h->Rp[mode]) * h->ldo[DOWN];
        pe = mode == STEP ? h->prof_begin() : -1;
        if (l + 1 < h->L) {
            CK(resid_norm_launch<T>(h->h, h->part, h->planes[mode][DOWN], ss_dn, h->ldo[DOWN], h->d,
                                    static_cast<const T *>(h->attn_norm[l + 1]), eps, nullptr, nrows,
                                    static_cast<T *>(h->xn), bh * h->d, s));
        } else if (want_logits) {
            const int *map = mode == STEP ? h->used : h->iota + (nrows - 1);
            const int rows = mode == STEP ? h->U : 1;
            CK(resid_norm_launch<T>(h->h, h->part, h->planes[mode][DOWN], ss_dn, h->ldo[DOWN], h->d,
                                    static_cast<const T *>(h->final_norm), eps, map, rows,
                                    static_cast<T *>(h->xu), static_cast<long long>(h->bh_u) * h->d, s));
        }
        h->prof_end(pe, 2, 0.0);
    }
    return LA_OK;
}

int forward_any(la_handle *h, Mode mode, const int *tok, int nrows, int P, bool want_logits) {
    return h->bf16 ? forward<__nv_bfloat16>(h, mode, tok, nrows, P, want_logits)
                   : forward<float>(h, mode, tok, nrows, P, want_logits);
}

int kv_commit(la_handle *h) {
    if (h->bf16)
        CK(kv_commit_split_launch(h->spec(), h->kcs, h->vcs, h->L, h->nkv, h->hd, h->seq, h->stream));
    else
        CK(kv_commit_launch(h->spec(), static_cast<float *>(h->cache), h->L, h->nkv, h->hd, h->stream));
    return LA_OK;
}

int check_device_error(la_handle *h) {
    if (h->st_host->err) {
        const unsigned e = h->st_host->err;
        h->prefilled = false;
        // A gate/up launch whose waits gave up may have left arrival counts
        // (the next step's row build also clears them).
        if (h->fuse_cnt) cudaMemsetAsync(h->fuse_cnt, 0, sizeof(int) * h->fuse_tiles, h->stream);
        return fail(LA_ERR_DEVICE_TIMEOUT, "device error bits 0x%x (bounded wait gave up or pool full)", e);
    }
    return LA_OK;
}

// KV of tokens_log[0 .. n) in prefill chunks; logits of the last row if asked.
int run_prefix(la_handle *h, int n, bool want_logits) {
    for (int c0 = 0; c0 < n; c0 += kPrefillRows) {
        const int rows = std::min(kPrefillRows, n - c0);
        const bool last = c0 + rows >= n;
        int rc = forward_any(h, PREFILL, h->tokens_log + c0, rows, c0, want_logits && last);
        if (rc != LA_OK) return rc;
    }
    if (want_logits) {
        int rc = run_lm_head(h, 1, false);
        if (rc != LA_OK) return rc;
        CK(argmax_launch(h->lm_part, h->planes_lm, h->lm_stride, h->ldo_lm, h->logits, 1, h->V,
                         h->opts.temperature > 0.f ? 1.f / h->opts.temperature : 0.f, h->amax,
                         h->lmax, h->lsum, h->opts.top_k, h->opts.top_p, h->thr_key, h->thr_cut, h->stream));
    }
    return LA_OK;
}

int reset_pool(la_handle *h) {
    const size_t nslots = static_cast<size_t>(1) << h->nslots_log2;
    CK(cudaMemsetAsync(h->pkeys, 0xFF, nslots * sizeof(int), h->stream));
    CK(cudaMemsetAsync(h->pcnt, 0, nslots * sizeof(int), h->stream));
    CK(cudaMemsetAsync(h->phead, 0, nslots * sizeof(int), h->stream));
    return LA_OK;
}

// Uploads one stream-K schedule over tile groups (tp consecutive 128-row
// weight tiles of one matrix: a 256-feature tile of the 2-SM kernel when
// tp = 2); returns per-128-column-tile plane counts for the consumers, the
// max plane count and each matrix's first group.
int upload_schedule(la_handle *h, const int *tiles, int nseg, int tp, int n_kb, int ctas, TcGemm &g,
                    int **planes_dev, int *max_planes, int *group0, bool whole_first = false) {
    int ngroups = 0;
    for (int i = 0; i < nseg; ++i) {
        group0[i] = ngroups;
        ngroups += (tiles[i] + tp - 1) / tp;
    }
    group0[nseg] = ngroups;
    std::vector<int> segs, first, gplanes;
    if (whole_first) hybrid_schedule(ngroups, n_kb, ctas, segs, first, gplanes);
    else stream_k_schedule(ngroups, n_kb, ctas, segs, first, gplanes);
    std::vector<int> planes;   // per 128-column tile, in column order
    for (int i = 0; i < nseg; ++i)
        for (int t = 0; t < tiles[i]; ++t) planes.push_back(gplanes[group0[i] + t / tp]);
    int *dsegs = nullptr, *dfirst = nullptr, *dplanes = nullptr;
    int rc;
    if ((rc = h->alloc(&dsegs, segs.size())) != LA_OK || (rc = h->alloc(&dfirst, first.size())) != LA_OK ||
        (rc = h->alloc(&dplanes, planes.size())) != LA_OK)
        return rc;
    CK(cudaMemcpy(dsegs, segs.data(), segs.size() * sizeof(int), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dfirst, first.data(), first.size() * sizeof(int), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dplanes, planes.data(), planes.size() * sizeof(int), cudaMemcpyHostToDevice));
    g.p.segs = reinterpret_cast<const int4 *>(dsegs);
    g.p.cta_first = dfirst;
    g.ctas = static_cast<int>(first.size()) - 1;
    *planes_dev = dplanes;
    *max_planes = *std::max_element(gplanes.begin(), gplanes.end());
    return LA_OK;
}

int build_plans(la_handle *h) {
    int dev = 0;
    CK(cudaGetDevice(&dev));
    // SwiGLU in the step's gate/up GEMM epilogue (rows of 4-feature groups).
    h->fuse_swiglu = h->F % 4 == 0;
    if (h->fuse_swiglu) {
        h->fuse_tiles = 2 * h->tg;
        int rc = h->alloc(&h->fuse_cnt, static_cast<size_t>(h->fuse_tiles));
        if (rc != LA_OK) return rc;
        CK(cudaMemset(h->fuse_cnt, 0, sizeof(int) * h->fuse_tiles));
    }
    int nsm = 0;
    CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
    const int bhs[2] = {h->bh_step, h->bh_pf};
    void *xs[4] = {h->xn, h->ao, h->xn, h->fa};
    const int Ks[4] = {h->d, h->qd, h->d, h->F};
    size_t part_max = 0;
    // 2-SM UMMA over 256-feature tiles, one CTA pair per two SMs.
    int pairs = std::min(nsm / 2, tc_gemm2_max_pairs());
    if (pairs < 1) return fail(LA_ERR_CUDA, "no CTA pair of the 2-SM GEMM fits on this device");
    for (int mode = 0; mode < 2; ++mode) {
        const int bhm = bhs[mode];
        const int bn = 2 * bhm;             // hi rows + lo rows
        for (int kind = 0; kind < 4; ++kind) {
            const int K = Ks[kind];
            const bool fuse = h->fuse_swiglu && mode == STEP && kind == GATEUP;
            CUtensorMap bmap;
            // box: a CTA's input rows of one row tile (bh in a step, 128 per tile in a prefill pass)
            if (make_tmap_bf16(&bmap, xs[kind], K, bn, static_cast<uint64_t>(K) * 2, kBlockK,
                               mode == STEP ? bhm : kTileM))
                return fail(LA_ERR_CUDA, "tensor map for activations failed");
            int outs[3], col0[3], nseg;
            if (kind == QKV) {
                nseg = 3;
                outs[0] = h->qd;
                outs[1] = outs[2] = h->kvd;
                col0[0] = 0;
                col0[1] = h->k_off;
                col0[2] = h->v_off;
            } else if (kind == GATEUP && fuse) {
                // one segment of 2 tg 128-row tiles: tile 2 t + r = gate and
                // up rows 128 t + 64 r .. + 63 (two 64-row boxes)
                nseg = 1;
                outs[0] = 2 * h->tg * kTileM;
                col0[0] = 0;
            } else if (kind == GATEUP) {
                nseg = 2;
                outs[0] = outs[1] = h->F;
                col0[0] = 0;
                col0[1] = h->up_off;
            } else {
                nseg = 1;
                outs[0] = h->d;
                col0[0] = 0;
            }
            int tiles[3];
            for (int i = 0; i < nseg; ++i) tiles[i] = (outs[i] + kTileM - 1) / kTileM;
            const int sub = mode == STEP ? kStepSub : 1;
            const int n_kb = (K + kBlockK * sub - 1) / (kBlockK * sub);
            TcGemm proto;
            std::memset(&proto.p, 0, sizeof(proto.p));
            proto.pair = true;
            int maxp = 1, rc, group0[4];
            if ((rc = upload_schedule(h, tiles, nseg, 2, n_kb, pairs, proto, &h->planes[mode][kind], &maxp, group0,
                                      fuse)) != LA_OK)
                return rc;
            part_max = std::max(part_max, static_cast<size_t>(maxp) * h->Rp[mode] * h->ldo[kind]);
            h->plan[mode][kind].resize(h->L);
            for (int l = 0; l < h->L; ++l) {
                TcGemm &g = h->plan[mode][kind][l];
                g = proto;
                const void *ws[3];
                if (kind == QKV) {
                    ws[0] = h->wq[l];
                    ws[1] = h->wk[l];
                    ws[2] = h->wv[l];
                } else if (kind == GATEUP) {
                    ws[0] = h->wg[l];
                    ws[1] = h->wu[l];
                } else {
                    ws[0] = kind == OPROJ ? h->wo[l] : h->wd[l];
                }
                if (fuse && (make_tmap_bf16(&g.p.a[0], h->wg[l], K, h->F, static_cast<uint64_t>(K) * 2, kBlockK, 64) ||
                             make_tmap_bf16(&g.p.a[1], h->wu[l], K, h->F, static_cast<uint64_t>(K) * 2, kBlockK, 64)))
                    return fail(LA_ERR_INVALID_ARG, "tensor map for a weight failed (16-byte alignment?)");
                for (int i = 0; i < nseg; ++i) {
                    if (!fuse &&
                        make_tmap_bf16(&g.p.a[i], ws[i], K, outs[i], static_cast<uint64_t>(K) * 2, kBlockK, kTileM))
                        return fail(LA_ERR_INVALID_ARG, "tensor map for a weight failed (16-byte alignment?)");
                    g.p.seg_tile0[i] = group0[i];
                    g.p.seg_out[i] = outs[i];
                    g.p.seg_col0[i] = col0[i];
                }
                g.p.seg_tile0[nseg] = group0[nseg];
                g.p.b = bmap;
                g.p.nseg = nseg;
                g.p.n_kb = n_kb;
                g.p.sub = sub;
                g.p.splits = 1;
                g.p.nrows = mode == STEP ? h->M : kPrefillRows;
                g.p.bn = bn;
                g.p.bh = bhm;
                g.p.ldo = h->ldo[kind];
                g.p.split_stride = static_cast<long long>(h->Rp[mode]) * h->ldo[kind];
                g.p.out = h->part;
                g.p.err = &h->st->err;
                if (fuse) {
                    g.p.fuse_cnt = h->fuse_cnt;
                    g.p.fuse_np = h->planes[mode][kind];
                    g.p.fuse_out = static_cast<__nv_bfloat16 *>(h->fa);
                    g.p.fuse_lo_off = static_cast<long long>(bhm) * h->F;
                    g.p.fuse_F = h->F;
                }
                tc_gemm_finalize(g);
            }
        }
    }
    for (int kind = 0; kind < 4; ++kind) {
        const int K = Ks[kind];
        CUtensorMap bmap;
        if (make_tmap_bf16(&bmap, xs[kind], K, 2 * h->bh_pf, static_cast<uint64_t>(K) * 2, kBlockK, kArRows))
            return fail(LA_ERR_CUDA, "tensor map for activations failed");
        h->plan_ar[kind] = h->plan[PREFILL][kind];
        for (TcGemm &g : h->plan_ar[kind]) {
            g.p.b = bmap;
            g.p.nrt = 1;
            g.p.bnh = kArRows;
            tc_gemm_finalize(g);
        }
    }
    // lm_head over the used rows
    {
        TcGemm &g = h->plan_lm;
        std::memset(&g.p, 0, sizeof(g.p));
        const int bn = 2 * h->bh_u;
        g.pair = true;
        if (make_tmap_bf16(&g.p.a[0], h->lm_head, h->d, h->V, static_cast<uint64_t>(h->d) * 2, kBlockK, kTileM) ||
            make_tmap_bf16(&g.p.b, h->xu, h->d, bn, static_cast<uint64_t>(h->d) * 2, kBlockK, h->bh_u))
            return fail(LA_ERR_INVALID_ARG, "tensor map for lm_head failed");
        const int n_kb = (h->d + kBlockK * kStepSub - 1) / (kBlockK * kStepSub);
        int maxp = 1, rc, group0[2];
        if ((rc = upload_schedule(h, &h->tv, 1, 2, n_kb, pairs, g, &h->planes_lm, &maxp, group0)) != LA_OK) return rc;
        g.p.nseg = 1;
        g.p.seg_tile0[0] = 0;
        g.p.seg_tile0[1] = group0[1];
        g.p.seg_out[0] = h->V;
        g.p.seg_col0[0] = 0;
        g.p.n_kb = n_kb;
        g.p.sub = kStepSub;
        g.p.splits = 1;
        g.p.nrows = h->U;
        g.p.bn = bn;
        g.p.bh = h->bh_u;
        g.p.ldo = h->ldo_lm;
        g.p.split_stride = h->lm_stride;
        g.p.out = h->lm_part;
        g.p.err = &h->st->err;
        tc_gemm_finalize(g);
        h->lm_part_elems = static_cast<size_t>(maxp) * h->lm_stride;
    }
    h->part_elems = part_max;
    return LA_OK;
}

}  // namespace

// ======================================================================== C ABI
extern "C" {

const char *la_strerror(int code) {
    switch (code) {
        case LA_OK: return "ok";
        case LA_ERR_INVALID_ARG: return "invalid argument";
        case LA_ERR_OOM: return "out of memory";
        case LA_ERR_CAPACITY: return "capacity exceeded";
        case LA_ERR_CUDA: return "CUDA error";
        case LA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case LA_ERR_STATE: return "call out of order";
        case LA_ERR_UNSUPPORTED: return "unsupported configuration";
        default: return "unknown error";
    }
}

const char *la_last_error(void) { return g_last_error.c_str(); }

static int la_prefill_impl(la_handle *h, const int32_t *prompt, int32_t n, int32_t *first_token);

static int la_create_body(const la_model_dims *dims, const la_weights *w, const la_opts *opts, la_handle **out) {
    if (!dims || !w || !opts || !out) return fail(LA_ERR_INVALID_ARG, "null argument");
    *out = nullptr;
    const la_model_dims &D = *dims;
    if (D.n_layers < 1 || D.d_model < 64 || D.n_heads < 1 || D.n_kv_heads < 1 || D.n_heads % D.n_kv_heads ||
        D.ffn < 1 || D.vocab < 2 || !(D.rms_eps > 0.f) || !(D.rope_base > 1.f))
        return fail(LA_ERR_INVALID_ARG, "bad model dims");
    if (D.head_dim != 64 && D.head_dim != 128) return fail(LA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (D.dtype != LA_F32 && D.dtype != LA_BF16) return fail(LA_ERR_INVALID_ARG, "dtype");
    if (D.d_model % 8 || D.ffn % 8 || (D.n_heads * D.head_dim) % 8)
        return fail(LA_ERR_UNSUPPORTED, "d_model, ffn and n_heads*head_dim must be multiples of 8");
    const la_opts &O = *opts;
    if (O.N < 2 || O.N > 8 || O.W < 1 || O.G < 0 || O.G > 32 || O.pool_cap < 0 || O.pool_cap > 32 ||
        !(O.temperature >= 0.f) || O.top_k < 0 || O.top_p != O.top_p ||
        (O.pool_policy != LA_POOL_FIFO && O.pool_policy != LA_POOL_LRU && O.pool_policy != LA_POOL_LFU))
        return fail(LA_ERR_INVALID_ARG,
                    "bad options (N 2..8, W >= 1, G 0..32, pool_cap 0..32, temperature >= 0, top_k >= 0, "
                    "top_p a number, pool_policy FIFO, LRU or LFU)");
    const int M = 1 + (O.W + O.G) * (O.N - 1);
    if (M > 256) return fail(LA_ERR_UNSUPPORTED, "1 + (W+G)(N-1) must be <= 256");
    if (O.max_seq < O.N + M + 2) return fail(LA_ERR_INVALID_ARG, "max_seq too small");
    if (!w->embed || !w->final_norm || !w->lm_head || !w->attn_norm || !w->wq || !w->wk || !w->wv || !w->wo ||
        !w->ffn_norm || !w->w_gate || !w->w_up || !w->w_down)
        return fail(LA_ERR_INVALID_ARG, "null weight pointer");

    std::unique_ptr<la_handle> owner(new la_handle());   // freed on every early return
    la_handle *h = owner.get();
    h->dims = D;
    h->opts = O;
    h->stream = static_cast<cudaStream_t>(O.cuda_stream);
    h->prof_on = O.profile != 0;
    h->bf16 = D.dtype == LA_BF16;
    h->act = h->bf16 ? 2 : 4;
    h->L = D.n_layers;
    h->d = D.d_model;
    h->nh = D.n_heads;
    h->nkv = D.n_kv_heads;
    h->hd = D.head_dim;
    h->F = D.ffn;
    h->V = D.vocab;
    h->qd = h->nh * h->hd;
    h->kvd = h->nkv * h->hd;
    h->qkv_out = h->qd + 2 * h->kvd;
    h->N = O.N;
    h->W = O.W;
    h->G = O.G;
    h->M = M;
    h->U = 1 + O.W + O.G * (O.N - 1);
    h->cap = O.pool_cap > 0 ? O.pool_cap : std::max(O.G, 1);
    h->max_seq = O.max_seq;
    h->R = round_up(std::max(M, kPrefillRows), 16);
    h->Rp[STEP] = round_up(std::max(M, kTileM), 16);
    h->Rp[PREFILL] = kPrefillRows;
    h->bn_step = round_up(M, 16);
    h->bn_pf = kPrefillRows;
    h->bn_u = round_up(h->U, 16);
    // bf16 GEMM inputs: hi rows [0, bh), lo rows [bh, 2 bh) of each buffer; a
    // step's GEMMs multiply 2 bh rows (UMMA N), so bh follows the row count
    h->bh_step = round_up(M, 16);
    h->bh_pf = kPrefillRows;
    h->bh_u = round_up(std::max(h->U, 1), 16);
    h->act_rows = h->bf16 ? 2 * kPrefillRows : h->R;
    h->seq = h->bf16 ? round_up(h->max_seq, 64) : h->max_seq;
    h->qv_pad = kPrefillRows * (h->nh / h->nkv);
    h->tq = (h->qd + kTileM - 1) / kTileM;
    h->tk = (h->kvd + kTileM - 1) / kTileM;
    h->tg = (h->F + kTileM - 1) / kTileM;
    h->td = (h->d + kTileM - 1) / kTileM;
    h->tv = (h->V + kTileM - 1) / kTileM;
    h->k_off = h->tq * kTileM;
    h->v_off = (h->tq + h->tk) * kTileM;
    h->up_off = h->tg * kTileM;
    h->ldo[QKV] = (h->tq + 2 * h->tk) * kTileM;
    h->ldo[OPROJ] = h->td * kTileM;
    h->ldo[GATEUP] = 2 * h->tg * kTileM;
    h->ldo[DOWN] = h->td * kTileM;
    h->ldo_lm = h->tv * kTileM;
    h->lm_stride = static_cast<long long>(std::max(h->U, 1)) * h->ldo_lm;
    if (h->bf16 && M > kTileM) {
        return fail(LA_ERR_UNSUPPORTED, "bf16 models need 1 + (W+G)(N-1) <= 128");
    }
    h->embed = w->embed;
    h->final_norm = w->final_norm;
    h->lm_head = w->lm_head;
    auto grab = [&](std::vector<const void *> &v, const void *const *src) {
        v.assign(src, src + h->L);
        for (const void *p : v)
            if (!p || (reinterpret_cast<uintptr_t>(p) & 15)) return false;
        return true;
    };
    if (!grab(h->attn_norm, w->attn_norm) || !grab(h->wq, w->wq) || !grab(h->wk, w->wk) || !grab(h->wv, w->wv) ||
        !grab(h->wo, w->wo) || !grab(h->ffn_norm, w->ffn_norm) || !grab(h->wg, w->w_gate) || !grab(h->wu, w->w_up) ||
        !grab(h->wd, w->w_down)) {
        return fail(LA_ERR_INVALID_ARG, "null or misaligned per-layer weight pointer");
    }
    for (const void *p : {w->embed, w->final_norm, w->lm_head})
        if (reinterpret_cast<uintptr_t>(p) & 15) {
            return fail(LA_ERR_INVALID_ARG, "weights must be 16-byte aligned");
        }

    int rc = LA_OK;
    auto A = [&](int r) {
        if (rc == LA_OK) rc = r;
    };
    const size_t act = h->act;
    const int R = h->R;
    A(h->alloc(&h->h, static_cast<size_t>(R) * h->d));
    const size_t ar = static_cast<size_t>(h->act_rows);
    A(h->alloc_bytes(&h->xn, ar * h->d * act));
    A(h->alloc_bytes(&h->ao, ar * h->qd * act));
    A(h->alloc_bytes(&h->fa, ar * h->F * act));
    A(h->alloc_bytes(&h->xu, ar * h->d * act));
    A(h->alloc(&h->q, static_cast<size_t>(R) * h->qd));
    A(h->alloc(&h->logits, static_cast<size_t>(std::max(h->U, 1)) * h->V));
    A(h->alloc(&h->amax, std::max(h->U, 1)));
    A(h->alloc(&h->lmax, std::max(h->U, 1)));
    A(h->alloc(&h->lsum, std::max(h->U, 1)));
    A(h->alloc(&h->thr_key, std::max(h->U, 1)));
    A(h->alloc(&h->thr_cut, std::max(h->U, 1)));
    const size_t cache_bytes = static_cast<size_t>(h->L) * 2 * h->nkv * h->seq * h->hd * sizeof(float);
    if (h->bf16) {
        A(h->alloc(&h->attn_ws, 1));
        A(h->alloc(&h->qs, static_cast<size_t>(2) * h->nkv * h->qv_pad * h->hd));
    } else {
        const int nch_max = (h->max_seq + kAttnChunk - 1) / kAttnChunk;
        A(h->alloc(&h->attn_ws, static_cast<size_t>(nch_max) * R * h->nh * (h->hd + 4)));
    }
    A(h->alloc_bytes(&h->cache, cache_bytes));
    A(h->alloc(&h->rope, static_cast<size_t>(h->max_seq) * (h->hd / 2)));
    A(h->alloc(&h->tok, M));
    A(h->alloc(&h->depth, M));
    h->anc_stride = h->N + h->W;
    A(h->alloc(&h->anc, static_cast<size_t>(M) * h->anc_stride));
    A(h->alloc(&h->anc_cnt, M));
    A(h->alloc(&h->vis_bits, static_cast<size_t>(M) * 8));
    A(h->alloc(&h->used, h->U));
    A(h->alloc(&h->iota, R));
    A(h->alloc(&h->st, 1));
    A(h->alloc(&h->tokens_log, h->max_seq));
    A(h->alloc(&h->window, static_cast<size_t>(h->N - 1) * h->W));
    A(h->alloc(&h->cands, std::max(h->G * (h->N - 1), 1)));
    int log2n = 10;
    while ((1 << log2n) < 2 * h->V) ++log2n;
    h->nslots_log2 = log2n;
    const size_t nslots = static_cast<size_t>(1) << log2n;
    A(h->alloc(&h->pkeys, nslots));
    A(h->alloc(&h->pcnt, nslots));
    A(h->alloc(&h->phead, nslots));
    A(h->alloc(&h->pent, nslots * h->cap * (h->N - 1)));
    A(h->alloc(&h->puse, nslots * h->cap));
    if (rc == LA_OK && cudaMallocHost(&h->st_host, sizeof(SpecState)) != cudaSuccess)
        rc = fail(LA_ERR_OOM, "pinned host allocation failed");
    if (rc != LA_OK) return rc;
    cudaStream_t s = h->stream;
    // Static tables: rotary angles, step-row depths and in-step key lists.
    {
        std::vector<float2> rope(static_cast<size_t>(h->max_seq) * (h->hd / 2));
        for (int p = 0; p < h->max_seq; ++p)
            for (int i = 0; i < h->hd / 2; ++i) {
                const double th = std::pow(static_cast<double>(D.rope_base), -2.0 * i / h->hd);
                const double a = p * th;
                rope[static_cast<size_t>(p) * (h->hd / 2) + i] =
                    make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
            }
        std::vector<int> parent, depth, used;
        std::vector<uint32_t> bits;
        step_structure(h->N, h->W, h->G, parent, depth);
        step_tables(h->N, h->W, h->G, depth, bits, used);
        std::vector<int> anc(static_cast<size_t>(M) * h->anc_stride, 0), cnt(M, 0);
        for (int r = 0; r < M; ++r) {
            std::vector<int> chain;
            for (int x = r; x >= 0; x = parent[x]) chain.push_back(x);
            std::reverse(chain.begin(), chain.end());
            cnt[r] = static_cast<int>(chain.size());
            for (size_t i = 0; i < chain.size(); ++i) anc[static_cast<size_t>(r) * h->anc_stride + i] = chain[i];
        }
        std::vector<int> iota(R);
        for (int i = 0; i < R; ++i) iota[i] = i;
        if (cudaMemcpy(h->rope, rope.data(), rope.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemcpy(h->depth, depth.data(), M * sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemcpy(h->anc, anc.data(), anc.size() * sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemcpy(h->anc_cnt, cnt.data(), M * sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemcpy(h->vis_bits, bits.data(), bits.size() * sizeof(uint32_t), cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemcpy(h->used, used.data(), used.size() * sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemcpy(h->iota, iota.data(), R * sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
            return fail(LA_ERR_CUDA, "uploading static tables failed");
        }
    }
    // Zero activations once so padded rows never hold NaN bit patterns.
    if (cudaMemsetAsync(h->xn, 0, ar * h->d * act, s) != cudaSuccess ||
        cudaMemsetAsync(h->ao, 0, ar * h->qd * act, s) != cudaSuccess ||
        cudaMemsetAsync(h->fa, 0, ar * h->F * act, s) != cudaSuccess ||
        cudaMemsetAsync(h->xu, 0, ar * h->d * act, s) != cudaSuccess ||
        cudaMemsetAsync(h->st, 0, sizeof(SpecState), s) != cudaSuccess) {
        return fail(LA_ERR_CUDA, "memset failed");
    }
    if (h->bf16) {
        // The tensor-core attention reads whole 128-key chunks and 128-row
        // query tiles: slots and rows past the live ones must hold finite
        // values (they are masked, and 0 * finite = 0 in P V).
        h->kcs = static_cast<__nv_bfloat16 *>(h->cache);
        h->vcs = h->kcs + static_cast<size_t>(h->L) * 2 * h->nkv * h->seq * h->hd;
        if (cudaMemsetAsync(h->cache, 0, cache_bytes, s) != cudaSuccess ||
            cudaMemsetAsync(h->qs, 0, static_cast<size_t>(2) * h->nkv * h->qv_pad * h->hd * 2, s) != cudaSuccess) {
            return fail(LA_ERR_CUDA, "memset failed");
        }
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&h->nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            return fail(LA_ERR_CUDA, "device query failed");
        }
        AttnUmmaParams &ap = h->attn_proto;
        ap.nh = h->nh;
        ap.nkv = h->nkv;
        ap.gq = h->nh / h->nkv;
        ap.hd = h->hd;
        ap.qv_pad = h->qv_pad;
        ap.seq = h->seq;
        ap.out = static_cast<__nv_bfloat16 *>(h->ao);
        ap.err = &h->st->err;
        ap.k_off = h->k_off;
        ap.qkv_tiles = h->ldo[QKV] / kTileM;
        ap.v_off = h->v_off;
        ap.rope = h->rope;
        ap.q = h->qs;
        ap.kc = h->kcs;
        ap.vc = h->vcs;
        if (!attention_umma_maps(ap, h->qs, h->kcs, h->vcs, h->L)) {
            return fail(LA_ERR_CUDA, "tensor maps for the attention failed");
        }
    }
    if (h->bf16) {
        rc = build_plans(h);
    } else {
        h->part_elems = static_cast<size_t>(R) * std::max(std::max(h->ldo[QKV], h->ldo[GATEUP]), h->ldo[DOWN]);
        h->lm_part_elems = static_cast<size_t>(h->lm_stride);
    }
    if (rc == LA_OK) rc = h->alloc(&h->part, h->part_elems);
    if (rc == LA_OK) rc = h->alloc(&h->lm_part, h->lm_part_elems);
    if (rc == LA_OK && h->bf16) {
        for (int m = 0; m < 2; ++m)
            for (int k = 0; k < 4; ++k)
                for (auto &g : h->plan[m][k]) g.p.out = h->part;
        for (int k = 0; k < 4; ++k)
            for (auto &g : h->plan_ar[k]) g.p.out = h->part;
        h->plan_lm.p.out = h->lm_part;
    }
    if (rc == LA_OK) rc = reset_pool(h);
    if (rc == LA_OK && cudaStreamSynchronize(s) != cudaSuccess) rc = fail(LA_ERR_CUDA, "create sync failed");
    if (rc != LA_OK) return rc;
    *out = owner.release();
    return LA_OK;
}

void la_destroy(la_handle *h) {
    if (!h) return;
    if (h->stream) cudaStreamSynchronize(h->stream);
    else cudaDeviceSynchronize();
    delete h;
}

static int la_prefill_body(la_handle *h, const int32_t *prompt, int32_t n, int32_t *first_token) {
    nvtxRangePushA("la_prefill");
    const int rc = la_prefill_impl(h, prompt, n, first_token);
    nvtxRangePop();
    return rc;
}

static int la_prefill_impl(la_handle *h, const int32_t *prompt, int32_t n, int32_t *first_token) {
    if (!h || !prompt || !first_token) return fail(LA_ERR_INVALID_ARG, "null argument");
    if (n < h->N) return fail(LA_ERR_INVALID_ARG, "prompt shorter than N");
    if (n + h->M + h->N + 2 > h->max_seq) return fail(LA_ERR_CAPACITY, "prompt too long for max_seq");
    for (int i = 0; i < n; ++i)
        if (prompt[i] < 0 || prompt[i] >= h->V) return fail(LA_ERR_INVALID_ARG, "token id out of range at %d", i);
    cudaStream_t s = h->stream;
    h->prefilled = false;
    CK(cudaMemsetAsync(h->st, 0, sizeof(SpecState), s));
    int rc = reset_pool(h);
    if (rc != LA_OK) return rc;
    CK(cudaMemcpyAsync(h->tokens_log, prompt, static_cast<size_t>(n) * sizeof(int32_t), cudaMemcpyHostToDevice, s));
    if ((rc = run_prefix(h, n, true)) != LA_OK) return rc;
    CK(first_token_launch(h->spec(), n, s));
    // Initial window: prompt tokens picked by splitmix64(seed ^ (k*W + j)).
    std::vector<int> win(static_cast<size_t>(h->N - 1) * h->W);
    for (int k = 0; k < h->N - 1; ++k)
        for (int j = 0; j < h->W; ++j)
            win[static_cast<size_t>(k) * h->W + j] =
                prompt[splitmix64(h->opts.seed ^ static_cast<uint64_t>(k * h->W + j)) % static_cast<uint64_t>(n)];
    CK(cudaMemcpyAsync(h->window, win.data(), win.size() * sizeof(int), cudaMemcpyHostToDevice, s));
    if (h->opts.prompt_as_reference) CK(pool_seed_prompt_launch(h->spec(), n, s));
    CK(cudaMemcpyAsync(h->st_host, h->st, sizeof(SpecState), cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
    if ((rc = check_device_error(h)) != LA_OK) return rc;
    *first_token = h->st_host->o;
    h->P = n;
    h->prefilled = true;
    h->steps = 0;
    h->generated = 1;
    h->last_A = 0;
    h->last_g = 0;
    h->logits_rows = 1;
    h->launches = 0;
    h->ev_used = 0;
    for (int c = 0; c < 4; ++c) h->prof_ms[c] = h->prof_bytes[c] = 0, h->prof_launches[c] = 0;
    h->h2d_bytes = static_cast<int64_t>(n) * sizeof(int32_t) + static_cast<int64_t>(win.size()) * sizeof(int);
    h->d2h_bytes = sizeof(SpecState);
    return LA_OK;
}

namespace {
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};
}  // namespace

}  // extern "C"

namespace {

// Every launch of one step, then the read-back of the step state.
int enqueue_step(la_handle *h) {
    cudaStream_t s = h->stream;
    int pe = h->prof_begin();
    CK(build_rows_launch(h->spec(), s));
    h->prof_end(pe, 3, 0.0);
    int rc = forward_any(h, STEP, h->tok, h->M, h->P, true);
    if (rc != LA_OK) return rc;
    if ((rc = run_lm_head(h, h->U, true)) != LA_OK) return rc;
    pe = h->prof_begin();
    CK(argmax_launch(h->lm_part, h->planes_lm, h->lm_stride, h->ldo_lm, h->logits, h->U, h->V,
                     h->opts.temperature > 0.f ? 1.f / h->opts.temperature : 0.f, h->amax,
                     h->lmax, h->lsum, h->opts.top_k, h->opts.top_p, h->thr_key, h->thr_cut, s));
    CK(finish_step_launch(h->spec(), s));
    if ((rc = kv_commit(h)) != LA_OK) return rc;
    h->prof_end(pe, 3, 0.0);
    h->launches += 4;   // build_rows, argmax, finish_step, kv_commit
    CK(cudaMemcpyAsync(h->st_host, h->st, sizeof(SpecState), cudaMemcpyDeviceToHost, s));
    return LA_OK;
}

// Capture enqueue_step into h->step_graph.  Every kernel argument of a step
// is fixed except the prefix length, which the attention reads from the
// device step state, so the graph replays for every later step.  On any
// failure the handle falls back to direct launches for good.
void capture_step(la_handle *h) {
    cudaStream_t s = h->stream;
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaGetLastError();
        h->graph_off = true;
        return;
    }
    const int64_t l0 = h->launches;
    const int rc = enqueue_step(h);
    cudaGraph_t g = nullptr;
    const cudaError_t e = cudaStreamEndCapture(s, &g);
    h->graph_launches = h->launches - l0;
    h->launches = l0;
    if (rc != LA_OK || e != cudaSuccess || !g || cudaGraphInstantiate(&h->step_graph, g, 0) != cudaSuccess) {
        cudaGetLastError();
        h->step_graph = nullptr;
        h->graph_off = true;
    }
    if (g) cudaGraphDestroy(g);
}

}  // namespace

namespace {

// Error word of la_gemm_bf16's kernels on the current device: one per device,
// allocated on the first call there and kept until the process exits (a
// kernel may only write its own device's word).
// With create = false, *out stays nullptr while the device has no word yet.
cudaError_t gemm_err_word(unsigned **out, bool create = true) {
    static std::mutex mu;
    static unsigned *words[64] = {};
    *out = nullptr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!words[dev] && create) {
        e = cudaMalloc(&words[dev], sizeof(unsigned));
        if (e == cudaSuccess) e = cudaMemset(words[dev], 0, sizeof(unsigned));
        if (e != cudaSuccess) {
            if (words[dev]) cudaFree(words[dev]);
            words[dev] = nullptr;
            return e;
        }
    }
    *out = words[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

static int la_step_body(la_handle *h, int32_t *out_tokens, int32_t *out_n) {
    NvtxRange range("la_step");
    if (!h || !out_tokens || !out_n) return fail(LA_ERR_INVALID_ARG, "null argument");
    if (!h->prefilled) return fail(LA_ERR_STATE, "la_step before la_prefill");
    if (h->P + h->M + h->N + 2 > h->max_seq) return fail(LA_ERR_CAPACITY, "max_seq reached");
    cudaStream_t s = h->stream;
    int rc;
    // The first step of a handle runs directly (one-time kernel attributes are
    // set outside any capture); later non-profiled steps replay a graph.
    if (h->bf16 && !h->prof_on && !h->graph_off && h->steps > 0 && !h->step_graph) capture_step(h);
    if (h->step_graph) {
        CK(cudaGraphLaunch(h->step_graph, s));
        h->launches += h->graph_launches;
    } else if ((rc = enqueue_step(h)) != LA_OK) {
        return rc;
    }
    CK(cudaStreamSynchronize(s));
    if ((rc = check_device_error(h)) != LA_OK) return rc;
    h->prof_collect();
    const SpecState &st = *h->st_host;
    if (st.A < 1 || st.A > h->N) {
        h->prefilled = false;
        return fail(LA_ERR_STATE, "device reported A=%d", st.A);
    }
    for (int i = 0; i < st.A; ++i) out_tokens[i] = st.acc[i];
    *out_n = st.A;
    h->P = st.P;
    h->steps += 1;
    h->generated += st.A;
    h->d2h_bytes += sizeof(SpecState);
    h->last_A = st.A;
    h->last_g = st.g;
    h->logits_rows = h->U;
    return LA_OK;
}

static int la_ar_step_body(la_handle *h, int32_t *token) {
    NvtxRange range("la_ar_step");
    if (!h || !token) return fail(LA_ERR_INVALID_ARG, "null argument");
    if (!h->prefilled) return fail(LA_ERR_STATE, "la_ar_step before la_prefill");
    if (h->P + 2 > h->max_seq) return fail(LA_ERR_CAPACITY, "max_seq reached");
    cudaStream_t s = h->stream;
    const int P = h->P;   // tokens_log[P] is the last committed token, at position P
    int rc = forward_any(h, PREFILL, h->tokens_log + P, 1, P, true);
    if (rc != LA_OK) return rc;
    if ((rc = run_lm_head(h, 1, false)) != LA_OK) return rc;
    CK(argmax_launch(h->lm_part, h->planes_lm, h->lm_stride, h->ldo_lm, h->logits, 1, h->V,
                     h->opts.temperature > 0.f ? 1.f / h->opts.temperature : 0.f, h->amax, h->lmax, h->lsum,
                     h->opts.top_k, h->opts.top_p, h->thr_key, h->thr_cut, s));
    CK(first_token_launch(h->spec(), P + 1, s));
    h->launches += 2;
    CK(cudaMemcpyAsync(h->st_host, h->st, sizeof(SpecState), cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
    if ((rc = check_device_error(h)) != LA_OK) return rc;
    *token = h->st_host->o;
    h->P = P + 1;
    h->generated += 1;
    h->d2h_bytes += sizeof(SpecState);
    h->logits_rows = 1;
    return LA_OK;
}

static int la_generate_body(la_handle *h, const int32_t *prompt, int32_t n, int32_t max_new, int32_t *out,
                            int32_t *out_n, int32_t *n_steps) {
    if (!h || !prompt || !out || max_new < 1) return fail(LA_ERR_INVALID_ARG, "bad argument");
    int32_t first = 0;
    int rc = la_prefill(h, prompt, n, &first);
    if (rc != LA_OK) return rc;
    int cnt = 0, steps = 0;
    out[cnt++] = first;
    int32_t buf[8];
    while (cnt < max_new) {
        int32_t a = 0;
        if ((rc = la_step(h, buf, &a)) != LA_OK) return rc;
        ++steps;
        for (int i = 0; i < a && cnt < max_new; ++i) out[cnt++] = buf[i];
    }
    if (out_n) *out_n = cnt;
    if (n_steps) *n_steps = steps;
    return LA_OK;
}

int la_stats(const la_handle *h, la_stats_t *o) {
    if (!h || !o) return fail(LA_ERR_INVALID_ARG, "null argument");
    o->steps = h->steps;
    o->generated = h->generated;
    o->last_accept = h->last_A;
    o->last_candidates = h->last_g;
    o->prefix_len = h->P;
    o->rows = h->M;
    o->gemm_ms = h->prof_ms[0];
    o->gemm_bytes = h->prof_bytes[0];
    o->gemm_launches = h->prof_launches[0];
    o->attn_ms = h->prof_ms[1];
    o->attn_bytes = h->prof_bytes[1];
    o->attn_launches = h->prof_launches[1];
    o->kernel_launches = h->launches;
    o->elem_ms = h->prof_ms[2];
    o->spec_ms = h->prof_ms[3];
    o->h2d_bytes = h->h2d_bytes;
    o->d2h_bytes = h->d2h_bytes;
    return LA_OK;
}

static int la_export_state_body(la_handle *h, la_state_t *stt) {
    if (!h || !stt || !stt->tokens || !stt->window || (!stt->records && stt->records_cap > 0))
        return fail(LA_ERR_INVALID_ARG, "null argument");
    if (!h->prefilled) return fail(LA_ERR_STATE, "no state before la_prefill");
    cudaStream_t s = h->stream;
    const int n = h->P + 1;
    const size_t nslots = static_cast<size_t>(1) << h->nslots_log2;
    const int L = h->N - 1;
    std::vector<int> keys(nslots), cnt(nslots), head(nslots), ent(nslots * h->cap * L), use(nslots * h->cap);
    std::vector<int> toks(n);
    CK(cudaMemcpyAsync(toks.data(), h->tokens_log, n * sizeof(int), cudaMemcpyDeviceToHost, s));
    CK(cudaMemcpyAsync(stt->window, h->window, static_cast<size_t>(L) * h->W * sizeof(int), cudaMemcpyDeviceToHost, s));
    CK(cudaMemcpyAsync(keys.data(), h->pkeys, nslots * sizeof(int), cudaMemcpyDeviceToHost, s));
    CK(cudaMemcpyAsync(cnt.data(), h->pcnt, nslots * sizeof(int), cudaMemcpyDeviceToHost, s));
    CK(cudaMemcpyAsync(head.data(), h->phead, nslots * sizeof(int), cudaMemcpyDeviceToHost, s));
    CK(cudaMemcpyAsync(ent.data(), h->pent, ent.size() * sizeof(int), cudaMemcpyDeviceToHost, s));
    CK(cudaMemcpyAsync(use.data(), h->puse, use.size() * sizeof(int), cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
    std::map<int, size_t> order;
    for (size_t i = 0; i < nslots; ++i)
        if (keys[i] >= 0) order[keys[i]] = i;
    int nrec = 0;
    for (auto &kv : order) nrec += cnt[kv.second];
    stt->n_tokens = n;
    stt->n_records = nrec;
    if (n > stt->tokens_cap || nrec > stt->records_cap)
        return fail(LA_ERR_CAPACITY, "state buffers too small (tokens %d, records %d)", n, nrec);
    std::memcpy(stt->tokens, toks.data(), n * sizeof(int));
    int r = 0;
    for (auto &kv : order) {
        const size_t sl = kv.second;
        for (int e = 0; e < cnt[sl]; ++e) {
            int *rec = stt->records + static_cast<size_t>(r) * h->N;
            rec[0] = kv.first;
            const size_t at = sl * h->cap + (head[sl] + e) % h->cap;
            const int *src = ent.data() + at * L;
            for (int m = 0; m < L; ++m) rec[1 + m] = src[m];
            if (stt->uses) stt->uses[r] = h->opts.pool_policy == LA_POOL_LFU ? use[at] : 0;
            ++r;
        }
    }
    return LA_OK;
}

static int la_import_state_body(la_handle *h, const la_state_t *stt) {
    if (!h || !stt || !stt->tokens || !stt->window || (stt->n_records > 0 && !stt->records))
        return fail(LA_ERR_INVALID_ARG, "null argument");
    const int n = stt->n_tokens;
    if (n < 2) return fail(LA_ERR_INVALID_ARG, "state needs at least two tokens");
    if (n - 1 + h->M + h->N + 2 > h->max_seq) return fail(LA_ERR_CAPACITY, "state too long for max_seq");
    for (int i = 0; i < n; ++i)
        if (stt->tokens[i] < 0 || stt->tokens[i] >= h->V) return fail(LA_ERR_INVALID_ARG, "token out of range");
    const int L = h->N - 1;
    for (int i = 0; i < L * h->W; ++i)
        if (stt->window[i] < 0 || stt->window[i] >= h->V) return fail(LA_ERR_INVALID_ARG, "window token out of range");
    for (int i = 0; i < stt->n_records * h->N; ++i)
        if (stt->records[i] < 0 || stt->records[i] >= h->V) return fail(LA_ERR_INVALID_ARG, "pool token out of range");
    cudaStream_t s = h->stream;
    h->prefilled = false;
    CK(cudaMemsetAsync(h->st, 0, sizeof(SpecState), s));
    int rc = reset_pool(h);
    if (rc != LA_OK) return rc;
    CK(cudaMemcpyAsync(h->tokens_log, stt->tokens, static_cast<size_t>(n) * sizeof(int), cudaMemcpyHostToDevice, s));
    if ((rc = run_prefix(h, n - 1, false)) != LA_OK) return rc;
    SpecState init{};
    init.P = n - 1;
    init.o = stt->tokens[n - 1];
    init.n_tokens = n;
    init.cstar = -1;
    *h->st_host = init;
    CK(cudaMemcpyAsync(h->st, h->st_host, sizeof(SpecState), cudaMemcpyHostToDevice, s));
    CK(cudaMemcpyAsync(h->window, stt->window, static_cast<size_t>(L) * h->W * sizeof(int), cudaMemcpyHostToDevice, s));
    if (stt->n_records > 0) {
        const size_t need = static_cast<size_t>(stt->n_records) * h->N;
        if (need > h->records_dev_cap) {
            int *p = nullptr;
            if ((rc = h->alloc(&p, need)) != LA_OK) return rc;
            h->records_dev = p;
            h->records_dev_cap = need;
        }
        CK(cudaMemcpyAsync(h->records_dev, stt->records, need * sizeof(int), cudaMemcpyHostToDevice, s));
        const int *uses = nullptr;
        if (stt->uses && h->opts.pool_policy == LA_POOL_LFU) {
            for (int i = 0; i < stt->n_records; ++i)
                if (stt->uses[i] < 0) return fail(LA_ERR_INVALID_ARG, "negative use count");
            const size_t nu = static_cast<size_t>(stt->n_records);
            if (nu > h->uses_dev_cap) {
                int *p = nullptr;
                if ((rc = h->alloc(&p, nu)) != LA_OK) return rc;
                h->uses_dev = p;
                h->uses_dev_cap = nu;
            }
            CK(cudaMemcpyAsync(h->uses_dev, stt->uses, nu * sizeof(int), cudaMemcpyHostToDevice, s));
            uses = h->uses_dev;
        }
        CK(pool_insert_launch(h->spec(), h->records_dev, uses, stt->n_records, s));
    }
    CK(cudaMemcpyAsync(h->st_host, h->st, sizeof(SpecState), cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
    if ((rc = check_device_error(h)) != LA_OK) return rc;
    h->P = n - 1;
    h->prefilled = true;
    h->logits_rows = 0;
    return LA_OK;
}

static int la_debug_logits_body(la_handle *h, float *host, int32_t *rows, int32_t *vocab) {
    if (!h || !rows || !vocab) return fail(LA_ERR_INVALID_ARG, "null argument");
    *rows = h->logits_rows;
    *vocab = h->V;
    if (host && h->logits_rows > 0) {
        CK(cudaMemcpyAsync(host, h->logits, static_cast<size_t>(h->logits_rows) * h->V * sizeof(float),
                           cudaMemcpyDeviceToHost, h->stream));
        CK(cudaStreamSynchronize(h->stream));
    }
    return LA_OK;
}

static int la_gemm_bf16_body(const void *x, const void *w, float *y, int32_t rows, int32_t out, int32_t k,
                             int32_t splits, float *workspace, void *stream) {
    if (!x || !w || !y || rows < 1 || rows > 256 || out < 1 || k < 8 || k % 8 || splits < 1)
        return fail(LA_ERR_INVALID_ARG, "bad GEMM arguments");
    const int n_kb = (k + kBlockK - 1) / kBlockK;
    if (splits > n_kb) return fail(LA_ERR_INVALID_ARG, "splits > k / 64");
    if (splits > 1 && !workspace) return fail(LA_ERR_INVALID_ARG, "workspace required when splits > 1");
    unsigned *err = nullptr;
    CK(gemm_err_word(&err));
    TcGemm g;
    std::memset(&g.p, 0, sizeof(g.p));
    const int bn = round_up(rows, 16);
    if (make_tmap_bf16(&g.p.a[0], w, k, out, static_cast<uint64_t>(k) * 2, kBlockK, kTileM) ||
        make_tmap_bf16(&g.p.b, x, k, rows, static_cast<uint64_t>(k) * 2, kBlockK, bn))
        return fail(LA_ERR_INVALID_ARG, "tensor map creation failed (16-byte alignment?)");
    g.p.nseg = 1;
    g.p.seg_tile0[0] = 0;
    g.p.seg_tile0[1] = (out + kTileM - 1) / kTileM;
    g.p.seg_out[0] = out;
    g.p.seg_col0[0] = 0;
    g.p.n_kb = n_kb;
    g.p.splits = splits;
    g.p.nrows = rows;
    g.p.bn = bn;
    g.p.ldo = out;
    g.p.stages = tc_gemm_stages_for(bn);
    g.p.split_stride = static_cast<long long>(rows) * out;
    g.p.out = splits > 1 ? workspace : y;
    g.p.err = err;
    tc_gemm_finalize(g);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CK(tc_gemm_launch(g, s));
    if (splits > 1) CK(reduce_splits_launch(workspace, splits, g.p.split_stride, rows, out, y, s));
    return LA_OK;
}

static int la_gemm_status_body(void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned *w = nullptr, bits = 0, bits_na = 0;
    CK(gemm_err_word(&w, false));
    if (w) {
        CK(cudaMemcpyAsync(&bits, w, sizeof(unsigned), cudaMemcpyDeviceToHost, s));
        CK(cudaMemsetAsync(w, 0, sizeof(unsigned), s));
    }
    CK(noalloc_err_take(s, &bits_na));
    CK(cudaStreamSynchronize(s));
    if (bits | bits_na)
        return fail(LA_ERR_DEVICE_TIMEOUT,
                    "a bounded wait of an earlier GEMM call gave up (error bits 0x%x la_gemm_bf16, 0x%x "
                    "la_gemm_bf16_noalloc); that call's output is void", bits, bits_na);
    return LA_OK;
}

static int la_selftest_timeout_body(la_handle *h, int64_t limit_ns, void *stream) {
    if (limit_ns < 1000 || limit_ns > static_cast<int64_t>(kWaitNs))
        return fail(LA_ERR_INVALID_ARG, "limit_ns must lie in [1000, %llu]", static_cast<unsigned long long>(kWaitNs));
    const unsigned long long lim = static_cast<unsigned long long>(limit_ns);
    if (h) {
        CK(wait_selftest_launch(&h->st->err, nullptr, lim, h->stream));
        return LA_OK;
    }
    unsigned *w = nullptr, *wna = nullptr;
    CK(gemm_err_word(&w));
    CK(noalloc_err_word(&wna));
    CK(wait_selftest_launch(w, wna, lim, static_cast<cudaStream_t>(stream)));
    return LA_OK;
}

static int la_step_tables_body(int32_t N, int32_t W, int32_t G, int32_t *depth, uint32_t *vis, int32_t *used,
                               int32_t max_rows, int32_t *m_out, int32_t *u_out) {
    if (N < 2 || W < 1 || G < 0 || !depth || !vis || !used || !m_out || !u_out)
        return fail(LA_ERR_INVALID_ARG, "la_step_tables: N >= 2, W >= 1, G >= 0 and non-null pointers");
    const long long M = 1 + static_cast<long long>(W + G) * (N - 1);
    if (M > 256 || M > max_rows) return fail(LA_ERR_CAPACITY, "la_step_tables: %lld rows (at most 256 and max_rows)", M);
    std::vector<int> dp, us;
    std::vector<uint32_t> bits;
    step_tables(N, W, G, dp, bits, us);
    std::copy(dp.begin(), dp.end(), depth);
    std::copy(bits.begin(), bits.end(), vis);
    std::copy(us.begin(), us.end(), used);
    *m_out = static_cast<int32_t>(dp.size());
    *u_out = static_cast<int32_t>(us.size());
    return LA_OK;
}

static int la_gemm_schedule_body(int32_t tiles, int32_t n_kb, int32_t ctas, int32_t whole_first, int32_t *segs,
                                 int32_t max_segs, int32_t *nseg_out, int32_t *cta_first, int32_t *ctas_used,
                                 int32_t *planes) {
    if (tiles < 1 || n_kb < 1 || ctas < 1 || max_segs < 0 || !segs || !nseg_out || !cta_first || !ctas_used || !planes)
        return fail(LA_ERR_INVALID_ARG, "la_gemm_schedule: sizes must be >= 1 and pointers non-null");
    std::vector<int> sg, first, tp;
    if (whole_first) hybrid_schedule(tiles, n_kb, ctas, sg, first, tp);
    else stream_k_schedule(tiles, n_kb, ctas, sg, first, tp);
    const int nseg = static_cast<int>(sg.size() / 4);
    if (nseg > max_segs) return fail(LA_ERR_CAPACITY, "la_gemm_schedule: %d segments, room for %d", nseg, max_segs);
    std::copy(sg.begin(), sg.end(), segs);
    std::copy(first.begin(), first.end(), cta_first);
    std::copy(tp.begin(), tp.end(), planes);
    *ctas_used = static_cast<int32_t>(first.size()) - 1;
    *nseg_out = nseg;
    return LA_OK;
}

// Exported entry points: each runs its body under abi_guard, so no C++
// exception crosses the C ABI.
int la_create(const la_model_dims *dims, const la_weights *w, const la_opts *opts, la_handle **out) {
    return abi_guard("la_create", [&] { return la_create_body(dims, w, opts, out); });
}

int la_prefill(la_handle *h, const int32_t *prompt, int32_t n, int32_t *first_token) {
    return abi_guard("la_prefill", [&] { return la_prefill_body(h, prompt, n, first_token); });
}

int la_step(la_handle *h, int32_t *out_tokens, int32_t *out_n) {
    return abi_guard("la_step", [&] { return la_step_body(h, out_tokens, out_n); });
}

int la_ar_step(la_handle *h, int32_t *token) {
    return abi_guard("la_ar_step", [&] { return la_ar_step_body(h, token); });
}

int la_generate(la_handle *h, const int32_t *prompt, int32_t n, int32_t max_new, int32_t *out, int32_t *out_n,
                int32_t *n_steps) {
    return abi_guard("la_generate", [&] { return la_generate_body(h, prompt, n, max_new, out, out_n, n_steps); });
}

int la_export_state(la_handle *h, la_state_t *stt) {
    return abi_guard("la_export_state", [&] { return la_export_state_body(h, stt); });
}

int la_import_state(la_handle *h, const la_state_t *stt) {
    return abi_guard("la_import_state", [&] { return la_import_state_body(h, stt); });
}

int la_debug_logits(la_handle *h, float *host, int32_t *rows, int32_t *vocab) {
    return abi_guard("la_debug_logits", [&] { return la_debug_logits_body(h, host, rows, vocab); });
}

int la_gemm_bf16(const void *x, const void *w, float *y, int32_t rows, int32_t out, int32_t k, int32_t splits,
                 float *workspace, void *stream) {
    return abi_guard("la_gemm_bf16",
                     [&] { return la_gemm_bf16_body(x, w, y, rows, out, k, splits, workspace, stream); });
}

int la_gemm_status(void *stream) {
    return abi_guard("la_gemm_status", [&] { return la_gemm_status_body(stream); });
}

int la_selftest_timeout(la_handle *h, int64_t limit_ns, void *stream) {
    return abi_guard("la_selftest_timeout", [&] { return la_selftest_timeout_body(h, limit_ns, stream); });
}

int la_step_tables(int32_t N, int32_t W, int32_t G, int32_t *depth, uint32_t *vis, int32_t *used, int32_t max_rows,
                   int32_t *m_out, int32_t *u_out) {
    return abi_guard("la_step_tables",
                     [&] { return la_step_tables_body(N, W, G, depth, vis, used, max_rows, m_out, u_out); });
}

int la_gemm_schedule(int32_t tiles, int32_t n_kb, int32_t ctas, int32_t whole_first, int32_t *segs,
                     int32_t max_segs, int32_t *nseg, int32_t *cta_first, int32_t *ctas_used, int32_t *planes) {
    return abi_guard("la_gemm_schedule", [&] {
        return la_gemm_schedule_body(tiles, n_kb, ctas, whole_first, segs, max_segs, nseg, cta_first, ctas_used,
                                     planes);
    });
}

}  // extern "C"
