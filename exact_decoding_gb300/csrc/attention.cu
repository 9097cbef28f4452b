// Lookahead-masked attention ("Integrated Forward Pass", Figure 2b of the
// paper-graph-ui page): every step row attends to the whole cached prefix
// [0, P) and, inside the step, only to itself and its ancestors (its own
// Jacobi column and the oldest level's left context for lookahead rows, its
// own n-gram's earlier tokens for candidate rows).  The mask is never
// materialised: the prefix part is dense and shared by all rows, the in-step
// part is a short per-row key list.
//
// Pass 1 (k_attn_prefix): split-KV over the prefix.  A CTA stages one 64-key
//   chunk of one KV head in shared memory once and applies it to every query
//   row and every query head of that KV head (all M rows share the prefix,
//   so each prefix K/V byte is read from HBM once per step).  It writes the
//   chunk's (max, sum, unnormalised output) per query.
// Pass 2 (k_attn_final): one warp per (row, head) merges the chunk partials
//   in fixed order, then adds the row's in-step keys with an online softmax
//   (warp-shuffle dot products) and writes the normalised output.
#include <algorithm>
#include <atomic>

#include "la_kernels.h"

namespace la {

template <typename T, int HD>
__global__ void __launch_bounds__(256) k_attn_prefix(const float *q, const T *kc, const T *vc, int max_seq, int P,
                                                     int nrows, int nh, int nkv, float *ws) {
    pdl_trigger();
    pdl_wait();
    constexpr int CH = kAttnChunk;
    constexpr int KT = CH + 4;      // Kt row stride (floats), keeps float4 alignment
    constexpr int QS = HD + 1;      // Qs row stride
    constexpr int PS = CH + 1;      // Ps row stride
    extern __shared__ float sm[];
    float *Kt = sm;                  // [HD][KT]
    float *Vs = Kt + HD * KT;        // [CH][HD]
    float *Qs = Vs + CH * HD;        // [32][QS]
    float *Ps = Qs + 32 * QS;        // [32][PS]
    float *ms = Ps + 32 * PS;        // [32]
    float *ls = ms + 32;             // [32]

    const int kvh = blockIdx.x, chunk = blockIdx.y;
    const int c0 = chunk * CH;
    const int nkeys = min(CH, P - c0);
    const int gq = nh / nkv;
    const int QV = nrows * gq;
    const float scale = rsqrtf(static_cast<float>(HD));
    const T *kb = kc + (static_cast<long long>(kvh) * max_seq + c0) * HD;
    const T *vb = vc + (static_cast<long long>(kvh) * max_seq + c0) * HD;
    for (int t = threadIdx.x; t < CH * HD; t += 256) {
        const int kk = t / HD, i = t % HD;
        const bool in = kk < nkeys;
        Kt[i * KT + kk] = in ? to_f32(kb[t]) : 0.f;
        Vs[kk * HD + i] = in ? to_f32(vb[t]) : 0.f;
    }
    const int tid = threadIdx.x;
    for (int qb = 0; qb < QV; qb += 32) {
        __syncthreads();
        for (int t = tid; t < 32 * HD; t += 256) {
            const int qi = t / HD, i = t % HD;
            const int qv = qb + qi;
            float v = 0.f;
            if (qv < QV) {
                const int r = qv / gq, hq = kvh * gq + qv % gq;
                v = q[(static_cast<long long>(r) * nh + hq) * HD + i] * scale;
            }
            Qs[qi * QS + i] = v;
        }
        __syncthreads();
        // scores: thread -> queries 2*qg, 2*qg+1 and keys 4*kg .. 4*kg+3
        {
            const int qg = tid >> 4, kg = tid & 15;
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            const float *q0 = Qs + (2 * qg) * QS, *q1 = q0 + QS;
#pragma unroll 8
            for (int i = 0; i < HD; ++i) {
                const float4 k4 = *reinterpret_cast<const float4 *>(Kt + i * KT + 4 * kg);
                const float a0 = q0[i], a1 = q1[i];
                acc[0][0] = fmaf(a0, k4.x, acc[0][0]);
                acc[0][1] = fmaf(a0, k4.y, acc[0][1]);
                acc[0][2] = fmaf(a0, k4.z, acc[0][2]);
                acc[0][3] = fmaf(a0, k4.w, acc[0][3]);
                acc[1][0] = fmaf(a1, k4.x, acc[1][0]);
                acc[1][1] = fmaf(a1, k4.y, acc[1][1]);
                acc[1][2] = fmaf(a1, k4.z, acc[1][2]);
                acc[1][3] = fmaf(a1, k4.w, acc[1][3]);
            }
#pragma unroll
            for (int a = 0; a < 2; ++a) {
                float m = -INFINITY;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (4 * kg + j >= nkeys) acc[a][j] = -INFINITY;
                    m = fmaxf(m, acc[a][j]);
                }
#pragma unroll
                for (int o = 8; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                float l = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float pj = (4 * kg + j < nkeys) ? expf(acc[a][j] - m) : 0.f;
                    Ps[(2 * qg + a) * PS + 4 * kg + j] = pj;
                    l += pj;
                }
#pragma unroll
                for (int o = 8; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
                if (kg == 0) {
                    ms[2 * qg + a] = m;
                    ls[2 * qg + a] = l;
                }
            }
        }
        __syncthreads();
        // P . V: thread -> query qo, dims dg*4 + 32*jj + (0..3)
        {
            const int qo = tid >> 3, dg = tid & 7;
            constexpr int NJ = HD / 32;
            float acc[NJ][4];
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) acc[jj][0] = acc[jj][1] = acc[jj][2] = acc[jj][3] = 0.f;
            const float *pr = Ps + qo * PS;
            for (int k = 0; k < CH; ++k) {
                const float pk = pr[k];
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) {
                    const float4 v4 = *reinterpret_cast<const float4 *>(Vs + k * HD + dg * 4 + 32 * jj);
                    acc[jj][0] = fmaf(pk, v4.x, acc[jj][0]);
                    acc[jj][1] = fmaf(pk, v4.y, acc[jj][1]);
                    acc[jj][2] = fmaf(pk, v4.z, acc[jj][2]);
                    acc[jj][3] = fmaf(pk, v4.w, acc[jj][3]);
                }
            }
            const int qv = qb + qo;
            if (qv < QV) {
                const int r = qv / gq, hq = kvh * gq + qv % gq;
                float *w = ws + ((static_cast<long long>(chunk) * nrows + r) * nh + hq) * (HD + 4);
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj)
                    *reinterpret_cast<float4 *>(w + dg * 4 + 32 * jj) =
                        make_float4(acc[jj][0], acc[jj][1], acc[jj][2], acc[jj][3]);
                if (dg == 0) {
                    w[HD] = ms[qo];
                    w[HD + 1] = ls[qo];
                }
            }
        }
    }
}

template <typename T, int HD>
__global__ void __launch_bounds__(256) k_attn_final(const float *q, const T *kc, const T *vc, int max_seq, int P,
                                                    int nrows, int nh, int nkv, const float *ws, int nch,
                                                    const int *anc, const int *anc_cnt, int anc_stride, T *out) {
    pdl_trigger();
    pdl_wait();
    constexpr int DPL = HD / 32;   // dims per lane
    const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= nrows * nh) return;
    const int r = gw / nh, h = gw % nh;
    const int kvh = h / (nh / nkv);
    const float scale = rsqrtf(static_cast<float>(HD));
    float qv[DPL], o[DPL];
    const float *qr = q + (static_cast<long long>(r) * nh + h) * HD + lane * DPL;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
        qv[j] = qr[j] * scale;
        o[j] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int c = 0; c < nch; ++c) {
        const float *w = ws + ((static_cast<long long>(c) * nrows + r) * nh + h) * (HD + 4);
        const float pm = w[HD], pl = w[HD + 1];
        const float nm = fmaxf(m, pm);
        const float a = (m == -INFINITY) ? 0.f : expf(m - nm);
        const float b = expf(pm - nm);
        l = l * a + pl * b;
#pragma unroll
        for (int j = 0; j < DPL; ++j) o[j] = o[j] * a + w[lane * DPL + j] * b;
        m = nm;
    }
    const int cnt = anc ? anc_cnt[r] : r + 1;
    const T *kb = kc + static_cast<long long>(kvh) * max_seq * HD;
    const T *vb = vc + static_cast<long long>(kvh) * max_seq * HD;
    for (int t = 0; t < cnt; ++t) {
        const int a_row = anc ? anc[r * anc_stride + t] : t;
        const long long slot = static_cast<long long>(P + a_row) * HD + lane * DPL;
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < DPL; ++j) s = fmaf(qv[j], to_f32(kb[slot + j]), s);
        s = warp_sum(s);
        const float nm = fmaxf(m, s);
        const float a = (m == -INFINITY) ? 0.f : expf(m - nm);
        const float b = expf(s - nm);
        l = l * a + b;
#pragma unroll
        for (int j = 0; j < DPL; ++j) o[j] = o[j] * a + to_f32(vb[slot + j]) * b;
        m = nm;
    }
    const float inv = 1.f / l;
    T *orow = out + static_cast<long long>(r) * nh * HD + h * HD + lane * DPL;
#pragma unroll
    for (int j = 0; j < DPL; ++j) orow[j] = from_f32<T>(o[j] * inv);
}

// Kernel attributes are per device: bit d of `mask` says they are set on
// device d.  True (with *bit = the current device's bit) while they still
// have to be set there; a device index past 63 sets them on every call.
static bool attrs_needed(const std::atomic<unsigned long long> &mask, unsigned long long *bit) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *bit = 0;
        return true;
    }
    *bit = 1ull << dev;
    return !(mask.load() & *bit);
}

template <typename T, int HD>
static cudaError_t attention_launch_hd(const AttnArgs &a, cudaStream_t s) {
    constexpr int CH = kAttnChunk;
    if (a.nch > 0) {
        const size_t smem = (static_cast<size_t>(HD) * (CH + 4) + CH * HD + 32 * (HD + 1) + 32 * (CH + 1) + 64) *
                            sizeof(float);
        static std::atomic<unsigned long long> configured{0};
        unsigned long long bit = 0;
        if (attrs_needed(configured, &bit)) {
            cudaError_t e = cudaFuncSetAttribute(k_attn_prefix<T, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            configured.fetch_or(bit);
        }
        dim3 grid(a.nkv, a.nch);
        launch_k(k_attn_prefix<T, HD>, dim3(grid), dim3(256), smem, s, a.q, a.kc, a.vc,
                                                     a.max_seq, a.P, a.nrows, a.nh, a.nkv, a.ws);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const int warps = a.nrows * a.nh;
    launch_k(k_attn_final<T, HD>, dim3((warps + 7) / 8), dim3(256), 0, s, a.q, a.kc, a.vc, a.max_seq, a.P, a.nrows, a.nh,
                                                         a.nkv, a.ws, a.nch, a.anc, a.anc_cnt, a.anc_stride,
                                                         static_cast<T *>(a.out));
    return cudaGetLastError();
}

cudaError_t attention_launch(const AttnArgs &a, cudaStream_t s) {
    if (a.hd == 128) return attention_launch_hd<float, 128>(a, s);
    if (a.hd == 64) return attention_launch_hd<float, 64>(a, s);
    return cudaErrorInvalidValue;
}

// ========================================================================== tcgen05 path (bf16 models)
// One cluster of `cs` CTAs per (KV head g, tile of 128 query vectors).
// Prologue: the cluster's CTAs share the work of summing the QKV GEMM's
// partial planes for KV head g, rotating q and k, scaling q, and writing the
// (hi, lo) planes of the tile's query vectors and of this step's K/V rows
// (clusters of the same KV head write identical K/V bytes); a proxy fence and
// a cluster barrier then make those writes visible to the TMA loads.  CTA
// rank j of the cluster takes the 128-key chunks [j n / cs, (j + 1) n / cs)
// of the keys [0, P + nrows): the cached prefix, then this step's own rows.
// Per chunk:
//   TMA   K (hi, lo) [128 keys x hd] and V^T (hi, lo) [hd x 128 keys]
//   UMMA  S = Qh Kh^T + Qh Kl^T + Ql Kh^T          (TMEM columns 0..127)
//   TMA   as soon as S is done, the next chunk's K into the same buffer
//   warps 16 warps, each a 32-query x 32-key block of S (a warp reads only
//         its own quarter of the TMEM lanes): mask, running max through
//         shared memory, P = exp(S - m) split into (hi, lo) bf16 pairs and
//         stored into TMEM (columns 256.. and 320..) as the next UMMA's A
//         operand; O of earlier chunks rescaled in TMEM
//   UMMA  O += Ph Vh + Ph Vl + Pl Vh                (A from TMEM; O in TMEM columns 128..)
//   TMA   the next chunk's V
// The products keep about 16 mantissa bits (the lo * lo term is dropped),
// the softmax is fp32.  At the end each CTA leaves (O, m, l) per query
// vector in its shared memory, and after a cluster barrier CTA j merges
// rows [j 128 / cs, (j + 1) 128 / cs) of all cs partials, read through
// distributed shared memory, and writes the normalised output.
constexpr int kUKeys = 128;                  // keys per chunk
constexpr int kUQ = 128;                     // query vectors per tile (UMMA M)
constexpr int kUThreads = 512;               // 16 warps: 4 lane quarters x 4 column quarters
constexpr uint32_t kUBox = 128u * 128u;      // bytes of a [128 rows x 64 bf16] swizzled box
constexpr float kLog2e = 1.4426950408889634f;
// TMEM columns: S [0, 128), O [128, 128 + hd), P hi [256, 320), P lo [320, 384)
// (a bf16 pair of keys per 32-bit column).
constexpr uint32_t kTmemO = 128, kTmemPh = 256, kTmemPl = 320, kTmemCols = 512;

// O (+)= A * B^T with A (M x 16, bf16) read from tensor memory at a_tmem and
// B from shared memory (descriptor), one UMMA of shape M x N x 16.
static __device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

template <int HD>
struct AttnLayout {
    static constexpr uint32_t q_bytes = 2u * (HD / 64) * kUBox;          // (hi, lo) x d blocks of 64
    static constexpr uint32_t k_bytes = 2u * (HD / 64) * kUBox;
    static constexpr uint32_t kp_bytes = k_bytes;                        // K only: P lives in TMEM
    static constexpr uint32_t vbox = static_cast<uint32_t>(HD) * 128u;   // [hd rows x 64 keys]
    static constexpr uint32_t v_bytes = 2u * (kUKeys / 64) * vbox;
    static constexpr int o_ld = HD + 4;                                  // floats per merge row
    static constexpr uint32_t q_off = 0, kp_off = q_bytes, v_off = kp_off + kp_bytes;
    static constexpr uint32_t ml_off = v_off + v_bytes;                  // m[128], l[128]
    static constexpr uint32_t red_off = ml_off + 2u * kUQ * 4u;          // [4][128] per-quarter partials
    static constexpr uint32_t vis_off = red_off + 4u * kUQ * 4u;         // [128][8] visibility words; merge weights
    static constexpr uint32_t tab_off = vis_off + kUQ * 8u * 4u;         // [128] row depths, [256] plane counts
    static constexpr uint32_t bar_off = tab_off + (kUQ + 256u) * 4u;     // 4 mbarriers + TMEM slot
    static constexpr uint32_t bytes = bar_off + 64u + 1024u;             // + alignment slack
    static_assert(static_cast<uint32_t>(kUQ) * o_ld * 4u <= q_bytes + kp_bytes, "merge rows overlay Q and K/P");
};

static __device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}

template <int HD>
__global__ void __launch_bounds__(kUThreads, 1) k_attn_umma(const __grid_constant__ AttnUmmaParams p) {
    using Lay = AttnLayout<HD>;
    constexpr int kCW = HD / 4;   // O columns per warp
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t s_q = smem_u32(smem + Lay::q_off), s_kp = smem_u32(smem + Lay::kp_off);
    const uint32_t s_v = smem_u32(smem + Lay::v_off);
    float *sm_m = reinterpret_cast<float *>(smem + Lay::ml_off);
    float *sm_l = sm_m + kUQ;
    float *red = reinterpret_cast<float *>(smem + Lay::red_off);
    uint32_t *svis = reinterpret_cast<uint32_t *>(smem + Lay::vis_off);
    float *wsm = reinterpret_cast<float *>(smem + Lay::vis_off);   // merge weights, after the last chunk
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::bar_off);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 4);
    float *so = reinterpret_cast<float *>(smem);   // merge rows, over Q and K/P once the MMAs are done

    pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qw = warp & 3, cw = warp >> 2;   // TMEM lane quarter, column quarter
    const int row = 32 * qw + lane;            // this thread's query vector within the tile
    const uint32_t rank = cluster_ctarank();
    const int cs = static_cast<int>(gridDim.x);   // the cluster spans x
    const int g = static_cast<int>(blockIdx.y) / p.mtiles, qt = static_cast<int>(blockIdx.y) % p.mtiles;
    // Prefix length: from the device step state when given (a captured step
    // graph), else the launch parameter.  Written before this step began.
    const int P = p.P_dev ? *p.P_dev : p.P;
    const int nchunks = (P + p.nrows + kUKeys - 1) / kUKeys;
    const int c_beg = static_cast<int>(static_cast<long long>(rank) * nchunks / cs);
    const int c_end = static_cast<int>(static_cast<long long>(rank + 1) * nchunks / cs);
    // bar_ld: Q (first chunk) and K landed; bar_v: V landed; bar_s / bar_pv: MMAs done.
    const uint32_t bar_ld = smem_u32(&bars[0]), bar_s = smem_u32(&bars[1]), bar_pv = smem_u32(&bars[2]);
    const uint32_t bar_v = smem_u32(&bars[3]);

    if (tid == 0) {
        mbar_init(bar_ld, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_pv, 1);
        mbar_init(bar_v, 1);
        fence_barrier_init();
        prefetch_tensormap(&p.tq);
        prefetch_tensormap(&p.tk);
        prefetch_tensormap(&p.tv);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_off = static_cast<uint32_t>(32 * qw) << 16;
    const uint32_t t_s = tmem + lane_off + static_cast<uint32_t>(32 * cw);              // 32 S columns
    const uint32_t t_o = tmem + lane_off + kTmemO + static_cast<uint32_t>(kCW * cw);    // kCW O columns
    const uint32_t t_ph = tmem + lane_off + kTmemPh + static_cast<uint32_t>(16 * cw);   // this warp's 32 keys of P
    const uint32_t t_pl = tmem + lane_off + kTmemPl + static_cast<uint32_t>(16 * cw);

    const int QV = p.nrows * p.gq;
    const int qv = qt * kUQ + row;
    const bool valid = qv < QV;
    const int r = valid ? qv / p.gq : 0;

    const long long krows_plane = static_cast<long long>(p.nkv) * p.seq;   // K rows from hi to lo plane
    const int vrows_plane = p.nkv * HD;
    const int ky0 = (p.layer * 2 * p.nkv + g) * p.seq;
    const int vy0 = (p.layer * 2 * p.nkv + g) * HD;
    // K of chunk c completes on bar_ld (the caller accounts its bytes), V on
    // bar_v; S can start while V lands.  Issued by thread 0, which counts them.
    int k_issued = 0, v_issued = 0;
    auto issue_k = [&](int c, uint64_t pol) {
        const int key0 = c * kUKeys;
#pragma unroll
        for (int pl = 0; pl < 2; ++pl)
#pragma unroll
            for (int db = 0; db < HD / 64; ++db)
                tma_load_2d(s_kp + (pl * (HD / 64) + db) * kUBox, &p.tk, db * 64,
                            static_cast<int>(ky0 + pl * krows_plane + key0), bar_ld, pol);
        ++k_issued;
    };
    auto issue_v = [&](int c, uint64_t pol) {
        const int key0 = c * kUKeys;
        mbar_arrive_expect_tx(bar_v, Lay::v_bytes);
#pragma unroll
        for (int pl = 0; pl < 2; ++pl)
#pragma unroll
            for (int kb = 0; kb < kUKeys / 64; ++kb)
                tma_load_2d(s_v + (pl * (kUKeys / 64) + kb) * Lay::vbox, &p.tv, key0 + kb * 64, vy0 + pl * vrows_plane,
                            bar_v, pol);
        ++v_issued;
    };
    auto issue_kv = [&](int c, uint64_t pol) {
        issue_k(c, pol);
        issue_v(c, pol);
    };
    // Cached-prefix chunk first in line: its K/V were written before this
    // launch began, so they load while the prologue runs.
    const bool early = p.prefix_early && c_beg < c_end && (c_beg + 1) * kUKeys <= P;
    if (tid == 0 && early) {
        mbar_expect_tx(bar_ld, Lay::k_bytes);
        issue_kv(c_beg, policy_evict_normal());
    }
    // Tables written once at create time (safe to read before the wait):
    // the step rows' depths and the QKV tiles' partial-plane counts.
    int *sdep = reinterpret_cast<int *>(smem + Lay::tab_off);
    int *splanes = sdep + kUQ;
    for (int i = tid; i < kUQ + 256; i += kUThreads) {
        if (i < kUQ) sdep[i] = i < p.nrows ? (p.depth ? p.depth[i] : i) : 0;
        else splanes[i - kUQ] = (p.planes && i - kUQ < p.qkv_tiles) ? p.planes[i - kUQ] : 1;
    }
    __syncthreads();
    auto nplanes = [&](int col) -> int {
        const int t = col >> 7;
        return !p.planes ? 1 : (t < 256 ? splanes[t] : p.planes[t]);
    };
    pdl_wait();   // the QKV planes and the visibility bits come from earlier kernels
    {
        // Prologue work items (rows fastest for v, so the transposed stores of a
        // warp hit consecutive slots), two per iteration so that their loads
        // are in flight together:
        //   q: (query vector of this tile, 4 rotary pairs i..i+3)
        //   k: (step row, 4 rotary pairs)          v: (step row, 8 dims)
        constexpr int half = HD / 2, Q4 = HD / 8, D8 = HD / 8;
        const int qv0 = qt * kUQ, nqv = max(0, min(kUQ, QV - qv0));
        const int nq = nqv * Q4, nk = p.nrows * Q4, nv = p.nrows * D8, total = nq + nk + nv;
        const float scale = rsqrtf(static_cast<float>(HD));
        const int stride = cs * kUThreads;
        struct Item {
            float4 a, b, c01, c23;   // rotary: x1, x2, (cos, sin) pairs; v: dims 0..3, 4..7
            long long dst, lo;
            int kind, j;             // 0 q, 1 k, 2 v, -1 none
        };
        auto load = [&](int t, Item &it) {
            it.kind = -1;
            if (t >= total) return;
            if (t < nq + nk) {
                const bool isq = t < nq;
                const int u = isq ? t : t - nq;
                int r, col0;
                it.j = u % Q4;
                if (isq) {
                    const int qvv = qv0 + u / Q4;
                    r = qvv / p.gq;
                    col0 = (g * p.gq + qvv % p.gq) * HD;
                    it.dst = (static_cast<long long>(g) * p.qv_pad + qvv) * HD;
                    it.lo = static_cast<long long>(p.nkv) * p.qv_pad * HD;
                } else {
                    r = u / Q4;
                    col0 = p.k_off + g * HD;
                    it.dst = ((static_cast<long long>(p.layer) * 2 * p.nkv + g) * p.seq + P + r) * HD;
                    it.lo = static_cast<long long>(p.nkv) * p.seq * HD;
                }
                it.kind = isq ? 0 : 1;
                // step rows sit at P + depth (the table covers a step's <= 128
                // rows); prefill rows at P + r
                const float2 *rr = p.rope + static_cast<long long>(P + (p.depth ? sdep[r] : r)) * half + 4 * it.j;
                it.c01 = *reinterpret_cast<const float4 *>(rr);
                it.c23 = *reinterpret_cast<const float4 *>(rr + 2);
                const int np = nplanes(col0);
                const float *pr = p.part + static_cast<long long>(r) * p.ldp + col0 + 4 * it.j;
                sum_planes4x2(pr, np, pr + half, np, p.sstride, it.a, it.b);
            } else {
                const int u = t - nq - nk, r = u % p.nrows, d8 = u / p.nrows;
                const int col = p.v_off + g * HD + 8 * d8;
                const float *pr = p.part + static_cast<long long>(r) * p.ldp + col;
                const int np = nplanes(col);
                sum_planes4x2(pr, np, pr + 4, np, p.sstride, it.a, it.b);
                it.kind = 2;
                it.lo = static_cast<long long>(p.nkv) * HD * p.seq;
                it.dst = ((static_cast<long long>(p.layer) * 2 * p.nkv + g) * HD + 8 * d8) * p.seq + P + r;
            }
        };
        auto store = [&](const Item &it) {
            if (it.kind < 0) return;
            if (it.kind < 2) {
                const float4 x1 = it.a, x2 = it.b, c01 = it.c01, c23 = it.c23;
                float4 y1 = make_float4(x1.x * c01.x - x2.x * c01.y, x1.y * c01.z - x2.y * c01.w,
                                        x1.z * c23.x - x2.z * c23.y, x1.w * c23.z - x2.w * c23.w);
                float4 y2 = make_float4(x1.x * c01.y + x2.x * c01.x, x1.y * c01.w + x2.y * c01.z,
                                        x1.z * c23.y + x2.z * c23.x, x1.w * c23.w + x2.w * c23.z);
                if (it.kind == 0) {
                    y1 = make_float4(y1.x * scale, y1.y * scale, y1.z * scale, y1.w * scale);
                    y2 = make_float4(y2.x * scale, y2.y * scale, y2.z * scale, y2.w * scale);
                }
                __nv_bfloat16 *base = it.kind == 0 ? p.q : p.kc;
                store_act4(base, it.dst + 4 * it.j, y1, it.lo);
                store_act4(base, it.dst + half + 4 * it.j, y2, it.lo);
            } else {
                const float v[8] = {it.a.x, it.a.y, it.a.z, it.a.w, it.b.x, it.b.y, it.b.z, it.b.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) store_act(p.vc, it.dst + static_cast<long long>(e) * p.seq, v[e], it.lo);
            }
        };
        for (int t = static_cast<int>(rank) * kUThreads + tid; t < total; t += 2 * stride) {
            Item i0, i1;
            load(t, i0);
            load(t + stride, i1);
            store(i0);
            store(i1);
        }
        // These generic-proxy global writes are read next by TMA (async proxy)
        // in every CTA of the cluster.
        __threadfence();
        asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    cluster_sync_all();
    if (cw == 0) {
#pragma unroll
        for (int w = 0; w < 8; ++w) svis[row * 8 + w] = (valid && p.vis_bits) ? p.vis_bits[r * 8 + w] : 0u;
    }
    const uint32_t *myvis = svis + row * 8;
    // Visibility of keys [k0, k0 + 32) for this query vector, bit j = key k0 + j.
    auto vis_word = [&](int k0) -> uint32_t {
        if (!valid) return 0u;
        const int s0 = k0 - P;   // step index of bit 0 (negative: cached prefix)
        uint32_t pre = 0u;
        if (s0 <= -32) return 0xffffffffu;
        if (s0 < 0) pre = (1u << (-s0)) - 1u;
        // in-step keys: bit j is step index s0 + j, valid for 0 <= s0 + j < nrows
        uint32_t st;
        if (p.vis_bits) {
            if (s0 >= 0) {
                const int w = s0 >> 5, sh = s0 & 31;
                const uint32_t lo = w < 8 ? myvis[w] : 0u, hi = w + 1 < 8 ? myvis[w + 1] : 0u;
                st = __funnelshift_r(lo, hi, sh);
            } else {
                st = myvis[0] << (-s0);
            }
        } else {
            // causal: step indices 0..r
            const int last = r - s0;   // highest visible bit
            st = last < 0 ? 0u : (last >= 31 ? 0xffffffffu : ((2u << last) - 1u));
            if (s0 < 0) st &= ~pre;
        }
        const int lim = p.nrows - s0;   // bits at or above lim are past the step rows
        const uint32_t live = lim <= 0 ? 0u : (lim >= 32 ? 0xffffffffu : ((1u << lim) - 1u));
        return pre | (st & live & ~pre);
    };

    if (tid == 0 && c_beg < c_end) {
        asm volatile("fence.proxy.async.global;" ::: "memory");
        const uint64_t pol = policy_evict_normal();   // other query tiles of this KV head read the same chunks
        mbar_arrive_expect_tx(bar_ld, early ? Lay::q_bytes : Lay::q_bytes + Lay::k_bytes);
#pragma unroll
        for (int pl = 0; pl < 2; ++pl)
#pragma unroll
            for (int db = 0; db < HD / 64; ++db)
                tma_load_2d(s_q + (pl * (HD / 64) + db) * kUBox, &p.tq, db * 64, (pl * p.nkv + g) * p.qv_pad + qt * kUQ,
                            bar_ld, pol);
        if (!early) issue_kv(c_beg, pol);
    }

    const uint32_t idesc_s = umma_idesc_bf16(kUQ, kUKeys), idesc_o = umma_idesc_bf16(kUQ, HD);
    float m_run = -INFINITY, l_part = 0.f;   // l_part: this warp's quarter of the keys
    bool ok = true;
    int it = 0;
    for (int c = c_beg; c < c_end; ++c, ++it) {
        const uint32_t ph = static_cast<uint32_t>(it & 1);
        bool w0 = true;
        if (tid == 0) w0 = mbar_wait(bar_ld, ph, p.err, ERR_TIMEOUT_ATTN);
        ok = __syncthreads_and(ok && w0);
        if (!ok) break;
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int db = 0; db < HD / 64; ++db) {
                const uint64_t qh = umma_desc_sw128(s_q + db * kUBox), ql = umma_desc_sw128(s_q + (HD / 64 + db) * kUBox);
                const uint64_t kh = umma_desc_sw128(s_kp + db * kUBox), kl = umma_desc_sw128(s_kp + (HD / 64 + db) * kUBox);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    umma_bf16(tmem, qh + 2 * kk, kh + 2 * kk, idesc_s, (db | kk) ? 1u : 0u);
                    umma_bf16(tmem, qh + 2 * kk, kl + 2 * kk, idesc_s, 1u);
                    umma_bf16(tmem, ql + 2 * kk, kh + 2 * kk, idesc_s, 1u);
                }
            }
            umma_commit(bar_s);
            w0 = mbar_wait(bar_s, ph, p.err, ERR_TIMEOUT_ATTN);
            if (w0 && c + 1 < c_end) {   // S has read K: the next chunk's K loads during softmax and P.V
                mbar_arrive_expect_tx(bar_ld, Lay::k_bytes);
                issue_k(c + 1, policy_evict_normal());
            }
        }
        ok = __syncthreads_and(w0);
        if (!ok) break;
        tc_fence_after();

        // This warp's 32 x 32 block of S: masked max, shared with the other
        // three column quarters of the same query vectors.
        const int key0 = c * kUKeys;
        const uint32_t mw = vis_word(key0 + 32 * cw);
        uint32_t v[32];
        tmem_ld_32x32b_x32(t_s, v);
        tmem_ld_wait();
        float mc = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if ((mw >> j) & 1u) mc = fmaxf(mc, __uint_as_float(v[j]));
        red[cw * kUQ + row] = mc;
        __syncthreads();
        mc = fmaxf(fmaxf(red[row], red[kUQ + row]), fmaxf(red[2 * kUQ + row], red[3 * kUQ + row]));
        const float m_new = fmaxf(m_run, mc);
        const float alpha = m_run == -INFINITY ? 0.f : exp2f((m_run - m_new) * kLog2e);
        float pv[32];
        float ls = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            pv[j] = ((mw >> j) & 1u) ? exp2f((__uint_as_float(v[j]) - m_new) * kLog2e) : 0.f;
            ls += pv[j];
        }
        l_part = l_part * alpha + ls;
        // Keys 32 cw .. 32 cw + 31 of this query vector's P row, as (hi, lo)
        // bf16 pairs, into TMEM: column 16 cw + j holds keys 32 cw + 2j (low
        // half) and 32 cw + 2j + 1.
        {
            uint32_t hh[16], ll[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float a = pv[2 * e], b = pv[2 * e + 1];
                const __nv_bfloat162 hb = __floats2bfloat162_rn(a, b);
                const float2 hf = __bfloat1622float2(hb);
                hh[e] = *reinterpret_cast<const uint32_t *>(&hb);
                ll[e] = pack_bf16x2(a - hf.x, b - hf.y);
            }
            tmem_st_32x32b_x16(t_ph, hh);
            tmem_st_32x32b_x16(t_pl, ll);
        }
        // O of the earlier chunks (in TMEM) to the new running max.
        if (it > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
            if constexpr (kCW == 32) {
                uint32_t o[32];
                tmem_ld_32x32b_x32(t_o, o);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                tmem_st_32x32b_x32(t_o, o);
            } else {
                uint32_t o[16];
                tmem_ld_32x32b_x16(t_o, o);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                tmem_st_32x32b_x16(t_o, o);
            }
            tmem_st_wait();
        }
        m_run = m_new;
        tmem_st_wait();
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && mbar_wait(bar_v, ph, p.err, ERR_TIMEOUT_ATTN)) {
            tc_fence_after();
#pragma unroll
            for (int kb = 0; kb < kUKeys / 64; ++kb) {
                const uint64_t vh = umma_desc_sw128(s_v + kb * Lay::vbox);
                const uint64_t vl = umma_desc_sw128(s_v + (kUKeys / 64 + kb) * Lay::vbox);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t pc = static_cast<uint32_t>(kb * 32 + kk * 8);   // 16 keys = 8 columns
                    umma_bf16_tmem_a(tmem + kTmemO, tmem + kTmemPh + pc, vh + 2 * kk, idesc_o, (it | kb | kk) ? 1u : 0u);
                    umma_bf16_tmem_a(tmem + kTmemO, tmem + kTmemPh + pc, vl + 2 * kk, idesc_o, 1u);
                    umma_bf16_tmem_a(tmem + kTmemO, tmem + kTmemPl + pc, vh + 2 * kk, idesc_o, 1u);
                }
            }
            umma_commit(bar_pv);
            w0 = mbar_wait(bar_pv, ph, p.err, ERR_TIMEOUT_ATTN);
            if (w0 && c + 1 < c_end) issue_v(c + 1, policy_evict_normal());   // V is free again
        } else if (tid == 0) {
            w0 = false;   // V never landed
        }
        ok = __syncthreads_and(w0);
        if (!ok) break;
        tc_fence_after();
    }
    if (!ok) {   // a load or an MMA never completed: wait (bounded) for TMA still in flight
        m_run = -INFINITY;
        l_part = 0.f;
        if (tid == 0) {
            for (int j = it; j < k_issued; ++j) mbar_wait(bar_ld, static_cast<uint32_t>(j & 1), p.err, ERR_TIMEOUT_ATTN);
            for (int j = it; j < v_issued; ++j) mbar_wait(bar_v, static_cast<uint32_t>(j & 1), p.err, ERR_TIMEOUT_ATTN);
        }
    }

    // Partials to this CTA's shared memory: O rows, m, and l summed over the
    // four column quarters.
    __syncthreads();
    {
        float *orow = so + row * Lay::o_ld + kCW * cw;
        const bool have = ok && it > 0;
        if constexpr (kCW == 32) {
            uint32_t o[32];
            if (have) {
                tmem_ld_32x32b_x32(t_o, o);
                tmem_ld_wait();
            }
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4 *>(orow + j) =
                    have ? make_float4(__uint_as_float(o[j]), __uint_as_float(o[j + 1]), __uint_as_float(o[j + 2]),
                                       __uint_as_float(o[j + 3]))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            uint32_t o[16];
            if (have) {
                tmem_ld_32x32b_x16(t_o, o);
                tmem_ld_wait();
            }
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4 *>(orow + j) =
                    have ? make_float4(__uint_as_float(o[j]), __uint_as_float(o[j + 1]), __uint_as_float(o[j + 2]),
                                       __uint_as_float(o[j + 3]))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        red[cw * kUQ + row] = l_part;
        if (cw == 0) sm_m[row] = m_run;
    }
    __syncthreads();
    if (cw == 0) sm_l[row] = red[row] + red[kUQ + row] + red[2 * kUQ + row] + red[3 * kUQ + row];
    tc_fence_before();
    cluster_sync_all();
    // Merge rows [rank 128 / cs, (rank + 1) 128 / cs) of the cs partials:
    // per-row weights exp(m_j - max) / sum first, then float4 columns.
    const int r_beg = static_cast<int>(rank) * kUQ / cs, rows_per = (static_cast<int>(rank) + 1) * kUQ / cs - r_beg;
    for (int i = tid; i < rows_per; i += kUThreads) {
        const int mr = r_beg + i;
        float mj[8];
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            mj[j] = j < cs ? ld_cluster_f32(mapa_shared(smem_u32(&sm_m[mr]), static_cast<uint32_t>(j))) : -INFINITY;
            mx = fmaxf(mx, mj[j]);
        }
        float L = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            mj[j] = mj[j] == -INFINITY ? 0.f : exp2f((mj[j] - mx) * kLog2e);
            if (mj[j] != 0.f) L += mj[j] * ld_cluster_f32(mapa_shared(smem_u32(&sm_l[mr]), static_cast<uint32_t>(j)));
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) wsm[i * 8 + j] = mj[j] * inv;
    }
    __syncthreads();
    constexpr int G4 = HD / 4;
    for (int i = tid; i < rows_per * G4; i += kUThreads) {
        const int li = i / G4, d = (i % G4) * 4;
        const int mr = r_beg + li;
        const int qvr = qt * kUQ + mr;
        if (qvr >= QV) continue;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float w = wsm[li * 8 + j];
            if (w == 0.f) continue;
            const float4 x = ld_cluster_f32x4(mapa_shared(smem_u32(so + mr * Lay::o_ld + d), static_cast<uint32_t>(j)));
            acc.x += w * x.x;
            acc.y += w * x.y;
            acc.z += w * x.z;
            acc.w += w * x.w;
        }
        const int rr = qvr / p.gq, head = g * p.gq + qvr % p.gq;
        const long long ob = (static_cast<long long>(rr) * p.nh + head) * HD + d;
        const __nv_bfloat162 h01 = __floats2bfloat162_rn(acc.x, acc.y), h23 = __floats2bfloat162_rn(acc.z, acc.w);
        const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
        uint2 hv, lv;
        hv.x = *reinterpret_cast<const uint32_t *>(&h01);
        hv.y = *reinterpret_cast<const uint32_t *>(&h23);
        lv.x = pack_bf16x2(acc.x - f01.x, acc.y - f01.y);
        lv.y = pack_bf16x2(acc.z - f23.x, acc.w - f23.y);
        *reinterpret_cast<uint2 *>(p.out + ob) = hv;
        *reinterpret_cast<uint2 *>(p.out + ob + p.out_lo_off) = lv;
    }
    cluster_sync_all();   // peers are done reading this CTA's shared memory
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int HD>
static cudaError_t attention_umma_hd(const AttnUmmaParams &p, int cs, cudaStream_t s) {
    using Lay = AttnLayout<HD>;
    static std::atomic<unsigned long long> configured{0};
    unsigned long long bit = 0;
    if (attrs_needed(configured, &bit)) {
        cudaError_t e = cudaFuncSetAttribute(k_attn_umma<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(Lay::bytes));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k_attn_umma<HD>, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, p.nkv * p.mtiles);
    cfg.blockDim = dim3(kUThreads);
    cfg.dynamicSmemBytes = Lay::bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cs;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k_attn_umma<HD>, p);
}

bool attention_umma_maps(AttnUmmaParams &p, const void *q, const void *kc, const void *vc, int L) {
    const int hd = p.hd;
    if (make_tmap_bf16(&p.tq, q, hd, static_cast<uint64_t>(2) * p.nkv * p.qv_pad, static_cast<uint64_t>(hd) * 2, 64,
                       kUQ))
        return false;
    if (make_tmap_bf16(&p.tk, kc, hd, static_cast<uint64_t>(L) * 2 * p.nkv * p.seq, static_cast<uint64_t>(hd) * 2, 64,
                       kUKeys))
        return false;
    if (make_tmap_bf16(&p.tv, vc, p.seq, static_cast<uint64_t>(L) * 2 * p.nkv * hd, static_cast<uint64_t>(p.seq) * 2,
                       64, static_cast<uint32_t>(hd)))
        return false;
    return true;
}

cudaError_t attention_umma_launch(AttnUmmaParams p, int nsm, int P_max, cudaStream_t s) {
    const int nchunks = (std::max(P_max, p.P) + p.nrows + kUKeys - 1) / kUKeys;
    p.mtiles = (p.nrows * p.gq + kUQ - 1) / kUQ;
    const int units = p.nkv * p.mtiles;
    // One chunk per CTA where the SMs allow it (clusters of up to 8 CTAs).
    int cs = std::min(std::min(8, nchunks), std::max(1, nsm / units));
    if (p.hd == 128) return attention_umma_hd<128>(p, cs, s);
    if (p.hd == 64) return attention_umma_hd<64>(p, cs, s);
    return cudaErrorInvalidValue;
}

}  // namespace la
