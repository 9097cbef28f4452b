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
#include "la_kernels.h"

namespace la {

template <typename T, int HD>
__global__ void __launch_bounds__(256) k_attn_prefix(const float *q, const T *kc, const T *vc, int max_seq, int P,
                                                     int nrows, int nh, int nkv, float *ws) {
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

template <typename T, int HD>
static cudaError_t attention_launch_hd(const AttnArgs &a, cudaStream_t s) {
    constexpr int CH = kAttnChunk;
    if (a.nch > 0) {
        const size_t smem = (static_cast<size_t>(HD) * (CH + 4) + CH * HD + 32 * (HD + 1) + 32 * (CH + 1) + 64) *
                            sizeof(float);
        static bool configured = false;
        if (!configured) {
            cudaError_t e = cudaFuncSetAttribute(k_attn_prefix<T, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            configured = true;
        }
        dim3 grid(a.nkv, a.nch);
        k_attn_prefix<T, HD><<<grid, 256, smem, s>>>(a.q, static_cast<const T *>(a.kc), static_cast<const T *>(a.vc),
                                                     a.max_seq, a.P, a.nrows, a.nh, a.nkv, a.ws);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const int warps = a.nrows * a.nh;
    k_attn_final<T, HD><<<(warps + 7) / 8, 256, 0, s>>>(a.q, static_cast<const T *>(a.kc),
                                                         static_cast<const T *>(a.vc), a.max_seq, a.P, a.nrows, a.nh,
                                                         a.nkv, a.ws, a.nch, a.anc, a.anc_cnt, a.anc_stride,
                                                         static_cast<T *>(a.out));
    return cudaGetLastError();
}

template <typename T>
cudaError_t attention_launch(const AttnArgs &a, cudaStream_t s) {
    if (a.hd == 128) return attention_launch_hd<T, 128>(a, s);
    if (a.hd == 64) return attention_launch_hd<T, 64>(a, s);
    return cudaErrorInvalidValue;
}

template cudaError_t attention_launch<float>(const AttnArgs &, cudaStream_t);
template cudaError_t attention_launch<__nv_bfloat16>(const AttnArgs &, cudaStream_t);

}  // namespace la
