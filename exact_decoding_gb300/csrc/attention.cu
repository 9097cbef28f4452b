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

template <typename T>
cudaError_t attention_launch(const AttnArgs &a, cudaStream_t s) {
    if (a.hd == 128) return attention_launch_hd<T, 128>(a, s);
    if (a.hd == 64) return attention_launch_hd<T, 64>(a, s);
    return cudaErrorInvalidValue;
}

template cudaError_t attention_launch<float>(const AttnArgs &, cudaStream_t);

// ========================================================================== tensor-core path (bf16 models)
// One CTA = (KV head, 64-key chunk, 64 query vectors); 4 warps x 16 queries.
// Chunks [0, nch_prefix) cover the cached prefix [0, P), visible to every
// row.  Chunks from nch_prefix on cover this step's own rows (slots P + s):
// row r sees step key s iff bit s of vis_bits[r] is set (tree mode) or s <= r
// (causal mode).
//
// Precision: K, V and q are fp32.  Each is split into bf16 planes hi + lo in
// shared memory and every product runs as three bf16 MMAs (hi*hi + hi*lo +
// lo*hi, fp32 accumulate) on mma.sync m16n8k16, which keeps about 16
// mantissa bits; the softmax is fp32 in registers and P is split the same
// way for P V.  Each CTA writes the chunk's (unnormalised O, max, sum) per
// query; k_attn_merge combines the chunks in order.
namespace {

constexpr int kTcChunk = 64;
constexpr int kTcQ = 64;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// bf16 pair (lo element first) for hi and for the remainder lo.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

template <int HD>
__global__ void __launch_bounds__(128) k_attn_tc(const float *q, const float *kc, const float *vc, int max_seq, int P,
                                                 int nrows, int nh, int nkv, int nch_prefix, const uint32_t *vis_bits,
                                                 float *ws) {
    pdl_trigger();
    pdl_wait();
    constexpr int LD = HD + 8;   // smem row stride (bf16): 16-byte aligned rows, conflict-free ldmatrix
    extern __shared__ __align__(16) __nv_bfloat16 smb[];
    __nv_bfloat16 *Kh = smb;                     // [kTcChunk][LD] each
    __nv_bfloat16 *Kl = Kh + kTcChunk * LD;
    __nv_bfloat16 *Vh = Kl + kTcChunk * LD;
    __nv_bfloat16 *Vl = Vh + kTcChunk * LD;

    const int kvh = blockIdx.x, chunk = blockIdx.y, qb = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = nh / nkv;
    const int QV = nrows * gq;
    const bool step_chunk = chunk >= nch_prefix;
    const int key0 = step_chunk ? (chunk - nch_prefix) * kTcChunk : chunk * kTcChunk;   // step index or position
    const int slot0 = step_chunk ? P + key0 : key0;
    const int nkeys = step_chunk ? min(kTcChunk, nrows - key0) : min(kTcChunk, P - key0);

    // K / V chunk -> shared hi/lo planes (keys past the chunk are zero).
    // All of a thread's loads are issued before any conversion.  Plain
    // (coherent) loads: with programmatic dependent launch this kernel's
    // lifetime overlaps the kernel that writes q, K and V, so the
    // read-only cache path must not be used for them.
    {
        const float *kb = kc + (static_cast<long long>(kvh) * max_seq + slot0) * HD;
        const float *vb = vc + (static_cast<long long>(kvh) * max_seq + slot0) * HD;
        constexpr int PER = kTcChunk * (HD / 4) / 128;   // float4 per thread per tensor
        float4 kx[PER], vx[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int t = tid + j * 128;
            const int key = t / (HD / 4), c = (t % (HD / 4)) * 4;
            if (key < nkeys) {
                kx[j] = *reinterpret_cast<const float4 *>(kb + static_cast<long long>(key) * HD + c);
                vx[j] = *reinterpret_cast<const float4 *>(vb + static_cast<long long>(key) * HD + c);
            } else {
                kx[j] = vx[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int t = tid + j * 128;
            const int key = t / (HD / 4), c = (t % (HD / 4)) * 4;
            uint2 h, l;
            split2(kx[j].x, kx[j].y, h.x, l.x);
            split2(kx[j].z, kx[j].w, h.y, l.y);
            *reinterpret_cast<uint2 *>(Kh + key * LD + c) = h;
            *reinterpret_cast<uint2 *>(Kl + key * LD + c) = l;
            split2(vx[j].x, vx[j].y, h.x, l.x);
            split2(vx[j].z, vx[j].w, h.y, l.y);
            *reinterpret_cast<uint2 *>(Vh + key * LD + c) = h;
            *reinterpret_cast<uint2 *>(Vl + key * LD + c) = l;
        }
    }
    // This warp's 16 query vectors: A fragments straight from global memory
    // (fp32, scaled, split into hi/lo), rows ra = lane/4 and rb = ra + 8.
    const int qv0 = qb * kTcQ + warp * 16;
    const int qa_v = qv0 + (lane >> 2), qb_v = qa_v + 8;
    const int ra = qa_v < QV ? qa_v / gq : -1, rb = qb_v < QV ? qb_v / gq : -1;
    const float scale = rsqrtf(static_cast<float>(HD));
    uint32_t qh[HD / 16][4], ql[HD / 16][4];
    {
        const float *qpa = ra >= 0 ? q + (static_cast<long long>(ra) * nh + kvh * gq + qa_v % gq) * HD : nullptr;
        const float *qpb = rb >= 0 ? q + (static_cast<long long>(rb) * nh + kvh * gq + qb_v % gq) * HD : nullptr;
        const int c0 = 2 * (lane & 3);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
            const int c = ks * 16 + c0;
            const float2 a0 = qpa ? *reinterpret_cast<const float2 *>(qpa + c) : make_float2(0.f, 0.f);
            const float2 a2 = qpa ? *reinterpret_cast<const float2 *>(qpa + c + 8) : make_float2(0.f, 0.f);
            const float2 b0 = qpb ? *reinterpret_cast<const float2 *>(qpb + c) : make_float2(0.f, 0.f);
            const float2 b2 = qpb ? *reinterpret_cast<const float2 *>(qpb + c + 8) : make_float2(0.f, 0.f);
            split2(a0.x * scale, a0.y * scale, qh[ks][0], ql[ks][0]);
            split2(b0.x * scale, b0.y * scale, qh[ks][1], ql[ks][1]);
            split2(a2.x * scale, a2.y * scale, qh[ks][2], ql[ks][2]);
            split2(b2.x * scale, b2.y * scale, qh[ks][3], ql[ks][3]);
        }
    }
    __syncthreads();
    if (qv0 >= QV) return;   // whole warp past the last query (no later block-wide sync)

    // S = Q K^T : 16 queries x 64 keys (8 n-tiles of 8 keys), three passes
    float sacc[kTcChunk / 8][4];
#pragma unroll
    for (int j = 0; j < kTcChunk / 8; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
    {
        const int krow = (lane & 7) + 8 * (lane >> 4);
        const int kcol = 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
            for (int np = 0; np < kTcChunk / 16; ++np) {
                uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
                ldsm_x4(smem_u32(Kh + (np * 16 + krow) * LD + ks * 16 + kcol), h0, h1, h2, h3);
                ldsm_x4(smem_u32(Kl + (np * 16 + krow) * LD + ks * 16 + kcol), l0, l1, l2, l3);
                mma_bf16(sacc[2 * np], qh[ks], h0, h1);
                mma_bf16(sacc[2 * np], qh[ks], l0, l1);
                mma_bf16(sacc[2 * np], ql[ks], h0, h1);
                mma_bf16(sacc[2 * np + 1], qh[ks], h2, h3);
                mma_bf16(sacc[2 * np + 1], qh[ks], l2, l3);
                mma_bf16(sacc[2 * np + 1], ql[ks], h2, h3);
            }
        }
    }
    // mask + softmax
    float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
    for (int j = 0; j < kTcChunk / 8; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int kk = j * 8 + 2 * (lane & 3) + e;
            bool va = kk < nkeys && ra >= 0, vb2 = kk < nkeys && rb >= 0;
            if (step_chunk) {
                const int sidx = key0 + kk;
                if (vis_bits) {
                    va = va && ((vis_bits[ra * 8 + (sidx >> 5)] >> (sidx & 31)) & 1u);
                    vb2 = vb2 && ((vis_bits[rb * 8 + (sidx >> 5)] >> (sidx & 31)) & 1u);
                } else {
                    va = va && sidx <= ra;
                    vb2 = vb2 && sidx <= rb;
                }
            }
            if (!va) sacc[j][e] = -INFINITY;
            if (!vb2) sacc[j][2 + e] = -INFINITY;
            ma = fmaxf(ma, sacc[j][e]);
            mb = fmaxf(mb, sacc[j][2 + e]);
        }
    }
    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    float la_ = 0.f, lb = 0.f;
#pragma unroll
    for (int j = 0; j < kTcChunk / 8; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float pa = ma == -INFINITY ? 0.f : expf(sacc[j][e] - ma);
            const float pb = mb == -INFINITY ? 0.f : expf(sacc[j][2 + e] - mb);
            sacc[j][e] = pa;
            sacc[j][2 + e] = pb;
            la_ += pa;
            lb += pb;
        }
    }
    la_ += __shfl_xor_sync(0xffffffffu, la_, 1);
    la_ += __shfl_xor_sync(0xffffffffu, la_, 2);
    lb += __shfl_xor_sync(0xffffffffu, lb, 1);
    lb += __shfl_xor_sync(0xffffffffu, lb, 2);
    // O = P V : 16 queries x HD dims, three passes
    float oacc[HD / 8][4];
#pragma unroll
    for (int j = 0; j < HD / 8; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;
    {
        const int vrow = (lane & 7) + 8 * ((lane >> 3) & 1);
        const int vcol = 8 * (lane >> 4);
#pragma unroll
        for (int kk = 0; kk < kTcChunk / 16; ++kk) {
            uint32_t ph[4], pl[4];
            split2(sacc[2 * kk][0], sacc[2 * kk][1], ph[0], pl[0]);
            split2(sacc[2 * kk][2], sacc[2 * kk][3], ph[1], pl[1]);
            split2(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1], ph[2], pl[2]);
            split2(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3], ph[3], pl[3]);
#pragma unroll
            for (int dp = 0; dp < HD / 16; ++dp) {
                uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
                ldsm_x4_t(smem_u32(Vh + (kk * 16 + vrow) * LD + dp * 16 + vcol), h0, h1, h2, h3);
                ldsm_x4_t(smem_u32(Vl + (kk * 16 + vrow) * LD + dp * 16 + vcol), l0, l1, l2, l3);
                mma_bf16(oacc[2 * dp], ph, h0, h1);
                mma_bf16(oacc[2 * dp], ph, l0, l1);
                mma_bf16(oacc[2 * dp], pl, h0, h1);
                mma_bf16(oacc[2 * dp + 1], ph, h2, h3);
                mma_bf16(oacc[2 * dp + 1], ph, l2, l3);
                mma_bf16(oacc[2 * dp + 1], pl, h2, h3);
            }
        }
    }
    // partials: ws[chunk][r][h][HD + 4] = (O, max, sum)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int qvv = half ? qb_v : qa_v;
        if (qvv >= QV) continue;
        const int r = qvv / gq, hq = kvh * gq + qvv % gq;
        float *w = ws + ((static_cast<long long>(chunk) * nrows + r) * nh + hq) * (HD + 4);
#pragma unroll
        for (int j = 0; j < HD / 8; ++j)
            *reinterpret_cast<float2 *>(w + j * 8 + 2 * (lane & 3)) =
                make_float2(oacc[j][2 * half], oacc[j][2 * half + 1]);
        if ((lane & 3) == 0) {
            w[HD] = half ? mb : ma;
            w[HD + 1] = half ? lb : la_;
        }
    }
}

template <int HD>
__global__ void __launch_bounds__(256) k_attn_merge(const float *ws, int nch, int nrows, int nh, __nv_bfloat16 *out,
                                                    long long lo_off) {
    pdl_trigger();
    pdl_wait();
    constexpr int DPL = HD / 32;
    const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= nrows * nh) return;
    const int r = gw / nh, h = gw % nh;
    float m = -INFINITY, l = 0.f, o[DPL];
#pragma unroll
    for (int j = 0; j < DPL; ++j) o[j] = 0.f;
    for (int c = 0; c < nch; ++c) {
        const float *w = ws + ((static_cast<long long>(c) * nrows + r) * nh + h) * (HD + 4);
        const float pm = w[HD];
        if (pm == -INFINITY) continue;
        const float pl = w[HD + 1];
        const float nm = fmaxf(m, pm);
        const float a = (m == -INFINITY) ? 0.f : expf(m - nm);
        const float b = expf(pm - nm);
        l = l * a + pl * b;
#pragma unroll
        for (int j = 0; j < DPL; ++j) o[j] = o[j] * a + w[lane * DPL + j] * b;
        m = nm;
    }
    const float inv = 1.f / l;
    const long long base = static_cast<long long>(r) * nh * HD + h * HD + lane * DPL;
#pragma unroll
    for (int j = 0; j < DPL; ++j) store_act(out, base + j, o[j] * inv, lo_off);
}

template <int HD>
cudaError_t attention_tc_hd(const AttnArgs &a, cudaStream_t s) {
    const int nch_prefix = (a.P + kTcChunk - 1) / kTcChunk;
    const int nch = nch_prefix + (a.nrows + kTcChunk - 1) / kTcChunk;
    const int gq = a.nh / a.nkv;
    const size_t smem = static_cast<size_t>(4 * kTcChunk) * (HD + 8) * sizeof(__nv_bfloat16);
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_attn_tc<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    dim3 grid(a.nkv, nch, (a.nrows * gq + kTcQ - 1) / kTcQ);
    launch_k(k_attn_tc<HD>, dim3(grid), dim3(128), smem, s, a.q, a.kc, a.vc, a.max_seq, a.P, a.nrows, a.nh, a.nkv, nch_prefix,
                                          a.vis_bits, a.ws);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int warps = a.nrows * a.nh;
    launch_k(k_attn_merge<HD>, dim3((warps + 7) / 8), dim3(256), 0, s, a.ws, nch, a.nrows, a.nh, static_cast<__nv_bfloat16 *>(a.out),
                                                     a.out_lo_off);
    return cudaGetLastError();
}

}  // namespace

int attention_tc_chunks(int P, int nrows) {
    return (P + kTcChunk - 1) / kTcChunk + (nrows + kTcChunk - 1) / kTcChunk;
}

template <>
cudaError_t attention_launch<__nv_bfloat16>(const AttnArgs &a, cudaStream_t s) {
    if (a.hd == 128) return attention_tc_hd<128>(a, s);
    if (a.hd == 64) return attention_tc_hd<64>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace la
