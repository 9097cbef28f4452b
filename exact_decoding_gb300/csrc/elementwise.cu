// Row-wise kernels between the projection GEMMs of one decoder layer:
//   embedding gather + RMSNorm, split-K reduction + rotary embedding + KV
//   write, split-K reduction + residual add + RMSNorm, split-K reduction +
//   SwiGLU, and the vocabulary argmax (with softmax statistics for sampling).
// The residual stream h stays fp32; T is the GEMM-input / KV-cache type.
#include "la_kernels.h"

namespace la {

template <int NT>
__device__ __forceinline__ float block_sum(float v, float *red) {
    v = warp_sum(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    if (w == 0) {
        t = (l < NT / 32) ? red[l] : 0.f;
        t = warp_sum(t);
        if (l == 0) red[0] = t;
    }
    __syncthreads();
    t = red[0];
    __syncthreads();
    return t;
}

// ------------------------------------------------------------------ embed + norm
template <typename T>
__global__ void __launch_bounds__(256) k_embed_norm(const T *embed, const int *tok, int d, const T *gain, float eps,
                                                    float *h, T *xn) {
    __shared__ float red[32];
    const int r = blockIdx.x;
    const T *e = embed + static_cast<long long>(tok[r]) * d;
    float *hr = h + static_cast<long long>(r) * d;
    float ss = 0.f;
    for (int i = threadIdx.x; i < d; i += 256) {
        const float v = to_f32(e[i]);
        hr[i] = v;
        ss += v * v;
    }
    const float inv = rsqrtf(block_sum<256>(ss, red) / d + eps);
    for (int i = threadIdx.x; i < d; i += 256) xn[static_cast<long long>(r) * d + i] = from_f32<T>(hr[i] * inv * to_f32(gain[i]));
}

template <typename T>
cudaError_t embed_norm_launch(const T *embed, const int *tok, int nrows, int d, const T *gain, float eps, float *h,
                              T *xn, cudaStream_t s) {
    k_embed_norm<T><<<nrows, 256, 0, s>>>(embed, tok, d, gain, eps, h, xn);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ qkv + rope + KV write
// part: [S][nrows][ldp] with q | k | v columns.  Row r sits at position
// P + depth[r] (P + r when depth is null) and its K/V go to cache slot P + r.
template <typename T>
__global__ void __launch_bounds__(128) k_qkv_rope(const float *part, int S, long long sstride, int ldp, int nh,
                                                  int nkv, int hd, const float2 *rope, int P, const int *depth,
                                                  float *q, T *kc, T *vc, int max_seq) {
    const int r = blockIdx.x;
    const int pos = P + (depth ? depth[r] : r);
    const int half = hd / 2;
    const float *pr = part + static_cast<long long>(r) * ldp;
    const float2 *cs = rope + static_cast<long long>(pos) * half;
    // q and k: rotate pairs (i, i + hd/2)
    const int nq_pairs = nh * half, nk_pairs = nkv * half;
    for (int t = threadIdx.x; t < nq_pairs + nk_pairs; t += blockDim.x) {
        const bool isq = t < nq_pairs;
        const int tt = isq ? t : t - nq_pairs;
        const int head = tt / half, i = tt % half;
        const int col = (isq ? 0 : nh * hd) + head * hd + i;
        float x1 = 0.f, x2 = 0.f;
        for (int sp = 0; sp < S; ++sp) {
            x1 += pr[sp * sstride + col];
            x2 += pr[sp * sstride + col + half];
        }
        const float2 c = cs[i];
        const float y1 = x1 * c.x - x2 * c.y, y2 = x1 * c.y + x2 * c.x;
        if (isq) {
            float *qr = q + (static_cast<long long>(r) * nh + head) * hd;
            qr[i] = y1;
            qr[i + half] = y2;
        } else {
            T *kr = kc + (static_cast<long long>(head) * max_seq + P + r) * hd;
            kr[i] = from_f32<T>(y1);
            kr[i + half] = from_f32<T>(y2);
        }
    }
    const int vcol0 = (nh + nkv) * hd;
    for (int t = threadIdx.x; t < nkv * hd; t += blockDim.x) {
        const int head = t / hd, i = t % hd;
        float v = 0.f;
        for (int sp = 0; sp < S; ++sp) v += pr[sp * sstride + vcol0 + t];
        vc[(static_cast<long long>(head) * max_seq + P + r) * hd + i] = from_f32<T>(v);
    }
}

template <typename T>
cudaError_t qkv_rope_launch(const float *part, int S, long long sstride, int ldp, int nrows, int nh, int nkv, int hd,
                            const float2 *rope, int P, const int *depth, float *q, T *kc, T *vc, int max_seq,
                            cudaStream_t s) {
    k_qkv_rope<T><<<nrows, 128, 0, s>>>(part, S, sstride, ldp, nh, nkv, hd, rope, P, depth, q, kc, vc, max_seq);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ residual + norm
// Output row i reads residual row r = row_map[i] (or i): h[r] += sum_s part[s][r];
// xout[i] = rmsnorm(h[r]) * gain.
template <typename T>
__global__ void __launch_bounds__(256) k_resid_norm(float *h, const float *part, int S, long long sstride, int ldp,
                                                    int d, const T *gain, float eps, const int *row_map, T *xout) {
    __shared__ float red[32];
    const int i = blockIdx.x;
    const int r = row_map ? row_map[i] : i;
    float *hr = h + static_cast<long long>(r) * d;
    const float *pr = part + static_cast<long long>(r) * ldp;
    float ss = 0.f;
    for (int c = threadIdx.x; c < d; c += 256) {
        float v = hr[c];
        for (int sp = 0; sp < S; ++sp) v += pr[sp * sstride + c];
        hr[c] = v;
        ss += v * v;
    }
    const float inv = rsqrtf(block_sum<256>(ss, red) / d + eps);
    T *xo = xout + static_cast<long long>(i) * d;
    for (int c = threadIdx.x; c < d; c += 256) xo[c] = from_f32<T>(hr[c] * inv * to_f32(gain[c]));
}

template <typename T>
cudaError_t resid_norm_launch(float *h, const float *part, int S, long long sstride, int ldp, int d, const T *gain,
                              float eps, const int *row_map, int nrows, T *xout, cudaStream_t s) {
    k_resid_norm<T><<<nrows, 256, 0, s>>>(h, part, S, sstride, ldp, d, gain, eps, row_map, xout);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ SwiGLU
// part columns: gate [0, F) | up [F, 2F).  out[r][f] = silu(gate) * up.
template <typename T>
__global__ void k_swiglu(const float *part, int S, long long sstride, int ldp, int nrows, int F, T *out) {
    const long long n = static_cast<long long>(nrows) * F;
    for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < n;
         t += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(t / F), f = static_cast<int>(t % F);
        const float *pr = part + static_cast<long long>(r) * ldp;
        float g = 0.f, u = 0.f;
        for (int sp = 0; sp < S; ++sp) {
            g += pr[sp * sstride + f];
            u += pr[sp * sstride + F + f];
        }
        out[t] = from_f32<T>(g / (1.f + expf(-g)) * u);
    }
}

template <typename T>
cudaError_t swiglu_launch(const float *part, int S, long long sstride, int ldp, int nrows, int F, T *out,
                          cudaStream_t s) {
    const long long n = static_cast<long long>(nrows) * F;
    int blocks = static_cast<int>((n + 255) / 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    k_swiglu<T><<<blocks, 256, 0, s>>>(part, S, sstride, ldp, nrows, F, out);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ argmax / softmax stats
// Per row: index of the largest logit (lowest index among equals), the max,
// and sum_v exp((l_v - max) * invT) when invT > 0.
__global__ void __launch_bounds__(1024) k_argmax(const float *logits, int V, float invT, int *amax, float *lmax,
                                                 float *lsum) {
    __shared__ float sv[32];
    __shared__ int si[32];
    __shared__ float red[32];
    const int r = blockIdx.x;
    const float *l = logits + static_cast<long long>(r) * V;
    float best = -INFINITY;
    int bi = 0x7fffffff;
    for (int v = threadIdx.x; v < V; v += 1024) {
        const float x = l[v];
        if (x > best) {
            best = x;
            bi = v;
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ob > best || (ob == best && oi < bi)) {
            best = ob;
            bi = oi;
        }
    }
    const int w = threadIdx.x >> 5, ln = threadIdx.x & 31;
    if (ln == 0) {
        sv[w] = best;
        si[w] = bi;
    }
    __syncthreads();
    if (w == 0) {
        best = sv[ln];
        bi = si[ln];
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ob > best || (ob == best && oi < bi)) {
                best = ob;
                bi = oi;
            }
        }
        if (ln == 0) {
            sv[0] = best;
            si[0] = bi;
        }
    }
    __syncthreads();
    best = sv[0];
    if (threadIdx.x == 0) {
        amax[r] = si[0];
        lmax[r] = best;
    }
    if (invT > 0.f) {
        float s = 0.f;
        for (int v = threadIdx.x; v < V; v += 1024) s += expf((l[v] - best) * invT);
        s = block_sum<1024>(s, red);
        if (threadIdx.x == 0) lsum[r] = s;
    }
}

cudaError_t argmax_launch(const float *logits, int rows, int V, float invT, int *amax, float *lmax, float *lsum,
                          cudaStream_t s) {
    k_argmax<<<rows, 1024, 0, s>>>(logits, V, invT, amax, lmax, lsum);
    return cudaGetLastError();
}

#define LA_INST(T)                                                                                                   \
    template cudaError_t embed_norm_launch<T>(const T *, const int *, int, int, const T *, float, float *, T *,       \
                                              cudaStream_t);                                                         \
    template cudaError_t qkv_rope_launch<T>(const float *, int, long long, int, int, int, int, int, const float2 *,   \
                                            int, const int *, float *, T *, T *, int, cudaStream_t);                 \
    template cudaError_t resid_norm_launch<T>(float *, const float *, int, long long, int, int, const T *, float,    \
                                              const int *, int, T *, cudaStream_t);                                  \
    template cudaError_t swiglu_launch<T>(const float *, int, long long, int, int, int, T *, cudaStream_t);
LA_INST(float)
LA_INST(__nv_bfloat16)
#undef LA_INST

}  // namespace la
