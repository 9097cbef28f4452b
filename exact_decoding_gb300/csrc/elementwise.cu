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
                                                    float *h, T *xn, long long lo_off) {
    pdl_trigger();
    pdl_wait();
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
    for (int i = threadIdx.x; i < d; i += 256)
        store_act(xn, static_cast<long long>(r) * d + i, hr[i] * inv * to_f32(gain[i]), lo_off);
}

template <typename T>
cudaError_t embed_norm_launch(const T *embed, const int *tok, int nrows, int d, const T *gain, float eps, float *h,
                              T *xn, long long lo_off, cudaStream_t s) {
    launch_k(k_embed_norm<T>, dim3(nrows), dim3(256), 0, s, embed, tok, d, gain, eps, h, xn, lo_off);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ qkv + rope + KV write
// part: [S][nrows][ldp] with q | k | v columns.  Row r sits at position
// P + depth[r] (P + r when depth is null) and its K/V go to cache slot P + r.
// One thread per work item: a rotated (q or k) pair, or one v element.
// Partial planes of column col, added in plane order.  Beyond two planes the
// loads go out in predicated batches of 4 so that they are in flight together.
__device__ __forceinline__ float sum_planes(const float *pr, const int *planes, long long sstride, int col) {
    const int n = planes ? planes[col >> 7] : 1;
    if (n <= 2) return n == 2 ? pr[col] + pr[sstride + col] : pr[col];
    float v = 0.f;
    for (int b = 0; b < n; b += 4) {
        float x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = (b + j < n) ? pr[(b + j) * sstride + col] : 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) v += x[j];
    }
    return v;
}

__global__ void __launch_bounds__(256) k_qkv_rope(const float *part, const int *planes, long long sstride, int ldp,
                                                  int nh, int nkv, int hd, int k_off, int v_off, const float2 *rope,
                                                  int P, const int *depth, float *q, float *kc, float *vc,
                                                  int max_seq) {
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.y;
    const int t = blockIdx.x * 256 + threadIdx.x;
    const int half = hd / 2;
    const int nq_pairs = nh * half, nk_pairs = nkv * half;
    const float *pr = part + static_cast<long long>(r) * ldp;
    if (t < nq_pairs + nk_pairs) {
        const int pos = P + (depth ? depth[r] : r);
        const bool isq = t < nq_pairs;
        const int tt = isq ? t : t - nq_pairs;
        const int head = tt / half, i = tt % half;
        const int col = (isq ? 0 : k_off) + head * hd + i;
        const float x1 = sum_planes(pr, planes, sstride, col);
        const float x2 = sum_planes(pr, planes, sstride, col + half);
        const float2 c = rope[static_cast<long long>(pos) * half + i];
        const float y1 = x1 * c.x - x2 * c.y, y2 = x1 * c.y + x2 * c.x;
        if (isq) {
            float *qr = q + (static_cast<long long>(r) * nh + head) * hd;
            qr[i] = y1;
            qr[i + half] = y2;
        } else {
            float *kr = kc + (static_cast<long long>(head) * max_seq + P + r) * hd;
            kr[i] = y1;
            kr[i + half] = y2;
        }
    } else if (t < nq_pairs + nk_pairs + nkv * hd) {
        const int tv = t - nq_pairs - nk_pairs;
        const int head = tv / hd, i = tv % hd;
        const float v = sum_planes(pr, planes, sstride, v_off + tv);
        vc[(static_cast<long long>(head) * max_seq + P + r) * hd + i] = v;
    }
}

cudaError_t qkv_rope_launch(const float *part, const int *planes, long long sstride, int ldp, int nrows, int nh,
                            int nkv, int hd, int k_off, int v_off, const float2 *rope, int P, const int *depth,
                            float *q, float *kc, float *vc, int max_seq, cudaStream_t s) {
    const int items = (nh + nkv) * (hd / 2) + nkv * hd;
    dim3 grid((items + 255) / 256, nrows);
    launch_k(k_qkv_rope, dim3(grid), dim3(256), 0, s, part, planes, sstride, ldp, nh, nkv, hd, k_off, v_off, rope, P, depth, q, kc, vc,
                                    max_seq);
    return cudaGetLastError();
}

// bf16 models: one CTA = 32 rows x one head slot (a q, k or v head).  The
// tile is summed into shared memory with coalesced row reads; q and k are
// rotated and written along d, v is written transposed (consecutive rows are
// consecutive cache columns).
template <int HD>
__global__ void __launch_bounds__(256) k_qkv_rope_split(const float *part, const int *planes, long long sstride,
                                                        int ldp, int nrows, int nh, int nkv, int k_off, int v_off,
                                                        const float2 *rope, int P, const int *depth,
                                                        __nv_bfloat16 *q, int qv_pad, __nv_bfloat16 *kc,
                                                        __nv_bfloat16 *vc, int layer, int seq) {
    pdl_trigger();
    pdl_wait();
    __shared__ float t[32][HD + 1];
    const int r0 = blockIdx.x * 32, hs = blockIdx.y;
    const bool isq = hs < nh, isk = !isq && hs < nh + nkv;
    const int col0 = isq ? hs * HD : isk ? k_off + (hs - nh) * HD : v_off + (hs - nh - nkv) * HD;
    // A head's columns start on a 128-column tile, so the whole tile has one
    // plane count; each plane's loads are all issued before they are added.
    {
        constexpr int PER = 32 * HD / 256;
        const int np = planes ? planes[col0 >> 7] : 1;
        float acc[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) acc[j] = 0.f;
        for (int pl = 0; pl < np; ++pl) {
            const float *base = part + pl * sstride + col0;
            float x[PER];
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const int i = threadIdx.x + j * 256, rr = i / HD, d = i % HD, r = r0 + rr;
                x[j] = r < nrows ? base[static_cast<long long>(r) * ldp + d] : 0.f;
            }
#pragma unroll
            for (int j = 0; j < PER; ++j) acc[j] += x[j];
        }
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int i = threadIdx.x + j * 256;
            t[i / HD][i % HD] = acc[j];
        }
    }
    __syncthreads();
    constexpr int half = HD / 2;
    if (isq || isk) {
        const int gq = nh / nkv;
        const float scale = rsqrtf(static_cast<float>(HD));
        for (int i = threadIdx.x; i < 32 * half; i += 256) {
            const int rr = i / half, ii = i % half, r = r0 + rr;
            if (r >= nrows) continue;
            const int pos = P + (depth ? depth[r] : r);
            const float2 c = rope[static_cast<long long>(pos) * half + ii];
            const float x1 = t[rr][ii], x2 = t[rr][ii + half];
            float y1 = x1 * c.x - x2 * c.y, y2 = x1 * c.y + x2 * c.x;
            if (isq) {
                const int g = hs / gq, qv = r * gq + hs % gq;
                const long long base = (static_cast<long long>(g) * qv_pad + qv) * HD;
                const long long lo = static_cast<long long>(nkv) * qv_pad * HD;
                store_act(q, base + ii, y1 * scale, lo);
                store_act(q, base + ii + half, y2 * scale, lo);
            } else {
                const long long base = ((static_cast<long long>(layer) * 2 * nkv + (hs - nh)) * seq + P + r) * HD;
                const long long lo = static_cast<long long>(nkv) * seq * HD;
                store_act(kc, base + ii, y1, lo);
                store_act(kc, base + ii + half, y2, lo);
            }
        }
    } else {
        const int vh = hs - nh - nkv;
        const long long lo = static_cast<long long>(nkv) * HD * seq;
        for (int i = threadIdx.x; i < 32 * HD; i += 256) {
            const int d = i / 32, rr = i % 32, r = r0 + rr;
            if (r >= nrows) continue;
            const long long idx = ((static_cast<long long>(layer) * 2 * nkv + vh) * HD + d) * seq + P + r;
            store_act(vc, idx, t[rr][d], lo);
        }
    }
}

cudaError_t qkv_rope_split_launch(const float *part, const int *planes, long long sstride, int ldp, int nrows,
                                  int nh, int nkv, int hd, int k_off, int v_off, const float2 *rope, int P,
                                  const int *depth, __nv_bfloat16 *q, int qv_pad, __nv_bfloat16 *kc,
                                  __nv_bfloat16 *vc, int layer, int seq, cudaStream_t s) {
    dim3 grid((nrows + 31) / 32, nh + 2 * nkv);
    if (hd == 128)
        launch_k(k_qkv_rope_split<128>, grid, dim3(256), 0, s, part, planes, sstride, ldp, nrows, nh, nkv, k_off,
                 v_off, rope, P, depth, q, qv_pad, kc, vc, layer, seq);
    else if (hd == 64)
        launch_k(k_qkv_rope_split<64>, grid, dim3(256), 0, s, part, planes, sstride, ldp, nrows, nh, nkv, k_off,
                 v_off, rope, P, depth, q, qv_pad, kc, vc, layer, seq);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

// ------------------------------------------------------------------ residual + norm
// Output row i reads residual row r = row_map[i] (or i): h[r] += sum_s part[s][r];
// xout[i] = rmsnorm(h[r]) * gain.  d % 4 == 0; float4 accesses, all loads of
// a thread issued before the reduction.
template <typename T>
__global__ void __launch_bounds__(1024) k_resid_norm(float *h, const float *part, const int *planes,
                                                     long long sstride, int ldp,
                                                     int d, const T *gain, float eps, const int *row_map, T *xout,
                                                     long long lo_off) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[32];
    const int i = blockIdx.x;
    const int r = row_map ? row_map[i] : i;
    float4 *hr = reinterpret_cast<float4 *>(h + static_cast<long long>(r) * d);
    const float *pr = part + static_cast<long long>(r) * ldp;
    const int d4 = d / 4;
    constexpr int kMaxPer = 4;   // d <= 16384
    float4 v[kMaxPer];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxPer; ++j) {
        const int c = threadIdx.x + j * 1024;
        if (c < d4) {
            float4 a = hr[c];
            const int np = planes ? planes[(4 * c) >> 7] : 1;
            for (int b0 = 0; b0 < np; b0 += 8) {
                float4 x[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    x[j] = (b0 + j < np) ? *reinterpret_cast<const float4 *>(pr + (b0 + j) * sstride + 4 * c)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    a.x += x[j].x;
                    a.y += x[j].y;
                    a.z += x[j].z;
                    a.w += x[j].w;
                }
            }
            v[j] = a;
            hr[c] = a;
            ss += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w;
        }
    }
    const float inv = rsqrtf(block_sum<1024>(ss, red) / d + eps);
    const long long o = static_cast<long long>(i) * d;
#pragma unroll
    for (int j = 0; j < kMaxPer; ++j) {
        const int c = threadIdx.x + j * 1024;
        if (c < d4) {
            const float4 a = v[j];
            store_act(xout, o + 4 * c + 0, a.x * inv * to_f32(gain[4 * c + 0]), lo_off);
            store_act(xout, o + 4 * c + 1, a.y * inv * to_f32(gain[4 * c + 1]), lo_off);
            store_act(xout, o + 4 * c + 2, a.z * inv * to_f32(gain[4 * c + 2]), lo_off);
            store_act(xout, o + 4 * c + 3, a.w * inv * to_f32(gain[4 * c + 3]), lo_off);
        }
    }
}

template <typename T>
cudaError_t resid_norm_launch(float *h, const float *part, const int *planes, long long sstride, int ldp, int d,
                              const T *gain, float eps, const int *row_map, int nrows, T *xout, long long lo_off,
                              cudaStream_t s) {
    if (d % 4 || d > 16384) return cudaErrorInvalidValue;
    launch_k(k_resid_norm<T>, dim3(nrows), dim3(1024), 0, s, h, part, planes, sstride, ldp, d, gain, eps, row_map, xout, lo_off);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ SwiGLU
// part columns: gate [0, F) | up [F, 2F).  out[r][f] = silu(gate) * up.
template <typename T>
__global__ void k_swiglu(const float *part, const int *planes, long long sstride, int ldp, int nrows, int F,
                         int up_off, T *out, long long lo_off) {
    pdl_trigger();
    pdl_wait();
    const long long n = static_cast<long long>(nrows) * F;
    for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < n;
         t += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(t / F), f = static_cast<int>(t % F);
        const float *pr = part + static_cast<long long>(r) * ldp;
        const float g = sum_planes(pr, planes, sstride, f);
        const float u = sum_planes(pr, planes, sstride, up_off + f);
        store_act(out, t, g / (1.f + expf(-g)) * u, lo_off);
    }
}

template <typename T>
cudaError_t swiglu_launch(const float *part, const int *planes, long long sstride, int ldp, int nrows, int F,
                          int up_off, T *out, long long lo_off, cudaStream_t s) {
    const long long n = static_cast<long long>(nrows) * F;
    int blocks = static_cast<int>((n + 255) / 256);
    if (blocks > 152 * 64) blocks = 152 * 64;
    launch_k(k_swiglu<T>, dim3(blocks), dim3(256), 0, s, part, planes, sstride, ldp, nrows, F, up_off, out, lo_off);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ argmax / softmax stats
// Per row: index of the largest logit (lowest index among equals), the max,
// and sum_v exp((l_v - max) * invT) when invT > 0.
__global__ void __launch_bounds__(1024) k_argmax(const float *part, const int *planes, long long sstride, int ldp,
                                                 float *logits, int V, float invT, int *amax, float *lmax,
                                                 float *lsum) {
    pdl_trigger();
    pdl_wait();
    __shared__ float sv[32];
    __shared__ int si[32];
    __shared__ float red[32];
    const int r = blockIdx.x;
    const float *pr = part + static_cast<long long>(r) * ldp;
    float *l = logits + static_cast<long long>(r) * V;
    float best = -INFINITY;
    int bi = 0x7fffffff;
    for (int v = threadIdx.x; v < V; v += 1024) {
        const float x = sum_planes(pr, planes, sstride, v);
        l[v] = x;
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

cudaError_t argmax_launch(const float *part, const int *planes, long long sstride, int ldp, float *logits, int rows,
                          int V, float invT, int *amax, float *lmax, float *lsum, cudaStream_t s) {
    launch_k(k_argmax, dim3(rows), dim3(1024), 0, s, part, planes, sstride, ldp, logits, V, invT, amax, lmax, lsum);
    return cudaGetLastError();
}

#define LA_INST(T)                                                                                                   \
    template cudaError_t embed_norm_launch<T>(const T *, const int *, int, int, const T *, float, float *, T *,       \
                                              long long, cudaStream_t);                                              \
    template cudaError_t resid_norm_launch<T>(float *, const float *, const int *, long long, int, int, const T *,   \
                                              float, const int *, int, T *, long long, cudaStream_t);                \
    template cudaError_t swiglu_launch<T>(const float *, const int *, long long, int, int, int, int, T *, long long, \
                                          cudaStream_t);
LA_INST(float)
LA_INST(__nv_bfloat16)
#undef LA_INST

}  // namespace la
