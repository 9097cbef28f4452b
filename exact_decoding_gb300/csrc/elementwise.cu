// Row-wise kernels between the projection GEMMs of one decoder layer:
//   embedding gather + RMSNorm, split-K reduction + rotary embedding + KV
//   write (fp32 models; bf16 models do this in the attention kernel's
//   prologue), split-K reduction + residual add + RMSNorm, split-K
//   reduction + SwiGLU, and the vocabulary argmax with, for sampling, each
//   row's top-k / top-p keep rule and kept softmax mass.
// The residual stream h stays fp32; T is the GEMM-input / KV-cache type.
#include <algorithm>
#include <climits>

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

// Resident-SM count of the current device (cached per device): the grids
// below are sized to run in one wave beside a resident GEMM CTA.
static int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 152;
    }
    return cached[dev];
}

// ------------------------------------------------------------------ residual + norm
// Output row i reads residual row r = row_map[i] (or i): h[r] += sum_s part[s][r];
// xout[i] = rmsnorm(h[r]) * gain.  One CTA of 512 threads per row, PER float4
// columns per thread (d <= 2048 PER), the planes of all of a thread's
// columns loaded together.  512 threads keep the CTA small enough to sit
// beside a resident GEMM CTA.
constexpr int kNormThreads = 512;
template <typename T, int PER>
__global__ void __launch_bounds__(kNormThreads) k_resid_norm(float *h, const float *part, const int *planes,
                                                             long long sstride, int ldp, int d, const T *gain,
                                                             float eps, const int *row_map, T *xout,
                                                             long long lo_off) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[32];
    const int i = blockIdx.x;
    const int r = row_map ? row_map[i] : i;
    float4 *hr = reinterpret_cast<float4 *>(h + static_cast<long long>(r) * d);
    const float *pr = part + static_cast<long long>(r) * ldp;
    const int d4 = d / 4;
    float4 acc[PER];
    int np[PER];
    int npmax = 1;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int c = threadIdx.x + j * kNormThreads;
        acc[j] = c < d4 ? hr[c] : make_float4(0.f, 0.f, 0.f, 0.f);
        np[j] = c < d4 ? (planes ? planes[(4 * c) >> 7] : 1) : 0;
        npmax = max(npmax, np[j]);
    }
    // Planes in batches: up to 8 / PER planes of every column in flight.
    constexpr int BP = PER >= 8 ? 1 : 8 / PER;
    for (int b0 = 0; b0 < npmax; b0 += BP) {
        float4 x[PER][BP];
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int c = threadIdx.x + j * kNormThreads;
#pragma unroll
            for (int k = 0; k < BP; ++k)
                x[j][k] = b0 + k < np[j] ? *reinterpret_cast<const float4 *>(pr + (b0 + k) * sstride + 4 * c)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < PER; ++j)
#pragma unroll
            for (int k = 0; k < BP; ++k)
                if (b0 + k < np[j]) add4(acc[j], x[j][k]);
    }
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int c = threadIdx.x + j * kNormThreads;
        if (c < d4) {
            hr[c] = acc[j];
            ss += acc[j].x * acc[j].x + acc[j].y * acc[j].y + acc[j].z * acc[j].z + acc[j].w * acc[j].w;
        }
    }
    const float inv = rsqrtf(block_sum<kNormThreads>(ss, red) / d + eps);
    const long long o = static_cast<long long>(i) * d;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int c = threadIdx.x + j * kNormThreads;
        if (c < d4) {
            const float4 a = acc[j];
            store_act4(xout, o + 4 * c,
                       make_float4(a.x * inv * to_f32(gain[4 * c + 0]), a.y * inv * to_f32(gain[4 * c + 1]),
                                   a.z * inv * to_f32(gain[4 * c + 2]), a.w * inv * to_f32(gain[4 * c + 3])),
                       lo_off);
        }
    }
}

template <typename T>
cudaError_t resid_norm_launch(float *h, const float *part, const int *planes, long long sstride, int ldp, int d,
                              const T *gain, float eps, const int *row_map, int nrows, T *xout, long long lo_off,
                              cudaStream_t s) {
    if (d % 4 || d > 16384) return cudaErrorInvalidValue;
    const int per = (d / 4 + kNormThreads - 1) / kNormThreads;
    const dim3 g(nrows), b(kNormThreads);
    switch (per) {
        case 1: launch_k(k_resid_norm<T, 1>, g, b, 0, s, h, part, planes, sstride, ldp, d, gain, eps, row_map, xout, lo_off); break;
        case 2: launch_k(k_resid_norm<T, 2>, g, b, 0, s, h, part, planes, sstride, ldp, d, gain, eps, row_map, xout, lo_off); break;
        case 3: launch_k(k_resid_norm<T, 3>, g, b, 0, s, h, part, planes, sstride, ldp, d, gain, eps, row_map, xout, lo_off); break;
        case 4: launch_k(k_resid_norm<T, 4>, g, b, 0, s, h, part, planes, sstride, ldp, d, gain, eps, row_map, xout, lo_off); break;
        default: launch_k(k_resid_norm<T, 8>, g, b, 0, s, h, part, planes, sstride, ldp, d, gain, eps, row_map, xout, lo_off); break;
    }
    return cudaGetLastError();
}

// ------------------------------------------------------------------ SwiGLU
// part columns: gate [0, F) | up [up_off, up_off + F).  out[r][f] = silu(gate) * up.
// Items of four columns, grid-stride over a grid sized to the SMs; F % 4 == 0.
// A thread takes its items kSwigluBatch at a time and issues the plane loads
// of all of them before it adds any (the loads are L2 hits whose latency,
// not bandwidth, sets the kernel's time).
constexpr int kSwigluBatch = 3;

template <typename T>
__global__ void __launch_bounds__(256) k_swiglu(const float *__restrict__ part, const int *__restrict__ planes,
                                                long long sstride, int ldp, int nrows, int F, int up_off,
                                                T *__restrict__ out, long long lo_off) {
    pdl_trigger();
    pdl_wait();
    const int F4 = F / 4;
    const long long n = static_cast<long long>(nrows) * F4;
    const long long stride = gridDim.x * 256ll;
    for (long long t0 = blockIdx.x * 256ll + threadIdx.x; t0 < n; t0 += kSwigluBatch * stride) {
        float4 g[kSwigluBatch], u[kSwigluBatch];
        int row[kSwigluBatch], col[kSwigluBatch];
#pragma unroll
        for (int b = 0; b < kSwigluBatch; ++b) {
            const long long t = t0 + b * stride;
            const long long tt = t < n ? t : t0;   // past the end: repeat the first item, not stored
            row[b] = static_cast<int>(tt / F4);
            col[b] = 4 * static_cast<int>(tt % F4);
        }
        // planes 0 and 1 of every item first (a tile rarely has more), then the rest
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        float4 xg[kSwigluBatch][2], xu[kSwigluBatch][2];
        int npg[kSwigluBatch], npu[kSwigluBatch];
#pragma unroll
        for (int b = 0; b < kSwigluBatch; ++b) {
            const float *pr = part + static_cast<long long>(row[b]) * ldp;
            const int f = col[b];
            npg[b] = planes ? planes[f >> 7] : 1;
            npu[b] = planes ? planes[(up_off + f) >> 7] : 1;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                xg[b][k] = k < npg[b] ? *reinterpret_cast<const float4 *>(pr + f + k * sstride) : z;
                xu[b][k] = k < npu[b] ? *reinterpret_cast<const float4 *>(pr + up_off + f + k * sstride) : z;
            }
        }
#pragma unroll
        for (int b = 0; b < kSwigluBatch; ++b) {
            g[b] = xg[b][0];
            u[b] = xu[b][0];
            if (npg[b] > 1) add4(g[b], xg[b][1]);
            if (npu[b] > 1) add4(u[b], xu[b][1]);
            if (npg[b] > 2 || npu[b] > 2) {
                const float *pr = part + static_cast<long long>(row[b]) * ldp + 2 * sstride;
                float4 rg, ru;
                sum_planes4x2(pr + col[b], npg[b] - 2, pr + up_off + col[b], npu[b] - 2, sstride, rg, ru);
                if (npg[b] > 2) add4(g[b], rg);
                if (npu[b] > 2) add4(u[b], ru);
            }
        }
#pragma unroll
        for (int b = 0; b < kSwigluBatch; ++b) {
            if (t0 + b * stride >= n) break;
            const float4 gg = g[b], uu = u[b];
            store_act4(out, static_cast<long long>(row[b]) * F + col[b],
                       make_float4(gg.x / (1.f + expf(-gg.x)) * uu.x, gg.y / (1.f + expf(-gg.y)) * uu.y,
                                   gg.z / (1.f + expf(-gg.z)) * uu.z, gg.w / (1.f + expf(-gg.w)) * uu.w),
                       lo_off);
        }
    }
}

template <typename T>
cudaError_t swiglu_launch(const float *part, const int *planes, long long sstride, int ldp, int nrows, int F,
                          int up_off, T *out, long long lo_off, cudaStream_t s) {
    if (F % 4) return cudaErrorInvalidValue;
    const long long n = static_cast<long long>(nrows) * (F / 4);
    const int blocks = static_cast<int>(std::min<long long>((n + 255) / 256, 3ll * sm_count()));
    launch_k(k_swiglu<T>, dim3(blocks), dim3(256), 0, s, part, planes, sstride, ldp, nrows, F, up_off, out, lo_off);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ argmax / softmax stats
// Exclusive prefix over the block's threads in thread order (fixed order, so
// the float version is deterministic); total in *tot.
template <typename X>
__device__ __forceinline__ X block_excl_scan(X v, X *wtot, X *tot) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    X incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const X y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wtot[w] = incl;
    __syncthreads();
    if (w == 0) {
        X x = lane < 32 ? wtot[lane] : X(0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const X y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        wtot[lane] = x;
    }
    __syncthreads();
    const X excl = (w > 0 ? wtot[w - 1] : X(0)) + incl - v;
    *tot = wtot[31];
    __syncthreads();
    return excl;
}

// Keep rule of one row's sampling distribution (top-k, then top-p on what
// top-k keeps; ranking by logit, ties to the lower id).  Thread t owns the
// contiguous ids [a, b).  top-k: 4-pass radix select of the k-th largest
// key with integer histograms, then the lowest ids among the tied keys;
// top-p: 32-step bisection on the key with fixed-order mass sums, then the
// tied keys in id order until the mass is reached.  Returns the kept mass.
__device__ float row_keep_rule(const float *l, int V, float mx, float invT, int top_k, float top_p, unsigned *thr_out,
                               int *cut_out) {
    __shared__ unsigned s_hist[256];
    __shared__ unsigned s_pref, s_rem;
    __shared__ int s_cut;
    __shared__ int s_wi[32];
    __shared__ float s_wf[32];
    const int tid = threadIdx.x;
    const int per = (V + 1023) / 1024, a = min(V, tid * per), b = min(V, a + per);
    unsigned thr = 0u;
    int cut = INT_MAX;
    if (top_k > 0 && top_k < V) {
        unsigned pref = 0u, pmask = 0u, rem = static_cast<unsigned>(top_k);
        for (int sh = 24; sh >= 0; sh -= 8) {
            for (int i = tid; i < 256; i += 1024) s_hist[i] = 0u;
            __syncthreads();
            for (int v = a; v < b; ++v) {
                const unsigned k = order_key(l[v]);
                if ((k & pmask) == pref) atomicAdd(&s_hist[(k >> sh) & 255u], 1u);
            }
            __syncthreads();
            if (tid == 0) {
                unsigned acc = 0u;
                for (int dd = 255; dd >= 0; --dd) {
                    if (acc + s_hist[dd] >= rem) {
                        s_pref = pref | (static_cast<unsigned>(dd) << sh);
                        s_rem = rem - acc;
                        break;
                    }
                    acc += s_hist[dd];
                }
            }
            __syncthreads();
            pref = s_pref;
            rem = s_rem;
            pmask |= 0xFFu << sh;
        }
        // the rem lowest ids among keys equal to pref
        int cnt = 0;
        for (int v = a; v < b; ++v) cnt += order_key(l[v]) == pref;
        int tot;
        const int excl = block_excl_scan<int>(cnt, s_wi, &tot);
        if (tid == 0) s_cut = INT_MAX;
        __syncthreads();
        if (cnt > 0 && excl < static_cast<int>(rem) && static_cast<int>(rem) <= excl + cnt) {
            int c = excl;
            for (int v = a; v < b; ++v)
                if (order_key(l[v]) == pref && ++c == static_cast<int>(rem)) {
                    s_cut = v;
                    break;
                }
        }
        __syncthreads();
        thr = pref;
        cut = s_cut;
    }
    if (top_p > 0.f && top_p < 1.f) {
        const unsigned thrk = thr;
        const int cutk = cut;
        float z = 0.f;
        for (int v = a; v < b; ++v)
            if (keep_token(l[v], v, thrk, cutk)) z += expf((l[v] - mx) * invT);
        float zk;
        block_excl_scan<float>(z, s_wf, &zk);
        const float target = top_p * zk;
        unsigned long long lo = 0ull, hi = 1ull << 32;   // largest key K with mass(key >= K) >= target
        for (int it = 0; it < 32; ++it) {
            const unsigned long long mid = (lo + hi) >> 1;
            float sm = 0.f;
            for (int v = a; v < b; ++v)
                if (keep_token(l[v], v, thrk, cutk) && order_key(l[v]) >= mid) sm += expf((l[v] - mx) * invT);
            float S;
            block_excl_scan<float>(sm, s_wf, &S);
            if (S >= target) lo = mid;
            else hi = mid;
        }
        const unsigned kp = static_cast<unsigned>(lo);
        float gt = 0.f, tie = 0.f;
        for (int v = a; v < b; ++v) {
            if (!keep_token(l[v], v, thrk, cutk)) continue;
            const unsigned k = order_key(l[v]);
            if (k > kp) gt += expf((l[v] - mx) * invT);
            else if (k == kp) tie += expf((l[v] - mx) * invT);
        }
        float Sgt, Stie;
        block_excl_scan<float>(gt, s_wf, &Sgt);
        const float excl = block_excl_scan<float>(tie, s_wf, &Stie);
        const float need = target - Sgt;   // tied mass still needed, in id order
        if (tid == 0) s_cut = INT_MIN;
        __syncthreads();
        if (tie > 0.f && excl < need && need <= excl + tie) {
            float c = excl;
            for (int v = a; v < b; ++v) {
                if (!keep_token(l[v], v, thrk, cutk) || order_key(l[v]) != kp) continue;
                c += expf((l[v] - mx) * invT);
                if (c >= need) {
                    atomicMax(&s_cut, -v);   // rounding may let two ranges claim: the lower id wins
                    break;
                }
            }
        }
        __syncthreads();
        int cp = s_cut == INT_MIN ? INT_MAX : -s_cut;   // no claim (rounding at the end): every tied token
        if (kp == thrk) cp = min(cp, cutk);
        thr = kp;
        cut = cp;
    }
    // kept mass, in the fixed order of the unfiltered sum
    float s = 0.f;
    for (int v = tid; v < V; v += 1024)
        if (keep_token(l[v], v, thr, cut)) s += expf((l[v] - mx) * invT);
    __syncthreads();
    *thr_out = thr;
    *cut_out = cut;
    return s;
}

// Per row: index of the largest logit (lowest index among equals), the max,
// and, when invT > 0, the row's top-k / top-p keep rule and the sum of
// exp((l_v - max) * invT) over the kept tokens.
__global__ void __launch_bounds__(1024) k_argmax(const float *part, const int *planes, long long sstride, int ldp,
                                                 float *logits, int V, float invT, int *amax, float *lmax,
                                                 float *lsum, int top_k, float top_p, unsigned *thr_key,
                                                 int *thr_cut) {
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
        // All-NaN logits leave no index: report token 0 rather than an id
        // outside the vocabulary (the step's tokens index the embedding).
        amax[r] = si[0] < V ? si[0] : 0;
        lmax[r] = best;
    }
    if (invT > 0.f) {
        __syncthreads();   // this CTA's logits stores are visible to all its threads
        unsigned thr;
        int cut;
        float s = row_keep_rule(l, V, best, invT, top_k, top_p, &thr, &cut);
        s = block_sum<1024>(s, red);
        if (threadIdx.x == 0) {
            lsum[r] = s;
            thr_key[r] = thr;
            thr_cut[r] = cut;
        }
    }
}

cudaError_t argmax_launch(const float *part, const int *planes, long long sstride, int ldp, float *logits, int rows,
                          int V, float invT, int *amax, float *lmax, float *lsum, int top_k, float top_p,
                          unsigned *thr_key, int *thr_cut, cudaStream_t s) {
    launch_k(k_argmax, dim3(rows), dim3(1024), 0, s, part, planes, sstride, ldp, logits, V, invT, amax, lmax, lsum,
             top_k, top_p, thr_key, thr_cut);
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
