// Speculation state of lookahead decoding on the device: candidate lookup
// and step-row build, verification (Algorithm 3 greedy / Algorithm 4
// sampling), n-gram harvest into the pool, window slide, bookkeeping and the
// KV commit of accepted rows.  Source: paper-graph-ui page, section 3.4,
// "The Lookahead Branch", "The Verification Branch", "Integrated Forward
// Pass".
//
// Step-row layout: row 0 is the last committed token o (position P);
// lookahead row (k, j) is 1 + k*W + j (window level k, column j, position
// P+1+j+k); candidate row (c, m), m = 1..N-1, is 1 + (N-1)*W + c*(N-1) + m-1
// (suffix token m of candidate c, position P+m).  "Used" rows (the ones
// whose logits are computed) are row 0, the top level's W rows and all
// candidate rows, in that order.
//
// n-gram pool: open-addressed hash table keyed by the n-gram's first token
// (Fibonacci hashing, linear probing, >= 2x as many slots as the vocabulary
// so it never fills).  Each slot keeps a ring of up to `cap` distinct
// (N-1)-token suffixes in eviction order (the next to be dropped at the
// head); a new suffix goes to the tail, and into a full ring it replaces
// the head.  FIFO: a suffix that is present stays where it is, candidates
// are read from the head.  LRU (section 7 of the same page leaves the
// eviction policy open): a suffix harvested again, or the step's winning
// candidate, moves to the tail, and candidates are read from the tail.  LFU
// (frequency-based eviction, the same passage): every ring entry carries a
// use count, and the ring is kept ordered by (count, time of the last use or
// entry) ascending; a use adds one to the count and moves the entry behind
// every entry whose count is not larger, a new suffix enters with count 0
// behind the count-0 entries after the head has been dropped from a full
// ring, and candidates are read from the tail.  Since a moved or new entry
// always carries the newest time, the ring order alone keeps the times.  All
// pool operations run in one warp: lanes probe 32 slots, or compare 32
// ring entries, at once; inserts keep their sequential order.
#include <climits>

#include "la_kernels.h"

namespace la {

constexpr unsigned FULL = 0xffffffffu;

// ------------------------------------------------------------------ Philox4x32-10
// Counter-based generator of Salmon, Moraes, Dror and Shaw (SC'11): ten
// rounds of two 32x32->64 multiplies, key bumped by the Weyl constants.
__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c[0], hi0 = __umulhi(0xD2511F53u, c[0]);
        const uint32_t lo1 = 0xCD9E8D57u * c[2], hi1 = __umulhi(0xCD9E8D57u, c[2]);
        const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = lo1;
        c[2] = n2;
        c[3] = lo0;
    }
}
// Sampling draw for (position, draw index): 24 high bits of the first word.
__device__ __forceinline__ float draw_uniform(unsigned long long seed, int position, int draw) {
    uint32_t c[4] = {static_cast<uint32_t>(position), static_cast<uint32_t>(draw), 0u, 0u};
    philox4x32_10(c, static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
    return static_cast<float>(c[0] >> 8) * (1.0f / 16777216.0f);
}

// ------------------------------------------------------------------ pool (one warp)
__device__ __forceinline__ int hash_slot(int key, int log2n) {
    return static_cast<int>((static_cast<uint32_t>(key) * 2654435761u) >> (32 - log2n));
}

// Slot holding `key` (>= 0), or -(first empty slot + 1) if absent, INT_MIN if full.
__device__ int pool_find(const SpecDev &d, int key, int lane) {
    const int n = 1 << d.nslots_log2, mask = n - 1;
    const int base = hash_slot(key, d.nslots_log2);
    for (int probe = 0; probe < n; probe += 32) {
        const int s = (base + probe + lane) & mask;
        const int k = d.pkeys[s];
        const unsigned hit = __ballot_sync(FULL, k == key);
        const unsigned emp = __ballot_sync(FULL, k == -1);
        const unsigned any = hit | emp;
        if (any) {
            const int i = __ffs(any) - 1;
            const int slot = (base + probe + i) & mask;
            return ((hit >> i) & 1u) ? slot : -(slot + 1);
        }
    }
    return INT_MIN;
}

// Ring entry `i` (0 = head) of `slot` moves to the tail; entries i+1..cnt-1
// move one place towards the head.  Lane l holds list entry l (cap <= 32)
// in registers (N - 1 <= 7 tokens); `i` and the counts are warp-uniform, so
// the early return leaves no lane behind in the shuffles.
__device__ void pool_move_to_tail_warp(const SpecDev &d, int slot, int i, int lane) {
    const int L = d.N - 1, cap = d.cap;
    const int cnt = d.pcnt[slot], head = d.phead[slot];
    if (i < 0 || i >= cnt - 1) return;   // absent, or already at the tail
    int *ring = d.pent + static_cast<long long>(slot) * cap * L;
    int e[7];
#pragma unroll
    for (int m = 0; m < 7; ++m) e[m] = (lane < cnt && m < L) ? ring[((head + lane) % cap) * L + m] : 0;
    const int src = lane < i ? lane : (lane < cnt - 1 ? lane + 1 : i);
#pragma unroll
    for (int m = 0; m < 7; ++m) e[m] = __shfl_sync(FULL, e[m], src & 31);
    __syncwarp();
    if (lane < cnt)
        for (int m = 0; m < L; ++m) ring[((head + lane) % cap) * L + m] = e[m];
    __syncwarp();
}

// List index of the entry of `slot` equal to suf, or -1 (every lane gets it).
__device__ int pool_index_warp(const SpecDev &d, int slot, const int *suf, int lane) {
    const int L = d.N - 1, cap = d.cap;
    const int cnt = d.pcnt[slot], head = d.phead[slot];
    bool same = false;
    if (lane < cnt) {
        const int *e = d.pent + (static_cast<long long>(slot) * cap + (head + lane) % cap) * L;
        same = true;
        for (int m = 0; m < L; ++m) same = same && (e[m] == suf[m]);
    }
    const unsigned hit = __ballot_sync(FULL, same);
    return hit ? __ffs(hit) - 1 : -1;
}

// LFU: entry `i` of `slot` is used: its count grows by one and it moves
// behind every other entry whose count is at most the new count (they are
// older).  Lane l holds list entry l; `i` and the counts are warp-uniform.
__device__ void pool_lfu_use_warp(const SpecDev &d, int slot, int i, int lane) {
    const int L = d.N - 1, cap = d.cap;
    const int cnt = d.pcnt[slot], head = d.phead[slot];
    if (i < 0 || i >= cnt) return;
    int *ring = d.pent + static_cast<long long>(slot) * cap * L;
    int *uses = d.puse + static_cast<long long>(slot) * cap;
    int e[7], u = 0;
    const int r = (head + lane) % cap;
#pragma unroll
    for (int m = 0; m < 7; ++m) e[m] = (lane < cnt && m < L) ? ring[r * L + m] : 0;
    if (lane < cnt) u = uses[r];
    const int newc = __shfl_sync(FULL, u, i) + 1;
    // final index of entry i: behind entries 0..i-1 (counts <= newc - 1) and
    // behind the run after i whose counts are <= newc
    const int pos = __popc(__ballot_sync(FULL, lane < cnt && lane != i && u <= newc));
    const int src = lane < i ? lane : (lane < pos ? lane + 1 : (lane == pos ? i : lane));
#pragma unroll
    for (int m = 0; m < 7; ++m) e[m] = __shfl_sync(FULL, e[m], src & 31);
    u = __shfl_sync(FULL, u, src & 31);
    if (lane == pos) u = newc;
    __syncwarp();
    if (lane < cnt) {
        for (int m = 0; m < L; ++m) ring[r * L + m] = e[m];
        uses[r] = u;
    }
    __syncwarp();
}

// LFU: a new suffix with use count c0 enters `slot` (known absent).  A full
// ring first drops its head (fewest uses, oldest among equals); the new entry
// goes behind every entry whose count is at most c0.
__device__ void pool_lfu_insert_warp(const SpecDev &d, int slot, const int *suf, int c0, int lane) {
    const int L = d.N - 1, cap = d.cap;
    int cnt = d.pcnt[slot], head = d.phead[slot];
    if (cnt == cap) {
        head = (head + 1) % cap;
        cnt -= 1;
    }
    int *ring = d.pent + static_cast<long long>(slot) * cap * L;
    int *uses = d.puse + static_cast<long long>(slot) * cap;
    int e[7], u = 0;
    const int r = (head + lane) % cap;
#pragma unroll
    for (int m = 0; m < 7; ++m) e[m] = (lane < cnt && m < L) ? ring[r * L + m] : 0;
    if (lane < cnt) u = uses[r];
    const int pos = __popc(__ballot_sync(FULL, lane < cnt && u <= c0));
    const int src = lane <= pos ? lane : lane - 1;
#pragma unroll
    for (int m = 0; m < 7; ++m) e[m] = __shfl_sync(FULL, e[m], src & 31);
    u = __shfl_sync(FULL, u, src & 31);
    if (lane == pos) {
        for (int m = 0; m < L; ++m) e[m] = suf[m];
        u = c0;
    }
    __syncwarp();
    if (lane <= cnt) {
        for (int m = 0; m < L; ++m) ring[r * L + m] = e[m];
        uses[r] = u;
    }
    __syncwarp();
    if (lane == 0) {
        d.pcnt[slot] = cnt + 1;
        d.phead[slot] = head;
    }
    __syncwarp();
}

// A use of the suffix `suf` of `key` (if present): LRU moves it to the tail,
// LFU counts it and re-orders; FIFO ignores it.
__device__ void pool_use_warp(const SpecDev &d, int key, const int *suf, int lane) {
    if (d.policy == kPoolFifo) return;
    const int f = pool_find(d, key, lane);
    if (f < 0) return;
    const int i = pool_index_warp(d, f, suf, lane);
    if (d.policy == kPoolLru)
        pool_move_to_tail_warp(d, f, i, lane);
    else
        pool_lfu_use_warp(d, f, i, lane);
}

// suf: N-1 tokens, identical in every lane; c0: LFU use count of a new entry.
__device__ void pool_insert_warp(const SpecDev &d, int key, const int *suf, int lane, int c0 = 0) {
    const int L = d.N - 1, cap = d.cap;
    const int f = pool_find(d, key, lane);
    if (f == INT_MIN) {
        if (lane == 0) atomicOr(&d.st->err, ERR_POOL);
        return;
    }
    int slot = f;
    if (f < 0) {
        slot = -f - 1;
        if (lane == 0) {
            d.pkeys[slot] = key;
            d.pcnt[slot] = 0;
            d.phead[slot] = 0;
        }
        __syncwarp();
    }
    const int cnt = d.pcnt[slot], head = d.phead[slot];
    const int present = pool_index_warp(d, slot, suf, lane);
    if (present >= 0) {
        if (d.policy == kPoolLru) pool_move_to_tail_warp(d, slot, present, lane);
        if (d.policy == kPoolLfu) pool_lfu_use_warp(d, slot, present, lane);
        return;
    }
    if (d.policy == kPoolLfu) {
        pool_lfu_insert_warp(d, slot, suf, c0, lane);
        return;
    }
    if (lane == 0) {
        int pos;
        if (cnt < cap) {
            pos = (head + cnt) % cap;
            d.pcnt[slot] = cnt + 1;
        } else {
            pos = head;
            d.phead[slot] = (head + 1) % cap;
        }
        int *e = d.pent + (static_cast<long long>(slot) * cap + pos) * L;
        for (int m = 0; m < L; ++m) e[m] = suf[m];
    }
    __syncwarp();
}

// ------------------------------------------------------------------ candidate lookup + step rows
__global__ void __launch_bounds__(256) k_build_rows(SpecDev d) {
    pdl_trigger();
    pdl_wait();
    // Every kernel of the previous step has completed: its gate/up GEMMs'
    // arrival counts start this step from 0 (a step adds at most layers x
    // planes to each, far from overflow).
    for (int i = threadIdx.x; i < d.n_step_zero; i += blockDim.x) d.step_zero[i] = 0;
    __shared__ int s_g;
    __shared__ int s_c[32 * 8];
    const int L = d.N - 1;
    const int tid = threadIdx.x, lane = tid & 31;
    const int o = d.st->o;
    if (tid < 32) {
        int g = 0;
        if (d.G > 0) {
            const int f = pool_find(d, o, lane);
            if (f >= 0) {
                const int cnt = d.pcnt[f], head = d.phead[f];
                g = min(cnt, d.G);
                for (int t = lane; t < g * L; t += 32) {
                    const int c = t / L, m = t % L;
                    const int li = d.policy != kPoolFifo ? cnt - 1 - c : c;   // LRU / LFU: from the tail
                    s_c[t] = d.pent[(static_cast<long long>(f) * d.cap + (head + li) % d.cap) * L + m];
                }
            }
        }
        if (lane == 0) s_g = g;
    }
    __syncthreads();
    const int g = s_g;
    const int look_end = 1 + L * d.W;
    for (int r = tid; r < d.M; r += blockDim.x) {
        int t;
        if (r == 0) {
            t = o;
        } else if (r < look_end) {
            t = d.window[r - 1];   // level-major: (k, j) -> k*W + j = r - 1
        } else {
            const int idx = r - look_end, c = idx / L;
            t = c < g ? s_c[idx] : 0;
        }
        d.tok[r] = t;
    }
    for (int t = tid; t < d.G * L; t += blockDim.x) d.cands[t] = (t / L) < g ? s_c[t] : -1;
    if (tid == 0) d.st->g = g;
}

// ------------------------------------------------------------------ inverse CDF (one block)
// Smallest id whose ascending cumulative weight exceeds u * total, with
// weight exp((l_v - mx) * invT) for the tokens the row's keep rule (thr,
// cut) keeps and the ids in rej[0..nrej) removed.
template <int NT>
__device__ int block_inverse_cdf(const float *l, int V, float mx, float invT, const int *rej, int nrej, float u,
                                 unsigned thr, int cut) {
    __shared__ float s_part[NT];
    __shared__ float s_warp[NT / 32];
    __shared__ int s_ans;
    const int tid = threadIdx.x;
    const int per = (V + NT - 1) / NT;
    const int a = min(V, tid * per), b = min(V, a + per);
    float part = 0.f;
    for (int v = a; v < b; ++v) {
        bool r = false;
        for (int i = 0; i < nrej; ++i) r = r || (rej[i] == v);
        part += (r || !keep_token(l[v], v, thr, cut)) ? 0.f : expf((l[v] - mx) * invT);
    }
    // inclusive warp scan, then across warps (fixed order)
    float incl = part;
    const int lane = tid & 31, w = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[w] = incl;
    if (tid == 0) s_ans = INT_MAX;
    __syncthreads();
    if (w == 0) {
        float x = lane < NT / 32 ? s_warp[lane] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(FULL, x, o);
            if (lane >= o) x += y;
        }
        if (lane < NT / 32) s_warp[lane] = x;
    }
    __syncthreads();
    const float excl = (w > 0 ? s_warp[w - 1] : 0.f) + (incl - part);
    const float total = s_warp[NT / 32 - 1];
    const float t = u * total;
    s_part[tid] = part;
    if (part > 0.f && excl <= t && t < excl + part) {
        float s = 0.f;
        int ans = b - 1;
        for (int v = a; v < b; ++v) {
            bool r = false;
            for (int i = 0; i < nrej; ++i) r = r || (rej[i] == v);
            s += (r || !keep_token(l[v], v, thr, cut)) ? 0.f : expf((l[v] - mx) * invT);
            if (excl + s > t) {
                ans = v;
                break;
            }
        }
        atomicMin(&s_ans, ans);   // rounding can make two ranges claim t: lowest id wins
    }
    __syncthreads();
    if (tid == 0 && s_ans == INT_MAX) {
        // t rounded up to the total: take the last id with weight
        for (int i = NT - 1; i >= 0; --i)
            if (s_part[i] > 0.f) {
                const int aa = min(V, i * per), bb = min(V, aa + per);
                for (int v = bb - 1; v >= aa; --v) {
                    bool r = false;
                    for (int k = 0; k < nrej; ++k) r = r || (rej[k] == v);
                    if (!r && keep_token(l[v], v, thr, cut) && expf((l[v] - mx) * invT) > 0.f) {
                        s_ans = v;
                        break;
                    }
                }
                break;
            }
    }
    __syncthreads();
    return s_ans;
}

// ------------------------------------------------------------------ verify + harvest + slide
constexpr int kFinishThreads = 1024;

__global__ void __launch_bounds__(kFinishThreads) k_finish_step(SpecDev d) {
    pdl_trigger();
    pdl_wait();
    __shared__ int s_acc[8];
    __shared__ int s_A, s_win, s_need_draw, s_dist_u, s_nrej;
    __shared__ int s_rej[32];
    __shared__ float s_u;
    const int L = d.N - 1;
    const int tid = threadIdx.x;
    const int P = d.st->P;
    const int g = d.st->g;
    const int cand_u0 = 1 + d.W;   // used index of candidate 0, depth 1
    if (tid == 0) {
        int A = 0, win = -1;
        unsigned surv = g >= 32 ? FULL : ((1u << g) - 1u);
        if (d.T <= 0.f) {
            // Algorithm 3: progressive filter against the argmax chain.
            int tau = d.amax[0];
            for (int depth = 1;; ++depth) {
                unsigned nxt = 0;
                for (int c = 0; c < g; ++c)
                    if (((surv >> c) & 1u) && d.cands[c * L + depth - 1] == tau) nxt |= 1u << c;
                s_acc[A++] = tau;
                if (!nxt) break;
                surv = nxt;
                const int c0 = __ffs(surv) - 1;
                const int nt = d.amax[cand_u0 + c0 * L + depth - 1];
                if (depth == L) {
                    s_acc[A++] = nt;
                    break;
                }
                tau = nt;
            }
            if (A > 1) win = __ffs(surv) - 1;
            s_need_draw = 0;
        } else {
            // Algorithm 4 with greedy drafts: accept x with probability
            // dist(x); on rejection remove x from dist; draw from dist at the end.
            const float invT = 1.f / d.T;
            int dist_u = 0, depth = 1;
            for (;;) {
                const int pos = P + depth;
                int nd = 0, accepted = -1, nrej = 0;
                float rej_mass = 0.f;
                const float *lr = d.logits + static_cast<long long>(dist_u) * d.V;
                const float mx = d.lmax[dist_u], Z = d.lsum[dist_u];   // Z: mass the keep rule keeps
                const unsigned thr = d.thr_key[dist_u];
                const int cut = d.thr_cut[dist_u];
                if (depth <= L && surv) {
                    for (int c = 0; c < g; ++c) {
                        if (!((surv >> c) & 1u)) continue;
                        const int x = d.cands[c * L + depth - 1];
                        bool seen = false;
                        for (int i = 0; i < nrej; ++i) seen = seen || (s_rej[i] == x);
                        if (seen) continue;
                        const float r = draw_uniform(d.seed, pos, nd++);
                        const float ex = keep_token(lr[x], x, thr, cut) ? expf((lr[x] - mx) * invT) : 0.f;
                        const float px = ex / (Z - rej_mass);
                        if (r <= px) {
                            accepted = x;
                            break;
                        }
                        s_rej[nrej++] = x;
                        rej_mass += ex;
                    }
                }
                if (accepted >= 0) {
                    s_acc[A++] = accepted;
                    unsigned nxt = 0;
                    for (int c = 0; c < g; ++c)
                        if (((surv >> c) & 1u) && d.cands[c * L + depth - 1] == accepted) nxt |= 1u << c;
                    surv = nxt;
                    dist_u = cand_u0 + (__ffs(surv) - 1) * L + depth - 1;
                    ++depth;
                    continue;
                }
                s_dist_u = dist_u;
                s_nrej = nrej;
                s_u = draw_uniform(d.seed, pos, nd);
                break;
            }
            if (A > 0) win = __ffs(surv) - 1;
            s_need_draw = 1;
        }
        s_A = A;
        s_win = win;
    }
    __syncthreads();
    if (s_need_draw) {
        const int u = s_dist_u;
        const int x = block_inverse_cdf<kFinishThreads>(d.logits + static_cast<long long>(u) * d.V, d.V, d.lmax[u],
                                                        1.f / d.T, s_rej, s_nrej, s_u, d.thr_key[u], d.thr_cut[u]);
        if (tid == 0) {
            s_acc[s_A] = x;
            s_A = s_A + 1;
        }
        __syncthreads();
    }
    // LRU / LFU: the winning candidate was used (before the harvest); then
    // harvest the window's n-grams (column order) and slide the window.
    if (tid < 32) {
        int suf[8];
        if (d.policy != kPoolFifo && s_win >= 0) {
            for (int m = 0; m < L; ++m) suf[m] = d.cands[s_win * L + m];
            pool_use_warp(d, d.st->o, suf, tid);
        }
        for (int j = 0; j < d.W; ++j) {
            for (int k = 1; k < L; ++k) suf[k - 1] = d.window[k * d.W + j];
            suf[L - 1] = d.amax[1 + j];
            pool_insert_warp(d, d.window[j], suf, tid);
        }
    }
    __syncthreads();
    for (int j = tid; j < d.W; j += blockDim.x) {
        for (int k = 0; k + 1 < L; ++k) d.window[k * d.W + j] = d.window[(k + 1) * d.W + j];
        d.window[(L - 1) * d.W + j] = d.amax[1 + j];
    }
    if (tid == 0) {
        const int A = s_A;
        SpecState *st = d.st;
        st->P_old = P;
        st->A = A;
        st->cstar = s_win;
        for (int i = 0; i < A; ++i) {
            st->acc[i] = s_acc[i];
            d.tokens_log[P + 1 + i] = s_acc[i];
        }
        st->P = P + A;
        st->o = s_acc[A - 1];
        st->n_tokens = P + A + 1;
    }
}

// Copy K/V of the winning candidate's rows m = 1..A-1 (slot P_old + its row)
// to slots P_old + m.  Row 0 already sits at P_old.
__global__ void k_kv_commit(SpecDev d, float *cache, int nkv, int hd) {
    pdl_trigger();
    pdl_wait();
    const int A = d.st->A, cs = d.st->cstar, P0 = d.st->P_old;
    if (A <= 1 || cs < 0) return;
    const int L = d.N - 1;
    const long long plane = static_cast<long long>(blockIdx.x);   // (layer, k|v, kv head)
    float *base = cache + plane * d.max_seq * hd;
    for (int t = threadIdx.x; t < (A - 1) * hd; t += blockDim.x) {
        const int m = 1 + t / hd, i = t % hd;
        const int src = P0 + 1 + L * d.W + cs * L + (m - 1);
        base[static_cast<long long>(P0 + m) * hd + i] = base[static_cast<long long>(src) * hd + i];
    }
}

// bf16 plane layouts: block = (layer, hi|lo, KV head); K rows move like the
// fp32 cache, V^T moves column runs (the accepted rows are consecutive slots
// on both sides, and the source run lies past the destination run).
__global__ void k_kv_commit_split(SpecDev d, __nv_bfloat16 *kc, __nv_bfloat16 *vc, int hd, int seq) {
    pdl_trigger();
    pdl_wait();
    const int A = d.st->A, cs = d.st->cstar, P0 = d.st->P_old;
    if (A <= 1 || cs < 0) return;
    const int n = A - 1;
    const int span = d.N - 1;
    const int src0 = P0 + 1 + span * d.W + cs * span;   // slot of the first accepted candidate token
    const long long plane = static_cast<long long>(blockIdx.x);
    __nv_bfloat16 *kb = kc + plane * seq * hd;
    for (int t = threadIdx.x; t < n * hd; t += blockDim.x) {
        const int m = t / hd, i = t % hd;
        kb[static_cast<long long>(P0 + 1 + m) * hd + i] = kb[static_cast<long long>(src0 + m) * hd + i];
    }
    __nv_bfloat16 *vb = vc + plane * hd * seq;
    for (int t = threadIdx.x; t < n * hd; t += blockDim.x) {
        const int i = t / n, m = t % n;
        vb[static_cast<long long>(i) * seq + P0 + 1 + m] = vb[static_cast<long long>(i) * seq + src0 + m];
    }
}

// ------------------------------------------------------------------ pool seeding / import
__global__ void k_pool_insert(SpecDev d, const int *records, const int *uses, int n) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x;
    const int N = d.N;
    for (int i = 0; i < n; ++i)
        pool_insert_warp(d, records[i * N], records + i * N + 1, lane, uses ? uses[i] : 0);
}

__global__ void k_pool_seed_prompt(SpecDev d, int n) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x;
    const int N = d.N;
    for (int i = 0; i + N <= n; ++i) pool_insert_warp(d, d.tokens_log[i], d.tokens_log + i + 1, lane);
}

__global__ void __launch_bounds__(kFinishThreads) k_first_token(SpecDev d, int n) {
    pdl_trigger();
    pdl_wait();
    int y;
    if (d.T <= 0.f) {
        y = d.amax[0];
    } else {
        const float u = draw_uniform(d.seed, n, 0);
        y = block_inverse_cdf<kFinishThreads>(d.logits, d.V, d.lmax[0], 1.f / d.T, nullptr, 0, u, d.thr_key[0],
                                              d.thr_cut[0]);
    }
    if (threadIdx.x == 0) {
        d.tokens_log[n] = y;
        d.st->o = y;
        d.st->P = n;
        d.st->n_tokens = n + 1;
        d.st->A = 0;
        d.st->g = 0;
        d.st->cstar = -1;
    }
}

// ------------------------------------------------------------------ launchers
cudaError_t build_rows_launch(const SpecDev &d, cudaStream_t s) {
    launch_k(k_build_rows, dim3(1), dim3(256), 0, s, d);
    return cudaGetLastError();
}
cudaError_t finish_step_launch(const SpecDev &d, cudaStream_t s) {
    launch_k(k_finish_step, dim3(1), dim3(kFinishThreads), 0, s, d);
    return cudaGetLastError();
}
cudaError_t kv_commit_launch(const SpecDev &d, float *cache, int L, int nkv, int hd, cudaStream_t s) {
    launch_k(k_kv_commit, dim3(L * 2 * nkv), dim3(128), 0, s, d, cache, nkv, hd);
    return cudaGetLastError();
}

cudaError_t kv_commit_split_launch(const SpecDev &d, __nv_bfloat16 *kc, __nv_bfloat16 *vc, int L, int nkv, int hd,
                                   int seq, cudaStream_t s) {
    launch_k(k_kv_commit_split, dim3(L * 2 * nkv), dim3(128), 0, s, d, kc, vc, hd, seq);
    return cudaGetLastError();
}

cudaError_t pool_insert_launch(const SpecDev &d, const int *records, const int *uses, int n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    launch_k(k_pool_insert, dim3(1), dim3(32), 0, s, d, records, uses, n);
    return cudaGetLastError();
}
cudaError_t pool_seed_prompt_launch(const SpecDev &d, int n, cudaStream_t s) {
    launch_k(k_pool_seed_prompt, dim3(1), dim3(32), 0, s, d, n);
    return cudaGetLastError();
}
cudaError_t first_token_launch(const SpecDev &d, int n, cudaStream_t s) {
    launch_k(k_first_token, dim3(1), dim3(kFinishThreads), 0, s, d, n);
    return cudaGetLastError();
}

}  // namespace la
