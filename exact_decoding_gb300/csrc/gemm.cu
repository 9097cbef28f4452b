// Projection GEMMs of the lookahead step: every weight byte is read once per
// step and multiplied against all M = 1 + (W+G)(N-1) step rows at once
// (the "extra tokens per step" of section 4 of the paper-graph-ui page ride
// on the same weight stream).
//
// bf16 path -- tcgen05 tensor cores, swap-AB: the weight matrix [out][K] is
// the UMMA A operand (K-major), the step rows [rows][K] are the B operand as
// bf16 (hi, lo) pairs stacked along N, the fp32 accumulator lives in TMEM.
// k_gemm_tc2 (the step's GEMMs) runs one 2-SM UMMA (cta_group::2, M = 256
// features, N = 256 = hi rows + lo rows) per CTA pair of a thread-block
// cluster: each CTA streams its 128 weight rows and its half of the input
// rows through a TMA ring, the pair leader issues the UMMAs, four warps per
// CTA drain TMEM and add the hi and lo columns.  k_gemm_tc is the 1-SM form
// (M = 128), used by la_gemm_bf16.  The flattened tile x k-block work is
// split evenly over the SMs (stream-K); partial sums go to a workspace and
// are added in a fixed order by the consumer kernel, so results are
// deterministic.
//
// fp32 path -- a plain SIMT kernel (fp32 FMA, no tf32) for fp32 models.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <vector>

#include "la_kernels.h"

namespace la {

// ------------------------------------------------------------------ tcgen05 kernel
// Work: a list of segments (tile, k-block range, partial plane).  With a
// segment table each CTA runs the contiguous run of segments the host gave
// it (stream-K: the flattened tile x k-block work split evenly over the
// SMs); without one, CTA b runs the single segment (tile b / splits, split b
// % splits, plane = split).  The accumulator is double-buffered in TMEM so a
// segment's epilogue overlaps the next segment's main loop.
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

struct SegInfo {
    int seg, row0, kb0, kb1, plane;
};

__device__ __forceinline__ SegInfo segment(const TcGemmParams &p, int i) {
    int tile, kb0, kb1, plane;
    if (p.segs) {
        const int4 s = p.segs[i];
        tile = s.x;
        kb0 = s.y;
        kb1 = s.z;
        plane = s.w;
    } else {
        tile = i / p.splits;
        const int split = i % p.splits;
        kb0 = static_cast<int>((static_cast<long long>(split) * p.n_kb) / p.splits);
        kb1 = static_cast<int>((static_cast<long long>(split + 1) * p.n_kb) / p.splits);
        plane = split;
    }
    int seg = 0;
    while (seg + 1 < p.nseg && tile >= p.seg_tile0[seg + 1]) ++seg;
    return SegInfo{seg, (tile - p.seg_tile0[seg]) * kTileM, kb0, kb1, plane};
}

__global__ void __launch_bounds__(192, 1) k_gemm_tc(const __grid_constant__ TcGemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int bn = p.bn;
    const uint32_t a_bytes = kTileM * kBlockK * 2;
    const uint32_t b_bytes = static_cast<uint32_t>(bn) * kBlockK * 2;
    const uint32_t stage_bytes = a_bytes + b_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.stages * stage_bytes);
    uint64_t *full = bars;
    uint64_t *empty = bars + p.stages;
    uint64_t *accfull = bars + 2 * p.stages;       // [2]
    uint64_t *accempty = bars + 2 * p.stages + 2;  // [2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * p.stages + 4);

    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int sbeg, send;
    if (p.segs) {
        sbeg = p.cta_first[blockIdx.x];
        send = p.cta_first[blockIdx.x + 1];
    } else {
        sbeg = blockIdx.x;
        send = blockIdx.x + 1;
    }
    // Two accumulator buffers when this CTA runs more than one segment.
    const int nbuf = (send - sbeg) > 1 ? 2 : 1;
    uint32_t ncols = 32;
    while (ncols < static_cast<uint32_t>(nbuf * bn)) ncols <<= 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&accfull[b]), 1);
            mbar_init(smem_u32(&accempty[b]), 4);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // TMA producer: weights stream through L2 once (evict first); the
            // small row block is re-read by every CTA (evict last).
            for (int sg = 0; sg < p.nseg; ++sg) prefetch_tensormap(&p.a[sg]);
            prefetch_tensormap(&p.b);
            const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
            // Weights do not depend on the previous kernel: fill the ring's
            // weight halves before waiting for it, then load the input rows.
            int it = 0;
            for (int i = sbeg; i < send && it < p.stages; ++i) {
                const SegInfo g = segment(p, i);
                for (int kb = g.kb0; kb < g.kb1 && it < p.stages; ++kb, ++it) {
                    const uint32_t fb = smem_u32(&full[it]);
                    mbar_arrive_expect_tx(fb, stage_bytes);
                    tma_load_2d(smem_u32(smem + it * stage_bytes), &p.a[g.seg], kb * kBlockK, g.row0, fb, pol_w);
                }
            }
            const int npre = it;
            pdl_wait();
            it = 0;
            bool ok = true;
            for (int i = sbeg; i < send && ok; ++i) {
                const SegInfo g = segment(p, i);
                for (int kb = g.kb0; kb < g.kb1; ++kb, ++it) {
                    const int st = it % p.stages;
                    const uint32_t sa = smem_u32(smem + st * stage_bytes);
                    const uint32_t fb = smem_u32(&full[st]);
                    if (it < npre) {
                        tma_load_2d(sa + a_bytes, &p.b, kb * kBlockK, 0, fb, pol_x);
                        continue;
                    }
                    if (!mbar_wait(smem_u32(&empty[st]), ((it / p.stages) & 1) ^ 1, p.err, ERR_TIMEOUT_EMPTY)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(fb, stage_bytes);
                    tma_load_2d(sa, &p.a[g.seg], kb * kBlockK, g.row0, fb, pol_w);
                    tma_load_2d(sa + a_bytes, &p.b, kb * kBlockK, 0, fb, pol_x);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // UMMA issuer: 4 instructions of K = 16 per 64-wide stage.
            const uint32_t idesc = umma_idesc_bf16(kTileM, bn);
            int it = 0, ul = 0;
            bool ok = true;
            for (int i = sbeg; i < send; ++i, ++ul) {
                const SegInfo g = segment(p, i);
                const int buf = ul & 1;
                if (ok && ul >= 2)
                    ok = mbar_wait(smem_u32(&accempty[buf]), ((ul >> 1) & 1) ^ 1, p.err, ERR_TIMEOUT_ACCUM);
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(buf * bn);
                for (int kb = g.kb0; kb < g.kb1 && ok; ++kb, ++it) {
                    const int st = it % p.stages;
                    if (!mbar_wait(smem_u32(&full[st]), (it / p.stages) & 1, p.err, ERR_TIMEOUT_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + st * stage_bytes);
                    const uint64_t da = umma_desc_sw128(sa), db = umma_desc_sw128(sa + a_bytes);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk)
                        umma_bf16(d, da + 2 * kk, db + 2 * kk, idesc, (kb != g.kb0 || kk != 0) ? 1u : 0u);
                    umma_commit(smem_u32(&empty[st]));
                }
                umma_commit(smem_u32(&accfull[buf]));
            }
        }
    } else {
        // Epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 = output features.
        const int q = warp & 3;
        int ul = 0;
        for (int i = sbeg; i < send; ++i, ++ul) {
            const SegInfo g = segment(p, i);
            const int buf = ul & 1;
            bool ok = mbar_wait(smem_u32(&accfull[buf]), (ul >> 1) & 1, p.err, ERR_TIMEOUT_ACCUM);
            ok = __all_sync(0xffffffffu, ok);
            __syncwarp();
            tc_fence_after();
            if (!ok) break;
            const int f = g.row0 + 32 * q + lane;
            const bool fv = f < p.seg_out[g.seg];
            float *out = p.out + static_cast<long long>(g.plane) * p.split_stride + p.seg_col0[g.seg] + f;
            const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(buf * bn);
            if (p.bh > 0) {
                // columns c (hi rows) + columns c + bh (lo rows) = one output row
                for (int c0 = 0; c0 < p.bh; c0 += 32) {
                    uint32_t r[32], s2[32];
                    tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(c0), r);
                    tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(c0 + p.bh), s2);
                    tmem_ld_wait();
                    if (fv) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int row = c0 + j;
                            if (row < p.nrows)
                                out[static_cast<long long>(row) * p.ldo] = __uint_as_float(r[j]) + __uint_as_float(s2[j]);
                        }
                    }
                }
            } else {
                for (int c0 = 0; c0 < bn; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(c0), r);
                    tmem_ld_wait();
                    if (fv) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int row = c0 + j;
                            if (row < p.nrows) out[static_cast<long long>(row) * p.ldo] = __uint_as_float(r[j]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&accempty[buf]));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

// ------------------------------------------------------------------ 2-SM (cta_group::2) kernel
// A cluster of two CTAs computes a 256-feature tile: UMMA M = 256 weight rows
// (128 in each CTA's shared memory), N = 256 input rows (hi rows 0..127 held
// by rank 0, lo rows 128..255 by rank 1), K = 16.  Rank 0 issues every MMA;
// both CTAs' TMA loads complete on rank 0's full barrier; the MMA commits are
// multicast to both CTAs.  Each CTA's TMEM holds D for its 128 weight rows
// (columns c = hi row c, c + 128 = lo row c), drained by its own epilogue.
// Compared with the 1-SM kernel, a shared-memory stage per SM is half as
// large (16 KB weights + 16 KB rows) and one MMA covers twice the weights.
// With nrt = 2 (prefill chunks of 256 rows) a stage carries two row tiles:
// each weight k-block feeds two MMAs, into the two TMEM accumulators
// (columns t * 256 ..), so the accumulators are no longer double-buffered
// across segments; the ring is 4 stages of 48 KB.
//
// With SUB = 2 a stage holds two adjacent 64-column k-blocks of the same
// weight rows (and rows), loaded back to back: the weight rows are read 256
// contiguous bytes at a time instead of 128, and the producer waits once per
// two k-blocks.  The schedule's k units are then 128 columns wide; a unit
// past K reads zeros (TMA fill), which add nothing.
// Named barrier over the `n` threads of the calling warps (id != 0); the
// .red form returns the AND of every thread's predicate.
__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ bool named_bar_and(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// Fused SwiGLU of rows [r0, r1) of one split 128-column tile t2 of the
// gate/up GEMM, run by the epilogue's 128 threads (e = 0..127) of one CTA
// that contributed a piece of the tile, once every piece has arrived: gate =
// sum of the tile's planes at columns 128 t2 + j, up = at 128 t2 + 64 + j
// (j < 64), in plane order; feature f = 64 t2 + j.  Two items (a row's four
// features) per thread per pass, four planes of both loaded together.  Loads
// bypass L1: other SMs wrote the planes during this launch.
__device__ __noinline__ void swiglu_fixup(const TcGemmParams &p, int t2, int r0, int r1, int e) {
    const int np = p.fuse_np[t2];
    const long long ss = p.split_stride;
    const float *base = p.out + static_cast<long long>(r0) * p.ldo + t2 * kTileM;
    const int fbase = t2 * 64, nit = (r1 - r0) * 16;
    for (int i0 = e; i0 < nit; i0 += 2 * 128) {
        const float *pr[2];
        float4 g[2], u[2];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int i = i0 + b * 128 < nit ? i0 + b * 128 : i0;
            pr[b] = base + static_cast<long long>(i >> 4) * p.ldo + 4 * (i & 15);
            g[b] = make_float4(0.f, 0.f, 0.f, 0.f);
            u[b] = g[b];
        }
        for (int k0 = 0; k0 < np; k0 += 4) {   // four planes of both items in flight, added in plane order
            float4 xg[2][4], xu[2][4];
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (k0 + k < np) {
                        xg[b][k] = __ldcg(reinterpret_cast<const float4 *>(pr[b] + (k0 + k) * ss));
                        xu[b][k] = __ldcg(reinterpret_cast<const float4 *>(pr[b] + 64 + (k0 + k) * ss));
                    }
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (k0 + k < np) {
                        add4(g[b], xg[b][k]);
                        add4(u[b], xu[b][k]);
                    }
        }
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int i = i0 + b * 128;
            const int f = fbase + 4 * (i & 15);
            const float4 gg = g[b], uu = u[b];
            if (i < nit && f < p.fuse_F)
                store_act4(p.fuse_out, static_cast<long long>(r0 + (i >> 4)) * p.fuse_F + f,
                           make_float4(__fdividef(gg.x, 1.f + __expf(-gg.x)) * uu.x,
                                       __fdividef(gg.y, 1.f + __expf(-gg.y)) * uu.y,
                                       __fdividef(gg.z, 1.f + __expf(-gg.z)) * uu.z,
                                       __fdividef(gg.w, 1.f + __expf(-gg.w)) * uu.w),
                           p.fuse_lo_off);
        }
    }
}

template <int NRT, int SUB, bool FUSE = false>
__global__ void __launch_bounds__(192, 1) k_gemm_tc2(const __grid_constant__ TcGemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    constexpr uint32_t box_bytes = kTileM * kBlockK * 2;   // 128 rows x 64 columns
    constexpr uint32_t a_bytes = SUB * box_bytes;          // 128 weight rows, SUB k-blocks
    // Input rows per CTA and row tile (hi rows in rank 0, lo rows in rank 1):
    // bnh when set (a one-row forward), else bh for a single row tile of at
    // most 128 rows (a step, the lm_head), else 128; the UMMA N is twice that.
    const int nhalf = NRT == 1 && p.bnh > 0 ? p.bnh : gemm2_nhalf(NRT, p.bh);
    const uint32_t bbox_bytes = static_cast<uint32_t>(nhalf) * kBlockK * 2;
    const uint32_t b_bytes = SUB * bbox_bytes;             // this CTA's input rows of one row tile
    constexpr int nrt = NRT;
    constexpr int nbuf = nrt == 1 ? 2 : 1;                 // accumulators in flight
    const uint32_t stage_bytes = a_bytes + static_cast<uint32_t>(nrt) * b_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.stages * stage_bytes);
    uint64_t *full = bars;
    uint64_t *empty = bars + p.stages;
    uint64_t *accfull = bars + 2 * p.stages;       // [2]
    uint64_t *accempty = bars + 2 * p.stages + 2;  // [2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * p.stages + 4);

    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int sbeg = p.cta_first[pair], send = p.cta_first[pair + 1];
    constexpr uint32_t ncols = 512;   // two 256-column accumulators

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&accfull[b]), 1);
            mbar_init(smem_u32(&accempty[b]), 8);    // 4 epilogue warps in each CTA
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), ncols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();   // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            for (int sg = 0; sg < p.nseg; ++sg) prefetch_tensormap(&p.a[sg]);
            prefetch_tensormap(&p.b);
            const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
            const int brow = static_cast<int>(rank) * p.bh;     // hi rows (rank 0) or lo rows (rank 1)
            auto weight_row = [&](const SegInfo &g) { return 2 * g.row0 + static_cast<int>(rank) * kTileM; };
            // The weight half of one stage: SUB boxes of 128 rows, or with
            // FUSE a 64-row gate box and the matching 64-row up box each.
            auto load_w = [&](uint32_t sa, const SegInfo &g, int kb, uint32_t fl) {
#pragma unroll
                for (int s = 0; s < SUB; ++s) {
                    const int col = (kb * SUB + s) * kBlockK;
                    if constexpr (FUSE) {
                        const int f0 = g.row0 + 64 * static_cast<int>(rank);
                        tma_load_2d_pair(sa + s * box_bytes, &p.a[0], col, f0, fl, pol_w);
                        tma_load_2d_pair(sa + s * box_bytes + box_bytes / 2, &p.a[1], col, f0, fl, pol_w);
                    } else {
                        tma_load_2d_pair(sa + s * box_bytes, &p.a[g.seg], col, weight_row(g), fl, pol_w);
                    }
                }
            };
            int it = 0;
            for (int i = sbeg; i < send && it < p.stages; ++i) {
                const SegInfo g = segment(p, i);
                for (int kb = g.kb0; kb < g.kb1 && it < p.stages; ++kb, ++it) {
                    const uint32_t fl = mapa_shared(smem_u32(&full[it]), 0);
                    if (leader) mbar_arrive_expect_tx(smem_u32(&full[it]), 2 * stage_bytes);
                    load_w(smem_u32(smem + it * stage_bytes), g, kb, fl);
                }
            }
            const int npre = it;
            pdl_wait();
            it = 0;
            bool ok = true;
            for (int i = sbeg; i < send && ok; ++i) {
                const SegInfo g = segment(p, i);
                for (int kb = g.kb0; kb < g.kb1; ++kb, ++it) {
                    const int st = it % p.stages;
                    const uint32_t sa = smem_u32(smem + st * stage_bytes);
                    const uint32_t fl = mapa_shared(smem_u32(&full[st]), 0);
                    if (it < npre) {
#pragma unroll
                        for (int t = 0; t < nrt; ++t)
#pragma unroll
                            for (int s = 0; s < SUB; ++s)
                                tma_load_2d_pair(sa + a_bytes + t * b_bytes + s * bbox_bytes, &p.b,
                                                 (kb * SUB + s) * kBlockK, brow + t * kTileM, fl, pol_x);
                        continue;
                    }
                    if (!mbar_wait_cluster(smem_u32(&empty[st]), ((it / p.stages) & 1) ^ 1, p.err, ERR_TIMEOUT_EMPTY)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(smem_u32(&full[st]), 2 * stage_bytes);
                    load_w(sa, g, kb, fl);
#pragma unroll
                    for (int t = 0; t < nrt; ++t)
#pragma unroll
                        for (int s = 0; s < SUB; ++s)
                            tma_load_2d_pair(sa + a_bytes + t * b_bytes + s * bbox_bytes, &p.b,
                                             (kb * SUB + s) * kBlockK, brow + t * kTileM, fl, pol_x);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // Pair UMMA issuer: M = 256, N = 256, 4 k-steps of 16 per k-block.
            const uint32_t idesc = umma_idesc_bf16(2 * kTileM, 2 * nhalf);
            int it = 0, ul = 0;
            bool ok = true;
            for (int i = sbeg; i < send; ++i, ++ul) {
                const SegInfo g = segment(p, i);
                const int buf = ul % nbuf, use = ul / nbuf;   // use-th time this accumulator is filled
                if (ok && use >= 1)
                    ok = mbar_wait_cluster(smem_u32(&accempty[buf]), (use - 1) & 1, p.err, ERR_TIMEOUT_ACCUM);
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(buf * 2 * kTileM);
                for (int kb = g.kb0; kb < g.kb1 && ok; ++kb, ++it) {
                    const int st = it % p.stages;
                    if (!mbar_wait_cluster(smem_u32(&full[st]), (it / p.stages) & 1, p.err, ERR_TIMEOUT_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + st * stage_bytes);
#pragma unroll
                    for (int t = 0; t < nrt; ++t) {
                        const uint32_t dt = d + static_cast<uint32_t>(t * 2 * kTileM);
#pragma unroll
                        for (int s = 0; s < SUB; ++s) {
                            const uint64_t da = umma_desc_sw128(sa + s * box_bytes);
                            const uint64_t db = umma_desc_sw128(sa + a_bytes + t * b_bytes + s * bbox_bytes);
#pragma unroll
                            for (int kk = 0; kk < kBlockK / 16; ++kk)
                                umma_pair_bf16(dt, da + 2 * kk, db + 2 * kk, idesc,
                                               (kb != g.kb0 || s != 0 || kk != 0) ? 1u : 0u);
                        }
                    }
                    umma_pair_commit(smem_u32(&empty[st]), 0x3);
                }
                umma_pair_commit(smem_u32(&accfull[buf]), 0x3);
            }
        }
    } else {
        // Epilogue: TMEM lanes 32*(w%4).. = this CTA's weight rows; columns c
        // and c + 128 are the hi and lo input row c.
        const int q = warp & 3;
        const uint32_t acc_leader[2] = {mapa_shared(smem_u32(&accempty[0]), 0), mapa_shared(smem_u32(&accempty[1]), 0)};
        // FUSE: split tiles this CTA has published a piece of, waiting for
        // the rest: (tile, arrival count that completes it, share = plane).
        // Every piece is published before any wait, so no CTA waits on a
        // CTA that is itself waiting.
        __shared__ int4 s_pend[8];
        __shared__ int s_ok;
        int npend = 0;
        auto flush = [&]() {
            named_bar_sync(1, 128);   // s_pend written by thread 64
            for (int k = 0; k < npend; ++k) {
                const int4 pd = s_pend[k];
                if (threadIdx.x == 64) {
                    bool arrived = ld_acquire_gpu(p.fuse_cnt + pd.x) - pd.y >= 0;
                    const uint64_t t0 = globaltimer();
                    while (!arrived) {
                        __nanosleep(64);
                        arrived = ld_acquire_gpu(p.fuse_cnt + pd.x) - pd.y >= 0;
                        if (!arrived && globaltimer() - t0 > kWaitNs) {
                            atomicOr(p.err, ERR_TIMEOUT_TILE);
                            break;
                        }
                    }
                    s_ok = arrived;
                }
                named_bar_sync(1, 128);
                if (s_ok) {
                    const int np = p.fuse_np[pd.x];
                    swiglu_fixup(p, pd.x, pd.z * p.nrows / np, (pd.z + 1) * p.nrows / np,
                                 static_cast<int>(threadIdx.x) - 64);
                }
                named_bar_sync(1, 128);   // s_ok is rewritten for the next entry
            }
            npend = 0;
        };
        int ul = 0;
        for (int i = sbeg; i < send; ++i, ++ul) {
            const SegInfo g = segment(p, i);
            const int buf = ul % nbuf;
            if constexpr (FUSE) {
                // before waiting for a whole tile's accumulator, finish the
                // split tiles (their other pieces are done early in every run)
                if (npend > 0 && (npend == 8 || p.fuse_np[2 * g.row0 / kTileM + static_cast<int>(rank)] == 1)) flush();
            }
            bool ok = mbar_wait_cluster(smem_u32(&accfull[buf]), (ul / nbuf) & 1, p.err, ERR_TIMEOUT_ACCUM);
            ok = __all_sync(0xffffffffu, ok);
            // With FUSE the four epilogue warps meet at named barriers below,
            // so they take the same branch here.
            if constexpr (FUSE) ok = named_bar_and(1, 128, ok);
            __syncwarp();
            tc_fence_after();
            if (!ok) break;
            if constexpr (FUSE) {
                // A tile no other CTA touched (one plane): SwiGLU straight
                // from TMEM.  Lanes 0..63 hold gate rows, 64..127 the up rows
                // of the same features; the up warps pass their sums through
                // shared memory, 32 input rows at a time.
                const int t2 = 2 * g.row0 / kTileM + static_cast<int>(rank);
                if (p.fuse_np[t2] == 1) {
                    // [128 lanes][33]: this chunk's gate (lanes 0..63) and up
                    // (64..127) sums; then thread e takes features 2 (e % 32),
                    // + 1 of rows e / 32 + 4 k, so a warp stores 64 bf16 of one row.
                    __shared__ float xch[128 * 33];
                    const uint32_t lb = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(buf * 2 * kTileM);
                    const int e = static_cast<int>(threadIdx.x) - 64, fp = 2 * (e & 31), f = 64 * t2 + fp;
                    for (int c0 = 0; c0 < kTileM && c0 < p.nrows; c0 += 32) {
                        uint32_t r[32], s2[32];
                        tmem_ld_32x32b_x32(lb + static_cast<uint32_t>(c0), r);
                        tmem_ld_32x32b_x32(lb + static_cast<uint32_t>(c0 + nhalf), s2);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            xch[(32 * q + lane) * 33 + j] = __uint_as_float(r[j]) + __uint_as_float(s2[j]);
                        named_bar_sync(1, 128);
                        if (f < p.fuse_F) {
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const int j = (e >> 5) + 4 * k, row = c0 + j;
                                if (row < p.nrows) {
                                    const float g0 = xch[fp * 33 + j], g1 = xch[(fp + 1) * 33 + j];
                                    const float u0 = xch[(64 + fp) * 33 + j], u1 = xch[(65 + fp) * 33 + j];
                                    store_act2(p.fuse_out, static_cast<long long>(row) * p.fuse_F + f,
                                               __fdividef(g0, 1.f + __expf(-g0)) * u0,
                                               __fdividef(g1, 1.f + __expf(-g1)) * u1, p.fuse_lo_off);
                                }
                            }
                        }
                        named_bar_sync(1, 128);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(acc_leader[buf]);
                    continue;
                }
            }
            const int f = 2 * g.row0 + static_cast<int>(rank) * kTileM + 32 * q + lane;
            const bool fv = f < p.seg_out[g.seg];
            float *out = p.out + static_cast<long long>(g.plane) * p.split_stride + p.seg_col0[g.seg] + f;
            const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(buf * 2 * kTileM);
            for (int c0 = 0; c0 < nrt * kTileM && c0 < p.nrows; c0 += 32) {
                // rows c0 .. c0 + 31: tile t = c0 / 128 at columns t * 256 + (c0 % 128) (hi) and + 128 (lo)
                const uint32_t col = static_cast<uint32_t>((c0 / kTileM) * 2 * kTileM + c0 % kTileM);
                uint32_t r[32], s2[32];
                tmem_ld_32x32b_x32(lane_base + col, r);
                tmem_ld_32x32b_x32(lane_base + col + static_cast<uint32_t>(nhalf), s2);
                tmem_ld_wait();
                if (fv && c0 < p.nrows) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int row = c0 + j;
                        if (row < p.nrows)
                            out[static_cast<long long>(row) * p.ldo] = __uint_as_float(r[j]) + __uint_as_float(s2[j]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc_leader[buf]);
            if constexpr (FUSE) {
                // Publish this partial and count the arrival.  The count only
                // grows (by the tile's planes per launch): the pieces of this
                // launch are complete when it reaches the next multiple of them.
                const int t2 = 2 * g.row0 / kTileM + static_cast<int>(rank);
                __threadfence();
                named_bar_sync(1, 128);
                if (threadIdx.x == 64) {
                    const int np = p.fuse_np[t2];
                    const int old = atomicAdd(p.fuse_cnt + t2, 1);
                    s_pend[npend] = make_int4(t2, (old / np + 1) * np, g.plane, 0);
                }
                ++npend;
            }
        }
        if constexpr (FUSE) {
            if (npend > 0) flush();
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // the leader's MMAs read both CTAs' shared memory: finish together
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, ncols);
    }
}

// Stage: SUB k-blocks of 128 weight rows and of nrt row tiles of `nhalf`
// input rows (nhalf as in the kernel: bnh, bh or 128).
static size_t gemm2_stage_bytes(int nrt, int sub, int nhalf) {
    return static_cast<size_t>(sub) * (kTileM + nrt * nhalf) * kBlockK * 2;
}

size_t tc_gemm2_smem_bytes(int stages, int nrt, int sub, int nhalf) {
    return static_cast<size_t>(stages) * gemm2_stage_bytes(nrt, sub, nhalf) + 1024 + 256;
}

int tc_gemm2_stages(int nrt, int sub, int nhalf) {
    // as many stages as fit in 200 KB, at most 8 (128-row halves: 6 for one row
    // tile, 4 for two, 3 for one row tile with two k-blocks per stage)
    const int n = static_cast<int>((200 * 1024) / gemm2_stage_bytes(nrt, sub, nhalf));
    return n > 8 ? 8 : n;
}

// Raise a kernel's dynamic shared-memory limit to the device's opt-in
// maximum less its static shared memory.  Function attributes are per
// device, so `done` keeps one bit per device index (indices past 63 set the
// attribute on every call).
static cudaError_t smem_attr_per_device(const void *fn, std::atomic<unsigned long long> &done) {
    int dev = 0, mx = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit && (done.load() & bit)) return cudaSuccess;
    cudaFuncAttributes fa;
    e = cudaDeviceGetAttribute(&mx, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, fn);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 mx - static_cast<int>(fa.sharedSizeBytes));
    if (e == cudaSuccess) done.fetch_or(bit);
    return e;
}

static cudaError_t gemm2_smem_attr() {
    static std::atomic<unsigned long long> done1{0}, done2{0}, done3{0}, done4{0};
    cudaError_t e = smem_attr_per_device(reinterpret_cast<const void *>(k_gemm_tc2<1, 1>), done1);
    if (e == cudaSuccess) e = smem_attr_per_device(reinterpret_cast<const void *>(k_gemm_tc2<2, 1>), done2);
    if (e == cudaSuccess) e = smem_attr_per_device(reinterpret_cast<const void *>(k_gemm_tc2<1, 2>), done3);
    if (e == cudaSuccess) e = smem_attr_per_device(reinterpret_cast<const void *>(k_gemm_tc2<1, 2, true>), done4);
    return e;
}

int tc_gemm2_max_pairs() {
    if (gemm2_smem_attr() != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 512);
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = tc_gemm2_smem_bytes(tc_gemm2_stages());
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_gemm_tc2<1, 1>, &cfg) != cudaSuccess) return 0;
    return n;
}

cudaError_t tc_gemm2_launch(const TcGemm &g, cudaStream_t s) {
    cudaError_t e = gemm2_smem_attr();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * g.ctas);
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = g.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (g.p.fuse_out) {   // fused SwiGLU: step mode only (one row tile, two k-blocks per stage)
        if (g.p.nrt != 1 || g.p.sub != 2) return cudaErrorInvalidValue;
        return cudaLaunchKernelEx(&cfg, k_gemm_tc2<1, 2, true>, g.p);
    }
    if (g.p.nrt == 2) return cudaLaunchKernelEx(&cfg, k_gemm_tc2<2, 1>, g.p);
    if (g.p.sub == 2) return cudaLaunchKernelEx(&cfg, k_gemm_tc2<1, 2>, g.p);
    return cudaLaunchKernelEx(&cfg, k_gemm_tc2<1, 1>, g.p);
}

size_t tc_gemm_smem_bytes(int bn, int stages) {
    return static_cast<size_t>(stages) * (kTileM * kBlockK * 2 + bn * kBlockK * 2) + 1024 + 256;
}

// Stream-K schedule: the flattened (tile, k-block) work split into `ctas`
// contiguous, equal runs (+-1 k-block); a run is cut at tile boundaries into
// segments.  Partial plane of a segment = how many earlier CTAs touched its
// tile, so tile t has tile_planes[t] planes, added in plane order.
void stream_k_schedule(int tiles, int n_kb, int ctas, std::vector<int> &segs, std::vector<int> &cta_first,
                       std::vector<int> &tile_planes) {
    const long long W = static_cast<long long>(tiles) * n_kb;
    if (ctas > W) ctas = static_cast<int>(W);
    segs.clear();
    cta_first.assign(ctas + 1, 0);
    tile_planes.assign(tiles, 0);
    for (int c = 0; c < ctas; ++c) {
        cta_first[c] = static_cast<int>(segs.size() / 4);
        long long s = W * c / ctas;
        const long long e = W * (c + 1) / ctas;
        while (s < e) {
            const int t = static_cast<int>(s / n_kb);
            const int k0 = static_cast<int>(s % n_kb);
            const int k1 = static_cast<int>(std::min<long long>(n_kb, k0 + (e - s)));
            segs.push_back(t);
            segs.push_back(k0);
            segs.push_back(k1);
            segs.push_back(tile_planes[t]++);
            s += k1 - k0;
        }
    }
    cta_first[ctas] = static_cast<int>(segs.size() / 4);
}

// Whole tiles first, stream-K for the rest: each CTA takes an even share of
// the k-blocks of the last `tiles % ctas` tiles (split as above, planes in
// CTA order), then `tiles / ctas` whole tiles of its own (one plane each).
// Split tiles are done early in every CTA's run, so the CTAs that share one
// can finish it (the fused SwiGLU) while their whole tiles stream.
void hybrid_schedule(int tiles, int n_kb, int ctas, std::vector<int> &segs, std::vector<int> &cta_first,
                     std::vector<int> &tile_planes) {
    const int whole = ctas > 0 ? tiles / ctas : 0;
    if (whole == 0) {
        stream_k_schedule(tiles, n_kb, ctas, segs, cta_first, tile_planes);
        return;
    }
    const int t_split = whole * ctas;   // tiles [t_split, tiles) are split
    const long long W = static_cast<long long>(tiles - t_split) * n_kb;
    segs.clear();
    cta_first.assign(ctas + 1, 0);
    tile_planes.assign(tiles, 0);
    for (int c = 0; c < ctas; ++c) {
        cta_first[c] = static_cast<int>(segs.size() / 4);
        long long s = W * c / ctas;
        const long long e = W * (c + 1) / ctas;
        while (s < e) {
            const int t = t_split + static_cast<int>(s / n_kb);
            const int k0 = static_cast<int>(s % n_kb);
            const int k1 = static_cast<int>(std::min<long long>(n_kb, k0 + (e - s)));
            segs.push_back(t);
            segs.push_back(k0);
            segs.push_back(k1);
            segs.push_back(tile_planes[t]++);
            s += k1 - k0;
        }
        for (int w = 0; w < whole; ++w) {
            const int t = c * whole + w;
            segs.push_back(t);
            segs.push_back(0);
            segs.push_back(n_kb);
            segs.push_back(tile_planes[t]++);
        }
    }
    cta_first[ctas] = static_cast<int>(segs.size() / 4);
}

int tc_gemm_stages_for(int bn) {
    // Two CTAs per SM when they fit (about 113 KB each), else one deep ring.
    const size_t stage = kTileM * kBlockK * 2 + static_cast<size_t>(bn) * kBlockK * 2;
    int s = static_cast<int>((113 * 1024 - 1280) / stage);
    if (s >= 3) return s > 6 ? 6 : s;
    s = static_cast<int>((220 * 1024 - 1280) / stage);
    return s > 8 ? 8 : (s < 2 ? 2 : s);
}

// The 1-SM kernel's limit, per device like the 2-SM kernel's.
static cudaError_t gemm_smem_attr() {
    static std::atomic<unsigned long long> done{0};
    return smem_attr_per_device(reinterpret_cast<const void *>(k_gemm_tc), done);
}

int tc_gemm_ctas_per_sm(int bn, int stages) {
    const size_t sm = tc_gemm_smem_bytes(bn, stages);
    gemm_smem_attr();
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemm_tc, 192, sm) != cudaSuccess) n = 1;
    return n < 1 ? 1 : n;
}

int choose_splits(int tiles, int n_kb, int slots) {
    // The GEMM is bound by HBM, not by waves: it needs every SM streaming,
    // not every CTA slot filled.  Take the fewest K-splits that put at least
    // one CTA on (nearly) every SM, since each split adds S x rows x out fp32
    // partials that the consumer kernel must read back.  Keep >= 4 k-blocks
    // (256 K) per CTA.
    int nsm = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        nsm = 148;
    (void)slots;
    int s = 1;
    while (tiles * s < (nsm * 9) / 10 && n_kb / (s + 1) >= 4 && s < 16) ++s;
    return s;
}

void tc_gemm_finalize(TcGemm &g) {
    if (g.pair) {
        if (g.p.nrt < 1) g.p.nrt = 1;
        if (g.p.sub < 1 || g.p.nrt == 2) g.p.sub = 1;
        const int nhalf = g.p.nrt == 1 && g.p.bnh > 0 ? g.p.bnh : gemm2_nhalf(g.p.nrt, g.p.bh);
        g.p.stages = tc_gemm2_stages(g.p.nrt, g.p.sub, nhalf);
        g.grid = 2 * g.ctas;
        g.smem = tc_gemm2_smem_bytes(g.p.stages, g.p.nrt, g.p.sub, nhalf);
        return;
    }
    g.grid = g.p.segs ? g.ctas : g.p.seg_tile0[g.p.nseg] * g.p.splits;
    g.smem = tc_gemm_smem_bytes(g.p.bn, g.p.stages);
}

cudaError_t tc_gemm_launch(const TcGemm &g, cudaStream_t s) {
    if (g.pair) return tc_gemm2_launch(g, s);
    cudaError_t e = gemm_smem_attr();
    if (e != cudaSuccess) return e;
    launch_k(k_gemm_tc, dim3(g.grid), dim3(192), g.smem, s, g.p);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ bounded-wait self-test
// One thread waits, through the same mbar_wait as every kernel of the
// library, on a barrier that nothing arrives at.  The wait gives up after
// limit_ns, sets ERR_TIMEOUT_SELFTEST in *err (and in *err2 when given) and
// the kernel returns: the failure path of an in-kernel wait, exercised
// without a fault or an endless loop.  No TMA or MMA is in flight.
__global__ void k_wait_selftest(unsigned *err, unsigned *err2, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    if (!mbar_wait(b, 0, err, ERR_TIMEOUT_SELFTEST, limit_ns) && err2) atomicOr(err2, ERR_TIMEOUT_SELFTEST);
}

cudaError_t wait_selftest_launch(unsigned *err, unsigned *err2, unsigned long long limit_ns, cudaStream_t s) {
    k_wait_selftest<<<1, 32, 0, s>>>(err, err2, limit_ns);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

int make_tmap_bf16(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                   uint32_t box_inner, uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return -1;
    if ((reinterpret_cast<uintptr_t>(base) & 15) || (row_bytes & 15)) return -2;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : -3;
}

// ------------------------------------------------------------------ fp32 SIMT path
__global__ void k_gemm_simt(const SimtGemmParams p, int total_f) {
    pdl_trigger();
    pdl_wait();
    const int f = blockIdx.x * 64 + (threadIdx.x & 63);
    const int r = blockIdx.y * 4 + (threadIdx.x >> 6);
    if (f >= total_f || r >= p.nrows) return;
    int seg = 0;
    while (seg + 1 < p.nseg && f >= p.seg_f0[seg + 1]) ++seg;
    const int fl = f - p.seg_f0[seg];
    const float *w = p.a[seg] + static_cast<long long>(fl) * p.K;
    const float *x = p.x + static_cast<long long>(r) * p.ldx;
    float acc = 0.f;
    for (int k = 0; k < p.K; ++k) acc = fmaf(x[k], w[k], acc);
    p.out[static_cast<long long>(r) * p.ldo + p.seg_col0[seg] + fl] = acc;
}

cudaError_t simt_gemm_launch(const SimtGemmParams &p, int total_f, cudaStream_t s) {
    dim3 grid((total_f + 63) / 64, (p.nrows + 3) / 4);
    launch_k(k_gemm_simt, dim3(grid), dim3(256), 0, s, p, total_f);
    return cudaGetLastError();
}

__global__ void k_reduce_splits(const float *part, int splits, long long stride, long long n, float *y) {
    pdl_trigger();
    pdl_wait();
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        float acc = part[i];
        for (int s = 1; s < splits; ++s) acc += part[s * stride + i];
        y[i] = acc;
    }
}

cudaError_t reduce_splits_launch(const float *part, int splits, long long stride, int rows, int cols, float *y,
                                 cudaStream_t s) {
    const long long n = static_cast<long long>(rows) * cols;
    int blocks = static_cast<int>((n + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    launch_k(k_reduce_splits, dim3(blocks), dim3(256), 0, s, part, splits, stride, n, y);
    return cudaGetLastError();
}

}  // namespace la
