// Mixed dense/factorized decode attention, split-K over pages (shared part).
//
// "PuzzleKV: Page-Wise Low-Rank Decomposition for KV Cache Compression",
// §3.3 ④: a factorized page contributes the page-local softmax state of
// eq. (4), s = (q R_K^T) L_K^T / sqrt(d), o = (exp(s - m) L_V) R_V, computed
// with the small factors contracted first (no page is ever rebuilt); a dense
// page contributes the same state from its stored rows; all states merge by
// the online-softmax reduction of eq. (5).
//
// One CTA handles one (sequence, KV head, page range).  Its pages are cut
// into units -- a factorized page, or a half (a quarter for INT4 stores) of a
// dense page, keys and values -- each of which fits one shared-memory slot.  The CTA's warps
// take its units round-robin and stream them through private slots with one
// or two bulk copies per unit (mbarrier transaction counts), each keeping its
// own running (m, l, o) for the G query heads of the KV head.  At the end the
// warps' states are merged in shared memory, every CTA's state goes to the
// workspace, and the last CTA of the (sequence, KV head) to finish merges the
// splits and writes the output.
//
// bf16 storage: the four contractions of eq. (4) run on tensor cores
// (mma.sync m16n8k16 / m16n8k8, fp32 accumulate).  The G <= 8 query heads fill
// rows 0-7 of the 16-row tile; intermediate operands (q R_K^T, the softmax
// weights, and their product with L_V) are split into a bf16 high part in rows
// 0-7 and a bf16 residual in rows 8-15, so a single mma carries about 16
// mantissa bits and the two row halves are summed afterwards.
// INT4 factor records [PuzzleKV §4.3]: the 4-bit codes enter fp16 products
// as exact integers and the scales are folded into the small operands
// (factored_unit_q4).  Keys stored before RoPE [PuzzleKV §4.1, Appendix D.3]:
// each page's keys are rebuilt and turned at their positions
// (factored_unit_rope, dense_unit_rope).
// fp32 storage: CUDA-core fp32 arithmetic throughout.
#pragma once
#include <cuda_fp16.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace pkv {

constexpr int NWC = 4;            // consumer warps of the fp32 kernel
constexpr int CTAS_PER_SM = 1;    // resident bf16 decode CTAs per SM
constexpr int NS_MAX = 16;        // shared-memory stages (bf16 kernel), chosen at launch
constexpr int MAX_CHUNK = MAX_CHUNK_PAGES;
constexpr float LOG2E = 1.4426950408889634f;

// 2^x with the PTX ex2.approx instruction (max relative error about 2^-22;
// ex2(-inf) = +0), for the softmax weights of the tensor-core path.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Shape of the tensor-core decode kernel: warps (NWC), shared-memory slots
// each warp streams its units through (SPW) and units per dense page (DU).
// Two slots per warp keep its copies ahead of its arithmetic.  A bf16 record
// of at most 18 KB (ranks fixed at compile time) leaves room for 6 warps x 2
// slots, which hide more of each warp's latency than 4; larger or
// runtime-rank records keep 4 x 2.  An INT4 record (4.5 KB) fits a
// quarter-page slot, so 8 warps fit in the same shared memory; the per-page
// code expansion is the part that needs them.  Keys stored before RoPE make a
// factorized page several times the arithmetic of a bf16 one (rebuilding and
// turning its keys), so that path also runs 8 warps, with one slot each.
// Pages of 32 or fewer tokens carry half the bytes (or less) for the same
// work per unit; with ranks fixed at compile time and a record of at most
// 12 KB they run 8 warps x 2 slots as well.  A unit keeps a multiple of 8
// rows (the period of the dense pages' swizzle).
template <bool Q4, int P, bool ROPE = false, int D = 128, int RKT = 0, int RVT = 0>
struct DecodeShape {
    static constexpr int REC = RKT > 0 && RVT > 0 ? 16 * (RKT + RVT) * (P + D) : 0;  // bf16 record bytes
    static constexpr bool WIDE = !Q4 && !ROPE && P <= 32 && REC > 0 && REC <= 12288;
    static constexpr int NWC = Q4 || ROPE || WIDE ? 8 : (REC > 0 && REC <= 18432 ? 6 : 4);
    // bf16 stores cut dense pages in halves: quarter pages would make the
    // slots no larger than a 15 KB record, but in back-to-back fused steps
    // they stretched each layer's split-merge tail (1.9 us more per layer)
    static constexpr int SPW = ROPE ? 1 : 2, DU = Q4 && P >= 32 ? 4 : 2;
    // 256 threads x 192 registers leave room for a 256-thread, 64-register
    // background conversion CTA on the same SM (at 209 the INT4 kernel locked
    // conversions out of the SMs it held); the pre-RoPE kernel needs all 255
    static constexpr int MAXREG = NWC == 8 && !ROPE ? 192 : 255;
};

// One shared-memory slot: a factor record or one unit of a dense page (P / DU
// K rows and P / DU V rows).
template <int P, int D, int DU>
__host__ __device__ inline size_t decode_unit_bytes(const Layout &y) {
    const size_t unit = (size_t)(P / DU) * D * 2 * 2;
    return ((y.rec_bytes > unit ? y.rec_bytes : unit) + 15) & ~(size_t)15;
}
// ... followed, when keys precede RoPE, by the (cos, sin) row of the unit's
// page start (D / 2 float2).
template <int P, int D, int DU, bool ROPE>
__host__ __device__ inline size_t decode_stage_bytes(const Layout &y) {
    return (decode_unit_bytes<P, D, DU>(y) + (ROPE ? (size_t)D * 4 : 0) + 127) & ~(size_t)127;
}

// Rows of the dense-page unit starting at token `first` (units of PU rows)
// that a length-T sequence holds.
__device__ __forceinline__ int unit_valid(int T, int first, int PU) {
    const int v = T - first;
    return v < 0 ? 0 : (v > PU ? PU : v);
}

// The CTA's shared state beside its slots.  The dense-unit table holds at
// most every dense page of a sequence (sink, window, the page being filled)
// cut into DU units; it is sized by DU because a bf16 decode CTA and a
// background factorization CTA fit one SM's shared memory together only with
// a few hundred bytes to spare.
template <int DU>
struct DecodeShared {
    uint64_t merge_bar;  // completion of the split-merge bulk copies
    int failed;
    int last;
    int n_pre, n_dense;  // dense units before the factorized stretch, and in all
    int slot_info[NS_MAX];  // per slot: page << 3 | dense << 2 | unit
    // each dense unit in page order, as rel << 3 | 4 | unit: rel is the page
    // itself for sink pages (before the factorized stretch) and the page minus
    // the stretch's end after it; both stay below MAX_DENSE_PAGES
    short dense_units[MAX_DENSE_PAGES * DU];
};


// Split hand-off, eq. (5).  `comb` holds the NW warp states of a CTA
// ([warp][g][m, l, pad, pad, o...], D + 4 floats per row, 16-byte aligned, m
// in log2 units).  cta_state merges them into the CTA's state for element e
// = (head g, columns 4j .. 4j+3): o (a float4) and (m, l).
template <int D, int NW>
__device__ __forceinline__ void cta_state(const float *comb, int e, float4 &acc, float2 &ml) {
    const int g = e / (D / 4), j = e % (D / 4);
    float mw[NW], M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        mw[w] = comb[(w * 8 + g) * (D + 4)];
        M = fmaxf(M, mw[w]);
    }
    float L = 0.f;
    acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const float *row = comb + (w * 8 + g) * (D + 4);
        const float c = mw[w] == -INFINITY ? 0.f : ex2_approx(mw[w] - M);
        const float4 v = reinterpret_cast<const float4 *>(row + 4)[j];
        L = fmaf(c, row[1], L);
        acc.x = fmaf(c, v.x, acc.x);
        acc.y = fmaf(c, v.y, acc.y);
        acc.z = fmaf(c, v.z, acc.z);
        acc.w = fmaf(c, v.w, acc.w);
    }
    ml = make_float2(M, L);
}

// The merge of eq. (5) over the ns split states of each of the G query heads
// of (b, h), written to `out`.  One warp per head, everything in registers:
// lane t holds the m of splits t, t + 32, ...; their largest value and the
// weights 2^(m_s - m) and normaliser come from warp shuffles, and each lane
// sums one float4 of o over the splits in split order (at D = 64, two lanes
// per float4, even and odd splits, added in a fixed order).  The sums are the
// same whichever CTA merges, so results are bitwise reproducible.  ld1(g, s,
// k) and ld4(g, s, k) read float k (or floats k .. k+3) of split s's row of
// head g.
template <int D, typename LD1, typename LD4>
__device__ __forceinline__ void merge_states(const DecodeParams &prm, int b_idx, int h, int ns, LD1 ld1, LD4 ld4) {
    constexpr int NJ = D / 4, NSUB = 32 / NJ, NI = MAX_SPLITS / 32;
    const int G = prm.y.G;
    const int nwarps = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = lane % NJ, sub = lane / NJ;
    for (int g = warp; g < G; g += nwarps) {
        float m[NI], c[NI];
        float M = -INFINITY;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int sp = lane + 32 * i;
            m[i] = sp < ns ? ld1(g, sp, 0) : -INFINITY;
            M = fmaxf(M, m[i]);
        }
        M = warp_max(M);
        float L = 0.f;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int sp = lane + 32 * i;
            c[i] = m[i] == -INFINITY ? 0.f : ex2_approx(m[i] - M);
            if (sp < ns) L = fmaf(c[i], ld1(g, sp, 1), L);
        }
        L = warp_sum(L);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int n_here = min(32, ns - 32 * i);
            for (int t2 = 0; NSUB * t2 < n_here; ++t2) {  // the same trip count in every lane
                const int t = NSUB * t2 + sub;
                const float cs = __shfl_sync(0xffffffffu, c[i], t < 32 ? t : 31);
                if (t < n_here) {
                    const float4 v = ld4(g, 32 * i + t, 4 + 4 * j);
                    acc.x = fmaf(cs, v.x, acc.x);
                    acc.y = fmaf(cs, v.y, acc.y);
                    acc.z = fmaf(cs, v.z, acc.z);
                    acc.w = fmaf(cs, v.w, acc.w);
                }
            }
        }
        if constexpr (NSUB == 2) {  // odd splits' partial sums into the even lanes'
            acc.x += __shfl_down_sync(0xffffffffu, acc.x, NJ);
            acc.y += __shfl_down_sync(0xffffffffu, acc.y, NJ);
            acc.z += __shfl_down_sync(0xffffffffu, acc.z, NJ);
            acc.w += __shfl_down_sync(0xffffffffu, acc.w, NJ);
        }
        const float il = 1.f / L;
        if (sub == 0)
            reinterpret_cast<float4 *>(prm.out + ((size_t)b_idx * prm.y.Hq + h * G + g) * D)[j] =
                make_float4(acc.x * il, acc.y * il, acc.z * il, acc.w * il);
    }
}

// Reads of split states staged in shared memory at `rows` (rows of S
// floats, head g's ns rows contiguous): plain loads, which the compiler may
// batch (the staging barrier's wait orders them after the copies).
struct StagedRows {
    const float *rows;
    int ns, S;
    __device__ __forceinline__ float one(int g, int sp, int k) const { return rows[(g * ns + sp) * S + k]; }
    __device__ __forceinline__ float4 four(int g, int sp, int k) const {
        return *reinterpret_cast<const float4 *>(rows + (g * ns + sp) * S + k);
    }
};

// The merge bulk copies of a staged hand-off were issued on `bar`: wait for
// them (bounded by the launch's limit) and agree over the CTA whether they
// landed.  If a wait gave up, the copies are given one more bounded wait so
// that none is still writing when the CTA exits, and false is returned: the
// caller then skips the merge, leaves `out` and the ticket as they are, and
// the status word (set by the wait) tells the host, whose status check also
// clears the tickets.
__device__ __forceinline__ bool merge_copies_landed(const DecodeParams &prm, uint64_t *bar) {
    const uint64_t lim = prm.wait_ns ? prm.wait_ns : WAIT_NS;
    const bool ok = __syncthreads_and(mbar_wait_bounded(bar, 0, prm.status, lim) ? 1 : 0) != 0;
    if (!ok && threadIdx.x == 0) mbar_wait_bounded(bar, 0, nullptr);
    return ok;
}

// Publishing hand-off: the CTA's state goes to its workspace row and becomes
// visible before the CTA takes its arrival ticket for (b, h) with one
// acquire-release atomic; the CTA that takes the last ticket therefore sees
// every state, merges them and writes `out`, then resets the ticket.  With
// `merge_bar` (an mbarrier of count 1 in its first phase) and room in
// `stage_buf` (16-byte aligned shared memory, `stage_cap` bytes, may overlap
// `comb`) the states arrive by one bulk copy per query head; otherwise they
// are read from global memory.  Returns true in the CTA that merged.
template <int D, int NW>
__device__ bool finish_split(const DecodeParams &prm, const float *comb, int b_idx, int b, int h, int split, int ns,
                             int *last, float *stage_buf = nullptr, size_t stage_cap = 0,
                             uint64_t *merge_bar = nullptr) {
    const Layout &y = prm.y;
    const int G = y.G, S = y.part_stride;
    int *arrivals = prm.tickets + y.ticket_index(b, h);
    // the CTA's state, one float4 of o per thread, written straight to its
    // workspace row; j = 0 also writes m and l
    for (int e = threadIdx.x; e < G * (D / 4); e += blockDim.x) {
        float4 acc;
        float2 ml;
        cta_state<D, NW>(comb, e, acc, ml);
        const int g = e / (D / 4), j = e % (D / 4);
        float *prow = prm.partials + y.partial_index(b, h * G + g, split) * S;
        reinterpret_cast<float4 *>(prow + 4)[j] = acc;
        if (j == 0) reinterpret_cast<float4 *>(prow)[0] = make_float4(ml.x, ml.y, 0.f, 0.f);
    }
    // rows of head g are contiguous: partial_index(b, h G + g, 0 .. ns-1)
    const bool staged = merge_bar != nullptr && stage_buf != nullptr && (size_t)G * ns * S * 4 <= stage_cap;
    __syncthreads();
    if (threadIdx.x == 0) {
        // release: the CTA's state (ordered before this by the barrier) is
        // visible before its ticket; acquire: the last CTA sees every state
        const bool is_last = atom_add_acq_rel_gpu(arrivals, 1) == ns - 1;
        *last = is_last;
        if (is_last && staged) {  // the states were written through the generic proxy
            fence_proxy_async_global();
            fence_proxy_async_shared();  // the warp states in stage_buf have been read
            const uint32_t bytes = (uint32_t)ns * S * 4;
            mbar_arrive_expect_tx(merge_bar, (uint32_t)G * bytes + (prm.inject == 2 ? 16u : 0u));
            for (int g = 0; g < G; ++g)
                bulk_g2s(stage_buf + (size_t)g * ns * S, prm.partials + y.partial_index(b, h * G + g, 0) * S,
                         bytes, merge_bar);
        }
    }
    __syncthreads();
    if (!*last) return false;
    if (staged) {
        if (!merge_copies_landed(prm, merge_bar)) return false;
        const StagedRows rows{stage_buf, ns, S};
        merge_states<D>(prm, b_idx, h, ns, [&](int g, int sp, int k) { return rows.one(g, sp, k); },
                        [&](int g, int sp, int k) { return rows.four(g, sp, k); });
    } else {
        const float *rows = prm.partials + y.partial_index(b, h * G, 0) * S;  // head g at + g MAX_SPLITS S
        merge_states<D>(
            prm, b_idx, h, ns,
            [&](int g, int sp, int k) -> float { return __ldcg(rows + ((size_t)g * MAX_SPLITS + sp) * S + k); },
            [&](int g, int sp, int k) -> float4 {
                return __ldcg(reinterpret_cast<const float4 *>(rows + ((size_t)g * MAX_SPLITS + sp) * S + k));
            });
    }
    if (threadIdx.x == 0) arrivals[0] = 0;
    return true;
}

// ---------------------------------------------------------------- bf16 tensor-core path

template <int P, int D>
struct WarpState {
    uint32_t qf[D / 16][2];  // A fragments of q (rows 0-7), k-steps of 16
    uint32_t qh[D / 16][2];  // the same in fp16 (INT4 stores)
    float o[D / 8][4];       // rows 0-7: high-part products, rows 8-15: residual products
    float m, l;              // running max (log2 units) and this thread's partial sum
};

template <int P, int D>
__device__ __forceinline__ void online_softmax(WarpState<P, D> &w, float (*sv)[2], int ntile) {
    float mx = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < P / 8; ++nt)
        if (nt < ntile) mx = fmaxf(mx, fmaxf(sv[nt][0], sv[nt][1]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(w.m, mx);
    float ls = 0.f;
#pragma unroll
    for (int nt = 0; nt < P / 8; ++nt) {
        if (nt < ntile) {
            sv[nt][0] = ex2_approx(sv[nt][0] - m_new);
            sv[nt][1] = ex2_approx(sv[nt][1] - m_new);
            ls += sv[nt][0] + sv[nt][1];
        }
    }
    // the running max of a row rarely moves once a few pages are in: rescale
    // the accumulators only when it moved for some row of the warp
    if (!__all_sync(0xffffffffu, m_new == w.m)) {
        const float alpha = ex2_approx(w.m - m_new);
        w.l *= alpha;
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
            w.o[nt][0] *= alpha;
            w.o[nt][1] *= alpha;
            w.o[nt][2] *= alpha;
            w.o[nt][3] *= alpha;
        }
    }
    w.l += ls;
    w.m = m_new;
}

// o += A (16 x rk, split rows) * B where B^T rows live in `rows_base`
// (row = output column n, chunks = k in 8s), rk = 8 * nkt.
// A fragments: av[j] = per 8-wide k tile j, (hi, lo) packed pairs.
template <int NT_OUT, int MAXRT>
__device__ __forceinline__ void mma_rows(float (*acc)[4], const uint32_t (*ahi)[1], const uint32_t (*alo)[1],
                                         int nkt, uint32_t rows_base, int pitch, int lane) {
    const int ks_full = nkt >> 1;
#pragma unroll
    for (int ks = 0; ks < MAXRT / 2; ++ks) {
        if (ks < ks_full) {
            uint32_t a0 = ahi[2 * ks][0], a1 = alo[2 * ks][0], a2 = ahi[2 * ks + 1][0], a3 = alo[2 * ks + 1][0];
#pragma unroll
            for (int nt = 0; nt < NT_OUT; nt += 2) {
                int m = lane >> 3;
                int row = 8 * (nt + (m >> 1)) + (lane & 7);
                int ch = 2 * ks + (m & 1);
                uint32_t r0, r1, r2, r3;
                ldsm_x4(rows_base + swz_offset(row, ch * 16, pitch), r0, r1, r2, r3);
                Ops<false>::mma(acc[nt], a0, a1, a2, a3, r0, r1);
                Ops<false>::mma(acc[nt + 1], a0, a1, a2, a3, r2, r3);
            }
        }
    }
    if (nkt & 1) {
        const int j = nkt - 1;
        uint32_t a0 = 0u, a1 = 0u;
#pragma unroll
        for (int jj = 0; jj < MAXRT; ++jj)  // static register indices only
            if (jj == j) {
                a0 = ahi[jj][0];
                a1 = alo[jj][0];
            }
#pragma unroll
        for (int nt = 0; nt < NT_OUT; nt += 4) {
            int m = lane >> 3;
            int row = 8 * (nt + m) + (lane & 7);
            uint32_t r0, r1, r2, r3;
            if (NT_OUT - nt >= 4) {
                ldsm_x4(rows_base + swz_offset(row, j * 16, pitch), r0, r1, r2, r3);
                Ops<false>::mma8(acc[nt], a0, a1, r0);
                Ops<false>::mma8(acc[nt + 1], a0, a1, r1);
                Ops<false>::mma8(acc[nt + 2], a0, a1, r2);
                Ops<false>::mma8(acc[nt + 3], a0, a1, r3);
            } else {
                int row2 = 8 * (nt + (m & 1)) + (lane & 7);
                ldsm_x2(rows_base + swz_offset(row2, j * 16, pitch), r0, r1);
                Ops<false>::mma8(acc[nt], a0, a1, r0);
                Ops<false>::mma8(acc[nt + 1], a0, a1, r1);
            }
        }
    }
}

template <int P, int D, int RKT, int RVT>
__device__ __forceinline__ void factored_values(WarpState<P, D> &w, const float (*s)[4], uint32_t st,
                                                const Layout &y, int lane, float scale_log2);
template <int P, int D, int RKT, int RVT>
__device__ __forceinline__ void factored_values_sv(WarpState<P, D> &w, float (*sv)[2], uint32_t st,
                                                   const Layout &y, int lane);

// RKT / RVT: rank tiles (ranks / 8) when fixed at compile time, 0 = read
// from the layout (up to 8 tiles).
template <int P, int D, int RKT, int RVT>
__device__ __forceinline__ void factored_unit(WarpState<P, D> &w, uint32_t st, const Layout &y, int lane,
                                              float scale_log2) {
    using O = Ops<false>;
    const uint32_t(&qa)[D / 16][2] = w.qf;
    constexpr int MAXK = RKT ? RKT : 8;
    const int nkt = RKT ? RKT : (y.rkp >> 3);
    const uint32_t LK = st, RK = st + (uint32_t)P * nkt * 16;
    // 1. t = q R_K^T  (16 x rkp; rows 8-15 stay zero), as two accumulator
    // chains of half the head dim each, so the products of a rank tile do not
    // wait on one another D / 16 deep
    float t[MAXK][4], t2[MAXK][4];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
        t[j][0] = t[j][1] = t[j][2] = t[j][3] = 0.f;
        t2[j][0] = t2[j][1] = t2[j][2] = t2[j][3] = 0.f;
        if (j < nkt) {
#pragma unroll
            for (int k2 = 0; k2 < D / 32; ++k2) {
                int row = 8 * j + (lane & 7), ch = 4 * k2 + (lane >> 3);
                uint32_t r0, r1, r2, r3;
                ldsm_x4(RK + swz_offset(row, ch * 16, D * 2), r0, r1, r2, r3);
                O::mma(t[j], qa[2 * k2][0], 0u, qa[2 * k2][1], 0u, r0, r1);
                O::mma(t2[j], qa[2 * k2 + 1][0], 0u, qa[2 * k2 + 1][1], 0u, r2, r3);
            }
            t[j][0] += t2[j][0];
            t[j][1] += t2[j][1];
            t[j][2] += t2[j][2];
            t[j][3] += t2[j][3];
        }
    }
    // 2. s = t L_K^T  (16 x P), t split into high (rows 0-7) and residual (rows 8-15)
    uint32_t thi[MAXK][1], tlo[MAXK][1];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) O::split(t[j][0], t[j][1], thi[j][0], tlo[j][0]);
    float s[P / 8][4];
#pragma unroll
    for (int nt = 0; nt < P / 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    mma_rows<P / 8, MAXK>(s, thi, tlo, nkt, LK, nkt * 16, lane);
    factored_values<P, D, RKT, RVT>(w, s, st, y, lane, scale_log2);
}

// Stages 3-5 of a factorized page from its raw scores s (rows 0-7 and 8-15
// of each tile summed): the page-local softmax state merged into the running
// one, u = p L_V and o += u R_V, from the bf16 record at `st`.
template <int P, int D, int RKT, int RVT>
__device__ __forceinline__ void factored_values(WarpState<P, D> &w, const float (*s)[4], uint32_t st,
                                                const Layout &y, int lane, float scale_log2) {
    float sv[P / 8][2];
#pragma unroll
    for (int nt = 0; nt < P / 8; ++nt) {
        sv[nt][0] = (s[nt][0] + s[nt][2]) * scale_log2;
        sv[nt][1] = (s[nt][1] + s[nt][3]) * scale_log2;
    }
    factored_values_sv<P, D, RKT, RVT>(w, sv, st, y, lane);
}

// The same from the scaled scores sv (log2 units; head g, tokens 8 nt + 2c, +1).
template <int P, int D, int RKT, int RVT>
__device__ __forceinline__ void factored_values_sv(WarpState<P, D> &w, float (*sv)[2], uint32_t st,
                                                   const Layout &y, int lane) {
    using O = Ops<false>;
    constexpr int MAXV = RVT ? RVT : 8;
    const int nkt = RKT ? RKT : (y.rkp >> 3), nvt = RVT ? RVT : (y.rvp >> 3);
    const uint32_t off_RK = (uint32_t)P * nkt * 16, off_LV = off_RK + (uint32_t)nkt * 8 * D * 2;
    const uint32_t off_RV = off_LV + (uint32_t)nvt * 8 * P * 2;
    const uint32_t LV = st + off_LV, RV = st + off_RV;
    // 3. page-local softmax state merged into the running one
    online_softmax<P, D>(w, sv, P / 8);
    // 4. u = p L_V  (16 x rvp): A = p split by token k-steps, B = LVt rows (rank)
    float u[MAXV][4];
#pragma unroll
    for (int j = 0; j < MAXV; ++j) u[j][0] = u[j][1] = u[j][2] = u[j][3] = 0.f;
#pragma unroll
    for (int kt = 0; kt < P / 16; ++kt) {
        uint32_t h0, l0, h1, l1;
        O::split(sv[2 * kt][0], sv[2 * kt][1], h0, l0);
        O::split(sv[2 * kt + 1][0], sv[2 * kt + 1][1], h1, l1);
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
            if (j < nvt) {
                int row = 8 * j + (lane & 7), ch = 2 * kt + ((lane >> 3) & 1);
                uint32_t r0, r1;
                ldsm_x2(LV + swz_offset(row, ch * 16, P * 2), r0, r1);
                O::mma(u[j], h0, l0, h1, l1, r0, r1);
            }
        }
    }
    // 5. o += u R_V: A = u split by rank tiles, B = RVt rows (head dim)
    uint32_t uhi[MAXV][1], ulo[MAXV][1];
#pragma unroll
    for (int j = 0; j < MAXV; ++j) O::split(u[j][0] + u[j][2], u[j][1] + u[j][3], uhi[j][0], ulo[j][0]);
    mma_rows<D / 8, MAXV>(w.o, uhi, ulo, nvt, RV, nvt * 16, lane);
}

template <int P, int D, int PH>
__device__ __forceinline__ void dense_values(WarpState<P, D> &w, const float (*s)[4], uint32_t V, int valid,
                                             int lane, float scale_log2);

template <int P, int D, int PH>  // PH: tokens in the unit (a multiple of 8, at most P / 2)
__device__ __forceinline__ void dense_unit(WarpState<P, D> &w, uint32_t st, int valid, int lane,
                                           float scale_log2) {
    constexpr int NT = PH / 8;
    const uint32_t K = st, V = st + PH * D * 2;
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int k2 = 0; k2 < D / 32; ++k2) {
            int row = 8 * nt + (lane & 7), ch = 4 * k2 + (lane >> 3);
            uint32_t r0, r1, r2, r3;
            ldsm_x4(K + swz_offset(row, ch * 16, D * 2), r0, r1, r2, r3);
            mma16816(s[nt], w.qf[2 * k2][0], 0u, w.qf[2 * k2][1], 0u, r0, r1);
            mma16816(s[nt], w.qf[2 * k2 + 1][0], 0u, w.qf[2 * k2 + 1][1], 0u, r2, r3);
        }
    }
    dense_values<P, D, PH>(w, s, V, valid, lane, scale_log2);
}

// The rest of a dense unit from its raw scores s (rows 0-7 and 8-15 of each
// tile summed): rows at or past `valid` masked, the softmax state merged into
// the running one, o += p V from the unit's V rows at `V`.
template <int P, int D, int PH>
__device__ __forceinline__ void dense_values(WarpState<P, D> &w, const float (*s)[4], uint32_t V, int valid,
                                             int lane, float scale_log2) {
    constexpr int NT = PH / 8;
    float sv[P / 8][2];
    const int c2 = 2 * (lane & 3);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        int tok = 8 * nt + c2;
        sv[nt][0] = tok < valid ? (s[nt][0] + s[nt][2]) * scale_log2 : -INFINITY;
        sv[nt][1] = tok + 1 < valid ? (s[nt][1] + s[nt][3]) * scale_log2 : -INFINITY;
    }
    online_softmax<P, D>(w, sv, NT);
    // o += p V: V rows are tokens (k); transposed ldmatrix gives the col-major B
    if constexpr (PH >= 16) {
#pragma unroll
        for (int kt = 0; kt < PH / 16; ++kt) {
            uint32_t h0, l0, h1, l1;
            split_bf16(sv[2 * kt][0], sv[2 * kt][1], h0, l0);
            split_bf16(sv[2 * kt + 1][0], sv[2 * kt + 1][1], h1, l1);
#pragma unroll
            for (int nt = 0; nt < D / 8; nt += 2) {
                int m = lane >> 3;
                int row = 16 * kt + 8 * (m & 1) + (lane & 7);
                int ch = nt + (m >> 1);
                uint32_t r0, r1, r2, r3;
                ldsm_x4_t(V + swz_offset(row, ch * 16, D * 2), r0, r1, r2, r3);
                mma16816(w.o[nt], h0, l0, h1, l1, r0, r1);
                mma16816(w.o[nt + 1], h0, l0, h1, l1, r2, r3);
            }
        }
    } else {  // 8-token unit: one k8 step
        uint32_t h0, l0;
        split_bf16(sv[0][0], sv[0][1], h0, l0);
#pragma unroll
        for (int nt = 0; nt < D / 8; nt += 4) {
            int m = lane >> 3;
            int row = lane & 7;
            uint32_t r0, r1, r2, r3;
            ldsm_x4_t(V + swz_offset(row, (nt + m) * 16, D * 2), r0, r1, r2, r3);
            mma1688(w.o[nt], h0, l0, r0);
            mma1688(w.o[nt + 1], h0, l0, r1);
            mma1688(w.o[nt + 2], h0, l0, r2);
            mma1688(w.o[nt + 3], h0, l0, r3);
        }
    }
}


// One factorized page from an INT4 record [PuzzleKV §4.3] in shared memory.
// The codes enter the fp16 tensor-core products as exact small integers
// (layout.h: tensor-core operand order) and every scale is folded into the
// small operand beside it:
//   t = (q o s_RK) C_RK^T,  s = (t o s_LK) C_LK^T,
//   u = (p o s_LV) C_LV,    o += (u C_RV) o s_RV
// (o: elementwise; C: the code matrices), each scaled operand carried as an
// fp16 high part (rows 0-7) and residual (rows 8-15) of its m16 tile, so the
// products keep about 22 bits.  RKT / RVT: rank tiles when fixed at compile
// time, 0 = from the layout (INT4 ranks are at most P / 2).
template <int P, int D, int RKT, int RVT>
__device__ __forceinline__ void factored_unit_q4(WarpState<P, D> &w, const unsigned char *rec, const Layout &y,
                                                 int lane, float scale_log2) {
    using O = Ops<true>;
    constexpr int MAXK = RKT ? RKT : P / 16, MAXV = RVT ? RVT : P / 16;
    const int nkt = RKT ? RKT : (y.rkp >> 3), nvt = RVT ? RVT : (y.rvp >> 3);
    const int c = lane & 3;
    // word wd of this lane's part of a stream: slab wd / 2, word wd % 2
    const uint32_t *ks_ = reinterpret_cast<const uint32_t *>(rec) + 2 * lane;
    const uint32_t *vs_ = reinterpret_cast<const uint32_t *>(rec + y.q_off_V) + 2 * lane;
    auto breg = [](const uint32_t *st, int m) -> uint32_t {
        const int wd = m >> 2;
        return q4_reg(st[(wd >> 1) * 64 + (wd & 1)], m & 3);
    };
    // 1. t = (q o s_RK) C_RK^T: A = q o s_RK over the head dim (k-step ks holds
    // columns 16 ks + 2c, +1 and 16 ks + 8 + 2c, +1: one uint2 of lane c's
    // scales, the four lanes' uint2 contiguous)
    const uint2 *sRK = reinterpret_cast<const uint2 *>(rec + y.q_off_sRK) + c;
    float t[MAXK][4];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) t[j][0] = t[j][1] = t[j][2] = t[j][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint2 sc = sRK[4 * ks];
        uint32_t h0, l0, h1, l1;
        mul_split_f16(w.qh[ks][0], sc.x, h0, l0);
        mul_split_f16(w.qh[ks][1], sc.y, h1, l1);
#pragma unroll
        for (int j = 0; j < MAXK; ++j)
            if (j < nkt) {
                const int m = 2 * (ks * nkt + j);
                O::mma(t[j], h0, l0, h1, l1, breg(ks_, m), breg(ks_, m + 1));
            }
    }
    // 2. s = (t o s_LK) C_LK^T: this lane holds rank columns 8j + 2c, +1
    const __half2 *sLK = reinterpret_cast<const __half2 *>(rec + y.q_off_sLK) + c * nkt;
    uint32_t thi[MAXK][1], tlo[MAXK][1];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
        thi[j][0] = tlo[j][0] = 0u;
        if (j < nkt) {
            const float2 sc = __half22float2(sLK[j]);
            O::split((t[j][0] + t[j][2]) * sc.x, (t[j][1] + t[j][3]) * sc.y, thi[j][0], tlo[j][0]);
        }
    }
    float s[P / 8][4];
#pragma unroll
    for (int nt = 0; nt < P / 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    {
        const int m0 = nkt * (D / 8), kf = nkt >> 1;  // L_K's first register; full k-steps
#pragma unroll
        for (int ks = 0; ks < MAXK / 2; ++ks)
            if (ks < kf) {
#pragma unroll
                for (int nt = 0; nt < P / 8; ++nt) {
                    const int m = m0 + ks * (P / 4) + 2 * nt;
                    O::mma(s[nt], thi[2 * ks][0], tlo[2 * ks][0], thi[2 * ks + 1][0], tlo[2 * ks + 1][0],
                           breg(ks_, m), breg(ks_, m + 1));
                }
            }
        if (nkt & 1) {
            uint32_t a0 = 0u, a1 = 0u;
#pragma unroll
            for (int jj = 0; jj < MAXK; ++jj)  // static register indices only
                if (jj == nkt - 1) {
                    a0 = thi[jj][0];
                    a1 = tlo[jj][0];
                }
#pragma unroll
            for (int nt = 0; nt < P / 8; ++nt) O::mma8(s[nt], a0, a1, breg(ks_, m0 + kf * (P / 4) + nt));
        }
    }
    float sv[P / 8][2];
#pragma unroll
    for (int nt = 0; nt < P / 8; ++nt) {
        sv[nt][0] = (s[nt][0] + s[nt][2]) * scale_log2;
        sv[nt][1] = (s[nt][1] + s[nt][3]) * scale_log2;
    }
    // 3. page-local softmax state merged into the running one
    online_softmax<P, D>(w, sv, P / 8);
    // 4. u = (p o s_LV) C_LV: this lane holds tokens 8nt + 2c, +1
    const __half2 *sLV = reinterpret_cast<const __half2 *>(rec + y.q_off_sLV) + c * (P / 8);
    float u[MAXV][4];
#pragma unroll
    for (int j = 0; j < MAXV; ++j) u[j][0] = u[j][1] = u[j][2] = u[j][3] = 0.f;
#pragma unroll
    for (int kt = 0; kt < P / 16; ++kt) {
        const float2 s0 = __half22float2(sLV[2 * kt]), s1 = __half22float2(sLV[2 * kt + 1]);
        uint32_t h0, l0, h1, l1;
        O::split(sv[2 * kt][0] * s0.x, sv[2 * kt][1] * s0.y, h0, l0);
        O::split(sv[2 * kt + 1][0] * s1.x, sv[2 * kt + 1][1] * s1.y, h1, l1);
#pragma unroll
        for (int j = 0; j < MAXV; ++j)
            if (j < nvt) {
                const int m = 2 * (kt * nvt + j);
                O::mma(u[j], h0, l0, h1, l1, breg(vs_, m), breg(vs_, m + 1));
            }
    }
    // 5. o += (u C_RV) o s_RV, four head-dim tiles at a time
    uint32_t uhi[MAXV][1], ulo[MAXV][1];
#pragma unroll
    for (int j = 0; j < MAXV; ++j) O::split(u[j][0] + u[j][2], u[j][1] + u[j][3], uhi[j][0], ulo[j][0]);
    // head-dim tile nt's scales for lane c (columns 8 nt + 2c, +1): half2
    // (nt / 2) 8 + 2c + nt % 2 in k-step order
    const __half2 *sRV = reinterpret_cast<const __half2 *>(rec + y.q_off_sRV) + 2 * c;
    const int m0 = nvt * (P / 8), kf = nvt >> 1;  // R_V's first register; full k-steps
    uint32_t a0 = 0u, a1 = 0u;                    // the 8-wide last k-step's operand
#pragma unroll
    for (int jj = 0; jj < MAXV; ++jj)
        if (jj == nvt - 1) {
            a0 = uhi[jj][0];
            a1 = ulo[jj][0];
        }
#pragma unroll
    for (int n0 = 0; n0 < D / 8; n0 += 4) {
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < MAXV / 2; ++ks)
            if (ks < kf) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int m = m0 + ks * (D / 4) + 2 * (n0 + i);
                    O::mma(acc[i], uhi[2 * ks][0], ulo[2 * ks][0], uhi[2 * ks + 1][0], ulo[2 * ks + 1][0],
                           breg(vs_, m), breg(vs_, m + 1));
                }
            }
        if (nvt & 1) {
#pragma unroll
            for (int i = 0; i < 4; ++i) O::mma8(acc[i], a0, a1, breg(vs_, m0 + kf * (D / 4) + n0 + i));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 sc = __half22float2(sRV[((n0 + i) >> 1) * 8 + ((n0 + i) & 1)]);
            w.o[n0 + i][0] = fmaf(acc[i][0], sc.x, w.o[n0 + i][0]);
            w.o[n0 + i][1] = fmaf(acc[i][1], sc.y, w.o[n0 + i][1]);
            w.o[n0 + i][2] = fmaf(acc[i][2], sc.x, w.o[n0 + i][2]);
            w.o[n0 + i][3] = fmaf(acc[i][3], sc.y, w.o[n0 + i][3]);
        }
    }
}

// ---------------------------------------------------------------- keys stored before RoPE
//
// Keys given before RoPE [PuzzleKV §4.1, Appendix D.3] are factorized as
// they are and turned at attention: the key at absolute position n meets the
// (already rotated) query as q . R(n) k.  A page starting at n0 splits the
// rotation as R(n0 + delta) = R(n0) R(delta), so each unit turns the query
// back once by the page start, q_p = R(n0)^T q, and each key only by its
// offset delta < P inside the page.  R pairs dims (i, i + D/2) with angle
// n theta_i; `base` holds (cos, sin) of n0 theta_i (D/2 entries, copied with
// the unit) and `delta` the (cos, sin) of delta theta_i ([P][D/2], shared).

// q_p as fp16 high parts (A rows 0-7) and residuals (rows 8-15): this lane's
// q elements (head g, dims 16 ks + 8 b + 2c, +1) pair dim i < D/2 (k-step
// ks < D/32) with i + D/2 (k-step ks + D/32, same b and lane position).
template <int D>
__device__ __forceinline__ void rope_query(const uint32_t (&qf)[D / 16][2], const float2 *base, int lane,
                                           uint32_t (&qhi)[D / 16][2], uint32_t (&qlo)[D / 16][2]) {
    const int c2 = 2 * (lane & 3);
#pragma unroll
    for (int ks = 0; ks < D / 32; ++ks)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int i = 16 * ks + 8 * b + c2;
            const float4 cs = *reinterpret_cast<const float4 *>(base + i);  // (cos, sin) of dims i, i + 1
            const float x0 = bf16_lo_to_f32(qf[ks][b]), x1 = bf16_hi_to_f32(qf[ks][b]);
            const float y0 = bf16_lo_to_f32(qf[ks + D / 32][b]), y1 = bf16_hi_to_f32(qf[ks + D / 32][b]);
            // R^T turns (x, y) by minus the angle: x' = x c + y s, y' = y c - x s
            split_f16(fmaf(x0, cs.x, y0 * cs.y), fmaf(x1, cs.z, y1 * cs.w), qhi[ks][b], qlo[ks][b]);
            split_f16(fmaf(y0, cs.x, -x0 * cs.y), fmaf(y1, cs.z, -x1 * cs.w), qhi[ks + D / 32][b],
                      qlo[ks + D / 32][b]);
        }
}

// Turn the pair (x, y) = (k_i, k_{i + D/2}) by the angle whose (cos, sin) is cs.
__device__ __forceinline__ void rope_turn(float &x, float &y, float c, float s) {
    const float xr = fmaf(x, c, -y * s), yr = fmaf(y, c, x * s);
    x = xr;
    y = yr;
}

// acc (rows g: high parts of q_p, rows g + 8: residuals) += q_p . k over one
// k-step (q_p fragments qh0, ql0 for dims 2c, +1 and qh1, ql1 for 8 + 2c, +1
// of the step) for the 8 tokens of an n-tile, whose rotated keys this lane
// holds as fp32 pairs (x0, x1) (dims 2c, +1 of the step, token g) and
// (y0, y1) (dims 8 + 2c, +1); each key pair goes in as an fp16 high part and a
// residual (two products).
__device__ __forceinline__ void rope_score_step(float *acc, uint32_t qh0, uint32_t ql0, uint32_t qh1, uint32_t ql1,
                                                float x0, float x1, float y0, float y1) {
    uint32_t h0, l0, h1, l1;
    split_f16(x0, x1, h0, l0);
    split_f16(y0, y1, h1, l1);
    mma16816_f16(acc, qh0, ql0, qh1, ql1, h0, h1);
    mma16816_f16(acc, qh0, ql0, qh1, ql1, l0, l1);
}

// A factorized page of a store whose keys precede RoPE: K = L_K R_K rebuilt
// 16 tokens at a time on the tensor cores (bf16 x bf16 products are exact in
// fp32), each row turned by its offset, scored against q_p; then the value
// stages as for any factorized page.
template <int P, int D, int RKT, int RVT>
__device__ __forceinline__ void factored_unit_rope(WarpState<P, D> &w, uint32_t st, const float2 *base,
                                                   const float2 *delta, const Layout &y, int lane,
                                                   float scale_log2) {
    constexpr int MAXK = RKT ? RKT : P / 8;
    const int nkt = RKT ? RKT : (y.rkp >> 3);
    const uint32_t LK = st, RK = st + (uint32_t)P * nkt * 16;
    const int g = lane >> 2, c2 = 2 * (lane & 3), m = lane >> 3;
    uint32_t qhi[D / 16][2], qlo[D / 16][2];
    rope_query<D>(w.qf, base, lane, qhi, qlo);
    float sv[P / 8][2];
#pragma unroll
    for (int mt = 0; mt < P / 16; ++mt) {
        // kh[nt]: tokens 16 mt + g (elements 0, 1) and + 8 (2, 3), dims 8 nt + 2c, +1
        float kh[D / 8][4];
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) kh[nt][0] = kh[nt][1] = kh[nt][2] = kh[nt][3] = 0.f;
        const int arow = 16 * mt + 8 * (m & 1) + (lane & 7);
#pragma unroll
        for (int kr = 0; kr < MAXK / 2; ++kr)
            if (kr < (nkt >> 1)) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(LK + swz_offset(arow, (2 * kr + (m >> 1)) * 16, nkt * 16), a0, a1, a2, a3);
#pragma unroll
                for (int nt = 0; nt < D / 8; nt += 2) {
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4_t(RK + swz_offset(16 * kr + 8 * (m & 1) + (lane & 7), (nt + (m >> 1)) * 16, D * 2), r0,
                              r1, r2, r3);
                    mma16816(kh[nt], a0, a1, a2, a3, r0, r1);
                    mma16816(kh[nt + 1], a0, a1, a2, a3, r2, r3);
                }
            }
        if (nkt & 1) {  // an 8-wide last rank step
            const int kr = nkt - 1;
            uint32_t a0, a1;
            ldsm_x2(LK + swz_offset(arow, kr * 16, nkt * 16), a0, a1);
#pragma unroll
            for (int nt = 0; nt < D / 8; nt += 4) {
                uint32_t r0, r1, r2, r3;
                ldsm_x4_t(RK + swz_offset(8 * kr + (lane & 7), (nt + m) * 16, D * 2), r0, r1, r2, r3);
                mma1688(kh[nt], a0, a1, r0);
                mma1688(kh[nt + 1], a0, a1, r1);
                mma1688(kh[nt + 2], a0, a1, r2);
                mma1688(kh[nt + 3], a0, a1, r3);
            }
        }
        // turn each row by its offset (dims 8 nt + 2c + e, nt < D/16, pair with
        // nt + D/16) and score it: k-steps ks and ks + D/32 share their turns
        const float2 *d0 = delta + (16 * mt + g) * (D / 2), *d1 = d0 + 8 * (D / 2);
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};  // tokens 16 mt + 0..7, + 8..15
#pragma unroll
        for (int ks = 0; ks < D / 32; ++ks) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int nt = 2 * ks + b;
                const float4 ca = *reinterpret_cast<const float4 *>(d0 + 8 * nt + c2);
                const float4 cb = *reinterpret_cast<const float4 *>(d1 + 8 * nt + c2);
                rope_turn(kh[nt][0], kh[nt + D / 16][0], ca.x, ca.y);
                rope_turn(kh[nt][1], kh[nt + D / 16][1], ca.z, ca.w);
                rope_turn(kh[nt][2], kh[nt + D / 16][2], cb.x, cb.y);
                rope_turn(kh[nt][3], kh[nt + D / 16][3], cb.z, cb.w);
            }
            const int lo = 2 * ks, hi = 2 * ks + D / 16, kq = ks + D / 32;
            rope_score_step(sa, qhi[ks][0], qlo[ks][0], qhi[ks][1], qlo[ks][1], kh[lo][0], kh[lo][1], kh[lo + 1][0],
                            kh[lo + 1][1]);
            rope_score_step(sb, qhi[ks][0], qlo[ks][0], qhi[ks][1], qlo[ks][1], kh[lo][2], kh[lo][3], kh[lo + 1][2],
                            kh[lo + 1][3]);
            rope_score_step(sa, qhi[kq][0], qlo[kq][0], qhi[kq][1], qlo[kq][1], kh[hi][0], kh[hi][1], kh[hi + 1][0],
                            kh[hi + 1][1]);
            rope_score_step(sb, qhi[kq][0], qlo[kq][0], qhi[kq][1], qlo[kq][1], kh[hi][2], kh[hi][3], kh[hi + 1][2],
                            kh[hi + 1][3]);
        }
        sv[2 * mt][0] = (sa[0] + sa[2]) * scale_log2;
        sv[2 * mt][1] = (sa[1] + sa[3]) * scale_log2;
        sv[2 * mt + 1][0] = (sb[0] + sb[2]) * scale_log2;
        sv[2 * mt + 1][1] = (sb[1] + sb[3]) * scale_log2;
    }
    factored_values_sv<P, D, RKT, RVT>(w, sv, st, y, lane);
}

// A dense unit (PH rows from page offset `off`) of a store whose keys precede
// RoPE: each key row is turned by its offset inside the page and scored
// against q_p, then the value stages as for any dense unit.
template <int P, int D, int PH>
__device__ __forceinline__ void dense_unit_rope(WarpState<P, D> &w, uint32_t st, const float2 *base,
                                                const float2 *delta, int off, int valid, int lane,
                                                float scale_log2) {
    constexpr int NT = PH / 8;
    const uint32_t K = st, V = st + PH * D * 2;
    const int g = lane >> 2, c2 = 2 * (lane & 3);
    uint32_t qhi[D / 16][2], qlo[D / 16][2];
    rope_query<D>(w.qf, base, lane, qhi, qlo);
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
        uint32_t kr[D / 16][2];  // token 8 nt + g, dims 16 ks + 8 b + 2c, +1 (bf16 pairs)
#pragma unroll
        for (int k2 = 0; k2 < D / 32; ++k2) {
            int row = 8 * nt + (lane & 7), ch = 4 * k2 + (lane >> 3);
            ldsm_x4(K + swz_offset(row, ch * 16, D * 2), kr[2 * k2][0], kr[2 * k2][1], kr[2 * k2 + 1][0],
                    kr[2 * k2 + 1][1]);
        }
        const float2 *dr = delta + (off + 8 * nt + g) * (D / 2);
#pragma unroll
        for (int ks = 0; ks < D / 32; ++ks) {  // k-steps ks and ks + D/32 share their turns
            float x[2][2], yv[2][2];
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const float4 cs = *reinterpret_cast<const float4 *>(dr + 16 * ks + 8 * b + c2);
                x[b][0] = bf16_lo_to_f32(kr[ks][b]);
                x[b][1] = bf16_hi_to_f32(kr[ks][b]);
                yv[b][0] = bf16_lo_to_f32(kr[ks + D / 32][b]);
                yv[b][1] = bf16_hi_to_f32(kr[ks + D / 32][b]);
                rope_turn(x[b][0], yv[b][0], cs.x, cs.y);
                rope_turn(x[b][1], yv[b][1], cs.z, cs.w);
            }
            const int kq = ks + D / 32;
            rope_score_step(s[nt], qhi[ks][0], qlo[ks][0], qhi[ks][1], qlo[ks][1], x[0][0], x[0][1], x[1][0],
                            x[1][1]);
            rope_score_step(s[nt], qhi[kq][0], qlo[kq][0], qhi[kq][1], qlo[kq][1], yv[0][0], yv[0][1], yv[1][0],
                            yv[1][1]);
        }
    }
    dense_values<P, D, PH>(w, s, V, valid, lane, scale_log2);
}

// Fused append: page-table record of the call's new token (position T - 1),
// written by one thread per sequence.  Nothing in this launch reads it.
__device__ inline void append_page_table(const DecodeParams &prm, int b_idx, int b, int T) {
    const Layout &y = prm.y;
    const int pos = T - 1, pg = pos / y.P;
    prm.lengths_out[y.len_index(b, prm.layer)] = T;
    if (pos % y.P == 0) prm.desc_out[y.desc_index(b, prm.layer, pg)] = (KIND_DENSE << KIND_SHIFT) | y.dense_slot(pg);
    const int cp = prm.conv_page[b_idx];
    if (cp >= 0) prm.desc_out[y.desc_index(b, prm.layer, cp)] = (KIND_FACTORED << KIND_SHIFT) | cp;
}

// Fused append, bf16 path: the staged dense unit (PU key rows, then PU
// value rows) was copied before the new token reached the pool; write the
// token's key and value rows into the staged copy (row `srow` of the unit)
// and into the dense pool (row `prow` of the page in `slot`).  One warp.
template <int D, int PU>
__device__ __forceinline__ void patch_new_row(const DecodeParams &prm, unsigned char *stage, int b_idx, int b, int h,
                                              int slot, int prow, int srow, int lane) {
    const Layout &y = prm.y;
    const size_t in_off = ((size_t)b_idx * y.H + h) * D;
    const uint32_t *kin = reinterpret_cast<const uint32_t *>(reinterpret_cast<const __nv_bfloat16 *>(prm.k_new) + in_off);
    const uint32_t *vin = reinterpret_cast<const uint32_t *>(reinterpret_cast<const __nv_bfloat16 *>(prm.v_new) + in_off);
    unsigned char *kst = stage, *vst = stage + (size_t)PU * D * 2;
    char *kpool = const_cast<char *>(prm.dense_pool) + y.dense_offset(prm.layer, b, slot, h, 0);
    char *vpool = const_cast<char *>(prm.dense_pool) + y.dense_offset(prm.layer, b, slot, h, 1);
    for (int c2 = lane; c2 < D / 2; c2 += 32) {  // two bf16 per lane step
        const uint32_t kv = kin[c2], vv = vin[c2];
        *reinterpret_cast<uint32_t *>(kst + swz_offset(srow, c2 * 4, D * 2)) = kv;
        *reinterpret_cast<uint32_t *>(vst + swz_offset(srow, c2 * 4, D * 2)) = vv;
        *reinterpret_cast<uint32_t *>(kpool + swz_offset(prow, c2 * 4, D * 2)) = kv;
        *reinterpret_cast<uint32_t *>(vpool + swz_offset(prow, c2 * 4, D * 2)) = vv;
    }
    __syncwarp();
}

// One CTA of a (sequence, KV head) group of `gridDim.x` CTAs, streaming one
// contiguous, byte-balanced range of the sequence's pages.  The CTA's units
// are dealt round-robin to its NWC warps; each warp streams its own units
// through SPW private shared-memory slots, its lane 0 issuing the bulk copy of
// the warp's next unit into the slot the warp has just finished with (one
// mbarrier per slot, so a slot's phases are always consumed in order by the
// warp that fills it).  The slots' first fill, issued before the dependency
// wait, holds a large part of the range (NWC x SPW units); the rest is
// copied on demand.  Asking L2 to prefetch the rest of the range as well made
// back-to-back launches slower (the next launch's prefetches compete with the
// current one's last copies and its completion) and the single launch no
// faster, so the kernel does not; a CTA with a short range of bf16 records
// only keeps each warp's next factor record beyond its slots in flight to L2.
//
// Overlap with the neighbouring launches (programmatic dependent launch): a
// CTA lets the next launch start as soon as its own wait for the preceding
// launch has returned, so at most two decode grids are resident and the next
// one fetches while this one finishes.  Before that wait only bytes no earlier
// launch can still be writing are copied to shared memory: factor records
// (unless the preceding launch of this store was a conversion, a prefill or an
// append, in which case prm.wait_first makes the first copy wait) and dense
// rows below T - 2 (the rows the preceding launch may append are T - 2 and
// T - 1).  The query rows are prefetched into L2 before that wait: L2 is the
// point of coherence, so a row written after its prefetch is still read fresh.

template <int P, int D, int RKT, int RVT, bool Q4, bool ROPE>
__global__ void __launch_bounds__(DecodeShape<Q4, P, ROPE, D, RKT, RVT>::NWC * 32, CTAS_PER_SM)
    __maxnreg__((DecodeShape<Q4, P, ROPE, D, RKT, RVT>::MAXREG)) decode_bf16_kernel(const DecodeParams prm) {
    using Shape = DecodeShape<Q4, P, ROPE, D, RKT, RVT>;
    constexpr int NWC = Shape::NWC, SPW = Shape::SPW, NS = NWC * SPW;
    constexpr int DU = Shape::DU, PU = P / DU;  // dense units per page, rows per unit
    extern __shared__ __align__(128) unsigned char smem[];
    const Layout &y = prm.y;
    const int b_idx = blockIdx.z, b = prm.seqs[b_idx], h = blockIdx.y, rank = blockIdx.x;
    const int T = prm.lens[b_idx];
    const int ns = prm.nsplit[b_idx];  // CTAs taking part for this sequence (<= its pages)
    if (rank >= ns) return;            // uniform over the CTA

    const size_t stage_bytes = decode_stage_bytes<P, D, DU, ROPE>(y);
    const size_t base_off = decode_unit_bytes<P, D, DU>(y);  // RoPE: the page-start row in a slot
    unsigned char *stages = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * stage_bytes);
    DecodeShared<DU> &sh = *reinterpret_cast<DecodeShared<DU> *>(full + NS);
    // RoPE: the in-page offsets' (cos, sin) table [P][D/2], after the shared state
    float2 *rope_delta = reinterpret_cast<float2 *>(
        (reinterpret_cast<uintptr_t>(&sh + 1) + 15) & ~static_cast<uintptr_t>(15));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *wfull = full + warp * SPW;
    unsigned char *wstage = stages + (size_t)warp * SPW * stage_bytes;
    int *winfo = sh.slot_info + warp * SPW;  // per slot: page << 3 | dense << 2 | unit

    // this CTA's pages and their factorized stretch (split on the host)
    const int pb = prm.bounds[prm.boff[b_idx] + rank], pe = prm.bounds[prm.boff[b_idx] + rank + 1];
    const int a1 = min(max(pb, prm.fs[b_idx]), pe), a2 = max(a1, min(pe, prm.fw[b_idx]));
    const int n_fac = a2 - a1;
    bool waited = prm.wait_first != 0;
    uint64_t policy = 0;
    const char *fact = prm.factor_pool + y.record_offset(prm.layer, b, h, 0);
    // failure-path test hook: the very first unit of CTA (0, 0, 0) expects 16
    // bytes that no copy delivers, so its wait runs out
    bool poison = prm.inject == 1 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && warp == 0;
    // one unit (code page << 3 | dense << 2 | unit) into this warp's slot
    auto issue = [&](int slot, int info) {
        winfo[slot] = info;
        const int pg = info >> 3, hf = info & 3;
        unsigned char *dst = wstage + (size_t)slot * stage_bytes;
        const uint32_t extra = (ROPE ? (uint32_t)D * 4 : 0u) + (poison ? 16u : 0u);  // RoPE: the page start's (cos, sin) row
        poison = false;
        if (!(info & 4)) {
            mbar_arrive_expect_tx(&wfull[slot], (uint32_t)y.rec_bytes + extra);
            bulk_g2s_hint(dst, fact + (size_t)pg * y.rec_bytes, (uint32_t)y.rec_bytes, &wfull[slot], policy);
        } else {
            const int first = pg * P + hf * PU;
            if (!waited && first + unit_valid(T, first, PU) >= T - 1) {
                grid_dependency_wait();
                waited = true;
            }
            const int slot_d = y.dense_slot(pg);
            const uint32_t hb = (uint32_t)PU * D * 2;
            mbar_arrive_expect_tx(&wfull[slot], 2 * hb + extra);
            bulk_g2s_hint(dst, prm.dense_pool + y.dense_offset(prm.layer, b, slot_d, h, 0) + hf * hb, hb,
                          &wfull[slot], policy);
            bulk_g2s_hint(dst + hb, prm.dense_pool + y.dense_offset(prm.layer, b, slot_d, h, 1) + hf * hb, hb,
                          &wfull[slot], policy);
        }
        if (ROPE)  // constant table: no launch writes it
            bulk_g2s(dst + base_off, prm.rope_base + (size_t)pg * (D / 2), extra, &wfull[slot]);
    };
    if (ROPE) {  // constant table: read before any dependency wait
        const float4 *src = reinterpret_cast<const float4 *>(prm.rope_delta);
        float4 *dstt = reinterpret_cast<float4 *>(rope_delta);
        for (int i = threadIdx.x; i < P * D / 4; i += blockDim.x) dstt[i] = __ldg(src + i);
    }
    if (threadIdx.x == 0) {
        sh.failed = 0;
        // The CTA's units in page order: the dense units of [pb, a1) (sink
        // pages), one unit per factorized page of [a1, a2), the dense units of
        // [a2, pe) (window and incomplete pages).  The few dense ones are
        // listed here, before any dependency wait, so that taking a unit later
        // is a table lookup; units with no valid row are left out.
        int n = 0;
        for (int p = pb; p < pe; ++p) {
            if (p == a1) {
                sh.n_pre = n;
                p = a2;
                if (p >= pe) break;
            }
            for (int hf = 0; hf < DU; ++hf)
                if (T > p * P + hf * PU) sh.dense_units[n++] = (short)(((p < a1 ? p : p - a2) << 3) | 4 | hf);
        }
        if (a1 >= pe) sh.n_pre = n;
        sh.n_dense = n;
        for (int i = 0; i < NS; ++i) mbar_init(&full[i], 1);
        mbar_init(&sh.merge_bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    // unit u of the CTA goes to warp u mod NWC
    const int n_pre = sh.n_pre, n_units = sh.n_dense + n_fac;
    const int n_mine = n_units > warp ? (n_units - 1 - warp) / NWC + 1 : 0;
    // A short range (a few units per warp) is latency-bound: each warp's
    // factor record one unit beyond its slots also goes to L2 ahead of time
    // (32K tokens at batch 1: 427.5 -> 423.5 us per 32-layer step; two units
    // ahead: 444.5).  The first such request goes out with the first copies;
    // a refill's request pays only when the record that refill copies is in
    // L2 already (refill requests alone: 463 us).  Long ranges keep their
    // bandwidth for the slots' own copies (128K tokens and 16-request
    // batches were 1.5-3 % slower with it), and so do INT4 records, whose
    // kernel is bound by instruction issue (392.5 -> 412.5 us per step with
    // it).
    const bool ahead = !Q4 && n_units <= 6 * NWC;
    auto unit_of = [&](int u) -> int {
        return u < n_pre ? (int)sh.dense_units[u]
                         : (u < n_pre + n_fac ? (a1 + u - n_pre) << 3 : (a2 << 3) + sh.dense_units[u - n_fac]);
    };
    if (lane == 0) {
        policy = l2_evict_first();
        if (warp == 0)  // the query rows, read by every warp right after the dependency wait
            prefetch_l2(prm.q + ((size_t)b_idx * y.Hq + (size_t)h * y.G) * D * 2, (uint32_t)(y.G * D * 2));
        if (waited) grid_dependency_wait();
        for (int k = 0; k < SPW && k < n_mine; ++k) issue(k, unit_of(warp + NWC * k));
        if (ahead && SPW < n_mine) {
            const int nx = unit_of(warp + NWC * SPW);
            if (!(nx & 4)) prefetch_l2(fact + (size_t)(nx >> 3) * y.rec_bytes, (uint32_t)y.rec_bytes);
        }
    }

    // q, the appended token and the page table may come from the preceding grid
    grid_dependency_wait();
    if (threadIdx.x == 0) grid_launch_dependents();  // the next launch may now become resident
    if (prm.append && rank == 0 && h == 0 && threadIdx.x == 0) append_page_table(prm, b_idx, b, T);
    WarpState<P, D> w;
    {
        const int g = lane >> 2, c2 = 2 * (lane & 3);
        const __nv_bfloat16 *qrow =
            reinterpret_cast<const __nv_bfloat16 *>(prm.q) + ((size_t)b_idx * y.Hq + (size_t)h * y.G + g) * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            w.qf[kk][0] = g < y.G ? *reinterpret_cast<const uint32_t *>(qrow + kk * 16 + c2) : 0u;
            w.qf[kk][1] = g < y.G ? *reinterpret_cast<const uint32_t *>(qrow + kk * 16 + 8 + c2) : 0u;
            if constexpr (Q4) {  // bf16 -> fp16 is exact within fp16's range
                w.qh[kk][0] = pack_f16(bf16_lo_to_f32(w.qf[kk][0]), bf16_hi_to_f32(w.qf[kk][0]));
                w.qh[kk][1] = pack_f16(bf16_lo_to_f32(w.qf[kk][1]), bf16_hi_to_f32(w.qf[kk][1]));
            }
        }
    }
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) w.o[nt][0] = w.o[nt][1] = w.o[nt][2] = w.o[nt][3] = 0.f;
    w.m = -INFINITY;
    w.l = 0.f;
    const float scale_log2 = LOG2E * rsqrtf((float)D);
    const uint64_t wait_lim = prm.wait_ns ? prm.wait_ns : WAIT_NS;
    int slot = 0, k = 0;
    uint32_t ph = 0;
    for (; k < n_mine; ++k) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&wfull[slot], ph, prm.status, wait_lim))) break;
        const int info = winfo[slot];
        const int pg = info >> 3, part = info & 3;
        const uint32_t st = smem_u32(wstage + (size_t)slot * stage_bytes);
        if (!(info & 4)) {
            if constexpr (Q4) {
                factored_unit_q4<P, D, RKT, RVT>(w, wstage + (size_t)slot * stage_bytes, y, lane, scale_log2);
            } else if constexpr (ROPE) {
                factored_unit_rope<P, D, RKT, RVT>(
                    w, st, reinterpret_cast<const float2 *>(wstage + (size_t)slot * stage_bytes + base_off),
                    rope_delta, y, lane, scale_log2);
            } else {
                factored_unit<P, D, RKT, RVT>(w, st, y, lane, scale_log2);
            }
        } else {
            const int first = pg * P + part * PU;
            const int valid = unit_valid(T, first, PU);
            if (prm.append && first + valid == T)  // this unit ends with the appended token
                patch_new_row<D, PU>(prm, wstage + (size_t)slot * stage_bytes, b_idx, b, h, y.dense_slot(pg),
                                 T - 1 - pg * P, valid - 1, lane);
            if constexpr (ROPE)
                dense_unit_rope<P, D, PU>(
                    w, st, reinterpret_cast<const float2 *>(wstage + (size_t)slot * stage_bytes + base_off),
                    rope_delta, part * PU, valid, lane, scale_log2);
            else
                dense_unit<P, D, PU>(w, st, valid, lane, scale_log2);
        }
        __syncwarp();
        if (lane == 0 && k + SPW < n_mine) {  // the slot is free again: this warp's next unit goes into it
            fence_proxy_async_shared();
            issue(slot, unit_of(warp + NWC * (k + SPW)));
            if (ahead && k + SPW + 1 < n_mine) {
                const int nx = unit_of(warp + NWC * (k + SPW + 1));
                if (!(nx & 4)) prefetch_l2(fact + (size_t)(nx >> 3) * y.rec_bytes, (uint32_t)y.rec_bytes);
            }
        }
        if (++slot == SPW) {
            slot = 0;
            ph ^= 1;
        }
    }
    if (k < n_mine) {  // a bounded wait gave up: let this warp's copies land before the CTA exits
        if (lane == 0) {
            sh.failed = 1;
            const int issued = min(n_mine, k + SPW);  // units [0, issued) had their copies issued
            for (int kk = k; kk < issued; ++kk) mbar_wait_bounded(&wfull[kk % SPW], (kk / SPW) & 1, nullptr);
        }
        __syncwarp();
    }
    __syncthreads();  // the warp states go over slots that other warps may have been filling
    if (sh.failed) return;
    {  // per-warp state -> shared memory (every copy has landed and been read)
        const int g = lane >> 2, c2 = 2 * (lane & 3);
        float l = w.l;
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        float *comb = reinterpret_cast<float *>(stages) + (size_t)warp * 8 * (D + 4);
        if (g < y.G) {
            float *row = comb + g * (D + 4);
            if (c2 == 0) {
                row[0] = w.m;
                row[1] = l;
            }
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
                row[4 + 8 * nt + c2] = w.o[nt][0] + w.o[nt][2];
                row[4 + 8 * nt + c2 + 1] = w.o[nt][1] + w.o[nt][3];
            }
        }
    }
    __syncthreads();
    {
        // ring reuse: the warp states, over which the merging CTA stages the
        // other CTAs' states (it has merged its warps' states by then)
        float *comb = reinterpret_cast<float *>(stages);
        finish_split<D, NWC>(prm, comb, b_idx, b, h, rank, ns, &sh.last, comb, (size_t)NS * stage_bytes,
                             &sh.merge_bar);
    }
}

inline void choose_chunk(DecodeParams &p, long total_pages, int max_pages, int ctas_per_wave, int &splits) {
    int chunk = (int)((total_pages + ctas_per_wave - 1) / ctas_per_wave);
    chunk = chunk < 1 ? 1 : (chunk > MAX_CHUNK ? MAX_CHUNK : chunk);
    while ((max_pages + chunk - 1) / chunk > MAX_SPLITS) ++chunk;
    p.chunk = chunk;
    splits = (max_pages + chunk - 1) / chunk;
}

// Launch set-up of one kernel instantiation on the current device, computed
// once (shared-memory opt-in, ring depth, occupancy): none of it changes
// between calls, and querying it per launch costs more host time than a
// decode launch takes on the GPU.
struct LaunchSetup {
    int ready = 0;
    int stages = 0;
    size_t smem = 0;
    int occ = 1;
    cudaError_t err = cudaSuccess;
};

template <int P, int D, int RKT, int RVT, bool Q4 = false, bool ROPE = false>
cudaError_t launch_bf16(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st) {
    const Layout &y = p.y;
    using Shape = DecodeShape<Q4, P, ROPE, D, RKT, RVT>;
    const size_t stage_bytes = decode_stage_bytes<P, D, Shape::DU, ROPE>(y);
    auto k = decode_bf16_kernel<P, D, RKT, RVT, Q4, ROPE>;
    // one set-up per (device, record size): the ring depth depends on the record size
    static std::mutex mu;
    static LaunchSetup cache[64][4];
    static size_t cache_key[64][4];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    LaunchSetup setup;
    {
        std::lock_guard<std::mutex> lock(mu);
        int slot = -1;
        for (int i = 0; i < 4; ++i)
            if (cache[dev][i].ready && cache_key[dev][i] == stage_bytes) slot = i;
        if (slot < 0) {
            for (int i = 0; i < 4 && slot < 0; ++i)
                if (!cache[dev][i].ready) slot = i;
            if (slot < 0) slot = 0;
            LaunchSetup &c = cache[dev][slot];
            c = LaunchSetup{};
            constexpr int NS = Shape::NWC * Shape::SPW;
            const size_t tail_bytes = (size_t)Shape::NWC * 8 * (D + 4) * 4;  // the warp states
            if ((size_t)NS * stage_bytes < tail_bytes) return cudaErrorInvalidValue;
            c.stages = NS;
            c.smem = NS * stage_bytes + NS * sizeof(uint64_t) + sizeof(DecodeShared<Shape::DU>) +
                     (ROPE ? 16 + (size_t)P * D * 4 : 0);  // RoPE: the aligned in-page angle table
            c.err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem);
            // An SM's shared/L1 split is set when it takes a CTA and holds
            // while any CTA runs there: with the largest split a background
            // factorization CTA still fits beside a decode CTA.
            if (c.err == cudaSuccess)
                c.err = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             cudaSharedmemCarveoutMaxShared);
            if (c.err == cudaSuccess &&
                (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c.occ, k, Shape::NWC * 32, c.smem) != cudaSuccess ||
                 c.occ < 1))
                c.occ = 1;
            c.ready = 1;
            cache_key[dev][slot] = stage_bytes;
        }
        setup = cache[dev][slot];
    }
    if (setup.err != cudaSuccess) return setup.err;
    p.stages = setup.stages;
    // The CTAs of each KV head are shared out among the sequences in
    // proportion to their pages (largest remainder, at least one each, at most
    // one per page), each CTA streaming one byte-balanced range: about one CTA
    // per SM, or two waves when the sequences' lengths are so uneven that one
    // wave would leave a CTA with more than 1.3 times the mean load.
    int n[MAX_CALL_BATCH];
    {
        long tot = 0;
        for (int i = 0; i < p.nseq; ++i) tot += (p.lens[i] + P - 1) / P;
        auto share_out = [&](int target) {
            double rem[MAX_CALL_BATCH];
            int given = 0;
            for (int i = 0; i < p.nseq; ++i) {
                const int pages = (p.lens[i] + P - 1) / P;
                const double share = (double)target * pages / (double)tot;
                n[i] = std::max(1, std::min((int)share, std::min(MAX_SPLITS, pages)));
                rem[i] = share - (double)n[i];
                given += n[i];
            }
            while (given < target) {  // the rest by largest remainder
                int best = -1;
                for (int i = 0; i < p.nseq; ++i)
                    if (n[i] < std::min(MAX_SPLITS, (p.lens[i] + P - 1) / P) && (best < 0 || rem[i] > rem[best]))
                        best = i;
                if (best < 0) break;
                ++n[best];
                rem[best] -= 1.0;
                ++given;
            }
            double worst = 0.0;
            for (int i = 0; i < p.nseq; ++i) worst = std::max(worst, (double)((p.lens[i] + P - 1) / P) / n[i]);
            return worst / ((double)tot / std::max(given, 1));  // largest load over the mean
        };
        const int wave = std::max(p.nseq, num_sms / y.H);
        if (share_out(wave) > 1.3) share_out(2 * wave);
    }
    // page bounds of every CTA, ns + 1 per call entry (fewer CTAs if they do not fit)
    for (;;) {
        int need = 0;
        for (int i = 0; i < p.nseq; ++i) need += n[i] + 1;
        if (need <= MAX_BOUNDS) break;
        int big = 0;
        for (int i = 1; i < p.nseq; ++i)
            if (n[i] > n[big]) big = i;
        if (n[big] == 1) return cudaErrorInvalidValue;  // cannot happen: MAX_BOUNDS >= 2 MAX_CALL_BATCH
        --n[big];
    }
    int group = 1;
    for (int i = 0, off = 0; i < p.nseq; ++i) {
        const int T = p.lens[i];
        const PageSplit split(T, P, y.sink_pages, y.sink_tokens, y.W, (long long)y.rec_bytes,
                              (long long)P * D * 2, n[i]);
        p.nsplit[i] = n[i];
        p.boff[i] = off;
        p.fs[i] = split.fs;
        p.fw[i] = split.fw;
        for (int r = 0; r <= n[i]; ++r) p.bounds[off + r] = split.begin(r);
        off += n[i] + 1;
        group = std::max(group, n[i]);
    }
    const int splits = group;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)splits, (unsigned)y.H, (unsigned)p.nseq);
    cfg.blockDim = dim3(Shape::NWC * 32, 1, 1);
    cfg.dynamicSmemBytes = setup.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start while the previous grid finishes
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Per page size: picks the rank-specialised kernel (ranks <= 32 at d = 128) or
// the runtime-rank kernel; defined in decode_bf16_p*.cu.
cudaError_t launch_bf16_p16(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st);
cudaError_t launch_bf16_p32(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st);
cudaError_t launch_bf16_p64(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st);
// INT4 factor stores, all page sizes; defined in decode_bf16_q4.cu.
cudaError_t launch_bf16_q4(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st);
// Stores whose keys precede RoPE, P = 32 and 64; defined in decode_bf16_rope.cu.
cudaError_t launch_bf16_rope(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st);

}  // namespace pkv
