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
// into units -- a factorized page, or half of a dense page (keys and values of
// P/2 tokens) -- each of which fits one shared-memory stage.  A producer warp
// streams units through an NS-stage ring with one or two bulk copies per unit
// (mbarrier transaction counts); NWC consumer warps each take every NWC-th
// unit and keep their own running (m, l, o) for the G query heads of the KV
// head.  At the end the warps' states are merged in shared memory and the
// CTA's state goes to the workspace; a second kernel merges the splits.
//
// bf16 storage: the four contractions of eq. (4) run on tensor cores
// (mma.sync m16n8k16 / m16n8k8, fp32 accumulate).  The G <= 8 query heads fill
// rows 0-7 of the 16-row tile; intermediate operands (q R_K^T, the softmax
// weights, and their product with L_V) are split into a bf16 high part in rows
// 0-7 and a bf16 residual in rows 8-15, so a single mma carries about 16
// mantissa bits and the two row halves are summed afterwards.
// fp32 storage: CUDA-core fp32 arithmetic throughout.
#pragma once
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace pkv {

constexpr int NWC = 4;            // consumer warps of the fp32 kernel
constexpr int NWC_BF16 = 8;       // consumer warps of the bf16 kernel
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

struct DecodeShared {
    int desc[MAX_CHUNK];
    int cnt[MAX_CHUNK];
    int off[MAX_CHUNK];
    int unit[2 * MAX_CHUNK];
    int n_units;
    int issued;
    int failed;
    int last;
};

__device__ __forceinline__ int dense_half_valid(int T, int p, int P, int half) {
    int first = p * P + half * (P / 2);
    int v = T - first;
    return v < 0 ? 0 : (v > P / 2 ? P / 2 : v);
}

// Build the CTA's unit list: per page 1 unit (factorized) or one per non-empty
// dense half.  Page kinds follow page_kind() at the call's length, the rule
// the store's page table records (the host mirror passes the length, so no
// global load precedes the first bulk copy); a factorized page's record is
// its own preallocated slot, a dense page sits in dense_slot(page).
// Returns the page count of the CTA (0: nothing to do).
__device__ inline int build_units(DecodeShared &sh, const DecodeParams &prm, int b_idx, int split, int &T_out) {
    const Layout &y = prm.y;
    const int p0 = split * prm.chunk;
    const int T = prm.lens[b_idx];
    T_out = T;
    const int n_pages = (T + y.P - 1) / y.P;
    if (p0 >= n_pages) return 0;
    const int np = min(prm.chunk, n_pages - p0);
    for (int i = threadIdx.x; i < np; i += blockDim.x) {
        const int p = p0 + i;
        const int kind = page_kind(p, T, y.P, y.sink_tokens, y.W);
        sh.desc[i] = (kind << KIND_SHIFT) | (kind == KIND_FACTORED ? p : y.dense_slot(p));
        sh.cnt[i] = kind == KIND_FACTORED
                        ? 1
                        : (dense_half_valid(T, p0 + i, y.P, 0) > 0) + (dense_half_valid(T, p0 + i, y.P, 1) > 0);
    }
    __syncthreads();
    if (threadIdx.x < 32) {  // warp 0: exclusive scan over pages, lane-contiguous segments
        int lane = threadIdx.x;
        int seg = (np + 31) / 32;
        int lo = lane * seg, hi = min(lo + seg, np);
        int sum = 0;
        for (int i = lo; i < hi; ++i) sum += sh.cnt[i];
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int i = lo; i < hi; ++i) {
            sh.off[i] = run;
            run += sh.cnt[i];
        }
        if (lane == 31) sh.n_units = incl;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < np; i += blockDim.x) {
        int o = sh.off[i];
        int kind = sh.desc[i] >> KIND_SHIFT;
        if (kind == KIND_FACTORED) {
            sh.unit[o] = i << 1;
        } else {
            int k = 0;
            for (int half = 0; half < 2; ++half)
                if (dense_half_valid(T, p0 + i, y.P, half) > 0) sh.unit[o + k++] = (i << 1) | half;
        }
    }
    __syncthreads();
    return np;
}

// Write this CTA's state for the G query heads of (b, h) -- the NWC warp
// states in `comb` ([warp][g][m, l, o...], D + 2 floats per row) merged by
// eq. (5) -- to the workspace; then, if this CTA is the last of the `ns`
// CTAs of (b, h) to get there (atomic ticket, no waiting), merge all ns
// partial states into `out` and reset the ticket for the next launch.
// `scratch` holds 3 * MAX_SPLITS * 8 + 16 floats of shared memory; `stage_buf`
// (optional, `stage_cap` bytes) receives the partial rows for the merge.
template <int D, int NW>
__device__ void finish_split(const DecodeParams &prm, const float *comb, int b_idx, int b, int h, int split, int ns,
                             float *scratch, int *last, float *stage_buf = nullptr, size_t stage_cap = 0) {
    const Layout &y = prm.y;
    const int G = y.G, S = y.part_stride;
    for (int e = threadIdx.x; e < G * (D + 2); e += blockDim.x) {
        int gg = e / (D + 2), k = e % (D + 2);
        float M = -INFINITY;
        for (int w = 0; w < NW; ++w) M = fmaxf(M, comb[(w * 8 + gg) * (D + 2)]);
        float acc = 0.f;
        if (k == 0) {
            acc = M;
        } else {
            for (int w = 0; w < NW; ++w) {
                float mw = comb[(w * 8 + gg) * (D + 2)];
                acc += (mw == -INFINITY ? 0.f : exp2f(mw - M)) * comb[(w * 8 + gg) * (D + 2) + k];
            }
        }
        prm.partials[y.partial_index(b, h * G + gg, split) * S + (k < 2 ? k : k + 2)] = acc;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        int old = atomicAdd(prm.tickets + y.ticket_index(b, h), 1);
        *last = (old == ns - 1);
    }
    __syncthreads();
    if (!*last) return;
    __threadfence();
    float *sm = scratch, *sl = scratch + MAX_SPLITS * 8, *wt = sl + MAX_SPLITS * 8, *Mg = wt + MAX_SPLITS * 8;
    float *iL = Mg + 8;
    // all partial rows of the G heads, staged in shared memory when they fit:
    // every load is issued before any is used (one round trip instead of ns)
    const int rows = ns * G, row4 = S / 4;
    const bool staged = stage_buf != nullptr && (size_t)rows * S * 4 <= stage_cap;
    if (staged) {
        float4 *dst = reinterpret_cast<float4 *>(stage_buf);
        const int total = rows * row4;
        for (int base = threadIdx.x; base < total; base += blockDim.x * 12) {
            float4 v[12];
#pragma unroll
            for (int k = 0; k < 12; ++k) {
                int e = base + k * blockDim.x;
                if (e < total) {
                    int r = e / row4, c = e % row4, sp = r / G, g = r % G;
                    v[k] = __ldcg(reinterpret_cast<const float4 *>(prm.partials +
                                                                   y.partial_index(b, h * G + g, sp) * S) + c);
                }
            }
#pragma unroll
            for (int k = 0; k < 12; ++k) {
                int e = base + k * blockDim.x;
                if (e < total) dst[e] = v[k];
            }
        }
        __syncthreads();
    }
    auto row_ptr = [&](int sp, int g) -> const float * {
        return staged ? stage_buf + ((size_t)sp * G + g) * S : prm.partials + y.partial_index(b, h * G + g, sp) * S;
    };
    for (int e = threadIdx.x; e < ns * G; e += blockDim.x) {
        int sp = e / G, g = e % G;
        const float *row = row_ptr(sp, g);
        sm[sp * 8 + g] = staged ? row[0] : __ldcg(row);
        sl[sp * 8 + g] = staged ? row[1] : __ldcg(row + 1);
    }
    __syncthreads();
    if (threadIdx.x < G) {
        int g = threadIdx.x;
        float M = -INFINITY, L = 0.f;
        for (int sp = 0; sp < ns; ++sp) M = fmaxf(M, sm[sp * 8 + g]);
        for (int sp = 0; sp < ns; ++sp) {
            float m = sm[sp * 8 + g];
            L += (m == -INFINITY ? 0.f : exp2f(m - M)) * sl[sp * 8 + g];
        }
        Mg[g] = M;
        iL[g] = 1.f / L;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < ns * G; e += blockDim.x) {
        int sp = e / G, g = e % G;
        float m = sm[sp * 8 + g];
        wt[sp * 8 + g] = (m == -INFINITY ? 0.f : exp2f(m - Mg[g])) * iL[g];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < G * (D / 4); e += blockDim.x) {
        int g = e / (D / 4), k4 = e % (D / 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int sp = 0; sp < ns; ++sp) {
            const float4 *src = reinterpret_cast<const float4 *>(row_ptr(sp, g) + 4) + k4;
            const float4 v = staged ? *src : __ldcg(src);
            float c = wt[sp * 8 + g];
            acc.x = fmaf(c, v.x, acc.x);
            acc.y = fmaf(c, v.y, acc.y);
            acc.z = fmaf(c, v.z, acc.z);
            acc.w = fmaf(c, v.w, acc.w);
        }
        reinterpret_cast<float4 *>(prm.out + ((size_t)b_idx * y.Hq + h * G + g) * D)[k4] = acc;
    }
    if (threadIdx.x == 0) prm.tickets[y.ticket_index(b, h)] = 0;
}

// ---------------------------------------------------------------- bf16 tensor-core path

template <int P, int D>
struct WarpState {
    uint32_t qf[D / 16][2];  // A fragments of q (rows 0-7), k-steps of 16
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
                mma16816(acc[nt], a0, a1, a2, a3, r0, r1);
                mma16816(acc[nt + 1], a0, a1, a2, a3, r2, r3);
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
                mma1688(acc[nt], a0, a1, r0);
                mma1688(acc[nt + 1], a0, a1, r1);
                mma1688(acc[nt + 2], a0, a1, r2);
                mma1688(acc[nt + 3], a0, a1, r3);
            } else {
                int row2 = 8 * (nt + (m & 1)) + (lane & 7);
                ldsm_x2(rows_base + swz_offset(row2, j * 16, pitch), r0, r1);
                mma1688(acc[nt], a0, a1, r0);
                mma1688(acc[nt + 1], a0, a1, r1);
            }
        }
    }
}

// RKT / RVT: rank tiles (ranks / 8) when fixed at compile time, 0 = read
// from the layout (up to 8 tiles).
template <int P, int D, int RKT, int RVT>
__device__ __forceinline__ void factored_unit(WarpState<P, D> &w, uint32_t st, const Layout &y, int lane,
                                              float scale_log2) {
    constexpr int MAXK = RKT ? RKT : 8, MAXV = RVT ? RVT : 8;
    const int nkt = RKT ? RKT : (y.rkp >> 3), nvt = RVT ? RVT : (y.rvp >> 3);
    const uint32_t off_RK = (uint32_t)P * nkt * 16, off_LV = off_RK + (uint32_t)nkt * 8 * D * 2;
    const uint32_t off_RV = off_LV + (uint32_t)nvt * 8 * P * 2;
    const uint32_t LK = st, RK = st + off_RK, LV = st + off_LV, RV = st + off_RV;
    // 1. t = q R_K^T  (16 x rkp; rows 8-15 stay zero)
    float t[MAXK][4];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
        t[j][0] = t[j][1] = t[j][2] = t[j][3] = 0.f;
        if (j < nkt) {
#pragma unroll
            for (int k2 = 0; k2 < D / 32; ++k2) {
                int row = 8 * j + (lane & 7), ch = 4 * k2 + (lane >> 3);
                uint32_t r0, r1, r2, r3;
                ldsm_x4(RK + swz_offset(row, ch * 16, D * 2), r0, r1, r2, r3);
                mma16816(t[j], w.qf[2 * k2][0], 0u, w.qf[2 * k2][1], 0u, r0, r1);
                mma16816(t[j], w.qf[2 * k2 + 1][0], 0u, w.qf[2 * k2 + 1][1], 0u, r2, r3);
            }
        }
    }
    // 2. s = t L_K^T  (16 x P), t split into high (rows 0-7) and residual (rows 8-15)
    uint32_t thi[MAXK][1], tlo[MAXK][1];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) split_bf16(t[j][0], t[j][1], thi[j][0], tlo[j][0]);
    float s[P / 8][4];
#pragma unroll
    for (int nt = 0; nt < P / 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    mma_rows<P / 8, MAXK>(s, thi, tlo, nkt, LK, nkt * 16, lane);
    float sv[P / 8][2];
#pragma unroll
    for (int nt = 0; nt < P / 8; ++nt) {
        sv[nt][0] = (s[nt][0] + s[nt][2]) * scale_log2;
        sv[nt][1] = (s[nt][1] + s[nt][3]) * scale_log2;
    }
    // 3. page-local softmax state merged into the running one
    online_softmax<P, D>(w, sv, P / 8);
    // 4. u = p L_V  (16 x rvp): A = p split by token k-steps, B = LVt rows (rank)
    float u[MAXV][4];
#pragma unroll
    for (int j = 0; j < MAXV; ++j) u[j][0] = u[j][1] = u[j][2] = u[j][3] = 0.f;
#pragma unroll
    for (int kt = 0; kt < P / 16; ++kt) {
        uint32_t h0, l0, h1, l1;
        split_bf16(sv[2 * kt][0], sv[2 * kt][1], h0, l0);
        split_bf16(sv[2 * kt + 1][0], sv[2 * kt + 1][1], h1, l1);
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
            if (j < nvt) {
                int row = 8 * j + (lane & 7), ch = 2 * kt + ((lane >> 3) & 1);
                uint32_t r0, r1;
                ldsm_x2(LV + swz_offset(row, ch * 16, P * 2), r0, r1);
                mma16816(u[j], h0, l0, h1, l1, r0, r1);
            }
        }
    }
    // 5. o += u R_V: A = u split by rank tiles, B = RVt rows (head dim)
    uint32_t uhi[MAXV][1], ulo[MAXV][1];
#pragma unroll
    for (int j = 0; j < MAXV; ++j) split_bf16(u[j][0] + u[j][2], u[j][1] + u[j][3], uhi[j][0], ulo[j][0]);
    mma_rows<D / 8, MAXV>(w.o, uhi, ulo, nvt, RV, nvt * 16, lane);
}

template <int P, int D>
__device__ __forceinline__ void dense_unit(WarpState<P, D> &w, uint32_t st, int valid, int lane,
                                           float scale_log2) {
    constexpr int PH = P / 2;  // tokens in the unit
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
    float sv[P / 8][2];
    const int c2 = 2 * (lane & 3);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        int tok = 8 * nt + c2;
        sv[nt][0] = tok < valid ? s[nt][0] * scale_log2 : -INFINITY;
        sv[nt][1] = tok + 1 < valid ? s[nt][1] * scale_log2 : -INFINITY;
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

// Fused append, bf16 path: the staged half page was copied before the new
// token reached the pool; write the token's key and value rows into the
// staged copy (row `srow` of the unit) and into the dense pool (row `prow`
// of the page in `slot`).  One warp.
template <int D>
__device__ __forceinline__ void patch_new_row(const DecodeParams &prm, unsigned char *stage, int b_idx, int b, int h,
                                              int slot, int prow, int srow, int lane) {
    const Layout &y = prm.y;
    const size_t in_off = ((size_t)b_idx * y.H + h) * D;
    const uint32_t *kin = reinterpret_cast<const uint32_t *>(reinterpret_cast<const __nv_bfloat16 *>(prm.k_new) + in_off);
    const uint32_t *vin = reinterpret_cast<const uint32_t *>(reinterpret_cast<const __nv_bfloat16 *>(prm.v_new) + in_off);
    unsigned char *kst = stage, *vst = stage + (size_t)(y.P / 2) * D * 2;
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

template <int P, int D, int RKT, int RVT>
__global__ void __launch_bounds__((NWC_BF16 + 1) * 32) decode_bf16_kernel(const DecodeParams prm) {
    constexpr int NWC = NWC_BF16;
    extern __shared__ __align__(128) unsigned char smem[];
    const Layout &y = prm.y;
    const int b_idx = blockIdx.z, b = prm.seqs[b_idx], h = blockIdx.y, split = blockIdx.x;
    const int NS = prm.stages;

    const size_t stage_bytes = ((y.rec_bytes > (size_t)P * D * 2 ? y.rec_bytes : (size_t)P * D * 2) + 127) & ~(size_t)127;
    unsigned char *stages = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * stage_bytes);
    uint64_t *empty = full + NS_MAX;
    DecodeShared &sh = *reinterpret_cast<DecodeShared *>(empty + NS_MAX);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        sh.failed = 0;
        sh.issued = 0;
        fence_barrier_init();
    }
    int T = 0;
    const int np = build_units(sh, prm, b_idx, split, T);  // contains __syncthreads
    if (np == 0) return;
    const int n_pages = (T + P - 1) / P;
    const int p0 = split * prm.chunk;
    const int NU = sh.n_units;
    if (prm.append && split == 0 && h == 0 && threadIdx.x == 0) append_page_table(prm, b_idx, b, T);

    WarpState<P, D> w;
    if (warp == NWC) {  // producer
        if (lane == 0) {
            int u = 0;
            for (; u < NU; ++u) {
                int stg = u % NS;
                uint32_t ph = (u / NS) & 1;
                if (!mbar_wait_bounded(&empty[stg], ph ^ 1, prm.status)) {
                    sh.failed = 1;
                    break;
                }
                int info = sh.unit[u];
                int i = info >> 1, half = info & 1;
                int d = sh.desc[i];
                int slot = d & SLOT_MASK;
                unsigned char *dst = stages + (size_t)stg * stage_bytes;
                if ((d >> KIND_SHIFT) == KIND_FACTORED) {
                    mbar_arrive_expect_tx(&full[stg], (uint32_t)y.rec_bytes);
                    bulk_g2s(dst, prm.factor_pool + y.record_offset(prm.layer, b, h, slot), (uint32_t)y.rec_bytes,
                             &full[stg]);
                } else {
                    const uint32_t hb = (uint32_t)(P / 2) * D * 2;
                    mbar_arrive_expect_tx(&full[stg], 2 * hb);
                    bulk_g2s(dst, prm.dense_pool + y.dense_offset(prm.layer, b, slot, h, 0) + half * hb, hb, &full[stg]);
                    bulk_g2s(dst + hb, prm.dense_pool + y.dense_offset(prm.layer, b, slot, h, 1) + half * hb, hb,
                             &full[stg]);
                }
            }
            sh.issued = u;
        }
        __syncwarp();
    } else {  // consumers
        const int g = lane >> 2, c2 = 2 * (lane & 3);
        const __nv_bfloat16 *qrow =
            reinterpret_cast<const __nv_bfloat16 *>(prm.q) + ((size_t)b_idx * y.Hq + (size_t)h * y.G + g) * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            w.qf[kk][0] = g < y.G ? *reinterpret_cast<const uint32_t *>(qrow + kk * 16 + c2) : 0u;
            w.qf[kk][1] = g < y.G ? *reinterpret_cast<const uint32_t *>(qrow + kk * 16 + 8 + c2) : 0u;
        }
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) w.o[nt][0] = w.o[nt][1] = w.o[nt][2] = w.o[nt][3] = 0.f;
        w.m = -INFINITY;
        w.l = 0.f;
        const float scale_log2 = LOG2E * rsqrtf((float)D);
        for (int u = warp; u < NU; u += NWC) {
            int stg = u % NS;
            uint32_t ph = (u / NS) & 1;
            bool ok = mbar_wait_bounded(&full[stg], ph, prm.status);
            if (!__all_sync(0xffffffffu, ok)) {
                sh.failed = 1;
                break;
            }
            int info = sh.unit[u];
            int i = info >> 1, half = info & 1;
            int d = sh.desc[i];
            uint32_t st = smem_u32(stages + (size_t)stg * stage_bytes);
            if ((d >> KIND_SHIFT) == KIND_FACTORED) {
                factored_unit<P, D, RKT, RVT>(w, st, y, lane, scale_log2);
            } else {
                const int valid = dense_half_valid(T, p0 + i, P, half);
                const int first = (p0 + i) * P + half * (P / 2);
                if (prm.append && first + valid == T)  // this unit ends with the appended token
                    patch_new_row<D>(prm, stages + (size_t)stg * stage_bytes, b_idx, b, h, d & SLOT_MASK,
                                     T - 1 - (p0 + i) * P, valid - 1, lane);
                dense_unit<P, D>(w, st, valid, lane, scale_log2);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stg]);
        }
    }
    __syncthreads();
    if (sh.failed) {
        // a bounded wait gave up: let every issued copy land before the CTA exits
        if (threadIdx.x == 0) {
            for (int u = sh.issued - NS; u < sh.issued; ++u)
                if (u >= 0) mbar_wait_bounded(&full[u % NS], (u / NS) & 1, nullptr);
        }
        __syncthreads();
        return;
    }
    if (warp < NWC) {  // per-warp state -> shared memory (the ring is free: every copy has landed)
        const int g = lane >> 2, c2 = 2 * (lane & 3);
        float l = w.l;
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        float *comb = reinterpret_cast<float *>(stages) + (size_t)warp * 8 * (D + 2);
        if (g < y.G) {
            float *row = comb + g * (D + 2);
            if (c2 == 0) {
                row[0] = w.m;
                row[1] = l;
            }
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
                row[2 + 8 * nt + c2] = w.o[nt][0] + w.o[nt][2];
                row[2 + 8 * nt + c2 + 1] = w.o[nt][1] + w.o[nt][3];
            }
        }
    }
    __syncthreads();
    {
        const float *comb = reinterpret_cast<const float *>(stages);
        float *scratch = reinterpret_cast<float *>(stages) + NWC * 8 * (D + 2);
        float *stage_buf = scratch + 3 * MAX_SPLITS * 8 + 16;
        const size_t used = (size_t)(NWC * 8 * (D + 2) + 3 * MAX_SPLITS * 8 + 16) * 4;
        const size_t cap = (size_t)NS * stage_bytes > used ? (size_t)NS * stage_bytes - used : 0;
        const int ns = (n_pages + prm.chunk - 1) / prm.chunk;
        finish_split<D, NWC>(prm, comb, b_idx, b, h, split, ns, scratch, &sh.last, stage_buf, cap);
    }
}

inline void choose_chunk(DecodeParams &p, long total_pages, int max_pages, int ctas_per_wave, int &splits) {
    int chunk = (int)((total_pages + ctas_per_wave - 1) / ctas_per_wave);
    chunk = chunk < 1 ? 1 : (chunk > MAX_CHUNK ? MAX_CHUNK : chunk);
    while ((max_pages + chunk - 1) / chunk > MAX_SPLITS) ++chunk;
    p.chunk = chunk;
    splits = (max_pages + chunk - 1) / chunk;
}

template <int P, int D, int RKT, int RVT>
cudaError_t launch_bf16(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st) {
    const Layout &y = p.y;
    size_t stage_bytes = ((y.rec_bytes > (size_t)P * D * 2 ? y.rec_bytes : (size_t)P * D * 2) + 127) & ~(size_t)127;
    size_t tail_bytes = (size_t)NWC_BF16 * 8 * (D + 2) * 4 + (3 * MAX_SPLITS * 8 + 16) * 4;  // comb + merge scratch
    size_t fixed = 2 * NS_MAX * sizeof(uint64_t) + sizeof(DecodeShared);
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || optin <= 0)
        optin = 227 * 1024;
    // as many stages as fit: bytes in flight per SM are what hide HBM latency
    int ns = (int)(((size_t)optin - fixed) / stage_bytes);
    ns = ns > NS_MAX ? NS_MAX : ns;
    if (ns < 2 || ns * stage_bytes < tail_bytes) return cudaErrorInvalidValue;
    p.stages = ns;
    size_t smem = ns * stage_bytes + fixed;
    auto k = decode_bf16_kernel<P, D, RKT, RVT>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int occ = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, (NWC_BF16 + 1) * 32, smem) != cudaSuccess || occ < 1)
        occ = 1;
    int splits = 1;
    choose_chunk(p, total_pages, max_pages, num_sms * occ, splits);
    dim3 grid((unsigned)splits, (unsigned)y.H, (unsigned)p.nseq);
    k<<<grid, (NWC_BF16 + 1) * 32, smem, st>>>(p);
    return cudaGetLastError();
}

// Per page size: picks the rank-specialised kernel (ranks <= 32 at d = 128) or
// the runtime-rank kernel; defined in decode_bf16_p*.cu.
cudaError_t launch_bf16_p16(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st);
cudaError_t launch_bf16_p32(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st);
cudaError_t launch_bf16_p64(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st);

}  // namespace pkv
