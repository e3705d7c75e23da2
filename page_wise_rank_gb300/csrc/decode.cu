// Mixed dense/factorized decode attention, split-K over pages.
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
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace pkv {

constexpr int NWC = 4;            // consumer warps
constexpr int MAX_CHUNK = MAX_CHUNK_PAGES;
constexpr float LOG2E = 1.4426950408889634f;

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
// dense half.  Returns false if the CTA has no pages.
__device__ bool build_units(DecodeShared &sh, const DecodeParams &prm, int b, int h, int T, int p0, int np) {
    const Layout &y = prm.y;
    for (int i = threadIdx.x; i < np; i += blockDim.x) {
        int d = prm.desc[y.desc_index(b, prm.layer, p0 + i)];
        sh.desc[i] = d;
        int kind = d >> KIND_SHIFT;
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
    return true;
}


// Write this CTA's state for the G query heads of (b, h) -- the NWC warp
// states in `comb` ([warp][g][m, l, o...], D + 2 floats per row) merged by
// eq. (5) -- to the workspace; then, if this CTA is the last of the `ns`
// CTAs of (b, h) to get there (atomic ticket, no waiting), merge all ns
// partial states into `out` and reset the ticket for the next launch.
// `scratch` holds 3 * MAX_SPLITS * 8 + 16 floats of shared memory.
template <int D>
__device__ void finish_split(const DecodeParams &prm, const float *comb, int b_idx, int b, int h, int split, int ns,
                             float *scratch, int *last) {
    const Layout &y = prm.y;
    const int G = y.G, S = y.part_stride;
    for (int e = threadIdx.x; e < G * (D + 2); e += blockDim.x) {
        int gg = e / (D + 2), k = e % (D + 2);
        float M = -INFINITY;
        for (int w = 0; w < NWC; ++w) M = fmaxf(M, comb[(w * 8 + gg) * (D + 2)]);
        float acc = 0.f;
        if (k == 0) {
            acc = M;
        } else {
            for (int w = 0; w < NWC; ++w) {
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
    for (int e = threadIdx.x; e < ns * G; e += blockDim.x) {
        int sp = e / G, g = e % G;
        const float *row = prm.partials + y.partial_index(b, h * G + g, sp) * S;
        sm[sp * 8 + g] = __ldcg(row);
        sl[sp * 8 + g] = __ldcg(row + 1);
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
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                                        prm.partials + y.partial_index(b, h * G + g, sp) * S + 4) + k4);
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

template <int P, int D, int MAXRT>
struct WarpState {
    uint32_t qf[D / 16][2];  // A fragments of q (rows 0-7), k-steps of 16
    float o[D / 8][4];       // rows 0-7: high-part products, rows 8-15: residual products
    float m, l;              // running max (log2 units) and this thread's partial sum
};

template <int P, int D, int MAXRT>
__device__ __forceinline__ void online_softmax(WarpState<P, D, MAXRT> &w, float (*sv)[2], int ntile) {
    float mx = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < P / 8; ++nt)
        if (nt < ntile) mx = fmaxf(mx, fmaxf(sv[nt][0], sv[nt][1]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    float m_new = fmaxf(w.m, mx);
    float alpha = exp2f(w.m - m_new);
    float ls = 0.f;
#pragma unroll
    for (int nt = 0; nt < P / 8; ++nt) {
        if (nt < ntile) {
            sv[nt][0] = exp2f(sv[nt][0] - m_new);
            sv[nt][1] = exp2f(sv[nt][1] - m_new);
            ls += sv[nt][0] + sv[nt][1];
        }
    }
    w.l = w.l * alpha + ls;
    w.m = m_new;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
        w.o[nt][0] *= alpha;
        w.o[nt][1] *= alpha;
        w.o[nt][2] *= alpha;
        w.o[nt][3] *= alpha;
    }
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

template <int P, int D, int MAXRT>
__device__ __forceinline__ void factored_unit(WarpState<P, D, MAXRT> &w, uint32_t st, const Layout &y, int lane,
                                              float scale_log2) {
    const int nkt = y.rkp >> 3, nvt = y.rvp >> 3;
    const uint32_t LK = st, RK = st + (uint32_t)y.off_RK, LV = st + (uint32_t)y.off_LV, RV = st + (uint32_t)y.off_RV;
    // 1. t = q R_K^T  (16 x rkp; rows 8-15 stay zero)
    float t[MAXRT][4];
#pragma unroll
    for (int j = 0; j < MAXRT; ++j) {
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
    uint32_t thi[MAXRT][1], tlo[MAXRT][1];
#pragma unroll
    for (int j = 0; j < MAXRT; ++j) split_bf16(t[j][0], t[j][1], thi[j][0], tlo[j][0]);
    float s[P / 8][4];
#pragma unroll
    for (int nt = 0; nt < P / 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    mma_rows<P / 8, MAXRT>(s, thi, tlo, nkt, LK, y.rkp * 2, lane);
    float sv[P / 8][2];
#pragma unroll
    for (int nt = 0; nt < P / 8; ++nt) {
        sv[nt][0] = (s[nt][0] + s[nt][2]) * scale_log2;
        sv[nt][1] = (s[nt][1] + s[nt][3]) * scale_log2;
    }
    // 3. page-local softmax state merged into the running one
    online_softmax<P, D, MAXRT>(w, sv, P / 8);
    // 4. u = p L_V  (16 x rvp): A = p split by token k-steps, B = LVt rows (rank)
    float u[MAXRT][4];
#pragma unroll
    for (int j = 0; j < MAXRT; ++j) u[j][0] = u[j][1] = u[j][2] = u[j][3] = 0.f;
#pragma unroll
    for (int kt = 0; kt < P / 16; ++kt) {
        uint32_t h0, l0, h1, l1;
        split_bf16(sv[2 * kt][0], sv[2 * kt][1], h0, l0);
        split_bf16(sv[2 * kt + 1][0], sv[2 * kt + 1][1], h1, l1);
#pragma unroll
        for (int j = 0; j < MAXRT; ++j) {
            if (j < nvt) {
                int row = 8 * j + (lane & 7), ch = 2 * kt + ((lane >> 3) & 1);
                uint32_t r0, r1;
                ldsm_x2(LV + swz_offset(row, ch * 16, P * 2), r0, r1);
                mma16816(u[j], h0, l0, h1, l1, r0, r1);
            }
        }
    }
    // 5. o += u R_V: A = u split by rank tiles, B = RVt rows (head dim)
    uint32_t uhi[MAXRT][1], ulo[MAXRT][1];
#pragma unroll
    for (int j = 0; j < MAXRT; ++j) split_bf16(u[j][0] + u[j][2], u[j][1] + u[j][3], uhi[j][0], ulo[j][0]);
    mma_rows<D / 8, MAXRT>(w.o, uhi, ulo, nvt, RV, y.rvp * 2, lane);
}

template <int P, int D, int MAXRT>
__device__ __forceinline__ void dense_unit(WarpState<P, D, MAXRT> &w, uint32_t st, int valid, int lane,
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
    online_softmax<P, D, MAXRT>(w, sv, NT);
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

template <int P, int D, int MAXRT, int NS>
__global__ void __launch_bounds__((NWC + 1) * 32) decode_bf16_kernel(const DecodeParams prm) {
    extern __shared__ __align__(128) unsigned char smem[];
    const Layout &y = prm.y;
    const int b_idx = blockIdx.z, b = prm.seqs[b_idx], h = blockIdx.y, split = blockIdx.x;
    const int T = prm.lengths[y.len_index(b, prm.layer)];
    const int n_pages = (T + P - 1) / P;
    const int p0 = split * prm.chunk;
    if (p0 >= n_pages) return;
    const int np = min(prm.chunk, n_pages - p0);

    const size_t stage_bytes = ((y.rec_bytes > (size_t)P * D * 2 ? y.rec_bytes : (size_t)P * D * 2) + 127) & ~(size_t)127;
    unsigned char *stages = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + NS * stage_bytes);
    uint64_t *empty = full + NS;
    DecodeShared &sh = *reinterpret_cast<DecodeShared *>(empty + NS);
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
    build_units(sh, prm, b, h, T, p0, np);  // contains __syncthreads
    const int NU = sh.n_units;

    WarpState<P, D, MAXRT> w;
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
            if ((d >> KIND_SHIFT) == KIND_FACTORED)
                factored_unit<P, D, MAXRT>(w, st, y, lane, scale_log2);
            else
                dense_unit<P, D, MAXRT>(w, st, dense_half_valid(T, p0 + i, P, half), lane, scale_log2);
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
        const int ns = (n_pages + prm.chunk - 1) / prm.chunk;
        finish_split<D>(prm, comb, b_idx, b, h, split, ns, scratch, &sh.last);
    }
}

// ---------------------------------------------------------------- fp32 CUDA-core path

template <int P, int D>
__global__ void __launch_bounds__(NWC * 32) decode_f32_kernel(const DecodeParams prm) {
    const Layout &y = prm.y;
    const int b_idx = blockIdx.z, b = prm.seqs[b_idx], h = blockIdx.y, split = blockIdx.x;
    const int T = prm.lengths[y.len_index(b, prm.layer)];
    const int n_pages = (T + P - 1) / P;
    const int p0 = split * prm.chunk;
    if (p0 >= n_pages) return;
    const int p1 = min(p0 + prm.chunk, n_pages);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = y.G;
    constexpr int TPL = (P + 31) / 32;  // tokens per lane
    constexpr int DPL = D / 32;         // head dims per lane
    const float scale = rsqrtf((float)D);
    __shared__ float comb[NWC][8][D + 2];
    __shared__ float scratch[3 * MAX_SPLITS * 8 + 16];
    __shared__ int last;

    float q[8][DPL];  // this lane's head dims of each query row
    const float *qb = reinterpret_cast<const float *>(prm.q) + ((size_t)b_idx * y.Hq + (size_t)h * G) * D;
    for (int g = 0; g < 8; ++g)
        for (int e = 0; e < DPL; ++e) q[g][e] = g < G ? qb[g * D + lane + 32 * e] : 0.f;
    float m[8], l[8], o[8][DPL];
    for (int g = 0; g < 8; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
        for (int e = 0; e < DPL; ++e) o[g][e] = 0.f;
    }
    for (int p = p0 + warp; p < p1; p += NWC) {
        int d = prm.desc[y.desc_index(b, prm.layer, p)];
        int kind = d >> KIND_SHIFT, slot = d & SLOT_MASK;
        int valid = min(P, T - p * P);
        float s[8][TPL];
        if (kind == KIND_FACTORED) {
            const char *rec = prm.factor_pool + y.record_offset(prm.layer, b, h, slot);
            const int rkp = y.rkp;
            // t = q R_K^T: full dot products by warp reduction, one rank at a time
            float t[8][2];  // lane j holds rank j and j + 32
            for (int g = 0; g < 8; ++g) t[g][0] = t[g][1] = 0.f;
            for (int j = 0; j < rkp; ++j) {
                float part[8];
                for (int g = 0; g < 8; ++g) part[g] = 0.f;
                for (int e = 0; e < DPL; ++e) {
                    float r = *swz_ptr<float>(rec + y.off_RK, j, lane + 32 * e, D);
                    for (int g = 0; g < 8; ++g) part[g] = fmaf(q[g][e], r, part[g]);
                }
                for (int g = 0; g < 8; ++g) {
                    float v = warp_sum(part[g]);
                    if ((j & 31) == lane) t[g][j >> 5] = v;
                }
            }
            // s = t L_K^T / sqrt(d): lane = token
            for (int e = 0; e < TPL; ++e) {
                int i = lane + 32 * e;
                for (int g = 0; g < 8; ++g) s[g][e] = 0.f;
                for (int j = 0; j < rkp; ++j) {
                    float lk = i < P ? *swz_ptr<float>(rec, i, j, rkp) : 0.f;
                    for (int g = 0; g < 8; ++g) s[g][e] = fmaf(__shfl_sync(0xffffffffu, t[g][j >> 5], j & 31), lk, s[g][e]);
                }
                for (int g = 0; g < 8; ++g) s[g][e] = i < P ? s[g][e] * scale : -INFINITY;
            }
        } else {
            const char *kp = prm.dense_pool + y.dense_offset(prm.layer, b, slot, h, 0);
            for (int e = 0; e < TPL; ++e)
                for (int g = 0; g < 8; ++g) s[g][e] = 0.f;
            for (int i = 0; i < valid; ++i) {
                float part[8];
                for (int g = 0; g < 8; ++g) part[g] = 0.f;
                for (int e = 0; e < DPL; ++e) {
                    float kv = *swz_ptr<float>(kp, i, lane + 32 * e, D);
                    for (int g = 0; g < 8; ++g) part[g] = fmaf(q[g][e], kv, part[g]);
                }
                for (int g = 0; g < 8; ++g) {
                    float v = warp_sum(part[g]);
                    if ((i & 31) == lane) s[g][i >> 5] = v * scale;
                }
            }
            for (int e = 0; e < TPL; ++e)
                if (lane + 32 * e >= valid)
                    for (int g = 0; g < 8; ++g) s[g][e] = -INFINITY;
        }
        // online softmax per query row
        float pw[8][TPL];
        for (int g = 0; g < 8; ++g) {
            float mx = -INFINITY;
            for (int e = 0; e < TPL; ++e) mx = fmaxf(mx, s[g][e]);
            mx = warp_max(mx);
            float m_new = fmaxf(m[g], mx);
            float alpha = expf(m[g] - m_new);
            float ls = 0.f;
            for (int e = 0; e < TPL; ++e) {
                pw[g][e] = s[g][e] == -INFINITY ? 0.f : expf(s[g][e] - m_new);
                ls += pw[g][e];
            }
            l[g] = l[g] * alpha + warp_sum(ls);
            m[g] = m_new;
            for (int e = 0; e < DPL; ++e) o[g][e] *= alpha;
        }
        if (kind == KIND_FACTORED) {
            const char *rec = prm.factor_pool + y.record_offset(prm.layer, b, h, slot);
            const int rvp = y.rvp;
            for (int j = 0; j < rvp; ++j) {
                // u_j = sum_i p_i L_V[i][j]  (LVt row j)
                float part[8];
                for (int g = 0; g < 8; ++g) part[g] = 0.f;
                for (int e = 0; e < TPL; ++e) {
                    int i = lane + 32 * e;
                    float lv = i < P ? *swz_ptr<float>(rec + y.off_LV, j, i, P) : 0.f;
                    for (int g = 0; g < 8; ++g) part[g] = fmaf(pw[g][e], lv, part[g]);
                }
                for (int g = 0; g < 8; ++g) part[g] = warp_sum(part[g]);
                for (int e = 0; e < DPL; ++e) {
                    float rv = *swz_ptr<float>(rec + y.off_RV, lane + 32 * e, j, rvp);
                    for (int g = 0; g < 8; ++g) o[g][e] = fmaf(part[g], rv, o[g][e]);
                }
            }
        } else {
            const char *vp = prm.dense_pool + y.dense_offset(prm.layer, b, slot, h, 1);
            for (int i = 0; i < valid; ++i) {
                float pi[8];
                for (int g = 0; g < 8; ++g) pi[g] = __shfl_sync(0xffffffffu, pw[g][i >> 5], i & 31);
                for (int e = 0; e < DPL; ++e) {
                    float vv = *swz_ptr<float>(vp, i, lane + 32 * e, D);
                    for (int g = 0; g < 8; ++g) o[g][e] = fmaf(pi[g], vv, o[g][e]);
                }
            }
        }
    }
    // warp states -> shared (m kept in log2 units), then the split hand-off
    for (int g = 0; g < 8; ++g) {
        if (lane == 0) {
            comb[warp][g][0] = m[g] * LOG2E;
            comb[warp][g][1] = l[g];
        }
        for (int e = 0; e < DPL; ++e) comb[warp][g][2 + lane + 32 * e] = o[g][e];
    }
    __syncthreads();
    const int ns = (n_pages + prm.chunk - 1) / prm.chunk;
    finish_split<D>(prm, &comb[0][0][0], b_idx, b, h, split, ns, scratch, &last);
}

// ---------------------------------------------------------------- launch

static void choose_chunk(DecodeParams &p, long total_pages, int max_pages, int ctas_per_wave, int &splits) {
    int chunk = (int)((total_pages + ctas_per_wave - 1) / ctas_per_wave);
    chunk = chunk < 1 ? 1 : (chunk > MAX_CHUNK ? MAX_CHUNK : chunk);
    while ((max_pages + chunk - 1) / chunk > MAX_SPLITS) ++chunk;
    p.chunk = chunk;
    splits = (max_pages + chunk - 1) / chunk;
}

template <int P, int D, int MAXRT, int NS>
static cudaError_t launch_bf16(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st) {
    const Layout &y = p.y;
    size_t stage_bytes = ((y.rec_bytes > (size_t)P * D * 2 ? y.rec_bytes : (size_t)P * D * 2) + 127) & ~(size_t)127;
    size_t tail_bytes = (size_t)NWC * 8 * (D + 2) * 4 + (3 * MAX_SPLITS * 8 + 16) * 4;  // comb + merge scratch
    if (NS * stage_bytes < tail_bytes) return cudaErrorInvalidValue;
    size_t smem = NS * stage_bytes + 2 * NS * sizeof(uint64_t) + sizeof(DecodeShared);
    auto k = decode_bf16_kernel<P, D, MAXRT, NS>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int occ = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, (NWC + 1) * 32, smem) != cudaSuccess || occ < 1) occ = 1;
    int splits = 1;
    choose_chunk(p, total_pages, max_pages, num_sms * occ, splits);
    dim3 grid((unsigned)splits, (unsigned)y.H, (unsigned)p.nseq);
    k<<<grid, (NWC + 1) * 32, smem, st>>>(p);
    return cudaGetLastError();
}

template <int P, int D>
static cudaError_t launch_p_d(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st) {
    if (p.y.dtype == 0) {
        auto k = decode_f32_kernel<P, D>;
        int occ = 1;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, NWC * 32, 0) != cudaSuccess || occ < 1) occ = 1;
        int splits = 1;
        choose_chunk(p, total_pages, max_pages, num_sms * occ, splits);
        dim3 grid((unsigned)splits, (unsigned)p.y.H, (unsigned)p.nseq);
        k<<<grid, NWC * 32, 0, st>>>(p);
        return cudaGetLastError();
    }
    int maxrt = (p.y.rkp > p.y.rvp ? p.y.rkp : p.y.rvp) / 8;
    if (maxrt <= 4) return launch_bf16<P, D, 4, 8>(p, total_pages, max_pages, num_sms, st);
    return launch_bf16<P, D, 8, 4>(p, total_pages, max_pages, num_sms, st);
}

cudaError_t launch_decode(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st) {
#define PKV_DEC_CASE(PP, DD) \
    if (p.y.P == PP && p.y.d == DD) return launch_p_d<PP, DD>(p, total_pages, max_pages, num_sms, st);
    PKV_DEC_CASE(16, 64)
    PKV_DEC_CASE(32, 64)
    PKV_DEC_CASE(64, 64)
    PKV_DEC_CASE(16, 128)
    PKV_DEC_CASE(32, 128)
    PKV_DEC_CASE(64, 128)
#undef PKV_DEC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkv
