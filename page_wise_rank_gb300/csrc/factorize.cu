// Batched page factorization: one CTA per page.
//
// "PuzzleKV: Page-Wise Low-Rank Decomposition for KV Cache Compression",
// §3.3 ③ and eq. (2): for a P x d page X (P < d) the left singular subspace
// comes from the P x P Gram matrix G = X X^T; L = top-r eigenvectors Q_r,
// R = Q_r^T X.  Per CTA:
//   1. X -> shared memory (bf16 rows in the swizzled layout, or fp32 rows);
//   2. G = X X^T in fp32: bf16 pages on tensor cores (mma.sync m16n8k16,
//      bf16 products are exact in fp32), fp32 pages on CUDA cores;
//   3. the top-r eigenvectors of G: Householder reduction to tridiagonal
//      form, then for r <= P / 2 multisection for the eigenvalues, inverse
//      iteration for the r vectors of the tridiagonal and the reflections
//      applied to them; for larger r the reflections' product formed
//      explicitly and implicit QL on the tridiagonal with every rotation
//      applied to that product, eigenvalues ranked descending (ties: lower
//      index first);
//   4. L = Q_r, R = Q_r^T X in fp32, written as bf16 or fp32 into either a
//      factor record (swizzled store layout) or plain row-major arrays.
#include <cuda_fp16.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace pkv {

// An off-diagonal entry of the tridiagonal at or below this fraction of its
// norm counts as zero (the fp32 unit roundoff, 2^-23).
constexpr float QL_EPS = 1.1920929e-7f;
// The eigensolve works on G scaled to a largest diagonal entry in [1, 2).
// A column whose norm below the diagonal is at most NEGLIGIBLE gets no
// reflection, and a QL rotation whose radius is below it counts as a split:
// such entries change no eigenvalue by more than 1e-18, while reflecting or
// rotating by them would square them into the subnormal range (a block of
// repeated rows drives the trailing columns that low) and divide by that.
constexpr float NEGLIGIBLE = 1e-18f;

template <typename T, int P, int D>
struct FactorSmem {
    // The page X is needed for the Gram matrix and again for the projection,
    // the eigenvectors only in between: they share storage, and the page is
    // loaded a second time once the eigenvectors are taken out.
    union {
        alignas(128) unsigned char X[P * D * sizeof(T)];  // swizzled rows, pitch D * sizeof(T)
        float Z[P][P + 1];  // eigenvectors as columns: Z[i][j] = component i of vector j
    };
    // Gram matrix; during the reduction row k above the diagonal keeps beta_k
    // (G[k][k+1]) and the first entry of v_k (G[k][k+2]); after the
    // eigensolve, Q with its columns in eigenvalue order
    float G[P][P + 1];
    // scratch, each part live at its own time: the tridiagonal's diagonal
    // (then the eigenvalues, then per-column factors) in w[0, P), its
    // off-diagonal in w[P, 2P), the reduction's work vector in w[2P, 3P);
    // INT4 records' scales in w[0, P + D) once those are dead
    static constexpr int WN = 3 * P > P + D ? 3 * P : P + D;
    float w[WN];
    __device__ __forceinline__ float *lam() { return w; }
    __device__ __forceinline__ float *off() { return w + P; }
    __device__ __forceinline__ float *pv() { return w + 2 * P; }
    __device__ __forceinline__ float *sc() { return w; }
};

// Source page and destination of CTA `job` (mode chosen by the host).
struct JobView {
    const char *x;  // first row of X
    int x_pool;     // 1: rows in the swizzled dense-pool layout
    int kind;       // 0 = key, 1 = value (record destinations)
    int r;          // rank to keep
    char *rec;      // factor record (record modes) or nullptr
    char *L;        // plain outputs (batch mode)
    char *R;
    float *sigma;
    float *qL, *qR;  // batch INT4 mode: the absorbed fp32 factors (or nullptr)
};

__device__ __forceinline__ JobView job_view(const FactorParams &fp, long job) {
    JobView v{};
    const Layout &y = fp.y;
    if (fp.mode == FACT_MODE_BATCH) {
        v.x = fp.x_base + (size_t)job * fp.P * fp.d * fp.x_esz;
        v.x_pool = 0;
        v.kind = 0;
        v.r = fp.r;
        v.rec = nullptr;
        v.L = fp.L_out + (size_t)job * fp.P * fp.r * fp.out_esz;
        v.R = fp.R_out + (size_t)job * fp.r * fp.d * fp.out_esz;
        v.sigma = fp.sigma ? fp.sigma + (size_t)job * fp.P : nullptr;
    } else if (fp.mode == FACT_MODE_PREFILL) {
        // job -> (layer, head, kind, page) with pages innermost
        long np = fp.p_hi - fp.p_lo;
        long t = job;
        int pg = fp.p_lo + (int)(t % np); t /= np;
        int kind = (int)(t % 2); t /= 2;
        int h = (int)(t % y.H); t /= y.H;
        int lrel = (int)t;  // layer fp.layer0 + lrel, block lrel of the sources
        const char *src = kind == 0 ? fp.k_src : fp.v_src;
        v.x = src + (((size_t)lrel * y.H + h) * fp.T + (size_t)pg * y.P) * y.d * y.esz;
        v.x_pool = 0;
        v.kind = kind;
        v.r = kind == 0 ? y.rk : y.rv;
        v.rec = fp.factor_pool + y.record_offset(fp.layer0 + lrel, fp.seq, h, pg);
    } else if (fp.mode == FACT_MODE_BATCH_Q4) {
        const int rp = fp.q4_kind == 0 ? y.rkp : y.rvp;
        v.x = fp.x_base + (size_t)job * y.P * y.d * 2;
        v.x_pool = 0;
        v.kind = fp.q4_kind;
        v.r = fp.q4_kind == 0 ? y.rk : y.rv;
        v.rec = fp.q4_records + (size_t)job * y.rec_bytes;
        v.qL = fp.q4_L ? fp.q4_L + (size_t)job * y.P * rp : nullptr;
        v.qR = fp.q4_R ? fp.q4_R + (size_t)job * rp * y.d : nullptr;
    } else if (fp.mode == FACT_MODE_CONVERT_LIST) {  // job -> (list entry, head, kind)
        int kind = (int)(job % 2);
        long t = job / 2;
        int h = (int)(t % y.H);
        const int2 e = fp.conv_list[t / y.H];
        const int b = e.x >> 8, l = e.x & 255, pg = e.y;
        v.x = fp.dense_pool + y.dense_offset(l, b, y.dense_slot(pg), h, kind);
        v.x_pool = 1;
        v.kind = kind;
        v.r = kind == 0 ? y.rk : y.rv;
        v.rec = fp.factor_pool + y.record_offset(l, b, h, pg);
    } else {  // FACT_MODE_CONVERT: job -> (call entry, head, kind)
        int kind = (int)(job % 2);
        long t = job / 2;
        int h = (int)(t % y.H);
        int e = (int)(t / y.H);
        int b = fp.conv_seq[e], pg = fp.conv_page[e];
        v.x = fp.dense_pool + y.dense_offset(fp.layer, b, y.dense_slot(pg), h, kind);
        v.x_pool = 1;
        v.kind = kind;
        v.r = kind == 0 ? y.rk : y.rv;
        v.rec = fp.factor_pool + y.record_offset(fp.layer, b, h, pg);
    }
    return v;
}

template <typename T, int P, int D, int NT>
__device__ void load_page(FactorSmem<T, P, D> &s, const JobView &v) {
    // 16-byte vectors; pool pages are already swizzled, plain rows get swizzled here
    constexpr int PITCH = D * (int)sizeof(T);
    constexpr int NVEC = P * PITCH / 16;
    const uint4 *src = reinterpret_cast<const uint4 *>(v.x);
    for (int i = threadIdx.x; i < NVEC; i += NT) {
        uint4 val = src[i];
        int row = (i * 16) / PITCH, b = (i * 16) % PITCH;
        uint32_t off = v.x_pool ? (uint32_t)(i * 16) : swz_offset(row, b, PITCH);
        *reinterpret_cast<uint4 *>(s.X + off) = val;
    }
}

// G = X X^T, bf16 rows on tensor cores.
template <int P, int D, int NT>
__device__ void gram_bf16(FactorSmem<__nv_bfloat16, P, D> &s) {
    constexpr int MT = P / 16, NTL = P / 8, KS = D / 16, PITCH = D * 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t xb = smem_u32(s.X);
    for (int tile = warp; tile < MT * NTL; tile += NT / 32) {
        int mt = tile / NTL, nt = tile % NTL;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            uint32_t a0, a1, a2, a3, b0, b1;
            {   // A: rows mt*16 + (lane & 15), chunk 2kk + (lane >> 4)
                int row = mt * 16 + (lane & 15), ch = 2 * kk + (lane >> 4);
                ldsm_x4(xb + swz_offset(row, ch * 16, PITCH), a0, a1, a2, a3);
            }
            {   // B: rows nt*8 + (lane & 7), chunk 2kk + ((lane >> 3) & 1)
                int row = nt * 8 + (lane & 7), ch = 2 * kk + ((lane >> 3) & 1);
                ldsm_x2(xb + swz_offset(row, ch * 16, PITCH), b0, b1);
            }
            mma16816(acc, a0, a1, a2, a3, b0, b1);
        }
        int r0 = mt * 16 + (lane >> 2), c0 = nt * 8 + 2 * (lane & 3);
        s.G[r0][c0] = acc[0];
        s.G[r0][c0 + 1] = acc[1];
        s.G[r0 + 8][c0] = acc[2];
        s.G[r0 + 8][c0 + 1] = acc[3];
    }
}

// G = X X^T, fp32 rows on CUDA cores (upper triangle, mirrored).
template <int P, int D, int NT>
__device__ void gram_f32(FactorSmem<float, P, D> &s) {
    constexpr int PITCH = D * 4;
    for (int e = threadIdx.x; e < P * P; e += NT) {
        int i = e / P, j = e % P;
        if (j < i) continue;
        float acc = 0.f;
        for (int k = 0; k < D; ++k)
            acc = fmaf(*reinterpret_cast<const float *>(s.X + swz_offset(i, k * 4, PITCH)),
                       *reinterpret_cast<const float *>(s.X + swz_offset(j, k * 4, PITCH)), acc);
        s.G[i][j] = acc;
        s.G[j][i] = acc;
    }
}

// ---------------------------------------------------------------- eigensolve
// Eigenvectors of the symmetric P x P matrix in s.G (both triangles).  For
// ranks above P / 2, by three classical steps (smaller ranks replace steps 2
// and 3 by the top-r steps further down):
//   1. Householder reduction to tridiagonal form T = Q^T G Q, with P - 2
//      reflections H_k = I - beta_k v_k v_k^T (v_k supported on the indices
//      k+1 .. P-1), each applied to both sides of the trailing block as one
//      rank-2 update;
//   2. Q = H_0 H_1 ... H_{P-3} formed explicitly in s.Z, last reflection
//      first;
//   3. the implicit QL algorithm with Wilkinson shifts on T, every plane
//      rotation also applied to two columns of s.Z, whose columns so become
//      the eigenvectors of G (the tql2 scheme of Bowdler, Martin, Reinsch and
//      Wilkinson, "The QR and QL algorithms for symmetric matrices", 1968).
// Every sum is taken by a fixed set of lanes in a fixed order, whatever the
// block size, so every variant of the kernel gives the same bits.

// Sum over i in [0, n) of the products a(i) b(i), four lanes per output
// (lanes 4t .. 4t+3 of a warp; call with every lane of the warp): lane
// quarter q takes i = 8q + m + 32t (m < 8), which keeps the eight outputs of
// a warp on distinct banks when the products read row (or column) o + i of a
// matrix with pitch P + 1; the four partial sums meet by shuffles in a fixed
// order.  `active`: whether this lane's output exists (its products are
// skipped otherwise).
template <typename F>
__device__ __forceinline__ float quad_dot(int n, bool active, F prod) {
    const int q = threadIdx.x & 3;
    float acc = 0.f;
    if (active)
        for (int t = 0; 32 * t < n; ++t)
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int i = 32 * t + 8 * q + m;
                if (i < n) acc = prod(i, acc);
            }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    return acc;
}

// Step 1, on the lower triangle of s.G (the upper one is not read from the
// first reflection on).  On return lam[k] = T_kk, off[k] = T_{k,k+1}
// (off[P-1] = 0); v_k stays in column k of s.G from row k+2 on, its first
// entry in G[k][k+2], beta_k in G[k][k+1] (0: no reflection).
template <typename T, int P, int D, int NT>
__device__ void tridiagonalize(FactorSmem<T, P, D> &s) {
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int k = 0; k < P - 2; ++k) {
        const int n = P - 1 - k;  // order of the trailing block S = G[k+1.., k+1..]
        // every warp forms the reflection itself (the same sums in the same
        // order, hence the same bits): x = G[k+1.., k], x0 its first entry
        float sig = 0.f;
        for (int i = 1 + lane; i < n; i += 32) sig = fmaf(s.G[k + 1 + i][k], s.G[k + 1 + i][k], sig);
        sig = warp_sum(sig);
        const float x0 = s.G[k + 1][k];
        float alpha = x0, beta = 0.f, v0 = 0.f;
        if (sig > NEGLIGIBLE * NEGLIGIBLE) {  // H x = alpha e_1, v = x - alpha e_1, beta = 2 / |v|^2 <= 1 / sig
            alpha = -copysignf(sqrtf(fmaf(x0, x0, sig)), x0);
            v0 = x0 - alpha;  // |v0| = |x0| + |alpha|: no cancellation
            beta = -1.f / (alpha * v0);
        }
        if (tid == 0) {
            s.lam()[k] = s.G[k][k];
            s.off()[k] = alpha;
            s.G[k][k + 1] = beta;  // row k above the diagonal is no longer read
            s.G[k][k + 2] = v0;
        }
        if (beta == 0.f) continue;  // the same decision in every warp
        auto vv = [&](int i) { return i == 0 ? v0 : s.G[k + 1 + i][k]; };
        // entry (i, j) of S, from the lower triangle (the only one kept)
        auto S = [&](int i, int j) { return j <= i ? s.G[k + 1 + i][k + 1 + j] : s.G[k + 1 + j][k + 1 + i]; };
        // p = beta S v: four lanes per row (warp-uniform loop bounds)
        for (int base = 8 * warp; base < n; base += NT / 4) {
            const int i = base + (lane >> 2);
            const float acc = quad_dot(n, i < n, [&](int j, float a) { return fmaf(S(i, j), vv(j), a); });
            if ((lane & 3) == 0 && i < n) s.pv()[i] = beta * acc;
        }
        __syncthreads();
        // K = beta v.p / 2 (each warp), w = p - K v, S <- S - v w^T - w v^T on
        // the lower triangle.  Rows i and n - 1 - i share a warp pass (i + 1
        // and n - i entries: n + 1 together), so that short rows leave no
        // lanes idle.
        float vp = 0.f;
        for (int i = lane; i < n; i += 32) vp = fmaf(vv(i), s.pv()[i], vp);
        const float K = 0.5f * beta * warp_sum(vp);
        for (int pr = warp; 2 * pr < n; pr += NW) {
            const int i1 = pr, i2 = n - 1 - pr, len1 = i1 + 1, len = i1 == i2 ? len1 : n + 1;
            const float v1 = vv(i1), w1 = fmaf(-K, v1, s.pv()[i1]);
            const float v2 = vv(i2), w2 = fmaf(-K, v2, s.pv()[i2]);
            for (int t = lane; t < len; t += 32) {
                const bool first = t < len1;
                const int i = first ? i1 : i2, j = first ? t : t - len1;
                const float vi = first ? v1 : v2, wi = first ? w1 : w2;
                const float vj = vv(j), wj = fmaf(-K, vj, s.pv()[j]);
                s.G[k + 1 + i][k + 1 + j] -= fmaf(vi, wj, __fmul_rn(wi, vj));
            }
        }
        __syncthreads();
    }
    if (tid == 0) {
        s.lam()[P - 2] = s.G[P - 2][P - 2];
        s.lam()[P - 1] = s.G[P - 1][P - 1];
        s.off()[P - 2] = s.G[P - 1][P - 2];
        s.off()[P - 1] = 0.f;
    }
}

// Step 2: s.Z = H_0 ... H_{P-3} (H_k Z changes only the trailing block of
// rows and columns k+1 .. P-1 once the later reflections are in).
template <typename T, int P, int D, int NT>
__device__ void accumulate_q(FactorSmem<T, P, D> &s) {
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int e = tid; e < P * P; e += NT) s.Z[e / P][e % P] = e / P == e % P ? 1.f : 0.f;
    __syncthreads();
    for (int k = P - 3; k >= 0; --k) {
        const float beta = s.G[k][k + 1];
        if (beta == 0.f) continue;
        const int n = P - 1 - k;
        const float v0 = s.G[k][k + 2];
        auto vv = [&](int i) { return i == 0 ? v0 : s.G[k + 1 + i][k]; };
        // u = Z_S^T v (four lanes per column), then Z_S <- Z_S - beta v u^T
        for (int base = 8 * warp; base < n; base += NT / 4) {
            const int j = base + (lane >> 2);
            const float acc =
                quad_dot(n, j < n, [&](int i, float a) { return fmaf(vv(i), s.Z[k + 1 + i][k + 1 + j], a); });
            if ((lane & 3) == 0 && j < n) s.pv()[j] = beta * acc;
        }
        __syncthreads();
        for (int i = warp; i < n; i += NW) {
            const float vi = vv(i);
            for (int j = lane; j < n; j += 32) s.Z[k + 1 + i][k + 1 + j] = fmaf(-vi, s.pv()[j], s.Z[k + 1 + i][k + 1 + j]);
        }
        __syncthreads();
    }
}

// Step 3, run by one warp: the eigenvalues of the tridiagonal (lam, off)
// into lam, the rotations applied to the columns of s.Z (each lane its own
// rows).  Every lane computes the same scalar recurrence; lane 0 alone
// stores it (nothing in a pass reads back what the pass stored, and a
// __syncwarp publishes it before the next pass).  Shared-memory round trips
// stay off the recurrence: the search for the first negligible off-diagonal
// entry is one ballot, each lane carries the column it has just rotated in
// registers and loads the next one a rotation ahead.  Returns the rotations
// applied, or -1 once an eigenvalue took more than `max_it` QL iterations.
template <typename T, int P, int D>
__device__ int ql_implicit(FactorSmem<T, P, D> &s, int max_it) {
    constexpr int NR = (P + 31) / 32;  // rows of s.Z per lane
    const int lane = threadIdx.x & 31;
    float *d = s.lam(), *e = s.off();
    float tst = 0.f;
    int rotations = 0;
    for (int l = 0; l < P; ++l) {
        tst = fmaxf(tst, fabsf(d[l]) + fabsf(e[l]));
        for (int it = 0;; ++it) {
            // m: the first negligible off-diagonal entry from l on (e[P-1] = 0);
            // a NaN counts as negligible, as in a sequential scan
            int m = P - 1;
#pragma unroll
            for (int h = NR - 1; h >= 0; --h) {
                const int j = lane + 32 * h;
                const bool neg = j >= l && j < P - 1 && !(fabsf(e[j]) > QL_EPS * tst);
                const unsigned bal = __ballot_sync(0xffffffffu, neg);
                if (bal) m = 32 * h + __ffs(bal) - 1;
            }
            if (m == l) break;
            if (it == max_it) return -1;
            // shift: the eigenvalue of the leading 2 x 2 block nearer d[l]
            float g = __fsub_rn(d[l + 1], d[l]) / (2.f * e[l]);
            float r = sqrtf(fmaf(g, g, 1.f));
            g = __fadd_rn(__fsub_rn(d[m], d[l]), e[l] / __fadd_rn(g, copysignf(r, g)));
            float sn = 1.f, c = 1.f, p = 0.f;
            int i = m - 1;
            // d[i + 1], d[i] and e[i] of the coming rotation, and this lane's
            // entries of columns i + 1 (zc, rotated already in this pass)
            // and i (zi) of s.Z ride in registers (a rotation stores only
            // d[i + 1], e[i + 1] and column i + 1, which no later rotation of
            // the pass reads)
            float dn = d[m], di = d[m - 1], ei = e[m - 1];
            float zc[NR], zi[NR];
#pragma unroll
            for (int h = 0; h < NR; ++h) {
                const int row = lane + 32 * h;
                zc[h] = row < P ? s.Z[row][m] : 0.f;
                zi[h] = row < P ? s.Z[row][m - 1] : 0.f;
            }
            // unrolled so that the registers carried from one rotation to the
            // next are renamed instead of copied (a copy waits for the load
            // it moves): 720 K -> 611 K cycles of QL per 64 x 64 page job
#pragma unroll 4
            for (; i >= l; --i) {  // chase the bulge from the bottom of the block up
                const float di_next = i > l ? d[i - 1] : 0.f, ei_next = i > l ? e[i - 1] : 0.f;
                float zi_next[NR];
#pragma unroll
                for (int h = 0; h < NR; ++h) {
                    const int row = lane + 32 * h;
                    zi_next[h] = i > l && row < P ? s.Z[row][i - 1] : 0.f;
                }
                // every rounding is spelled out (no contraction left to the
                // compiler), so the recurrence gives the same bits however
                // the loop is scheduled
                const float f = __fmul_rn(sn, ei), b = __fmul_rn(c, ei);
                const float rr = fmaf(f, f, __fmul_rn(g, g));
                if (rr < NEGLIGIBLE * NEGLIGIBLE) {  // T splits: deflate and start again
                    if (lane == 0) e[i + 1] = sqrtf(rr);
                    break;
                }
                const float ir = rsqrtf(rr);  // one reciprocal square root gives r, sin and cos
                r = __fmul_rn(rr, ir);
                if (lane == 0) e[i + 1] = r;
                sn = __fmul_rn(f, ir);
                c = __fmul_rn(g, ir);
                g = __fsub_rn(dn, p);
                r = fmaf(__fsub_rn(di, g), sn, __fmul_rn(2.f * c, b));
                p = __fmul_rn(sn, r);
                if (lane == 0) d[i + 1] = __fadd_rn(g, p);
                g = fmaf(c, r, -b);
#pragma unroll
                for (int h = 0; h < NR; ++h) {
                    const int row = lane + 32 * h;
                    if (row < P) s.Z[row][i + 1] = fmaf(sn, zi[h], __fmul_rn(c, zc[h]));  // column i + 1 is final
                    zc[h] = fmaf(c, zi[h], -__fmul_rn(sn, zc[h]));                        // column i, carried
                    zi[h] = zi_next[h];
                }
                ++rotations;
                dn = di;
                di = di_next;
                ei = ei_next;
            }
#pragma unroll
            for (int h = 0; h < NR; ++h) {  // the carried column: i + 1 where the chase stopped
                const int row = lane + 32 * h;
                if (row < P) s.Z[row][i + 1] = zc[h];
            }
            if (lane == 0) {
                if (i >= l) {  // split at i + 1
                    d[i + 1] = __fsub_rn(d[i + 1], p);
                } else {
                    d[l] = __fsub_rn(d[l], p);
                    e[l] = g;
                }
                e[m] = 0.f;
            }
            __syncwarp();
        }
    }
    return rotations;
}

// ---------------------------------------------------------------- top-r eigenpairs
// A rank r <= P / 2 needs only the r largest eigenpairs (and every
// eigenvalue when the caller asks for the singular values), so the QL steps
// 2 and 3 above give way to three others that cost a fraction of them:
//   a. eigenvalues by multisection on Sturm counts (the number of negative
//      pivots of T - x I, formed by the recurrence q_i = (t_ii - x) -
//      t_{i-1,i}^2 / q_{i-1}, is the number of eigenvalues below x): one
//      warp per eigenvalue, 32 points a round, BIS_ROUNDS rounds from the
//      Gershgorin interval (33^6 > 2^30 subintervals, finer than fp32);
//   b. eigenvectors of T by inverse iteration: INV_ITERS solves with
//      T - lambda_k I by Gaussian elimination with partial pivoting, one
//      thread per vector, from fixed pseudo-random starts, each round
//      followed by modified Gram-Schmidt over the r vectors in descending
//      eigenvalue order, which keeps the vectors of a cluster of eigenvalues
//      apart;
//   c. the reflections applied to the r vectors: Y <- H_0 ... H_{P-3} Y.
// (Bisection on Sturm sequences: Barth, Martin and Wilkinson, "Calculation
// of the eigenvalues of a symmetric tridiagonal matrix by the method of
// bisection", 1967; inverse iteration: Wilkinson, "The Algebraic Eigenvalue
// Problem", 1965, ch. 5 and 9.)  As in the QL steps, every sum is taken by
// a fixed set of lanes in a fixed order and each eigenvalue and vector has
// its own warp or thread, so the block size does not change a bit.
constexpr int BIS_ROUNDS = 6;
constexpr int INV_ITERS = 3;
constexpr float PIVMIN = 1e-30f;  // a Sturm pivot at or below this counts as negative

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Entry i of start vector k: a fixed pseudo-random value in [-1, 1) (an
// integer hash of (i, k)).
__device__ __forceinline__ float start_entry(int i, int k) {
    uint32_t h = (uint32_t)i * 0x9E3779B1u + (uint32_t)k * 0x85EBCA77u + 0x165667B1u;
    h ^= h >> 15;
    h *= 0x2C1B3C6Du;
    h ^= h >> 12;
    return (float)(h & 0xFFFFFFu) * (1.f / 8388608.f) - 1.f;
}

// Step a for the NC eigenvalues k0 + u * NW (u < NC) of one warp, their
// multisection chains interleaved.
template <int P, int NW, int NC>
__device__ __forceinline__ void bisect_chains(const float *d, const float *e, float gl, float gu, int k0, float *out) {
    const int lane = threadIdx.x & 31;
    const float step = (float)(lane + 1) * (1.f / 33.f);
    float lo[NC], hi[NC];
#pragma unroll
    for (int u = 0; u < NC; ++u) {
        lo[u] = gl;
        hi[u] = gu;
    }
    for (int round = 0; round < BIS_ROUNDS; ++round) {
        float x[NC], q[NC];
        int c[NC];
#pragma unroll
        for (int u = 0; u < NC; ++u) {
            x[u] = fmaf(hi[u] - lo[u], step, lo[u]);
            q[u] = 1.f;
            c[u] = 0;
        }
#pragma unroll 2
        for (int i = 0; i < P; ++i) {
            const float di = d[i], e2 = i > 0 ? e[i - 1] * e[i - 1] : 0.f;
#pragma unroll
            for (int u = 0; u < NC; ++u) {
                const float t = fmaf(-e2, rcp_approx(q[u]), di - x[u]);
                const bool neg = t <= PIVMIN;
                c[u] += neg;
                q[u] = neg ? fminf(t, -PIVMIN) : t;
            }
        }
#pragma unroll
        for (int u = 0; u < NC; ++u) {  // the first point with more than j eigenvalues below it
            const int j = P - 1 - (k0 + u * NW);
            const unsigned bal = __ballot_sync(0xffffffffu, c[u] > j);
            const int a = bal ? __ffs(bal) - 1 : 32;
            const float xa = __shfl_sync(0xffffffffu, x[u], a & 31), xb = __shfl_sync(0xffffffffu, x[u], (a + 31) & 31);
            if (a < 32) hi[u] = xa;
            if (a > 0) lo[u] = xb;
        }
    }
    if (lane == 0)
#pragma unroll
        for (int u = 0; u < NC; ++u) out[k0 + u * NW] = 0.5f * (lo[u] + hi[u]);
}

// Step a: the nk largest eigenvalues of the tridiagonal (lam, off) into
// pv()[0 .. nk), descending.
template <typename T, int P, int D, int NT>
__device__ void eig_bisect(FactorSmem<T, P, D> &s, int nk) {
    constexpr int NW = NT / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *d = s.lam(), *e = s.off();
    float gl = INFINITY, gu = -INFINITY;
    for (int i = lane; i < P; i += 32) {
        const float a = (i > 0 ? fabsf(e[i - 1]) : 0.f) + (i < P - 1 ? fabsf(e[i]) : 0.f);
        gl = fminf(gl, d[i] - a);
        gu = fmaxf(gu, d[i] + a);
    }
    gl = -warp_max(-gl);
    gu = warp_max(gu);
    const float pad = fmaf(2e-6f, fmaxf(fabsf(gl), fabsf(gu)), 1e-30f);
    gl -= pad;
    gu += pad;
    for (int k0 = warp; k0 < nk; k0 += 4 * NW) {
        const int nc = min(4, (nk - k0 + NW - 1) / NW);
        if (nc == 4) bisect_chains<P, NW, 4>(d, e, gl, gu, k0, s.pv());
        else if (nc == 3) bisect_chains<P, NW, 3>(d, e, gl, gu, k0, s.pv());
        else if (nc == 2) bisect_chains<P, NW, 2>(d, e, gl, gu, k0, s.pv());
        else bisect_chains<P, NW, 1>(d, e, gl, gu, k0, s.pv());
    }
}

// Modified Gram-Schmidt over the r columns of Y (pitch yp), then unit
// length: column j loses its component along each earlier column k in turn.
template <int P, int NT>
__device__ void mgs_columns(float *Y, int yp, int r) {
    constexpr int NW = NT / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int k = 0; k < r - 1; ++k) {
        float nk = 0.f;  // |y_k|^2, every warp alike
        for (int i = lane; i < P; i += 32) nk = fmaf(Y[i * yp + k], Y[i * yp + k], nk);
        nk = warp_sum(nk);
        const float inv_nk = nk > 0.f ? 1.f / nk : 0.f;
        for (int j = k + 1 + warp; j < r; j += NW) {
            float dot = 0.f;
            for (int i = lane; i < P; i += 32) dot = fmaf(Y[i * yp + k], Y[i * yp + j], dot);
            const float c = warp_sum(dot) * inv_nk;
            for (int i = lane; i < P; i += 32) Y[i * yp + j] = fmaf(-c, Y[i * yp + k], Y[i * yp + j]);
        }
        __syncthreads();
    }
    for (int k = warp; k < r; k += NW) {
        float n2 = 0.f;
        for (int i = lane; i < P; i += 32) n2 = fmaf(Y[i * yp + k], Y[i * yp + k], n2);
        n2 = warp_sum(n2);
        const float sc = n2 > 0.f ? 1.f / sqrtf(n2) : 0.f;
        for (int i = lane; i < P; i += 32) Y[i * yp + k] *= sc;
    }
    __syncthreads();
}

// Step b: eigenvectors of the tridiagonal for the eigenvalues pv()[0 .. r)
// into the columns of Y (P x r, pitch yp).  Each solve factors
// T - lambda_k I = Pm L U by Gaussian elimination with partial pivoting
// (rows i and i + 1 swap when the entry below the pivot is larger; U then
// has a second superdiagonal, t_{i+1,i+2} at a swapped row), with b carried
// along, then back-substitutes.  The swap bits stay in the solving thread's
// registers and SC (P x r floats, pitch r) keeps one float per row: the
// multiplier of a swapped row, else the reciprocal pivot.  The back
// substitution recomputes the rest from the tridiagonal, bit for bit: a
// swapped row's pivot is t_{i+1,i} and its superdiagonal t_{i+1,i+1} -
// lambda; an unswapped row's superdiagonal is t_{i,i+1}, times minus the
// multiplier of row i - 1 if that one swapped.  A pivot below |T| 2^-23 is
// moved out to that size.  Rows swap whenever the entry below is the larger
// one and above 1e-30 (so that its reciprocal stays finite), however small:
// the trailing block of a page of rank r or less holds entries near the
// fp32 resolution of |T|, and without the swaps the cluster of eigenvalues
// there came out as a poorer basis of its subspace.
template <typename T, int P, int D, int NT>
__device__ void eig_vectors(FactorSmem<T, P, D> &s, int r, float *Y, int yp, float *SC) {
    static_assert(P <= 64, "swap bits of one solve in 64 bits");
    const int tid = threadIdx.x;
    const float *d = s.lam(), *e = s.off(), *lam = s.pv();
    for (int x = tid; x < P * r; x += NT) Y[(x / r) * yp + x % r] = start_entry(x / r, x % r);
    float tiny = 0.f;
    if (tid < r) {
        float tn = 0.f;
        for (int i = 0; i < P; ++i)
            tn = fmaxf(tn, fabsf(d[i]) + (i > 0 ? fabsf(e[i - 1]) : 0.f) + (i < P - 1 ? fabsf(e[i]) : 0.f));
        tiny = fmaxf(tn * 1.1920929e-7f, 1e-30f);
    }
    __syncthreads();
    for (int it = 0; it < INV_ITERS; ++it) {
        if (tid < r) {
            const int k = tid;
            const float lk = lam[k];
            auto moved = [&](float x) { return fabsf(x) < tiny ? (x < 0.f ? -tiny : tiny) : x; };
            // row i of the elimination: pivot cd, superdiagonal cu, right side cb
            float cd = d[0] - lk, cu = e[0], cb = Y[k];
            unsigned long long swaps = 0ull;
            for (int i = 0; i < P - 1; ++i) {
                const float sub = e[i], nd = d[i + 1] - lk, nu = i + 1 < P - 1 ? e[i + 1] : 0.f;
                const float nbv = Y[(i + 1) * yp + k];
                const bool sw = fabsf(sub) > fmaxf(fabsf(cd), 1e-30f);  // 1 / sub stays finite
                const float ip = rcp_approx(sw ? sub : moved(cd));
                const float f = (sw ? cd : sub) * ip;
                SC[i * r + k] = sw ? f : ip;
                Y[i * yp + k] = sw ? nbv : cb;
                swaps |= (unsigned long long)sw << i;
                const float a = sw ? cu : nd, bq = sw ? nd : cu;
                const float b0 = sw ? cb : nbv, b1 = sw ? nbv : cb;
                cd = fmaf(-f, bq, a);
                cu = sw ? -f * nu : nu;
                cb = fmaf(-f, b1, b0);
            }
            const float ipl = rcp_approx(moved(cd));
            // back substitution: y_i = (b_i - u1_i y_{i+1} - u2_i y_{i+2}) / u_ii,
            // u2_i = t_{i+1,i+2} where rows i and i + 1 swapped
            float y1 = cb * ipl, y2 = 0.f, amax = fabsf(y1);
            Y[(P - 1) * yp + k] = y1;
            float sl = SC[(P - 2) * r + k];
            for (int i = P - 2; i >= 0; --i) {
                const bool sw = (swaps >> i) & 1ull, swp = i > 0 && ((swaps >> (i - 1)) & 1ull);
                const float slp = i > 0 ? SC[(i - 1) * r + k] : 0.f;
                const float ip = sw ? rcp_approx(e[i]) : sl;
                const float u1 = sw ? d[i + 1] - lk : (swp ? -slp * e[i] : e[i]);
                const float u2 = sw ? e[i + 1] : 0.f;
                const float y = fmaf(-u1, y1, fmaf(-u2, y2, Y[i * yp + k])) * ip;
                Y[i * yp + k] = y;
                amax = fmaxf(amax, fabsf(y));
                y2 = y1;
                y1 = y;
                sl = slp;
            }
            // scaled to max |y| in [1, 2) by a power of two; a vector that
            // overflowed or vanished starts again from the unit vector e_k
            const bool ok = amax > 0.f && amax < INFINITY;
            const float sc = ok ? ldexpf(1.f, -ilogbf(amax)) : 0.f;
            for (int i = 0; i < P; ++i) Y[i * yp + k] = ok ? Y[i * yp + k] * sc : (i == k ? 1.f : 0.f);
        }
        __syncthreads();
        mgs_columns<P, NT>(Y, yp, r);
    }
}

// Step c: Y <- H_0 H_1 ... H_{P-3} Y, a warp per column (four columns of a
// warp interleaved); the reflections are read from s.G as the reduction left
// them.  They go two at a time, H_{m-1} H_m: with a = v_m^T y, b =
// v_{m-1}^T y and c = v_{m-1}^T v_m, one pass of sums gives
// y <- y - v_m (beta_m a) - v_{m-1} beta_{m-1} (b - c beta_m a),
// so the warp waits on one reduction per pair instead of one per reflection.
template <typename T, int P, int D, int NT>
__device__ void apply_reflections(FactorSmem<T, P, D> &s, float *Y, int yp, int r) {
    constexpr int NW = NT / 32, CW = 4;
    static_assert((P - 2) % 2 == 0, "the reflections pair up");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int k0 = warp; k0 < r; k0 += CW * NW) {
        for (int m = P - 3; m >= 1; m -= 2) {
            // H_m acts on rows m + 1 .., H_{m-1} on rows m ..; beta 0: no reflection
            const float b1 = s.G[m][m + 1], b0 = s.G[m - 1][m];
            if (b1 == 0.f && b0 == 0.f) continue;
            const float v1_0 = s.G[m][m + 2], v0_0 = s.G[m - 1][m + 1];
            // entries at absolute row R of v_m (R >= m + 1) and v_{m-1} (R >= m)
            auto v1 = [&](int R) { return R == m + 1 ? v1_0 : (R > m + 1 ? s.G[R][m] : 0.f); };
            auto v0 = [&](int R) { return R == m ? v0_0 : s.G[R][m - 1]; };
            float a[CW], b[CW], c = 0.f;
#pragma unroll
            for (int u = 0; u < CW; ++u) a[u] = b[u] = 0.f;
            for (int R = m + lane; R < P; R += 32) {
                const float x1 = v1(R), x0 = v0(R);
                c = fmaf(x0, x1, c);
#pragma unroll
                for (int u = 0; u < CW; ++u)
                    if (k0 + u * NW < r) {
                        const float yv = Y[R * yp + k0 + u * NW];
                        a[u] = fmaf(x1, yv, a[u]);
                        b[u] = fmaf(x0, yv, b[u]);
                    }
            }
            c = warp_sum(c);
            float t1[CW], t0[CW];
#pragma unroll
            for (int u = 0; u < CW; ++u) {
                t1[u] = b1 * warp_sum(a[u]);
                t0[u] = b0 * fmaf(-c, t1[u], warp_sum(b[u]));
            }
            for (int R = m + lane; R < P; R += 32) {
                const float x1 = v1(R), x0 = v0(R);
#pragma unroll
                for (int u = 0; u < CW; ++u)
                    if (k0 + u * NW < r) {
                        float &yv = Y[R * yp + k0 + u * NW];
                        yv = fmaf(-t0[u], x0, fmaf(-t1[u], x1, yv));
                    }
            }
        }
    }
    __syncthreads();
}

template <typename TO>
__device__ __forceinline__ void store_elem(char *base, size_t idx, float v) {
    reinterpret_cast<TO *>(base)[idx] = Elem<TO>::from_f32(v);
}

// INT4 record of one page's key or value factors [PuzzleKV §4.3], from the
// kept eigenvectors L (the first r columns of s.G, unit length) and the page
// X (s.X):
//   1. R = L^T X in fp32, written over X as Rf[rp][D] (X is read first; the
//      validated ranks keep rp <= P/2, so Rf fits in X's bf16 storage);
//   2. sigma_j = |row j of R| (R's rows are orthogonal: L holds eigenvectors),
//      Lt = L sigma^{1/2}, Rt = sigma^{-1/2} R (zero where sigma_j = 0);
//   3. one fp16 scale per group, max|x| / 7 rounded to fp16: columns of L_K
//      and of R_K / R_V (head-dim columns), rows of L_V (tokens), stored in
//      accumulator-column order (q4_scale_index; the head-dim vectors in
//      k-step order, q4_dscale_index);
//   4. codes round(x / scale) (IEEE division, round half to even) clamped to
//      [-7, 7], stored as code + 8 in the key or value stream's tensor-core
//      operand order (q4_operand_elem), one 32-bit word per thread step.
template <typename T, int P, int D, int NT>
__device__ void write_q4_record(FactorSmem<T, P, D> &s, const JobView &v, const Layout &y) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int NW = NT / 32;
    const int r = v.r, rp = v.kind == 0 ? y.rkp : y.rvp;
    static_assert(NT % D == 0, "one head-dim column per thread of a group");
    constexpr int GROUPS = NT / D, QMAX = (P / 2 + GROUPS - 1) / GROUPS;
    constexpr int PITCH = D * (int)sizeof(T);
    // 1. projection
    {
        const int k = tid % D, grp = tid / D;
        float acc[QMAX];
#pragma unroll
        for (int u = 0; u < QMAX; ++u) acc[u] = 0.f;
        for (int i = 0; i < P; ++i) {
            const float xv = Elem<T>::load(reinterpret_cast<const T *>(s.X + swz_offset(i, k * (int)sizeof(T), PITCH)));
#pragma unroll
            for (int u = 0; u < QMAX; ++u) {
                const int j = grp + u * GROUPS;
                if (j < r) acc[u] = fmaf(s.G[i][j], xv, acc[u]);
            }
        }
        __syncthreads();  // every thread is done with X
        float *Rf = reinterpret_cast<float *>(s.X);
#pragma unroll
        for (int u = 0; u < QMAX; ++u) {
            const int j = grp + u * GROUPS;
            if (j < rp) Rf[j * D + k] = j < r ? acc[u] : 0.f;
        }
    }
    __syncthreads();
    float *Rf = reinterpret_cast<float *>(s.X);
    // 2. sigma^{1/2} per rank (one warp per row, fixed summation order)
    for (int j = warp; j < rp; j += NW) {
        float a = 0.f;
        for (int k = lane; k < D; k += 32) a = fmaf(Rf[j * D + k], Rf[j * D + k], a);
        a = warp_sum(a);
        if (lane == 0) s.lam()[j] = sqrtf(sqrtf(a));
    }
    __syncthreads();
    for (int e = tid; e < P * rp; e += NT) {
        const int i = e / rp, j = e % rp;
        const float rs = s.lam()[j];
        s.G[i][j] = (j < r && rs > 0.f) ? s.G[i][j] * rs : 0.f;
    }
    for (int e = tid; e < rp * D; e += NT) {
        const float rs = s.lam()[e / D];
        Rf[e] = rs > 0.f ? Rf[e] / rs : 0.f;
    }
    __syncthreads();
    if (v.qL)  // the absorbed factors the codes below quantize
        for (int e = tid; e < P * rp; e += NT) v.qL[e] = s.G[e / rp][e % rp];
    if (v.qR)
        for (int e = tid; e < rp * D; e += NT) v.qR[e] = Rf[e];
    // 3. scales: fp16 in the record (accumulator-column order, the head-dim
    // vectors in k-step order), their fp32 values in the scratch for the
    // codes (sigma^{1/2} above is dead by now)
    float *scL = s.sc();       // per rank (keys) or per token (values): up to P
    float *scR = scL + P;      // per head-dim column: D
    unsigned char *rec = reinterpret_cast<unsigned char *>(v.rec);
    __half *hL = reinterpret_cast<__half *>(rec + (v.kind == 0 ? y.q_off_sLK : y.q_off_sLV));
    __half *hR = reinterpret_cast<__half *>(rec + (v.kind == 0 ? y.q_off_sRK : y.q_off_sRV));
    if (v.kind == 0) {
        for (int j = tid; j < rp; j += NT) {  // L_K column-wise
            float m = 0.f;
            for (int i = 0; i < P; ++i) m = fmaxf(m, fabsf(s.G[i][j]));
            const __half h = __float2half_rn(m / 7.f);
            hL[q4_scale_index(rp, j)] = h;
            scL[j] = __half2float(h);
        }
    } else {
        for (int i = tid; i < P; i += NT) {  // L_V row-wise
            float m = 0.f;
            for (int j = 0; j < rp; ++j) m = fmaxf(m, fabsf(s.G[i][j]));
            const __half h = __float2half_rn(m / 7.f);
            hL[q4_scale_index(P, i)] = h;
            scL[i] = __half2float(h);
        }
    }
    for (int k = tid; k < D; k += NT) {  // R_K and R_V column-wise
        float m = 0.f;
        for (int j = 0; j < rp; ++j) m = fmaxf(m, fabsf(Rf[j * D + k]));
        const __half h = __float2half_rn(m / 7.f);
        hR[q4_dscale_index(k)] = h;
        scR[k] = __half2float(h);
    }
    __syncthreads();
    // 4. codes: the key stream holds R_K as B[head dim][rank] then L_K as
    // B[rank][token]; the value stream L_V as B[token][rank] then R_V as
    // B[rank][head dim] (tensor-core operand order, see layout.h)
    auto q = [](float x, float sc) -> uint32_t {
        int c = sc > 0.f ? (int)rintf(x / sc) : 0;
        c = c < -7 ? -7 : (c > 7 ? 7 : c);
        return (uint32_t)(c + 8);
    };
    const int K0 = v.kind == 0 ? D : P, K1 = v.kind == 0 ? P : D;
    const int regs1 = q4_operand_regs(K0, rp), regs = regs1 + q4_operand_regs(rp, K1);
    auto code_of = [&](int m, int ln, int e) -> uint32_t {
        int k, n;
        if (m >= regs) return 8u;
        if (m < regs1) {
            q4_operand_elem(K0, rp, m, ln, e, k, n);
            return v.kind == 0 ? q(Rf[n * D + k], scR[k]) : q(s.G[k][n], scL[k]);
        }
        q4_operand_elem(rp, K1, m - regs1, ln, e, k, n);
        return v.kind == 0 ? q(s.G[n][k], scL[k]) : q(Rf[k * D + n], scR[n]);
    };
    uint32_t *words = reinterpret_cast<uint32_t *>(rec + (v.kind == 0 ? 0 : y.q_off_V));
    const int nwords = (v.kind == 0 ? y.q_kslabs : y.q_vslabs) * 64;
    for (int wi = tid; wi < nwords; wi += NT) {  // word wi: slab wi / 64, lane (wi % 64) / 2
        const int ln = (wi & 63) >> 1, w = 2 * (wi >> 6) + (wi & 1);
        uint32_t word = 0;
#pragma unroll
        for (int nu = 0; nu < 8; ++nu) word |= code_of(4 * w + (nu & 3), ln, nu >> 2) << (4 * nu);
        words[wi] = word;
    }
}

// Returns the QL rotations the page took (0 for a rank up to P / 2, which
// takes no QL, and if an eigenvalue hit the iteration cap, which the status
// word records).
template <typename T, int P, int D, int NT>
__device__ int factorize_one(FactorSmem<T, P, D> &s, const FactorParams &fp, long job) {
    const int tid = threadIdx.x, lane = tid & 31;
    const JobView v = job_view(fp, job);
    load_page<T, P, D, NT>(s, v);
    __syncthreads();
    if constexpr (sizeof(T) == 2) gram_bf16<P, D, NT>(s); else gram_f32<P, D, NT>(s);
    __syncthreads();
    // the tensor-core tiles of (i, j) and (j, i) may round differently:
    // symmetrise; and scale by a power of two (exact) that brings the largest
    // diagonal entry into [1, 2), so that no square in the eigensolve can
    // overflow
    float mx = 0.f;
    for (int i = lane; i < P; i += 32) mx = fmaxf(mx, s.G[i][i]);
    mx = warp_max(mx);
    const int ex = mx > 0.f ? ilogbf(mx) : 0;
    for (int e = tid; e < P * P; e += NT) {
        int i = e / P, j = e % P;
        if (j >= i) {
            const float g = ldexpf(s.G[i][j], -ex);
            s.G[i][j] = g;
            s.G[j][i] = g;
        }
    }
    __syncthreads();
    tridiagonalize<T, P, D, NT>(s);
    const int r = v.r;
    int rotations = 0;
    if (2 * r <= P) {  // the top r eigenpairs alone (steps a-c); X is dead here
        __syncthreads();
        eig_bisect<T, P, D, NT>(s, v.sigma ? P : r);
        __syncthreads();
        // Y (P x r, odd pitch) and the solves' scratch (P x r) in the
        // P x (P + 1) floats of s.Z: P (2r + 1) fits as r <= P / 2
        float *Y = &s.Z[0][0];
        const int yp = r | 1;
        eig_vectors<T, P, D, NT>(s, r, Y, yp, Y + P * yp);
        apply_reflections<T, P, D, NT>(s, Y, yp, r);
        if (v.sigma)
            for (int k = tid; k < P; k += NT) v.sigma[k] = sqrtf(fmaxf(ldexpf(s.pv()[k], ex), 0.f));
        for (int x = tid; x < P * r; x += NT) s.G[x / r][x % r] = Y[(x / r) * yp + x % r];
        __syncthreads();
    } else {
        accumulate_q<T, P, D, NT>(s);  // starts with a barrier; X is dead here (the page comes back below)
        if (tid < 32) {
            const int rot = ql_implicit<T, P, D>(s, fp.max_ql_iter);
            if (tid == 0) s.off()[0] = __int_as_float(rot);  // the off-diagonal is dead after QL
        }
        __syncthreads();
        rotations = __float_as_int(s.off()[0]);
        if (rotations < 0 && tid == 0 && fp.status) atomicAdd(fp.status + STATUS_NOT_CONVERGED, 1);
        // each thread t < P ranks eigenvalue t (descending, ties: lower index
        // first; a NaN ranks below every number, so the ranks stay a
        // permutation) and moves eigenvector t into column rank(t) of G
        if (tid < P) {
            auto key = [](float x) { return x == x ? x : -INFINITY; };
            const float li = key(s.lam()[tid]);
            int rank = 0;
            for (int j = 0; j < P; ++j) {
                const float lj = key(s.lam()[j]);
                rank += (lj > li) || (lj == li && j < tid);
            }
            if (v.sigma) v.sigma[rank] = sqrtf(fmaxf(ldexpf(s.lam()[tid], ex), 0.f));
            for (int i = 0; i < P; ++i) s.G[i][rank] = s.Z[i][tid];
        }
        __syncthreads();
    }
    // the eigenvectors are out: the page again, for the projection (the
    // barriers below order it before its first read)
    load_page<T, P, D, NT>(s, v);
    // A few thousand fp32 rotations leave the eigenvector norms off by about
    // 1e-6; scale the kept columns back to unit length (their mutual
    // orthogonality is at the same level).
    if (tid < v.r) {
        float n2 = 0.f;
        for (int i = 0; i < P; ++i) n2 = fmaf(s.G[i][tid], s.G[i][tid], n2);
        s.lam()[tid] = n2 > 0.f ? 1.f / sqrtf(n2) : 1.f;  // the eigenvalues are no longer needed
    }
    __syncthreads();
    for (int e = tid; e < P * v.r; e += NT) {
        int i = e / v.r, j = e % v.r;
        s.G[i][j] *= s.lam()[j];
    }
    __syncthreads();

    const Layout &y = fp.y;
    const bool rec = v.rec != nullptr;
    if (rec && y.q4) {
        write_q4_record<T, P, D, NT>(s, v, y);
        return rotations < 0 ? 0 : rotations;
    }
    const int rp = rec ? (v.kind == 0 ? y.rkp : y.rvp) : r;
    // L = Q_r  (record: keys LK[token][rank], values LVt[rank][token])
    for (int e = tid; e < P * rp; e += NT) {
        int i = e / rp, j = e % rp;
        float val = j < r ? s.G[i][j] : 0.f;
        if (rec) {
            using TS = T;
            if (v.kind == 0)
                *swz_ptr<TS>(v.rec, i, j, rp) = Elem<TS>::from_f32(val);
            else
                *swz_ptr<TS>(v.rec + y.off_LV, j, i, P) = Elem<TS>::from_f32(val);
        } else if (fp.out_esz == 2) {
            store_elem<__nv_bfloat16>(v.L, (size_t)i * r + j, val);
        } else {
            store_elem<float>(v.L, (size_t)i * r + j, val);
        }
    }
    // R = Q_r^T X in fp32: thread -> head-dim column k, a group of ranks
    constexpr int PITCH = D * (int)sizeof(T);
    constexpr int GROUPS = NT / D;
    const int k = tid % D, grp = tid / D;
    for (int j0 = grp; j0 < rp; j0 += GROUPS * 8) {
        float acc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = 0.f;
        for (int i = 0; i < P; ++i) {
            float xv = Elem<T>::load(reinterpret_cast<const T *>(s.X + swz_offset(i, k * (int)sizeof(T), PITCH)));
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                int j = j0 + u * GROUPS;
                if (j < r) acc[u] = fmaf(s.G[i][j], xv, acc[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            int j = j0 + u * GROUPS;
            if (j >= rp) continue;
            float val = j < r ? acc[u] : 0.f;
            if (rec) {
                if (v.kind == 0)
                    *swz_ptr<T>(v.rec + y.off_RK, j, k, D) = Elem<T>::from_f32(val);
                else
                    *swz_ptr<T>(v.rec + y.off_RV, k, j, rp) = Elem<T>::from_f32(val);
            } else if (fp.out_esz == 2) {
                store_elem<__nv_bfloat16>(v.R, (size_t)j * D + k, val);
            } else {
                store_elem<float>(v.R, (size_t)j * D + k, val);
            }
        }
    }
    return rotations < 0 ? 0 : rotations;
}

// The 256-thread variant keeps four CTAs per SM (64 registers): while one
// CTA's warps wait on a serial recurrence (a Sturm count, a solve, the QL
// chase) or a barrier, the other CTAs' reductions and updates fill the SM.
template <typename T, int P, int D, int NT>
__global__ void __launch_bounds__(NT, NT == 256 ? 4 : 1) factorize_kernel(const FactorParams fp) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    auto &s = *reinterpret_cast<FactorSmem<T, P, D> *>(smem_raw);
    unsigned long long jobs = 0, rotations = 0;
    for (long job = blockIdx.x; job < fp.n_jobs; job += gridDim.x) {
        rotations += (unsigned long long)factorize_one<T, P, D, NT>(s, fp, job);
        ++jobs;
        __syncthreads();
    }
    if (threadIdx.x == 0 && fp.status && jobs) {  // throughput accounting, once per CTA
        atomicAdd(reinterpret_cast<unsigned long long *>(fp.status + STATUS_JOBS), jobs);
        atomicAdd(reinterpret_cast<unsigned long long *>(fp.status + STATUS_ROTATIONS), rotations);
    }
}

template <typename T, int P, int D, int NT>
static cudaError_t launch_t(const FactorParams &fp, int num_sms, cudaStream_t st) {
    const size_t smem = sizeof(FactorSmem<T, P, D>);
    auto k = factorize_kernel<T, P, D, NT>;
    // the shared-memory opt-in is set once per device (per launch it costs
    // more host time than a small launch takes on the GPU)
    static std::atomic<int> attr_state[64];  // 0 = not set, 1 = set, 2 + error = failed
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int state = attr_state[dev].load(std::memory_order_acquire);
    if (state == 0) {
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        // the largest shared split, as the decode kernels ask: an SM set up
        // by either kernel then takes CTAs of the other beside its own
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        state = e == cudaSuccess ? 1 : 2 + (int)e;
        attr_state[dev].store(state, std::memory_order_release);
    }
    if (state != 1) return (cudaError_t)(state - 2);
    long blocks = fp.n_jobs;
    const long cap = fp.max_ctas > 0 ? fp.max_ctas : (long)num_sms * (NT >= 1024 ? 2 : 8);
    if (blocks > cap) blocks = cap;
    if (blocks < 1) return cudaSuccess;
    k<<<(unsigned)blocks, NT, smem, st>>>(fp);
    return cudaGetLastError();
}

// A few pages (conversions during decoding) are latency-bound: 1024 threads
// per page.  Many pages (prefill, batches) are throughput-bound: 256 threads,
// several pages per SM.  Background batches, which run between and beside
// decode launches (max_ctas set: one CTA per page job), never take 1024
// threads, which hold all of an SM's registers: a 256-thread CTA has 64
// registers and 36 KB of shared memory at P = 64, d = 128, bf16.  All
// variants give the same bits.
template <typename T, int P, int D>
static cudaError_t launch_nt(const FactorParams &fp, int num_sms, cudaStream_t st) {
    if (fp.n_jobs <= 2L * num_sms && fp.max_ctas <= 0) return launch_t<T, P, D, 1024>(fp, num_sms, st);
    return launch_t<T, P, D, 256>(fp, num_sms, st);
}

cudaError_t launch_factorize(const FactorParams &fp, int num_sms, cudaStream_t st) {
    if (fp.n_jobs <= 0) return cudaSuccess;
    const bool bf = fp.x_esz == 2;
#define PKV_FACT_CASE(PP, DD)                                                                    \
    if (fp.P == PP && fp.d == DD)                                                                \
        return bf ? launch_nt<__nv_bfloat16, PP, DD>(fp, num_sms, st) : launch_nt<float, PP, DD>(fp, num_sms, st);
    PKV_FACT_CASE(16, 64)
    PKV_FACT_CASE(32, 64)
    PKV_FACT_CASE(64, 64)
    PKV_FACT_CASE(16, 128)
    PKV_FACT_CASE(32, 128)
    PKV_FACT_CASE(64, 128)
#undef PKV_FACT_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkv
