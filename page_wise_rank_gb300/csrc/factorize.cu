// Batched page factorization: one CTA per page.
//
// "PuzzleKV: Page-Wise Low-Rank Decomposition for KV Cache Compression",
// §3.3 ③ and eq. (2): for a P x d page X (P < d) the left singular subspace
// comes from the P x P Gram matrix G = X X^T; L = top-r eigenvectors Q_r,
// R = Q_r^T X.  Per CTA:
//   1. X -> shared memory (bf16 rows in the swizzled layout, or fp32 rows);
//   2. G = X X^T in fp32: bf16 pages on tensor cores (mma.sync m16n8k16,
//      bf16 products are exact in fp32), fp32 pages on CUDA cores;
//   3. cyclic Jacobi on G with the round-robin (circle) pairing: each round
//      rotates P/2 disjoint pairs at once (2x2 blocks of G, pairs of
//      eigenvector rows); a sweep is P-1 rounds; stop after a sweep with no
//      rotation (relative threshold), or at the cap;
//   4. eigenvalues ranked descending (ties: lower index first);
//   5. L = Q_r, R = Q_r^T X in fp32, written as bf16 or fp32 into either a
//      factor record (swizzled store layout) or plain row-major arrays.
#include <cuda_fp16.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace pkv {

constexpr float JACOBI_TOL = 1e-6f;
// Stop the eigensolve once the kept subspace could gain at most this fraction
// of the energy it leaves out (reconstruction error excess about half of it:
// 5e-5, twenty times inside the 1e-3 bound on the excess).
constexpr float SUBSPACE_TOL = 1e-4f;

template <typename T, int P, int D>
struct FactorSmem {
    alignas(128) unsigned char X[P * D * sizeof(T)];  // swizzled rows, pitch D * sizeof(T)
    float G[P][P + 1];  // Gram matrix; after the eigensolve reused for Q[i][j] = Vt[order[j]][i]
    alignas(16) float Vt[P][P + 4];  // eigenvectors, one per row (rows stay 16-byte aligned)
    float4 pair[P / 2];              // per pair of the round: (p, q as int bits, cos, sin)
    float tn[P / 2];                 // tan of the pair's angle (0: no rotation)
    float lam[P];
    int order[P];
    float red[64];                   // per-warp partial sums (up to 32 warps, two sums)
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

// Cyclic Jacobi eigensolve of the symmetric P x P matrix in s.G (upper
// triangle, G[i][j] with i <= j, is the matrix); eigenvectors accumulate as
// the rows of s.Vt.  Returns the number of sweeps, or -1 at the cap.  A round
// rotates the P/2 disjoint pairs of the round-robin (circle) pairing at once:
// phase A computes the angles, phase B applies G <- J^T G J to the 2x2
// blocks of the upper triangle (each thread keeps its blocks for the whole
// solve) and rotates pairs of eigenvector rows with 16-byte vectors.  Blocks
// and rows of pairs that did not rotate are left alone.
// Energy the top-r subspace of the current diagonal can still gain, over the
// energy it leaves out: for every pair (i among the r largest diagonal
// entries, j among the rest) the exact gain of the 2 x 2 rotation,
// sqrt(h^2 + g_ij^2) - |h| with h = (g_ii - g_jj) / 2, summed, over the sum of
// the left-out diagonal.  Uses s.order (free during the solve) and s.red;
// every thread gets the result.
template <typename T, int P, int D, int NT>
__device__ float subspace_gain(FactorSmem<T, P, D> &s, int r) {
    const int tid = threadIdx.x;
    if (tid < P) {  // rank of each diagonal entry, descending (ties: lower index first)
        const float di = s.G[tid][tid];
        int rk = 0;
        for (int j = 0; j < P; ++j) {
            const float dj = s.G[j][j];
            rk += (dj > di) || (dj == di && j < tid);
        }
        s.order[rk] = tid;
    }
    __syncthreads();
    float gain = 0.f, left = 0.f;
    for (int e = tid; e < r * (P - r); e += NT) {
        const int i = s.order[e / (P - r)], j = s.order[r + e % (P - r)];
        const float h = 0.5f * (s.G[i][i] - s.G[j][j]);
        const float g = i < j ? s.G[i][j] : s.G[j][i];
        const float rad = sqrtf(fmaf(h, h, g * g));
        gain += rad > 0.f ? g * g / (rad + fabsf(h)) : 0.f;
    }
    for (int k = r + tid; k < P; k += NT) left += s.G[s.order[k]][s.order[k]];
    // block sums: warp shuffles, then one value per warp in s.lam
    gain = warp_sum(gain);
    left = warp_sum(left);
    const int warp = tid >> 5, lane = tid & 31;
    static_assert(NT / 32 <= 32, "two partial sums per warp in s.red");
    if (lane == 0) {
        s.red[warp] = gain;
        s.red[32 + warp] = left;
    }
    __syncthreads();
    float gs = 0.f, ls = 0.f;  // every thread sums the same values in the same order
    for (int w = 0; w < NT / 32; ++w) {
        gs += s.red[w];
        ls += s.red[32 + w];
    }
    __syncthreads();
    return ls > 0.f ? gs / ls : (gs > 0.f ? INFINITY : 0.f);
}

template <typename T, int P, int D, int NT>
__device__ int jacobi(FactorSmem<T, P, D> &s, int max_sweeps, int r) {
    constexpr int NP = P / 2;
    constexpr int NBLK = NP * (NP + 1) / 2;
    constexpr int BPT = (NBLK + NT - 1) / NT;  // blocks per thread
    constexpr int V4 = P / 4;                  // float4 per eigenvector row
    const int tid = threadIdx.x;
    for (int e = tid; e < P * P; e += NT) s.Vt[e / P][e % P] = (e / P == e % P) ? 1.f : 0.f;
    int my_al[BPT], my_be[BPT];
#pragma unroll
    for (int i = 0; i < BPT; ++i) {  // block e = tid + i * NT of the row-major upper triangle
        int e = tid + i * NT, be = 0;
        if (e < NBLK) {
            while ((be + 1) * (be + 2) / 2 <= e) ++be;
            my_al[i] = e - be * (be + 1) / 2;
            my_be[i] = be;
        } else {
            my_al[i] = my_be[i] = -1;
        }
    }
    const float tol2 = JACOBI_TOL * JACOBI_TOL;
    __syncthreads();
    for (int sweep = 0; sweep < max_sweeps; ++sweep) {
        int rotated_any = 0;
        for (int round = 0; round < P - 1; ++round) {
            // Phase A: slot 0 holds index 0, slot i >= 1 holds 1 + (i - 1 - round) mod (P - 1);
            // slot k meets slot P - 1 - k.
            int rot = 0;
            if (tid < NP) {
                int k = tid;
                int a = k == 0 ? 0 : 1 + ((k - 1 - round + 2 * (P - 1)) % (P - 1));
                int kb = P - 1 - k;
                int b = 1 + ((kb - 1 - round + 2 * (P - 1)) % (P - 1));
                int p = a < b ? a : b, q = a < b ? b : a;
                float gpp = s.G[p][p], gqq = s.G[q][q], gpq = s.G[p][q];
                float c = 1.f, sn = 0.f, t = 0.f;
                if (gpq * gpq > tol2 * fabsf(gpp * gqq) && gpq != 0.f) {
                    // tan of the angle that zeroes G_pq: smaller root of t^2 + 2 zeta t - 1 = 0
                    float zeta = __fdividef(gqq - gpp, 2.f * gpq);
                    float z2 = fmaf(zeta, zeta, 1.f);
                    t = copysignf(__fdividef(1.f, fabsf(zeta) + z2 * rsqrtf(z2)), zeta);
                    if (fabsf(zeta) > 1e18f) t = __fdividef(0.5f, zeta);  // z2 overflows
                    c = rsqrtf(fmaf(t, t, 1.f));
                    sn = t * c;
                    rot = 1;
                }
                s.pair[k] = make_float4(__int_as_float(p), __int_as_float(q), c, sn);
                s.tn[k] = t;
            }
            rotated_any |= __syncthreads_or(rot);
            // Phase B1: 2x2 blocks of the upper triangle of G
#pragma unroll
            for (int i = 0; i < BPT; ++i) {
                const int al = my_al[i], be = my_be[i];
                if (al < 0) continue;
                const float4 A = s.pair[al];
                const int pa = __float_as_int(A.x), qa = __float_as_int(A.y);
                if (al == be) {
                    const float t = s.tn[al];
                    if (t != 0.f) {
                        const float g00 = s.G[pa][pa], g01 = s.G[pa][qa], g11 = s.G[qa][qa];
                        s.G[pa][pa] = g00 - t * g01;
                        s.G[qa][qa] = g11 + t * g01;
                        s.G[pa][qa] = 0.f;
                    }
                    continue;
                }
                const float4 B = s.pair[be];
                if (A.w == 0.f && B.w == 0.f) continue;
                const int pb = __float_as_int(B.x), qb = __float_as_int(B.y);
                // element (x, y) of the symmetric matrix lives at G[min][max]
                float *e00 = pa < pb ? &s.G[pa][pb] : &s.G[pb][pa];
                float *e01 = pa < qb ? &s.G[pa][qb] : &s.G[qb][pa];
                float *e10 = qa < pb ? &s.G[qa][pb] : &s.G[pb][qa];
                float *e11 = qa < qb ? &s.G[qa][qb] : &s.G[qb][qa];
                const float ca = A.z, sa = A.w, cb = B.z, sb = B.w;
                const float g00 = *e00, g01 = *e01, g10 = *e10, g11 = *e11;
                const float h00 = ca * g00 - sa * g10, h01 = ca * g01 - sa * g11;
                const float h10 = sa * g00 + ca * g10, h11 = sa * g01 + ca * g11;
                *e00 = cb * h00 - sb * h01;
                *e01 = sb * h00 + cb * h01;
                *e10 = cb * h10 - sb * h11;
                *e11 = sb * h10 + cb * h11;
            }
            // Phase B2: eigenvector rows p, q of each pair, four components at a time
            for (int e = tid; e < NP * V4; e += NT) {
                const int k = e / V4, c4 = e % V4;
                const float4 A = s.pair[k];
                if (A.w == 0.f) continue;
                const int p = __float_as_int(A.x), q = __float_as_int(A.y);
                float4 *vp = reinterpret_cast<float4 *>(&s.Vt[p][0]) + c4;
                float4 *vq = reinterpret_cast<float4 *>(&s.Vt[q][0]) + c4;
                const float4 a = *vp, b = *vq;
                const float c = A.z, sn = A.w;
                *vp = make_float4(c * a.x - sn * b.x, c * a.y - sn * b.y, c * a.z - sn * b.z, c * a.w - sn * b.w);
                *vq = make_float4(sn * a.x + c * b.x, sn * a.y + c * b.y, sn * a.z + c * b.z, sn * a.w + c * b.w);
            }
            __syncthreads();
        }
        if (!rotated_any) return sweep + 1;
        // only the top-r subspace is kept: stop once no rotation could add
        // more than SUBSPACE_TOL of the energy it leaves out (rotations inside
        // the nearly degenerate noise bulk converge slowly and change nothing)
        if (r < P && subspace_gain<T, P, D, NT>(s, r) <= SUBSPACE_TOL) return sweep + 1;
    }
    return -1;
}

// INT4 records need the kept vectors to be eigenvectors (their sigma^{1/2}
// scaling), not just a basis of the kept subspace.  After the subspace stop
// the subspace is settled, so cyclic Jacobi restricted to the block of the r
// largest diagonal entries finishes the job: round-robin pairs among the
// block's indices (a dummy index when r is odd), each rotation applied to the
// block's entries of G and to the whole eigenvector rows.  Entries between
// the block and the rest are left alone: nothing reads them afterwards.
// Leaves s.order as the final ranking -- the block's indices by their
// polished eigenvalue (ties: lower index first), then the others in index
// order -- and returns the block sweeps taken (-1 at the cap).
template <typename T, int P, int D, int NT>
__device__ int polish_block(FactorSmem<T, P, D> &s, int r, int max_sweeps) {
    constexpr int V4 = P / 4;
    const int tid = threadIdx.x;
    const int n = (r + 1) & ~1, np = n / 2;
    if (tid < P) {
        const float li = s.G[tid][tid];
        int rank = 0;
        for (int j = 0; j < P; ++j) {
            const float lj = s.G[j][j];
            rank += (lj > li) || (lj == li && j < tid);
        }
        s.red[tid] = rank < r ? 1.f : 0.f;  // block membership
        if (rank < r) s.order[rank] = tid;
    }
    __syncthreads();
    const float tol2 = JACOBI_TOL * JACOBI_TOL;
    int done = -1;
    for (int sweep = 0; sweep < max_sweeps && done < 0; ++sweep) {
        int rotated_any = 0;
        for (int round = 0; round < n - 1; ++round) {
            int rot = 0;
            if (tid < np) {
                const int k = tid;
                const int a = k == 0 ? 0 : 1 + ((k - 1 - round + 2 * (n - 1)) % (n - 1));
                const int kb = n - 1 - k;
                const int b = 1 + ((kb - 1 - round + 2 * (n - 1)) % (n - 1));
                int p = -1, q = -1;
                float c = 1.f, sn = 0.f, t = 0.f;
                if (a < r && b < r) {
                    const int ia = s.order[a], ib = s.order[b];
                    p = ia < ib ? ia : ib;
                    q = ia < ib ? ib : ia;
                    const float gpp = s.G[p][p], gqq = s.G[q][q], gpq = s.G[p][q];
                    if (gpq * gpq > tol2 * fabsf(gpp * gqq) && gpq != 0.f) {
                        float zeta = __fdividef(gqq - gpp, 2.f * gpq);
                        float z2 = fmaf(zeta, zeta, 1.f);
                        t = copysignf(__fdividef(1.f, fabsf(zeta) + z2 * rsqrtf(z2)), zeta);
                        if (fabsf(zeta) > 1e18f) t = __fdividef(0.5f, zeta);
                        c = rsqrtf(fmaf(t, t, 1.f));
                        sn = t * c;
                        rot = 1;
                    }
                }
                s.pair[k] = make_float4(__int_as_float(p), __int_as_float(q), c, sn);  // p < 0: the dummy
                s.tn[k] = t;
            }
            rotated_any |= __syncthreads_or(rot);
            const int nblk = np * (np + 1) / 2;
            for (int e = tid; e < nblk; e += NT) {  // 2x2 blocks (al <= be) of this round's pairs
                int be = 0;
                while ((be + 1) * (be + 2) / 2 <= e) ++be;
                const int al = e - be * (be + 1) / 2;
                const float4 A = s.pair[al], B = s.pair[be];
                const int pa = __float_as_int(A.x), qa = __float_as_int(A.y);
                const int pb = __float_as_int(B.x), qb = __float_as_int(B.y);
                if (pa < 0 || pb < 0) continue;
                if (al == be) {
                    const float t = s.tn[al];
                    if (t != 0.f) {
                        const float g00 = s.G[pa][pa], g01 = s.G[pa][qa], g11 = s.G[qa][qa];
                        s.G[pa][pa] = g00 - t * g01;
                        s.G[qa][qa] = g11 + t * g01;
                        s.G[pa][qa] = 0.f;
                    }
                    continue;
                }
                if (A.w == 0.f && B.w == 0.f) continue;
                float *e00 = pa < pb ? &s.G[pa][pb] : &s.G[pb][pa];
                float *e01 = pa < qb ? &s.G[pa][qb] : &s.G[qb][pa];
                float *e10 = qa < pb ? &s.G[qa][pb] : &s.G[pb][qa];
                float *e11 = qa < qb ? &s.G[qa][qb] : &s.G[qb][qa];
                const float ca = A.z, sa = A.w, cb = B.z, sb = B.w;
                const float g00 = *e00, g01 = *e01, g10 = *e10, g11 = *e11;
                const float h00 = ca * g00 - sa * g10, h01 = ca * g01 - sa * g11;
                const float h10 = sa * g00 + ca * g10, h11 = sa * g01 + ca * g11;
                *e00 = cb * h00 - sb * h01;
                *e01 = sb * h00 + cb * h01;
                *e10 = cb * h10 - sb * h11;
                *e11 = sb * h10 + cb * h11;
            }
            for (int e = tid; e < np * V4; e += NT) {  // eigenvector rows p, q of each rotating pair
                const int k = e / V4, c4 = e % V4;
                const float4 A = s.pair[k];
                if (A.w == 0.f) continue;
                const int p = __float_as_int(A.x), q = __float_as_int(A.y);
                float4 *vp = reinterpret_cast<float4 *>(&s.Vt[p][0]) + c4;
                float4 *vq = reinterpret_cast<float4 *>(&s.Vt[q][0]) + c4;
                const float4 a = *vp, b = *vq;
                const float c = A.z, sn = A.w;
                *vp = make_float4(c * a.x - sn * b.x, c * a.y - sn * b.y, c * a.z - sn * b.z, c * a.w - sn * b.w);
                *vq = make_float4(sn * a.x + c * b.x, sn * a.y + c * b.y, sn * a.z + c * b.z, sn * a.w + c * b.w);
            }
            __syncthreads();
        }
        if (!rotated_any) done = sweep + 1;
    }
    // final ranking: the block by polished eigenvalue, then the rest by index
    if (tid < P) {
        const bool member = s.red[tid] != 0.f;
        const float li = s.G[tid][tid];
        int pos = member ? 0 : r;
        for (int j = 0; j < P; ++j) {
            const bool mj = s.red[j] != 0.f;
            if (member && mj) {
                const float lj = s.G[j][j];
                pos += (lj > li) || (lj == li && j < tid);
            } else if (!member && !mj) {
                pos += j < tid;
            }
        }
        s.lam[tid] = li;
        s.order[pos] = tid;
    }
    __syncthreads();
    return done;
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
//      accumulator-column order (q4_scale_index);
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
        if (lane == 0) s.lam[j] = sqrtf(sqrtf(a));
    }
    __syncthreads();
    for (int e = tid; e < P * rp; e += NT) {
        const int i = e / rp, j = e % rp;
        const float rs = s.lam[j];
        s.G[i][j] = (j < r && rs > 0.f) ? s.G[i][j] * rs : 0.f;
    }
    for (int e = tid; e < rp * D; e += NT) {
        const float rs = s.lam[e / D];
        Rf[e] = rs > 0.f ? Rf[e] / rs : 0.f;
    }
    __syncthreads();
    if (v.qL)  // the absorbed factors the codes below quantize
        for (int e = tid; e < P * rp; e += NT) v.qL[e] = s.G[e / rp][e % rp];
    if (v.qR)
        for (int e = tid; e < rp * D; e += NT) v.qR[e] = Rf[e];
    // 3. scales: fp16 in the record (accumulator-column order), their fp32
    // values in s.Vt for the codes
    float *scL = &s.Vt[0][0];  // per rank (keys) or per token (values): up to P
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
        hR[q4_scale_index(D, k)] = h;
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

// Returns the Jacobi sweeps the page took (the cap if it did not converge).
template <typename T, int P, int D, int NT>
__device__ int factorize_one(FactorSmem<T, P, D> &s, const FactorParams &fp, long job) {
    const int tid = threadIdx.x;
    const JobView v = job_view(fp, job);
    load_page<T, P, D, NT>(s, v);
    __syncthreads();
    if constexpr (sizeof(T) == 2) gram_bf16<P, D, NT>(s); else gram_f32<P, D, NT>(s);
    __syncthreads();
    // the tensor-core tiles of (i, j) and (j, i) may round differently: symmetrise
    for (int e = tid; e < P * P; e += NT) {
        int i = e / P, j = e % P;
        if (j > i) s.G[j][i] = s.G[i][j];
    }
    __syncthreads();
    // with singular values requested every eigenpair must converge; otherwise
    // only the kept subspace has to, and INT4 records (whose kept vectors
    // must be eigenvectors) then finish the kept block on its own
    const bool polish = !v.sigma && v.r < P && v.rec && fp.y.q4;
    int sweeps = jacobi<T, P, D, NT>(s, fp.max_sweeps, v.sigma ? P : v.r);
    if (polish && sweeps >= 0 && polish_block<T, P, D, NT>(s, v.r, fp.max_sweeps) < 0) sweeps = -1;
    if (sweeps < 0 && tid == 0 && fp.status) atomicAdd(fp.status + STATUS_NOT_CONVERGED, 1);
    if (!polish) {
        if (tid < P) s.lam[tid] = s.G[tid][tid];
        __syncthreads();
        if (tid < P) {
            float li = s.lam[tid];
            int rank = 0;
            for (int j = 0; j < P; ++j) {
                float lj = s.lam[j];
                rank += (lj > li) || (lj == li && j < tid);
            }
            s.order[rank] = tid;
        }
        __syncthreads();
    }
    const int r = v.r;
    if (v.sigma && tid < P) v.sigma[tid] = sqrtf(fmaxf(s.lam[s.order[tid]], 0.f));
    __syncthreads();
    for (int e = tid; e < P * P; e += NT) {
        int i = e / P, j = e % P;
        s.G[i][j] = s.Vt[s.order[j]][i];
    }
    __syncthreads();
    // Hundreds of rounds of fp32 rotations let the eigenvector norms drift by
    // ~1e-5; scale the kept columns back to unit length (their mutual
    // orthogonality is already at fp32 rounding level).
    if (tid < v.r) {
        float n2 = 0.f;
        for (int i = 0; i < P; ++i) n2 = fmaf(s.G[i][tid], s.G[i][tid], n2);
        s.lam[tid] = n2 > 0.f ? 1.f / sqrtf(n2) : 1.f;  // lam[] is free once order[] is set
    }
    __syncthreads();
    for (int e = tid; e < P * v.r; e += NT) {
        int i = e / v.r, j = e % v.r;
        s.G[i][j] *= s.lam[j];
    }
    __syncthreads();

    const Layout &y = fp.y;
    const bool rec = v.rec != nullptr;
    if (rec && y.q4) {
        write_q4_record<T, P, D, NT>(s, v, y);
        return sweeps < 0 ? fp.max_sweeps : sweeps;
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
    return sweeps < 0 ? fp.max_sweeps : sweeps;
}

// The 256-thread variant keeps four CTAs per SM (64 registers), which its
// shared memory also allows: four pages in flight keep the shared-memory
// pipe, which bounds the Jacobi rounds, busy through each round's barriers.
template <typename T, int P, int D, int NT>
__global__ void __launch_bounds__(NT, NT == 256 ? 4 : 1) factorize_kernel(const FactorParams fp) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    auto &s = *reinterpret_cast<FactorSmem<T, P, D> *>(smem_raw);
    unsigned long long jobs = 0, sweeps = 0;
    for (long job = blockIdx.x; job < fp.n_jobs; job += gridDim.x) {
        sweeps += (unsigned long long)factorize_one<T, P, D, NT>(s, fp, job);
        ++jobs;
        __syncthreads();
    }
    if (threadIdx.x == 0 && fp.status && jobs) {  // throughput accounting, once per CTA
        atomicAdd(reinterpret_cast<unsigned long long *>(fp.status + STATUS_JOBS), jobs);
        atomicAdd(reinterpret_cast<unsigned long long *>(fp.status + STATUS_SWEEPS), sweeps);
    }
}

template <typename T, int P, int D, int NT>
static cudaError_t launch_t(const FactorParams &fp, int num_sms, cudaStream_t st) {
    size_t smem = sizeof(FactorSmem<T, P, D>);
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
        state = e == cudaSuccess ? 1 : 2 + (int)e;
        attr_state[dev].store(state, std::memory_order_release);
    }
    if (state != 1) return (cudaError_t)(state - 2);
    long blocks = fp.n_jobs;
    long cap = (long)num_sms * (NT >= 1024 ? 2 : 8);
    if (fp.max_ctas > 0 && fp.max_ctas < cap) cap = fp.max_ctas;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) return cudaSuccess;
    k<<<(unsigned)blocks, NT, smem, st>>>(fp);
    return cudaGetLastError();
}

// A few pages (conversions during decoding) are latency-bound: 1024 threads
// per page.  Many pages (prefill, batches) are throughput-bound: 256 threads,
// several pages per SM.  Work capped to run beside decode launches (max_ctas,
// the background batches) always takes 256 threads: a 1024-thread CTA holds
// all of an SM's registers, so no decode CTA could share the SM with it.
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
