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
//      rotates P/2 disjoint pairs at once, every thread updating 2x2 blocks
//      of G and pairs of eigenvector entries; a sweep is P-1 rounds; stop
//      after a sweep with no rotation (relative threshold), or at the cap;
//   4. eigenvalues ranked descending (ties: lower index first);
//   5. L = Q_r, R = Q_r^T X in fp32, written as bf16 or fp32 into either a
//      factor record (swizzled store layout) or plain row-major arrays.
#include "common.cuh"
#include "kernels.h"

namespace pkv {

constexpr int FT_THREADS = 256;
constexpr float JACOBI_TOL = 1e-6f;

template <typename T, int P, int D>
struct FactorSmem {
    alignas(128) unsigned char X[P * D * sizeof(T)];  // swizzled rows, pitch D * sizeof(T)
    float G[P][P + 1];  // Gram matrix; after the eigensolve reused for Q[i][j] = V[i][order[j]]
    float V[P][P + 1];
    float cs[P / 2], sn[P / 2], tn[P / 2];
    int pp[P / 2], qq[P / 2];
    float lam[P];
    int order[P];
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
        int l = (int)t;
        const char *src = kind == 0 ? fp.k_src : fp.v_src;
        v.x = src + (((size_t)l * y.H + h) * fp.T + (size_t)pg * y.P) * y.d * y.esz;
        v.x_pool = 0;
        v.kind = kind;
        v.r = kind == 0 ? y.rk : y.rv;
        v.rec = fp.factor_pool + y.record_offset(l, fp.seq, h, pg);
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

template <typename T, int P, int D>
__device__ void load_page(FactorSmem<T, P, D> &s, const JobView &v) {
    // 16-byte vectors; pool pages are already swizzled, plain rows get swizzled here
    constexpr int PITCH = D * (int)sizeof(T);
    constexpr int NVEC = P * PITCH / 16;
    const uint4 *src = reinterpret_cast<const uint4 *>(v.x);
    for (int i = threadIdx.x; i < NVEC; i += FT_THREADS) {
        uint4 val = src[i];
        int row = (i * 16) / PITCH, b = (i * 16) % PITCH;
        uint32_t off = v.x_pool ? (uint32_t)(i * 16) : swz_offset(row, b, PITCH);
        *reinterpret_cast<uint4 *>(s.X + off) = val;
    }
}

// G = X X^T, bf16 rows on tensor cores.
template <int P, int D>
__device__ void gram_bf16(FactorSmem<__nv_bfloat16, P, D> &s) {
    constexpr int MT = P / 16, NT = P / 8, KS = D / 16, PITCH = D * 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t xb = smem_u32(s.X);
    for (int tile = warp; tile < MT * NT; tile += FT_THREADS / 32) {
        int mt = tile / NT, nt = tile % NT;
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
template <int P, int D>
__device__ void gram_f32(FactorSmem<float, P, D> &s) {
    constexpr int PITCH = D * 4;
    for (int e = threadIdx.x; e < P * P; e += FT_THREADS) {
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

// Cyclic Jacobi eigensolve of the symmetric P x P matrix in s.G; eigenvectors
// accumulate into s.V.  Returns the number of sweeps, or -1 at the cap.
template <typename T, int P, int D>
__device__ int jacobi(FactorSmem<T, P, D> &s, int max_sweeps) {
    constexpr int NP = P / 2;
    const int tid = threadIdx.x;
    for (int e = tid; e < P * P; e += FT_THREADS) s.V[e / P][e % P] = (e / P == e % P) ? 1.f : 0.f;
    __syncthreads();
    for (int sweep = 0; sweep < max_sweeps; ++sweep) {
        int rotated_any = 0;
        for (int round = 0; round < P - 1; ++round) {
            // Phase A: angles of the NP disjoint pairs of this round (circle method:
            // slot 0 holds index 0, slot i >= 1 holds 1 + (i - 1 - round) mod (P - 1);
            // slot k meets slot P - 1 - k).
            int rot = 0;
            if (tid < NP) {
                int k = tid;
                int a = k == 0 ? 0 : 1 + ((k - 1 - round + 2 * (P - 1)) % (P - 1));
                int kb = P - 1 - k;
                int b = 1 + ((kb - 1 - round + 2 * (P - 1)) % (P - 1));
                int p = a < b ? a : b, q = a < b ? b : a;
                float gpp = s.G[p][p], gqq = s.G[q][q], gpq = s.G[p][q];
                float c = 1.f, sn = 0.f, t = 0.f;
                if (gpq != 0.f && fabsf(gpq) > JACOBI_TOL * sqrtf(fabsf(gpp * gqq))) {
                    float zeta = (gqq - gpp) / (2.f * gpq);
                    t = copysignf(1.f, zeta) / (fabsf(zeta) + sqrtf(1.f + zeta * zeta));
                    c = 1.f / sqrtf(1.f + t * t);
                    sn = t * c;
                    rot = 1;
                }
                s.pp[k] = p;
                s.qq[k] = q;
                s.cs[k] = c;
                s.sn[k] = sn;
                s.tn[k] = t;
            }
            rotated_any |= __syncthreads_or(rot);
            // Phase B: G <- J^T G J on every 2x2 block, V <- V J.
            for (int bi = tid; bi < NP * NP; bi += FT_THREADS) {
                int al = bi % NP, be = bi / NP;
                int pa = s.pp[al], qa = s.qq[al], pb = s.pp[be], qb = s.qq[be];
                float g00 = s.G[pa][pb], g01 = s.G[pa][qb], g10 = s.G[qa][pb], g11 = s.G[qa][qb];
                if (al == be) {
                    float t = s.tn[al];
                    if (t != 0.f) {
                        s.G[pa][pa] = g00 - t * g01;
                        s.G[qa][qa] = g11 + t * g01;
                        s.G[pa][qa] = 0.f;
                        s.G[qa][pa] = 0.f;
                    }
                } else {
                    float ca = s.cs[al], sa = s.sn[al], cb = s.cs[be], sb = s.sn[be];
                    float h00 = ca * g00 - sa * g10, h01 = ca * g01 - sa * g11;
                    float h10 = sa * g00 + ca * g10, h11 = sa * g01 + ca * g11;
                    s.G[pa][pb] = cb * h00 - sb * h01;
                    s.G[pa][qb] = sb * h00 + cb * h01;
                    s.G[qa][pb] = cb * h10 - sb * h11;
                    s.G[qa][qb] = sb * h10 + cb * h11;
                }
            }
            for (int e = tid; e < P * NP; e += FT_THREADS) {
                int i = e % P, k = e / P;
                int p = s.pp[k], q = s.qq[k];
                float c = s.cs[k], sn = s.sn[k];
                float vp = s.V[i][p], vq = s.V[i][q];
                s.V[i][p] = c * vp - sn * vq;
                s.V[i][q] = sn * vp + c * vq;
            }
            __syncthreads();
        }
        if (!rotated_any) return sweep + 1;
    }
    return -1;
}

template <typename TO>
__device__ __forceinline__ void store_elem(char *base, size_t idx, float v) {
    reinterpret_cast<TO *>(base)[idx] = Elem<TO>::from_f32(v);
}

template <typename T, int P, int D>
__device__ void factorize_one(FactorSmem<T, P, D> &s, const FactorParams &fp, long job) {
    const int tid = threadIdx.x;
    const JobView v = job_view(fp, job);
    load_page<T, P, D>(s, v);
    __syncthreads();
    if constexpr (sizeof(T) == 2) gram_bf16<P, D>(s); else gram_f32<P, D>(s);
    __syncthreads();
    // the tensor-core tiles of (i, j) and (j, i) may round differently: symmetrise
    for (int e = tid; e < P * P; e += FT_THREADS) {
        int i = e / P, j = e % P;
        if (j > i) s.G[j][i] = s.G[i][j];
    }
    __syncthreads();
    int sweeps = jacobi<T, P, D>(s, fp.max_sweeps);
    if (sweeps < 0 && tid == 0 && fp.status) atomicAdd(fp.status + STATUS_NOT_CONVERGED, 1);
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
    const int r = v.r;
    if (v.sigma && tid < P) v.sigma[tid] = sqrtf(fmaxf(s.lam[s.order[tid]], 0.f));
    __syncthreads();
    for (int e = tid; e < P * P; e += FT_THREADS) {
        int i = e / P, j = e % P;
        s.G[i][j] = s.V[i][s.order[j]];
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
    for (int e = tid; e < P * v.r; e += FT_THREADS) {
        int i = e / v.r, j = e % v.r;
        s.G[i][j] *= s.lam[j];
    }
    __syncthreads();

    const Layout &y = fp.y;
    const bool rec = v.rec != nullptr;
    const int rp = rec ? (v.kind == 0 ? y.rkp : y.rvp) : r;
    // L = Q_r  (record: keys LK[token][rank], values LVt[rank][token])
    for (int e = tid; e < P * rp; e += FT_THREADS) {
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
    constexpr int GROUPS = FT_THREADS / D;
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
}

template <typename T, int P, int D>
__global__ void __launch_bounds__(FT_THREADS) factorize_kernel(const FactorParams fp) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    auto &s = *reinterpret_cast<FactorSmem<T, P, D> *>(smem_raw);
    for (long job = blockIdx.x; job < fp.n_jobs; job += gridDim.x) {
        factorize_one<T, P, D>(s, fp, job);
        __syncthreads();
    }
}

template <typename T, int P, int D>
static cudaError_t launch_t(const FactorParams &fp, int num_sms, cudaStream_t st) {
    size_t smem = sizeof(FactorSmem<T, P, D>);
    auto k = factorize_kernel<T, P, D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    long blocks = fp.n_jobs;
    long cap = (long)num_sms * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) return cudaSuccess;
    k<<<(unsigned)blocks, FT_THREADS, smem, st>>>(fp);
    return cudaGetLastError();
}

cudaError_t launch_factorize(const FactorParams &fp, int num_sms, cudaStream_t st) {
    if (fp.n_jobs <= 0) return cudaSuccess;
    const bool bf = fp.x_esz == 2;
#define PKV_FACT_CASE(PP, DD)                                                                    \
    if (fp.P == PP && fp.d == DD)                                                                \
        return bf ? launch_t<__nv_bfloat16, PP, DD>(fp, num_sms, st) : launch_t<float, PP, DD>(fp, num_sms, st);
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
