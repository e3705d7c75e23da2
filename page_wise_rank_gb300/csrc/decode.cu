// Decode attention: fp32 CUDA-core kernel and the launch dispatch.  The bf16
// tensor-core kernel and the split hand-off shared by both live in
// decode_impl.cuh (instantiated in decode_bf16_p*.cu).
#include "decode_impl.cuh"

namespace pkv {

// ---------------------------------------------------------------- fp32 CUDA-core path

template <int P, int D>
__global__ void __launch_bounds__(NWC * 32) decode_f32_kernel(const DecodeParams prm) {
    const Layout &y = prm.y;
    const int b_idx = blockIdx.z, b = prm.seqs[b_idx], h = blockIdx.y, split = blockIdx.x;
    const int T = prm.lens[b_idx];
    const int n_pages = (T + P - 1) / P;
    const int p0 = split * prm.chunk;
    if (p0 >= n_pages) return;
    if (prm.append && split == 0 && h == 0 && threadIdx.x == 0) append_page_table(prm, b_idx, b, T);
    const float *k_new = prm.append ? reinterpret_cast<const float *>(prm.k_new) + ((size_t)b_idx * y.H + h) * D : nullptr;
    const float *v_new = prm.append ? reinterpret_cast<const float *>(prm.v_new) + ((size_t)b_idx * y.H + h) * D : nullptr;
    const int p1 = min(p0 + prm.chunk, n_pages);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = y.G;
    constexpr int TPL = (P + 31) / 32;  // tokens per lane
    constexpr int DPL = D / 32;         // head dims per lane
    const float scale = rsqrtf((float)D);
    __shared__ __align__(16) float comb[NWC][8][D + 4];
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
        const int kind = page_kind(p, T, P, y.sink_tokens, y.W);
        const int slot = kind == KIND_FACTORED ? p : y.dense_slot(p);
        // fused append: the new token's rows come from the inputs (and go to the pool)
        const int new_row = (prm.append && p == (T - 1) / P) ? (T - 1) % P : -1;
        if (new_row >= 0) {
            float *kp = reinterpret_cast<float *>(const_cast<char *>(prm.dense_pool) + y.dense_offset(prm.layer, b, slot, h, 0));
            float *vp = reinterpret_cast<float *>(const_cast<char *>(prm.dense_pool) + y.dense_offset(prm.layer, b, slot, h, 1));
            for (int c = lane; c < D; c += 32) {
                *swz_ptr<float>(kp, new_row, c, D) = k_new[c];
                *swz_ptr<float>(vp, new_row, c, D) = v_new[c];
            }
        }
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
                    float kv = i == new_row ? k_new[lane + 32 * e] : *swz_ptr<float>(kp, i, lane + 32 * e, D);
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
                    float vv = i == new_row ? v_new[lane + 32 * e] : *swz_ptr<float>(vp, i, lane + 32 * e, D);
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
        for (int e = 0; e < DPL; ++e) comb[warp][g][4 + lane + 32 * e] = o[g][e];
    }
    __syncthreads();
    const int ns = (n_pages + prm.chunk - 1) / prm.chunk;
    finish_split<D, NWC>(prm, &comb[0][0][0], b_idx, b, h, split, ns, &last);
}

// ---------------------------------------------------------------- launch

template <int P, int D>
static cudaError_t launch_f32(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st) {
    auto k = decode_f32_kernel<P, D>;
    static int occ = 0;  // computed once (the kernel uses static shared memory only)
    if (occ == 0) {
        int o = 1;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, k, NWC * 32, 0) != cudaSuccess || o < 1) o = 1;
        occ = o;
    }
    int splits = 1;
    choose_chunk(p, total_pages, max_pages, num_sms * occ, splits);
    dim3 grid((unsigned)splits, (unsigned)p.y.H, (unsigned)p.nseq);
    k<<<grid, NWC * 32, 0, st>>>(p);
    return cudaGetLastError();
}

size_t decode_smem_bytes(const Layout &y) {
    if (y.dtype != 1) return 0;  // the fp32 kernel's shared memory is static and small
    const bool q4 = y.q4 != 0, rope = y.rope != 0;
    // the shape of the runtime-rank kernel of this path (DecodeShape): warps x
    // slots, units per dense page
    const int nwc = q4 || rope ? DecodeShape<true, 64>::NWC : DecodeShape<false, 64>::NWC;
    const int spw = rope ? DecodeShape<false, 64, true>::SPW : DecodeShape<false, 64>::SPW;
    const int du = q4 && y.P >= 32 ? DecodeShape<true, 64>::DU : DecodeShape<false, 64>::DU;
    const size_t unit = (size_t)(y.P / du) * y.d * 2 * 2;
    size_t stage = ((y.rec_bytes > unit ? y.rec_bytes : unit) + 15) & ~(size_t)15;
    if (rope) stage += (size_t)y.d * 4;
    stage = (stage + 127) & ~(size_t)127;
    const size_t ns = (size_t)nwc * spw;
    const size_t shared_state = du == 4 ? sizeof(DecodeShared<4>) : sizeof(DecodeShared<2>);
    return ns * stage + ns * sizeof(uint64_t) + shared_state + (rope ? 16 + (size_t)y.P * y.d * 4 : 0);
}

cudaError_t launch_decode(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st) {
    if (p.y.dtype == 1) {
        if (p.y.q4) return launch_bf16_q4(p, total_pages, max_pages, num_sms, st);
        if (p.y.rope) return launch_bf16_rope(p, total_pages, max_pages, num_sms, st);
        if (p.y.P == 64) return launch_bf16_p64(p, total_pages, max_pages, num_sms, st);
        if (p.y.P == 32) return launch_bf16_p32(p, total_pages, max_pages, num_sms, st);
        if (p.y.P == 16) return launch_bf16_p16(p, total_pages, max_pages, num_sms, st);
        return cudaErrorInvalidValue;
    }
#define PKV_DEC_CASE(PP, DD) \
    if (p.y.P == PP && p.y.d == DD) return launch_f32<PP, DD>(p, total_pages, max_pages, num_sms, st);
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
