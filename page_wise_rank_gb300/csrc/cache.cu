// Paged-cache maintenance kernels: sequence initialisation after prefill and
// per-token append ("PuzzleKV: Page-Wise Low-Rank Decomposition for KV Cache
// Compression", §3.3 ①② and ⑤).  Page kinds follow page_kind() in layout.h;
// the host mirror applies the same rule to decide which pages to factorize.
#include "common.cuh"
#include "kernels.h"

namespace pkv {

// Block (layer, head, K/V, dense page k): copy the page's valid rows from the
// prompt cache into its dense slot (swizzled rows) and zero the rest.  Block
// x == 0 of each layer also writes that layer's length and descriptors.
template <typename T>
__global__ void seq_init_kernel(const SeqInitParams p) {
    const Layout &y = p.y;
    const int lrel = blockIdx.z, layer = p.layer0 + lrel;
    const int n_pages = (p.T + y.P - 1) / y.P;
    if (blockIdx.x == 0 && blockIdx.y == 0) {
        if (threadIdx.x == 0) p.lengths[y.len_index(p.seq, layer)] = p.T;
        for (int pg = threadIdx.x; pg < y.n_pg_max; pg += blockDim.x) {
            int v = 0;
            if (pg < n_pages) {
                int kind = page_kind(pg, p.T, y.P, y.sink_tokens, y.W);
                v = kind == KIND_DENSE ? (KIND_DENSE << KIND_SHIFT) | y.dense_slot(pg) : pg;
            }
            p.desc[y.desc_index(p.seq, layer, pg)] = v;
        }
    }
    const int h = blockIdx.y / 2, kv = blockIdx.y % 2;
    const int k = blockIdx.x;
    if (k >= p.n_dense) return;
    const int pg = p.dense_pages[k];
    const T *src = reinterpret_cast<const T *>(kv == 0 ? p.k_src : p.v_src) +
                   (((size_t)lrel * y.H + h) * p.T + (size_t)pg * y.P) * y.d;
    char *dst = p.dense_pool + y.dense_offset(layer, p.seq, y.dense_slot(pg), h, kv);
    const int valid = min(y.P, p.T - pg * y.P);
    for (int e = threadIdx.x; e < y.P * y.d; e += blockDim.x) {
        int row = e / y.d, col = e % y.d;
        T v = row < valid ? src[(size_t)row * y.d + col] : Elem<T>::from_f32(0.f);
        *swz_ptr<T>(dst, row, col, y.d) = v;
    }
}

// Block (call entry, head): write the new key/value rows at position pos into
// the dense slot of page pos / P.  Block (entry, 0) thread 0 then advances the
// length and updates the descriptors: the new page (if pos starts one) becomes
// dense, and the page this call converts becomes factorized (its factors are
// written by the factorization launch that follows on the same stream, before
// any later attention call reads them).
template <typename T>
__global__ void append_kernel(const AppendParams p) {
    const Layout &y = p.y;
    const int e = blockIdx.x, h = blockIdx.y;
    const int b = p.seqs[e], pos = p.pos[e];
    const int pg = pos / y.P, row = pos % y.P;
    const int slot = y.dense_slot(pg);
    const T *ks = reinterpret_cast<const T *>(p.k) + ((size_t)e * y.H + h) * y.d;
    const T *vs = reinterpret_cast<const T *>(p.v) + ((size_t)e * y.H + h) * y.d;
    char *kd = p.dense_pool + y.dense_offset(p.layer, b, slot, h, 0);
    char *vd = p.dense_pool + y.dense_offset(p.layer, b, slot, h, 1);
    for (int c = threadIdx.x; c < y.d; c += blockDim.x) {
        *swz_ptr<T>(kd, row, c, y.d) = ks[c];
        *swz_ptr<T>(vd, row, c, y.d) = vs[c];
    }
    if (h == 0 && threadIdx.x == 0) {
        p.lengths[y.len_index(b, p.layer)] = pos + 1;
        if (row == 0) p.desc[y.desc_index(b, p.layer, pg)] = (KIND_DENSE << KIND_SHIFT) | slot;
        int cp = p.conv_page[e];
        if (cp >= 0) p.desc[y.desc_index(b, p.layer, cp)] = (KIND_FACTORED << KIND_SHIFT) | cp;
    }
}

cudaError_t launch_seq_init(const SeqInitParams &p, cudaStream_t st) {
    dim3 grid((unsigned)(p.n_dense > 0 ? p.n_dense : 1), (unsigned)(p.y.H * 2), (unsigned)p.n_layers);
    if (p.y.dtype == 1)
        seq_init_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(p);
    else
        seq_init_kernel<float><<<grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_append(const AppendParams &p, cudaStream_t st) {
    dim3 grid((unsigned)p.nseq, (unsigned)p.y.H);
    if (p.y.dtype == 1)
        append_kernel<__nv_bfloat16><<<grid, 128, 0, st>>>(p);
    else
        append_kernel<float><<<grid, 128, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
