// Kernel parameter blocks and launchers (private to the library).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "layout.h"

namespace pkv {

enum { FACT_MODE_BATCH = 0, FACT_MODE_PREFILL = 1, FACT_MODE_CONVERT = 2, FACT_MODE_CONVERT_LIST = 3,
       FACT_MODE_BATCH_Q4 = 4 };

struct FactorParams {
    int mode;
    long n_jobs;
    int max_ctas;  // grid size cap (0: the default, a few CTAs per SM looping over the jobs)
    int max_ql_iter;  // QL iterations allowed per eigenvalue
    int *status;  // device status words (may be null in batch mode)
    // batch mode: X[n][P][d] -> L[n][P][r], R[n][r][d], sigma[n][P]
    const char *x_base;
    int x_esz, out_esz, P, d, r;
    char *L_out, *R_out;
    float *sigma;
    // store modes
    Layout y;
    char *factor_pool;
    const char *dense_pool;
    // prefill: pages [p_lo, p_hi) of sequence `seq`, layers layer0 ..
    // layer0 + n_layers - 1, from k_src / v_src ([n_layers][H][T][d])
    const char *k_src, *v_src;
    int seq, T, p_lo, p_hi, layer0, n_layers;
    // convert: one page per call entry of `layer`
    int layer, n_conv;
    int conv_seq[MAX_CALL_BATCH], conv_page[MAX_CALL_BATCH];
    // convert list: device int2 {seq << 8 | layer, page} per page, 2 H jobs each
    const int2 *conv_list;
    // batch INT4 mode: pages X[n][P][d] (x_base) of one kind (0 key, 1 value)
    // -> INT4 records q4_records[n][y.rec_bytes] (that kind's code stream and
    // scales), and optionally the absorbed fp32 factors the codes quantize,
    // q4_L[n][P][rank padded to 8] and q4_R[n][rank padded][d]
    int q4_kind;
    char *q4_records;
    float *q4_L, *q4_R;
};

constexpr int MAX_BOUNDS = 384;  // page bounds of all CTAs of one bf16 decode launch

struct DecodeParams {
    Layout y;
    const char *factor_pool, *dense_pool;
    const int *lengths, *desc;
    const char *q;      // [B][Hq][d] storage dtype
    float *partials;    // workspace split partials
    int *tickets;       // workspace split tickets, zero between launches
    int wait_first;     // bf16 kernel: the preceding launch may have written factor records
    // failure-path test hook (0 = off): 1 = the first unit of CTA (0, 0, 0)
    // expects bytes no copy delivers, 2 = so does every split merge; the waits
    // of this launch give up after wait_ns (0 = the library's limit)
    int inject;
    unsigned long long wait_ns;
    float *out;         // [B][Hq][d]
    int *status;
    int layer, chunk, nseq;
    int stages;         // shared-memory ring depth (bf16 kernel)
    int seqs[MAX_CALL_BATCH];
    int lens[MAX_CALL_BATCH];       // tokens attended per call entry (host mirror, after any append)
    // fused append (decode step): the token at position lens - 1 comes from
    // k_new / v_new ([B][H][d]); the kernel writes it into its dense page and
    // updates the device page table (new page, page converted before launch)
    const char *k_new, *v_new;
    int append;
    int conv_page[MAX_CALL_BATCH];  // page converted before this launch, or -1
    // bf16 kernel, filled by its launcher: CTA r of call entry i streams pages
    // [bounds[boff[i] + r], bounds[boff[i] + r + 1]) (PageSplit), of which
    // [fs[i], fw[i]) are the sequence's factorized pages
    int boff[MAX_CALL_BATCH], fs[MAX_CALL_BATCH], fw[MAX_CALL_BATCH];
    int nsplit[MAX_CALL_BATCH];     // CTAs per (sequence, KV head) of call entry i
    int bounds[MAX_BOUNDS];
    int *lengths_out, *desc_out;    // device page table (written when append)
    const float2 *rope_base, *rope_delta;  // keys stored before RoPE: (cos, sin) tables (Layout)
};

constexpr int MAX_DENSE_PAGES = 64;  // dense pages of one sequence (sink + window + filling)

struct SeqInitParams {
    Layout y;
    int *lengths, *desc;
    char *dense_pool;
    const char *k_src, *v_src;  // [n_layers][H][T][d]: layers layer0 .. layer0 + n_layers - 1
    int seq, T, n_dense, layer0, n_layers;
    int dense_pages[MAX_DENSE_PAGES];
};

struct AppendParams {
    Layout y;
    int *lengths, *desc;
    char *dense_pool;
    const char *k, *v;  // [B][H][d]
    int layer, nseq;
    int seqs[MAX_CALL_BATCH];
    int pos[MAX_CALL_BATCH];       // token position written (old length)
    int conv_page[MAX_CALL_BATCH]; // page converted by this call, or -1
};

cudaError_t launch_factorize(const FactorParams &p, int num_sms, cudaStream_t st);
cudaError_t launch_seq_init(const SeqInitParams &p, cudaStream_t st);
cudaError_t launch_append(const AppendParams &p, cudaStream_t st);
// Chooses pages per CTA (p.chunk) for one wave over total_pages pages
// (all listed sequences and KV heads), then launches.
cudaError_t launch_decode(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st);
// Dynamic shared memory the tensor-core decode kernel of this layout's path
// needs in its runtime-rank form (0 for fp32 stores).
size_t decode_smem_bytes(const Layout &y);
constexpr size_t MAX_DECODE_SMEM = 227 * 1024;  // opt-in shared memory per CTA on sm_103a

}  // namespace pkv
