// C ABI of the PuzzleKV store (declared in include/puzzlekv.h).
//
// Host responsibilities: validate every argument before launching anything,
// keep a host mirror of each (sequence, layer) length so that page
// classification -- which pages are dense, which page an append converts --
// is decided without reading device memory, and launch the kernels on the
// caller's stream.  The library never allocates device memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <cmath>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/puzzlekv.h"
#include "kernels.h"
#include "layout.h"

using namespace pkv;

namespace {

thread_local std::string g_last_error;

puzzlekv_status fail(puzzlekv_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

puzzlekv_status cuda_fail(cudaError_t e, const char *what) {
    return fail(PUZZLEKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 132;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 132;
    return n;
}

int host_page_kind(int p, int T, int P, int sink, int W) { return page_kind(p, T, P, sink, W); }

void layout_from(Layout &y, const puzzlekv_config *c);

puzzlekv_status validate_config(const puzzlekv_config *c) {
    if (!c) return fail(PUZZLEKV_ERR_INVALID_ARG, "config is NULL");
    if (c->num_layers < 1 || c->num_kv_heads < 1 || c->num_q_heads < 1 || c->max_batch < 1 ||
        c->max_tokens_per_seq < 1)
        return fail(PUZZLEKV_ERR_INVALID_ARG, "layers, heads, max_batch and max_tokens_per_seq must be >= 1");
    if (c->num_q_heads % c->num_kv_heads != 0)
        return fail(PUZZLEKV_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
    int G = c->num_q_heads / c->num_kv_heads;
    if (G > 8) return fail(PUZZLEKV_ERR_UNSUPPORTED, "at most 8 query heads per KV head (got %d)", G);
    if (c->head_dim != 64 && c->head_dim != 128)
        return fail(PUZZLEKV_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", c->head_dim);
    if (c->page_size != 16 && c->page_size != 32 && c->page_size != 64)
        return fail(PUZZLEKV_ERR_UNSUPPORTED, "page_size must be 16, 32 or 64 (got %d)", c->page_size);
    if (c->page_size > c->head_dim) return fail(PUZZLEKV_ERR_UNSUPPORTED, "page_size must be <= head_dim");
    if (c->rank_k < 1 || c->rank_k > c->page_size || c->rank_v < 1 || c->rank_v > c->page_size)
        return fail(PUZZLEKV_ERR_INVALID_ARG, "ranks must be in [1, page_size]");
    if (c->sink_tokens < 0 || c->recent_tokens < 0)
        return fail(PUZZLEKV_ERR_INVALID_ARG, "sink_tokens and recent_tokens must be >= 0");
    if (c->kv_dtype != PUZZLEKV_F32 && c->kv_dtype != PUZZLEKV_BF16)
        return fail(PUZZLEKV_ERR_INVALID_ARG, "kv_dtype must be PUZZLEKV_F32 or PUZZLEKV_BF16");
    if (c->factor_int4 != 0 && c->factor_int4 != 1) return fail(PUZZLEKV_ERR_INVALID_ARG, "factor_int4 must be 0 or 1");
    if (c->factor_int4 && c->kv_dtype != PUZZLEKV_BF16)
        return fail(PUZZLEKV_ERR_UNSUPPORTED, "INT4 factors need kv_dtype = PUZZLEKV_BF16");
    if (c->factor_int4 && (c->rank_k > c->page_size / 2 || c->rank_v > c->page_size / 2))
        return fail(PUZZLEKV_ERR_UNSUPPORTED, "INT4 factors need rank_k, rank_v <= page_size / 2");
    if (!(c->rope_theta >= 0.f) || c->rope_theta > 1e30f)
        return fail(PUZZLEKV_ERR_INVALID_ARG, "rope_theta must be 0 (keys stored as given) or a positive base");
    if (c->rope_theta > 0.f && (c->kv_dtype != PUZZLEKV_BF16 || c->factor_int4 || c->page_size < 32))
        return fail(PUZZLEKV_ERR_UNSUPPORTED, "keys before RoPE need kv_dtype = PUZZLEKV_BF16, factor_int4 = 0 "
                                              "and page_size 32 or 64");
    if (c->max_batch > (1 << 16) || c->max_tokens_per_seq > (1 << 24) || c->num_layers > 255)
        return fail(PUZZLEKV_ERR_UNSUPPORTED, "max_batch, max_tokens_per_seq or num_layers too large");
    int P = c->page_size;
    int sink_pages = (c->sink_tokens + P - 1) / P;
    int ring = (c->recent_tokens + P - 1) / P + 2;
    if (sink_pages + ring > MAX_DENSE_PAGES)
        return fail(PUZZLEKV_ERR_UNSUPPORTED, "sink + window span more than %d dense pages", MAX_DENSE_PAGES - 2);
    int n_pg = (c->max_tokens_per_seq + P - 1) / P;
    if ((long)(n_pg + MAX_CHUNK_PAGES - 1) / MAX_CHUNK_PAGES > MAX_SPLITS)
        return fail(PUZZLEKV_ERR_UNSUPPORTED, "max_tokens_per_seq too large for the split-K workspace");
    Layout y;
    layout_from(y, c);
    const size_t smem = decode_smem_bytes(y);
    if (smem > MAX_DECODE_SMEM)
        return fail(PUZZLEKV_ERR_UNSUPPORTED, "factor records of %zu bytes need %zu bytes of decode shared memory "
                                              "(at most %zu): lower rank_k + rank_v", y.rec_bytes, smem,
                    MAX_DECODE_SMEM);
    return PUZZLEKV_OK;
}

void layout_from(Layout &y, const puzzlekv_config *c) {
    make_layout(y, c->num_layers, c->num_kv_heads, c->num_q_heads, c->head_dim, c->page_size, c->rank_k,
                c->rank_v, c->sink_tokens, c->recent_tokens, c->max_batch, c->max_tokens_per_seq, c->kv_dtype,
                c->factor_int4, c->rope_theta);
}

// An NVTX range around a call of the C ABI, seen by profilers (free when
// none is attached).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

}  // namespace

struct puzzlekv_store {
    puzzlekv_config cfg;
    Layout y;
    char *dense_pool, *factor_pool, *page_table, *workspace;
    std::vector<int> len;    // host mirror [seq][layer]; -1 = empty slot
    // Which pages have factor records, per (seq, layer): every page in
    // [sink_pages, conv_upto) and, above it, the pages marked in `marked`
    // (factorized out of order by a page-list call).
    std::vector<int> conv_upto;                   // [seq][layer]
    std::vector<std::vector<uint8_t>> marked;     // [seq][layer][page], allocated on first use
    std::vector<int2> job_host;  // staging of the batched-conversion job list
    bool after_decode = false;   // the store's latest launch was a decode launch
    int fail_next = 0;           // failure-path test hook for the next decode launch (0 = off)
    uint64_t fail_wait_ns = 0;   // its waits' limit
    int num_sms;
    // Batched conversions run on an internal low-priority stream.  A batch's
    // factor records are first read when one of its pages becomes
    // factorized, i.e. when its sequence reaches deadline[seq] tokens; the
    // first call that attends at or past that length makes the caller's
    // stream wait for the batch.
    struct ConvBatch {
        cudaEvent_t done = nullptr;
        bool pending = false;
        std::vector<int> deadline;  // [seq]: length at which the batch's first page is factorized
        std::vector<char> uses;     // [seq][layer]: the batch writes factor records of that layer
    };
    cudaStream_t conv_stream = nullptr;
    cudaEvent_t conv_ready = nullptr;  // caller's stream position a batch starts after
    std::vector<ConvBatch> batches;    // ring
    int next_batch = 0;
    ~puzzlekv_store() {
        if (conv_stream) cudaStreamSynchronize(conv_stream);
        for (auto &cb : batches)
            if (cb.done) cudaEventDestroy(cb.done);
        if (conv_ready) cudaEventDestroy(conv_ready);
        if (conv_stream) cudaStreamDestroy(conv_stream);
    }
};

constexpr int kConvBatches = 8;

// Make `strm` wait for every pending background conversion batch that the
// listed sequences (at the given lengths) reach, or for all of them when
// `all` is set.  Returns true if a wait was inserted.
static bool wait_conversions(puzzlekv_store *s, cudaStream_t strm, const int32_t *seq_ids, const int *lens, int B,
                             bool all = false) {
    bool waited = false;
    for (auto &cb : s->batches) {
        if (!cb.pending) continue;
        bool due = all;
        for (int i = 0; i < B && !due; ++i) due = lens[i] >= cb.deadline[seq_ids[i]];
        if (due) {
            cudaStreamWaitEvent(strm, cb.done, 0);
            cb.pending = false;
            waited = true;
        }
    }
    return waited;
}

// Background batches run on the store's internal lowest-priority stream,
// created on first use.  begin_batch takes the next ring entry (ordering the
// caller's stream after the entry's previous batch if that is still
// pending), clears its deadlines and orders the internal stream after the
// work already queued on `strm`; end_batch marks the batch's end.
static cudaError_t ensure_background(puzzlekv_store *s) {
    if (s->conv_stream) return cudaSuccess;
    int least = 0, greatest = 0;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&s->conv_stream, cudaStreamNonBlocking, least);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->conv_ready, cudaEventDisableTiming);
    s->batches.resize(kConvBatches);
    for (auto &cb : s->batches) {
        if (e == cudaSuccess && !cb.done) e = cudaEventCreateWithFlags(&cb.done, cudaEventDisableTiming);
        cb.deadline.assign(s->y.Bmax, INT_MAX);
        cb.uses.assign((size_t)s->y.Bmax * s->y.L, 0);
    }
    return e;
}

static cudaError_t begin_batch(puzzlekv_store *s, cudaStream_t strm, puzzlekv_store::ConvBatch *&out) {
    cudaError_t e = ensure_background(s);
    if (e != cudaSuccess) return e;
    puzzlekv_store::ConvBatch &cb = s->batches[s->next_batch];
    s->next_batch = (s->next_batch + 1) % kConvBatches;
    if (cb.pending) {  // its event is about to be reused: order the caller's stream after it now
        e = cudaStreamWaitEvent(strm, cb.done, 0);
        cb.pending = false;
    }
    std::fill(cb.deadline.begin(), cb.deadline.end(), INT_MAX);
    std::fill(cb.uses.begin(), cb.uses.end(), 0);
    // the batch reads what the caller's stream has written: start after it
    if (e == cudaSuccess) e = cudaEventRecord(s->conv_ready, strm);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s->conv_stream, s->conv_ready, 0);
    out = &cb;
    return e;
}

static cudaError_t end_batch(puzzlekv_store *s, puzzlekv_store::ConvBatch &cb) {
    cudaError_t e = cudaEventRecord(cb.done, s->conv_stream);
    if (e == cudaSuccess) cb.pending = true;
    return e;
}

static int *lengths_ptr(puzzlekv_store *s) { return reinterpret_cast<int *>(s->page_table); }
static int *desc_ptr(puzzlekv_store *s) { return reinterpret_cast<int *>(s->page_table + s->y.desc_offset); }
static int *status_ptr(puzzlekv_store *s) { return reinterpret_cast<int *>(s->workspace); }

// Factor-record bookkeeping of (seq b, layer l).
static bool has_factors(const puzzlekv_store *s, int b, int l, int p) {
    const size_t i = (size_t)b * s->y.L + l;
    if (p < s->conv_upto[i]) return p >= s->y.sink_pages;
    const std::vector<uint8_t> &m = s->marked[i];
    return (size_t)p < m.size() && m[p] != 0;
}
static void set_factors(puzzlekv_store *s, int b, int l, int p) {
    const size_t i = (size_t)b * s->y.L + l;
    int &upto = s->conv_upto[i];
    std::vector<uint8_t> &m = s->marked[i];
    if (p < upto) return;
    if (m.size() < (size_t)s->y.n_pg_max) m.assign(s->y.n_pg_max, 0);
    m[p] = 1;
    while (upto < s->y.n_pg_max && m[upto]) m[upto++] = 0;  // extend the prefix over marked pages
}
static void reset_factors(puzzlekv_store *s, int b, int l, int upto) {
    const size_t i = (size_t)b * s->y.L + l;
    s->conv_upto[i] = upto;
    std::vector<uint8_t>().swap(s->marked[i]);
}

extern "C" {

const char *puzzlekv_last_error(void) { return g_last_error.c_str(); }

int32_t puzzlekv_classify_pages(int32_t T, int32_t P, int32_t sink_tokens, int32_t recent_tokens, int32_t *kinds,
                                int32_t cap) {
    if (T < 0 || P < 1 || sink_tokens < 0 || recent_tokens < 0 || (!kinds && cap > 0)) return -1;
    int n = (T + P - 1) / P;
    if (n > cap) return -1;
    for (int p = 0; p < n; ++p) kinds[p] = host_page_kind(p, T, P, sink_tokens, recent_tokens);
    return n;
}

double puzzlekv_page_storage_ratio(int32_t P, int32_t d, int32_t rank_k, int32_t rank_v) {
    if (P < 1 || d < 1) return 0.0;
    return (double)(rank_k + rank_v) * (double)(P + d) / (2.0 * P * d);
}

puzzlekv_status puzzlekv_query_sizes(const puzzlekv_config *cfg, size_t *dense_pool_bytes, size_t *factor_pool_bytes,
                                     size_t *page_table_bytes, size_t *workspace_bytes) {
    puzzlekv_status st = validate_config(cfg);
    if (st != PUZZLEKV_OK) return st;
    Layout y;
    layout_from(y, cfg);
    if (dense_pool_bytes) *dense_pool_bytes = y.dense_pool_bytes;
    if (factor_pool_bytes) *factor_pool_bytes = y.factor_pool_bytes;
    if (page_table_bytes) *page_table_bytes = y.page_table_bytes;
    if (workspace_bytes) *workspace_bytes = y.workspace_bytes;
    return PUZZLEKV_OK;
}

puzzlekv_status puzzlekv_store_create(const puzzlekv_config *cfg, void *dense_pool, void *factor_pool,
                                      void *page_table, void *workspace, void *stream, puzzlekv_store **out) {
    NvtxRange nvtx_range("puzzlekv_store_create");
    if (!out) return fail(PUZZLEKV_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    puzzlekv_status st = validate_config(cfg);
    if (st != PUZZLEKV_OK) return st;
    if (!dense_pool || !factor_pool || !page_table || !workspace)
        return fail(PUZZLEKV_ERR_INVALID_ARG, "device buffers must not be NULL");
    if (!aligned256(dense_pool) || !aligned256(factor_pool) || !aligned256(page_table) || !aligned256(workspace))
        return fail(PUZZLEKV_ERR_INVALID_ARG, "device buffers must be 256-byte aligned");
    puzzlekv_store *s = new puzzlekv_store();
    s->cfg = *cfg;
    layout_from(s->y, cfg);
    s->dense_pool = static_cast<char *>(dense_pool);
    s->factor_pool = static_cast<char *>(factor_pool);
    s->page_table = static_cast<char *>(page_table);
    s->workspace = static_cast<char *>(workspace);
    s->len.assign((size_t)cfg->max_batch * cfg->num_layers, -1);
    s->conv_upto.assign((size_t)cfg->max_batch * cfg->num_layers, 0);
    s->marked.resize((size_t)cfg->max_batch * cfg->num_layers);
    s->num_sms = sm_count();
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(dense_pool, 0, s->y.dense_pool_bytes, strm);
    if (e == cudaSuccess) e = cudaMemsetAsync(page_table, 0, s->y.page_table_bytes, strm);
    if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, s->y.workspace_bytes, strm);
    if (e == cudaSuccess && s->y.rope) {  // (cos, sin) tables of the RoPE angles, from fp64
        const Layout &y = s->y;
        const int h = y.d / 2;
        std::vector<float2> base((size_t)y.n_pg_max * h), delta((size_t)y.P * h);
        for (int i = 0; i < h; ++i) {
            const double th = std::pow((double)y.rope_theta, -2.0 * i / y.d);
            for (int p = 0; p < y.n_pg_max; ++p) {
                const double a = (double)p * y.P * th;
                base[(size_t)p * h + i] = make_float2((float)std::cos(a), (float)std::sin(a));
            }
            for (int t = 0; t < y.P; ++t)
                delta[(size_t)t * h + i] = make_float2((float)std::cos(t * th), (float)std::sin(t * th));
        }
        // pageable sources: consumed when cudaMemcpyAsync returns
        e = cudaMemcpyAsync(s->workspace + y.rope_base_offset, base.data(), base.size() * sizeof(float2),
                            cudaMemcpyHostToDevice, strm);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(s->workspace + y.rope_delta_offset, delta.data(), delta.size() * sizeof(float2),
                                cudaMemcpyHostToDevice, strm);
    }
    if (e != cudaSuccess) {
        delete s;
        return cuda_fail(e, "store_create memset");
    }
    *out = s;
    return PUZZLEKV_OK;
}

puzzlekv_status puzzlekv_store_destroy(puzzlekv_store *store) {
    delete store;
    return PUZZLEKV_OK;
}

}  // extern "C"

// Prefill of layers [layer0, layer0 + n_layers) of sequence `seq` from
// k / v ([n_layers][H][T][d]): the dense pages and page table on `strm`, the
// eligible pages' factorization on `strm` or, with `async`, as a background
// batch that every later attention call on `seq` waits for.
static puzzlekv_status prefill(puzzlekv_store *s, int32_t seq, int32_t layer0, int32_t n_layers, const void *k,
                               const void *v, int32_t T, bool async, cudaStream_t strm) {
    const Layout &y = s->y;
    if (seq < 0 || seq >= y.Bmax) return fail(PUZZLEKV_ERR_INVALID_ARG, "seq %d out of range", seq);
    if (T < 1) return fail(PUZZLEKV_ERR_INVALID_ARG, "T must be >= 1");
    if (T > y.Tmax) return fail(PUZZLEKV_ERR_CAPACITY, "T=%d exceeds max_tokens_per_seq=%d", T, y.Tmax);
    if (!k || !v || !aligned16(k) || !aligned16(v))
        return fail(PUZZLEKV_ERR_INVALID_ARG, "k and v must be non-NULL and 16-byte aligned");
    const int n_pages = (T + y.P - 1) / y.P;
    SeqInitParams ip{};
    ip.y = y;
    ip.lengths = lengths_ptr(s);
    ip.desc = desc_ptr(s);
    ip.dense_pool = s->dense_pool;
    ip.k_src = static_cast<const char *>(k);
    ip.v_src = static_cast<const char *>(v);
    ip.seq = seq;
    ip.T = T;
    ip.layer0 = layer0;
    ip.n_layers = n_layers;
    int f_lo = -1, f_hi = -1;
    for (int p = 0; p < n_pages; ++p) {
        if (host_page_kind(p, T, y.P, y.sink_tokens, y.W) == KIND_DENSE) {
            if (ip.n_dense >= MAX_DENSE_PAGES) return fail(PUZZLEKV_ERR_UNSUPPORTED, "too many dense pages");
            ip.dense_pages[ip.n_dense++] = p;
        } else {
            if (f_lo < 0) f_lo = p;
            if (f_hi >= 0 && f_hi != p) return fail(PUZZLEKV_ERR_INVALID_ARG, "factorized pages not contiguous");
            f_hi = p + 1;
        }
    }
    // background work of an earlier use of these layers may still write
    // their records: order the new writes after it
    for (auto &cb : s->batches) {
        bool uses = false;
        for (int l = layer0; cb.pending && l < layer0 + n_layers && !uses; ++l) uses = cb.uses[(size_t)seq * y.L + l];
        if (uses) {
            cudaStreamWaitEvent(strm, cb.done, 0);
            cb.pending = false;
        }
    }
    cudaError_t e = launch_seq_init(ip, strm);
    s->after_decode = false;
    if (e != cudaSuccess) return cuda_fail(e, "seq_init launch");
    if (f_lo >= 0) {
        FactorParams fp{};
        fp.mode = FACT_MODE_PREFILL;
        fp.max_ql_iter = 30;
        fp.status = status_ptr(s);
        fp.y = y;
        fp.P = y.P;
        fp.d = y.d;
        fp.x_esz = y.esz;
        fp.factor_pool = s->factor_pool;
        fp.k_src = ip.k_src;
        fp.v_src = ip.v_src;
        fp.seq = seq;
        fp.T = T;
        fp.p_lo = f_lo;
        fp.p_hi = f_hi;
        fp.layer0 = layer0;
        fp.n_layers = n_layers;
        fp.n_jobs = (long)n_layers * y.H * 2 * (f_hi - f_lo);
        if (async) {
            puzzlekv_store::ConvBatch *cb = nullptr;
            e = begin_batch(s, strm, cb);
            if (e == cudaSuccess) {
                cb->deadline[seq] = 0;  // the sequence's next attention call waits for it
                for (int l = layer0; l < layer0 + n_layers; ++l) cb->uses[(size_t)seq * y.L + l] = 1;
                e = launch_factorize(fp, s->num_sms, s->conv_stream);
            }
            if (e == cudaSuccess) e = end_batch(s, *cb);
        } else {
            e = launch_factorize(fp, s->num_sms, strm);
        }
        s->after_decode = false;
        if (e != cudaSuccess) return cuda_fail(e, "factorize launch");
    }
    for (int l = layer0; l < layer0 + n_layers; ++l) {
        s->len[(size_t)seq * y.L + l] = T;
        reset_factors(s, seq, l, f_lo >= 0 ? f_hi : y.sink_pages);
    }
    return PUZZLEKV_OK;
}

extern "C" {

puzzlekv_status puzzlekv_load_prefill(puzzlekv_store *s, int32_t seq, const void *k, const void *v, int32_t T,
                                     void *stream) {
    NvtxRange nvtx_range("puzzlekv_load_prefill");
    if (!s) return fail(PUZZLEKV_ERR_INVALID_ARG, "store is NULL");
    return prefill(s, seq, 0, s->y.L, k, v, T, false, static_cast<cudaStream_t>(stream));
}

puzzlekv_status puzzlekv_factorize_layer(puzzlekv_store *s, int32_t seq, int32_t layer, const void *k, const void *v,
                                         int32_t T, int32_t async, void *stream) {
    NvtxRange nvtx_range("puzzlekv_factorize_layer");
    if (!s) return fail(PUZZLEKV_ERR_INVALID_ARG, "store is NULL");
    if (layer < 0 || layer >= s->y.L) return fail(PUZZLEKV_ERR_INVALID_ARG, "layer %d out of range", layer);
    return prefill(s, seq, layer, 1, k, v, T, async != 0, static_cast<cudaStream_t>(stream));
}

puzzlekv_status puzzlekv_wait_background(puzzlekv_store *s, void *stream) {
    if (!s) return fail(PUZZLEKV_ERR_INVALID_ARG, "store is NULL");
    wait_conversions(s, static_cast<cudaStream_t>(stream), nullptr, nullptr, 0, true);
    return PUZZLEKV_OK;
}

puzzlekv_status puzzlekv_background_stream(puzzlekv_store *s, void **stream) {
    if (!s || !stream) return fail(PUZZLEKV_ERR_INVALID_ARG, "store and stream must be non-NULL");
    cudaError_t e = ensure_background(s);
    if (e != cudaSuccess) return cuda_fail(e, "background stream setup");
    *stream = s->conv_stream;
    return PUZZLEKV_OK;
}

puzzlekv_status puzzlekv_factorize_batch(const void *X, int32_t x_dtype, int64_t n, int32_t P, int32_t d, int32_t r,
                                         void *L, void *R, int32_t out_dtype, float *sigma, int32_t *status,
                                         void *stream) {
    NvtxRange nvtx_range("puzzlekv_factorize_batch");
    if (n < 0) return fail(PUZZLEKV_ERR_INVALID_ARG, "n must be >= 0");
    if ((x_dtype != PUZZLEKV_F32 && x_dtype != PUZZLEKV_BF16) || (out_dtype != PUZZLEKV_F32 && out_dtype != PUZZLEKV_BF16))
        return fail(PUZZLEKV_ERR_INVALID_ARG, "dtype must be PUZZLEKV_F32 or PUZZLEKV_BF16");
    if ((P != 16 && P != 32 && P != 64) || (d != 64 && d != 128) || P > d)
        return fail(PUZZLEKV_ERR_UNSUPPORTED, "need P in {16,32,64}, d in {64,128}, P <= d");
    if (r < 1 || r > P) return fail(PUZZLEKV_ERR_INVALID_ARG, "rank must be in [1, P]");
    if (n == 0) return PUZZLEKV_OK;
    if (!X || !L || !R || !aligned16(X)) return fail(PUZZLEKV_ERR_INVALID_ARG, "X, L, R must be non-NULL, X 16-byte aligned");
    FactorParams fp{};
    fp.mode = FACT_MODE_BATCH;
    fp.n_jobs = (long)n;
    fp.max_ql_iter = 30;
    fp.status = status;
    fp.x_base = static_cast<const char *>(X);
    fp.x_esz = x_dtype == PUZZLEKV_BF16 ? 2 : 4;
    fp.out_esz = out_dtype == PUZZLEKV_BF16 ? 2 : 4;
    fp.P = P;
    fp.d = d;
    fp.r = r;
    fp.L_out = static_cast<char *>(L);
    fp.R_out = static_cast<char *>(R);
    fp.sigma = sigma;
    cudaError_t e = launch_factorize(fp, sm_count(), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "factorize_batch launch");
    return PUZZLEKV_OK;
}

puzzlekv_status puzzlekv_int4_record_bytes(int32_t P, int32_t d, int32_t rank_k, int32_t rank_v, int64_t *bytes) {
    if (!bytes) return fail(PUZZLEKV_ERR_INVALID_ARG, "bytes is NULL");
    if ((P != 16 && P != 32 && P != 64) || (d != 64 && d != 128) || P > d)
        return fail(PUZZLEKV_ERR_UNSUPPORTED, "need P in {16,32,64}, d in {64,128}, P <= d");
    if (rank_k < 1 || rank_v < 1 || rank_k > P / 2 || rank_v > P / 2)
        return fail(PUZZLEKV_ERR_UNSUPPORTED, "INT4 ranks must be in [1, P/2]");
    Layout y;
    make_layout(y, 1, 1, 1, d, P, rank_k, rank_v, 0, 0, 1, P, 1, 1);
    *bytes = (int64_t)y.rec_bytes;
    return PUZZLEKV_OK;
}

puzzlekv_status puzzlekv_factorize_batch_int4(const void *X, int64_t n, int32_t P, int32_t d, int32_t rank_k,
                                              int32_t rank_v, int32_t kind, void *records, float *L_absorbed,
                                              float *R_absorbed, int32_t *status, void *stream) {
    NvtxRange nvtx_range("puzzlekv_factorize_batch_int4");
    int64_t rec_bytes = 0;
    puzzlekv_status st = puzzlekv_int4_record_bytes(P, d, rank_k, rank_v, &rec_bytes);
    if (st != PUZZLEKV_OK) return st;
    if (n < 0) return fail(PUZZLEKV_ERR_INVALID_ARG, "n must be >= 0");
    if (kind != 0 && kind != 1) return fail(PUZZLEKV_ERR_INVALID_ARG, "kind must be 0 (key) or 1 (value)");
    if (n == 0) return PUZZLEKV_OK;
    if (!X || !records || !aligned16(X) || !aligned16(records) || !aligned16(L_absorbed) || !aligned16(R_absorbed))
        return fail(PUZZLEKV_ERR_INVALID_ARG, "X and records must be non-NULL; all pointers 16-byte aligned");
    FactorParams fp{};
    fp.mode = FACT_MODE_BATCH_Q4;
    fp.n_jobs = (long)n;
    fp.max_ql_iter = 30;
    fp.status = status;
    make_layout(fp.y, 1, 1, 1, d, P, rank_k, rank_v, 0, 0, 1, P, 1, 1);
    fp.P = P;
    fp.d = d;
    fp.x_esz = 2;
    fp.x_base = static_cast<const char *>(X);
    fp.q4_kind = kind;
    fp.q4_records = static_cast<char *>(records);
    fp.q4_L = L_absorbed;
    fp.q4_R = R_absorbed;
    cudaError_t e = launch_factorize(fp, sm_count(), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "factorize_batch_int4 launch");
    return PUZZLEKV_OK;
}

// [PuzzleKV §3.3 ⑤]: the page (if any) that growing a sequence from T to
// T + 1 tokens moves out of the dense region; at most one per step.
static int converted_page(const Layout &y, int T) {
    int conv = -1;
    const int n_old = (T + y.P - 1) / y.P;
    for (int p = std::max(0, (T - y.W) / y.P - 1); p < n_old; ++p)
        if (host_page_kind(p, T, y.P, y.sink_tokens, y.W) == KIND_DENSE &&
            host_page_kind(p, T + 1, y.P, y.sink_tokens, y.W) == KIND_FACTORED)
            conv = p;
    return conv;
}

// Decode-kernel parameters for one call (lengths from the host mirror).
static void fill_decode_params(puzzlekv_store *s, int32_t layer, const void *q, float *out, const int32_t *seq_ids,
                               int32_t B, int extra_tokens, DecodeParams &dp, long &total, int &max_pages) {
    const Layout &y = s->y;
    dp = DecodeParams{};
    dp.y = y;
    dp.factor_pool = s->factor_pool;
    dp.dense_pool = s->dense_pool;
    dp.lengths = reinterpret_cast<const int *>(s->page_table);
    dp.desc = reinterpret_cast<const int *>(s->page_table + y.desc_offset);
    dp.q = static_cast<const char *>(q);
    dp.partials = reinterpret_cast<float *>(s->workspace + y.partial_offset);
    dp.rope_base = reinterpret_cast<const float2 *>(s->workspace + y.rope_base_offset);
    dp.rope_delta = reinterpret_cast<const float2 *>(s->workspace + y.rope_delta_offset);
    dp.tickets = reinterpret_cast<int *>(s->workspace + y.ticket_offset);
    dp.wait_first = s->after_decode ? 0 : 1;
    dp.inject = s->fail_next;  // consumed by this launch
    dp.wait_ns = s->fail_next ? s->fail_wait_ns : 0;
    s->fail_next = 0;
    dp.out = out;
    dp.status = reinterpret_cast<int *>(s->workspace);
    dp.layer = layer;
    dp.nseq = B;
    total = 0;
    max_pages = 0;
    for (int i = 0; i < B; ++i) {
        const int T = s->len[(size_t)seq_ids[i] * y.L + layer] + extra_tokens;
        const int np = (T + y.P - 1) / y.P;
        total += (long)np * y.H;
        max_pages = std::max(max_pages, np);
        dp.seqs[i] = seq_ids[i];
        dp.lens[i] = T;
        dp.conv_page[i] = -1;
    }
}

static puzzlekv_status check_call(puzzlekv_store *s, int32_t layer, const int32_t *seq_ids, int32_t B) {
    if (!s) return fail(PUZZLEKV_ERR_INVALID_ARG, "store is NULL");
    if (layer < 0 || layer >= s->y.L) return fail(PUZZLEKV_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (B < 1 || B > MAX_CALL_BATCH) return fail(PUZZLEKV_ERR_INVALID_ARG, "B must be in [1, %d]", MAX_CALL_BATCH);
    if (!seq_ids) return fail(PUZZLEKV_ERR_INVALID_ARG, "seq_ids is NULL");
    for (int i = 0; i < B; ++i) {
        int b = seq_ids[i];
        if (b < 0 || b >= s->y.Bmax) return fail(PUZZLEKV_ERR_INVALID_ARG, "seq id %d out of range", b);
        if (s->len[(size_t)b * s->y.L + layer] < 1)
            return fail(PUZZLEKV_ERR_INVALID_ARG, "sequence %d holds no tokens", b);
        for (int j = 0; j < i; ++j)
            if (seq_ids[j] == b) return fail(PUZZLEKV_ERR_INVALID_ARG, "sequence %d listed twice", b);
    }
    return PUZZLEKV_OK;
}

puzzlekv_status puzzlekv_append_token(puzzlekv_store *s, int32_t layer, const void *k, const void *v,
                                      const int32_t *seq_ids, int32_t B, void *stream) {
    NvtxRange nvtx_range("puzzlekv_append_token");
    puzzlekv_status st = check_call(s, layer, seq_ids, B);
    if (st != PUZZLEKV_OK) return st;
    if (!k || !v || !aligned16(k) || !aligned16(v))
        return fail(PUZZLEKV_ERR_INVALID_ARG, "k and v must be non-NULL and 16-byte aligned");
    const Layout &y = s->y;
    AppendParams ap{};
    ap.y = y;
    ap.lengths = lengths_ptr(s);
    ap.desc = desc_ptr(s);
    ap.dense_pool = s->dense_pool;
    ap.k = static_cast<const char *>(k);
    ap.v = static_cast<const char *>(v);
    ap.layer = layer;
    ap.nseq = B;
    FactorParams fp{};
    fp.n_conv = 0;
    for (int i = 0; i < B; ++i) {
        const int T = s->len[(size_t)seq_ids[i] * y.L + layer];
        if (T + 1 > y.Tmax) return fail(PUZZLEKV_ERR_CAPACITY, "sequence %d is full (%d tokens)", seq_ids[i], T);
    }
    for (int i = 0; i < B; ++i) {
        int b = seq_ids[i];
        int T = s->len[(size_t)b * y.L + layer];
        ap.seqs[i] = b;
        ap.pos[i] = T;
        const int conv = converted_page(y, T);
        ap.conv_page[i] = conv;  // descriptor flip
        if (conv >= 0 && !has_factors(s, b, layer, conv)) {  // not factorized ahead of time: now, before attention
            fp.conv_seq[fp.n_conv] = b;
            fp.conv_page[fp.n_conv] = conv;
            fp.n_conv++;
            set_factors(s, b, layer, conv);
        }
    }
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_append(ap, strm);
    s->after_decode = false;
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    if (fp.n_conv > 0) {
        fp.mode = FACT_MODE_CONVERT;
        fp.max_ql_iter = 30;
        fp.status = status_ptr(s);
        fp.y = y;
        fp.P = y.P;
        fp.d = y.d;
        fp.x_esz = y.esz;
        fp.factor_pool = s->factor_pool;
        fp.dense_pool = s->dense_pool;
        fp.layer = layer;
        fp.n_jobs = (long)fp.n_conv * y.H * 2;
        e = launch_factorize(fp, s->num_sms, strm);
        s->after_decode = false;
        if (e != cudaSuccess) return cuda_fail(e, "conversion launch");
    }
    for (int i = 0; i < B; ++i) s->len[(size_t)seq_ids[i] * y.L + layer] += 1;
    return PUZZLEKV_OK;
}

puzzlekv_status puzzlekv_decode_attention(puzzlekv_store *s, int32_t layer, const void *q, float *out,
                                          const int32_t *seq_ids, int32_t B, void *stream) {
    NvtxRange nvtx_range("puzzlekv_decode_attention");
    puzzlekv_status st = check_call(s, layer, seq_ids, B);
    if (st != PUZZLEKV_OK) return st;
    if (!q || !out || !aligned16(q) || !aligned16(out))
        return fail(PUZZLEKV_ERR_INVALID_ARG, "q and out must be non-NULL and 16-byte aligned");
    DecodeParams dp;
    long total;
    int max_pages;
    fill_decode_params(s, layer, q, out, seq_ids, B, 0, dp, total, max_pages);
    if (wait_conversions(s, static_cast<cudaStream_t>(stream), seq_ids, dp.lens, B)) dp.wait_first = 1;
    cudaError_t e = launch_decode(dp, total, max_pages, s->num_sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    s->after_decode = true;
    return PUZZLEKV_OK;
}

puzzlekv_status puzzlekv_decode_step(puzzlekv_store *s, int32_t layer, const void *q, const void *k, const void *v,
                                     float *out, const int32_t *seq_ids, int32_t B, void *stream) {
    NvtxRange nvtx_range("puzzlekv_decode_step");
    puzzlekv_status st = check_call(s, layer, seq_ids, B);
    if (st != PUZZLEKV_OK) return st;
    if (!q || !out || !k || !v || !aligned16(q) || !aligned16(out) || !aligned16(k) || !aligned16(v))
        return fail(PUZZLEKV_ERR_INVALID_ARG, "q, k, v and out must be non-NULL and 16-byte aligned");
    const Layout &y = s->y;
    FactorParams fp{};
    fp.n_conv = 0;
    for (int i = 0; i < B; ++i) {
        const int b = seq_ids[i];
        const int T = s->len[(size_t)b * y.L + layer];
        if (T + 1 > y.Tmax) return fail(PUZZLEKV_ERR_CAPACITY, "sequence %d is full (%d tokens)", b, T);
    }
    DecodeParams dp;
    long total;
    int max_pages;
    fill_decode_params(s, layer, q, out, seq_ids, B, 1, dp, total, max_pages);
    dp.append = 1;
    dp.k_new = static_cast<const char *>(k);
    dp.v_new = static_cast<const char *>(v);
    dp.lengths_out = reinterpret_cast<int *>(s->page_table);
    dp.desc_out = reinterpret_cast<int *>(s->page_table + y.desc_offset);
    for (int i = 0; i < B; ++i) {
        const int b = seq_ids[i];
        const int conv = converted_page(y, s->len[(size_t)b * y.L + layer]);
        dp.conv_page[i] = conv;  // descriptor flip
        if (conv >= 0 && !has_factors(s, b, layer, conv)) {  // not factorized ahead of time: now, before attention
            fp.conv_seq[fp.n_conv] = b;
            fp.conv_page[fp.n_conv] = conv;
            fp.n_conv++;
            set_factors(s, b, layer, conv);
        }
    }
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (fp.n_conv > 0) {  // the page leaving the window is factorized before this step's attention
        fp.mode = FACT_MODE_CONVERT;
        fp.max_ql_iter = 30;
        fp.status = status_ptr(s);
        fp.y = y;
        fp.P = y.P;
        fp.d = y.d;
        fp.x_esz = y.esz;
        fp.factor_pool = s->factor_pool;
        fp.dense_pool = s->dense_pool;
        fp.layer = layer;
        fp.n_jobs = (long)fp.n_conv * y.H * 2;
        e = launch_factorize(fp, s->num_sms, strm);
        s->after_decode = false;
        if (e != cudaSuccess) return cuda_fail(e, "conversion launch");
    }
    if (fp.n_conv > 0) dp.wait_first = 1;
    if (wait_conversions(s, strm, seq_ids, dp.lens, B)) dp.wait_first = 1;
    e = launch_decode(dp, total, max_pages, s->num_sms, strm);
    if (e != cudaSuccess) return cuda_fail(e, "decode step launch");
    s->after_decode = true;
    for (int i = 0; i < B; ++i) s->len[(size_t)seq_ids[i] * y.L + layer] += 1;
    return PUZZLEKV_OK;
}

puzzlekv_status puzzlekv_factorize_pages(puzzlekv_store *s, const int32_t *seq_ids, const int32_t *page_ids,
                                         int32_t n, void *stream) {
    NvtxRange nvtx_range("puzzlekv_factorize_pages");
    if (!s) return fail(PUZZLEKV_ERR_INVALID_ARG, "store is NULL");
    if (n < -1) return fail(PUZZLEKV_ERR_INVALID_ARG, "n must be -1 (all eligible pages) or >= 0 (got %d)", n);
    if (n > 0 && (!seq_ids || !page_ids)) return fail(PUZZLEKV_ERR_INVALID_ARG, "seq_ids and page_ids must be non-NULL");
    const Layout &y = s->y;
    // every check first: a bad entry changes nothing
    auto complete_pages = [&](int b) {  // pages complete in every layer of sequence b (-1: empty slot)
        int c = INT_MAX;
        for (int l = 0; l < y.L; ++l) {
            const int T = s->len[(size_t)b * y.L + l];
            if (T < 1) return -1;
            c = std::min(c, T / y.P);
        }
        return c;
    };
    for (int i = 0; i < n; ++i) {
        const int b = seq_ids[i], p = page_ids[i];
        if (b < 0 || b >= y.Bmax) return fail(PUZZLEKV_ERR_INVALID_ARG, "entry %d: seq id %d out of range", i, b);
        const int c = complete_pages(b);
        if (c < 0) return fail(PUZZLEKV_ERR_INVALID_ARG, "entry %d: sequence %d holds no tokens", i, b);
        if (p < y.sink_pages || p >= c)
            return fail(PUZZLEKV_ERR_INVALID_ARG,
                        "entry %d: page %d of sequence %d is not eligible (sink pages end at %d, complete pages at %d)",
                        i, p, b, y.sink_pages, c);
    }
    // the jobs: every layer of each listed page without factors (a page
    // listed twice counts once); the pages are marked only once the list is
    // known to fit
    std::vector<int2> pages;
    if (n == -1) {
        for (int b = 0; b < y.Bmax; ++b) {
            const int c = complete_pages(b);
            for (int p = y.sink_pages; p < c; ++p) pages.push_back(make_int2(b, p));
        }
    } else {
        for (int i = 0; i < n; ++i) pages.push_back(make_int2(seq_ids[i], page_ids[i]));
        std::sort(pages.begin(), pages.end(), [](int2 u, int2 w) { return u.x != w.x ? u.x < w.x : u.y < w.y; });
        pages.erase(std::unique(pages.begin(), pages.end(), [](int2 u, int2 w) { return u.x == w.x && u.y == w.y; }),
                    pages.end());
    }
    s->job_host.clear();
    for (const int2 &bp : pages)
        for (int l = 0; l < y.L; ++l)
            if (!has_factors(s, bp.x, l, bp.y)) s->job_host.push_back(make_int2((bp.x << 8) | l, bp.y));
    if (s->job_host.empty()) return PUZZLEKV_OK;
    // cannot trigger (a page outside the window always has factors, so at
    // most ring + 1 pages per (seq, layer) lack them)
    if ((int)s->job_host.size() > y.max_conv_jobs)
        return fail(PUZZLEKV_ERR_CAPACITY, "internal: conversion list overflow");
    for (const int2 &j : s->job_host) set_factors(s, j.x >> 8, j.x & 255, j.y);
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    // the job list region is shared with the background batches: order this
    // call after every pending one (later batches start after this stream's work)
    wait_conversions(s, strm, nullptr, nullptr, 0, true);
    int2 *dev_jobs = reinterpret_cast<int2 *>(s->workspace + y.jobs_offset);
    // pageable source: the copy has consumed job_host when cudaMemcpyAsync returns
    cudaError_t e = cudaMemcpyAsync(dev_jobs, s->job_host.data(), s->job_host.size() * sizeof(int2),
                                    cudaMemcpyHostToDevice, strm);
    if (e != cudaSuccess) return cuda_fail(e, "page list upload");
    FactorParams fp{};
    fp.mode = FACT_MODE_CONVERT_LIST;
    fp.max_ql_iter = 30;
    fp.status = status_ptr(s);
    fp.y = y;
    fp.P = y.P;
    fp.d = y.d;
    fp.x_esz = y.esz;
    fp.factor_pool = s->factor_pool;
    fp.dense_pool = s->dense_pool;
    fp.conv_list = dev_jobs;
    fp.n_jobs = (long)s->job_host.size() * y.H * 2;
    e = launch_factorize(fp, s->num_sms, strm);
    s->after_decode = false;
    if (e != cudaSuccess) return cuda_fail(e, "page list factorization launch");
    return PUZZLEKV_OK;
}

puzzlekv_status puzzlekv_convert_ready_pages(puzzlekv_store *s, void *stream) {
    NvtxRange nvtx_range("puzzlekv_convert_ready_pages");
    if (!s) return fail(PUZZLEKV_ERR_INVALID_ARG, "store is NULL");
    const Layout &y = s->y;
    // every complete page without factors, with its slack: the decode steps
    // left before the page leaves the window (length (p + 1) P + W)
    struct Ready {
        int slack, b, l, p;
    };
    std::vector<Ready> ready;
    for (int b = 0; b < y.Bmax; ++b) {
        for (int l = 0; l < y.L; ++l) {
            const int T = s->len[(size_t)b * y.L + l];
            if (T < 1) continue;
            const int complete = T / y.P;  // pages whose P tokens are all present
            for (int p = std::max(s->conv_upto[(size_t)b * y.L + l], y.sink_pages); p < complete; ++p)
                if (!has_factors(s, b, l, p)) ready.push_back({(p + 1) * y.P + y.W - T, b, l, p});
        }
    }
    if (ready.empty()) return PUZZLEKV_OK;
    // Pacing.  A page is complete W tokens before it leaves the window, so
    // its conversion can spread over those steps.  A new batch starts only
    // when the previous one has finished, with about one CTA per SM (page
    // jobs of H heads x {K, V} per entry), so that few conversion CTAs ever
    // wait for SMs beside the decode launches; pages within kUrgentSteps of
    // their deadline go at once whatever else runs.
    constexpr int kUrgentSteps = 8;
    bool busy = false;
    if (s->conv_stream) {
        const puzzlekv_store::ConvBatch &last = s->batches[(s->next_batch + kConvBatches - 1) % kConvBatches];
        if (last.pending) {
            const cudaError_t q = cudaEventQuery(last.done);
            if (q == cudaErrorNotReady) {
                busy = true;
                (void)cudaGetLastError();  // not an error: leave nothing behind for later launch checks
            } else if (q != cudaSuccess) {
                return cuda_fail(q, "conversion batch query");
            }
        }
    }
    std::stable_sort(ready.begin(), ready.end(), [](const Ready &u, const Ready &w) { return u.slack < w.slack; });
    size_t take = 0;
    while (take < ready.size() && ready[take].slack <= kUrgentSteps) ++take;
    if (!busy) take = std::max(take, std::min(ready.size(), (size_t)std::max(1, s->num_sms / (2 * y.H))));
    if (take == 0) return PUZZLEKV_OK;
    if ((int)take > y.max_conv_jobs) return fail(PUZZLEKV_ERR_CAPACITY, "internal: conversion list overflow");
    s->job_host.clear();
    for (size_t i = 0; i < take; ++i) {
        const Ready &r = ready[i];
        s->job_host.push_back(make_int2((r.b << 8) | r.l, r.p));
        set_factors(s, r.b, r.l, r.p);
    }
    if (s->job_host.empty()) return PUZZLEKV_OK;
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    puzzlekv_store::ConvBatch *cbp = nullptr;
    cudaError_t e = begin_batch(s, strm, cbp);
    if (e != cudaSuccess) return cuda_fail(e, "conversion stream setup");
    puzzlekv_store::ConvBatch &cb = *cbp;
    for (const int2 &j : s->job_host) {  // page p is factorized from length (p + 1) P + W on
        const int b = j.x >> 8;
        cb.deadline[b] = std::min(cb.deadline[b], (j.y + 1) * y.P + y.W);
        cb.uses[(size_t)b * y.L + (j.x & 255)] = 1;
    }
    int2 *dev_jobs = reinterpret_cast<int2 *>(s->workspace + y.jobs_offset);
    // the list region is reused only in the internal stream's order; pageable
    // source: the copy has consumed job_host when cudaMemcpyAsync returns
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(dev_jobs, s->job_host.data(), s->job_host.size() * sizeof(int2), cudaMemcpyHostToDevice,
                            s->conv_stream);
    if (e != cudaSuccess) return cuda_fail(e, "conversion list upload");
    FactorParams fp{};
    fp.mode = FACT_MODE_CONVERT_LIST;
    fp.max_ql_iter = 30;
    fp.status = status_ptr(s);
    fp.y = y;
    fp.P = y.P;
    fp.d = y.d;
    fp.x_esz = y.esz;
    fp.factor_pool = s->factor_pool;
    fp.dense_pool = s->dense_pool;
    fp.conv_list = dev_jobs;
    fp.n_jobs = (long)s->job_host.size() * y.H * 2;
    // one CTA per page job: a conversion CTA holds its SM for one short job
    // only, so decode CTAs waiting for SMs get them back soon (one CTA per SM
    // looping over its share of jobs held SMs for whole milliseconds)
    fp.max_ctas = (int)std::min<long>(fp.n_jobs, 1L << 30);
    e = launch_factorize(fp, s->num_sms, s->conv_stream);
    if (e == cudaSuccess) e = end_batch(s, cb);
    if (e != cudaSuccess) return cuda_fail(e, "batched conversion launch");
    return PUZZLEKV_OK;
}

puzzlekv_status puzzlekv_store_stats(const puzzlekv_store *s, int32_t seq, int32_t layer, int32_t *length,
                                     int64_t *dense_pages, int64_t *factored_pages, int64_t *bytes_live) {
    if (!s) return fail(PUZZLEKV_ERR_INVALID_ARG, "store is NULL");
    const Layout &y = s->y;
    if (seq < 0 || seq >= y.Bmax || layer < 0 || layer >= y.L)
        return fail(PUZZLEKV_ERR_INVALID_ARG, "seq or layer out of range");
    int T = std::max(0, s->len[(size_t)seq * y.L + layer]);
    int64_t nd = 0, nf = 0, bytes = 0;
    int n = (T + y.P - 1) / y.P;
    for (int p = 0; p < n; ++p) {
        if (host_page_kind(p, T, y.P, y.sink_tokens, y.W) == KIND_DENSE) {
            ++nd;
            int rows = std::min(y.P, T - p * y.P);
            bytes += (int64_t)rows * 2 * y.d * y.esz * y.H;
        } else {
            ++nf;
            bytes += (int64_t)(y.rk + y.rv) * (y.P + y.d) * y.esz * y.H;
        }
    }
    if (length) *length = T;
    if (dense_pages) *dense_pages = nd;
    if (factored_pages) *factored_pages = nf;
    if (bytes_live) *bytes_live = bytes;
    return PUZZLEKV_OK;
}

puzzlekv_status puzzlekv_debug_fail_next_wait(puzzlekv_store *s, int32_t where, int64_t wait_ns) {
    if (!s) return fail(PUZZLEKV_ERR_INVALID_ARG, "store is NULL");
    if (where < 0 || where > 2) return fail(PUZZLEKV_ERR_INVALID_ARG, "where must be 0, 1 or 2 (got %d)", where);
    if (wait_ns < 1000 || wait_ns > (int64_t)1000000000)
        return fail(PUZZLEKV_ERR_INVALID_ARG, "wait_ns must be in [1e3, 1e9] (got %lld)", (long long)wait_ns);
    if (s->y.dtype != 1) return fail(PUZZLEKV_ERR_UNSUPPORTED, "the hook exists on the bf16 decode path only");
    s->fail_next = where;
    s->fail_wait_ns = (uint64_t)wait_ns;
    return PUZZLEKV_OK;
}

puzzlekv_status puzzlekv_check_device_status(puzzlekv_store *s, void *stream) {
    if (!s) return fail(PUZZLEKV_ERR_INVALID_ARG, "store is NULL");
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    int words[STATUS_WORDS] = {0};
    cudaError_t e = cudaStreamSynchronize(strm);
    if (e == cudaSuccess && s->conv_stream) e = cudaStreamSynchronize(s->conv_stream);
    if (e == cudaSuccess) e = cudaMemcpy(words, status_ptr(s), sizeof(words), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(status_ptr(s), 0, sizeof(int) * STATUS_JOBS);  // flags only
    if (e == cudaSuccess && words[STATUS_TIMEOUT])  // a CTA that gave up never took its split ticket
        e = cudaMemset(s->workspace + s->y.ticket_offset, 0, s->y.jobs_offset - s->y.ticket_offset);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (words[STATUS_TIMEOUT]) return fail(PUZZLEKV_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait ran out");
    if (words[STATUS_NOT_CONVERGED])
        return fail(PUZZLEKV_ERR_NOT_CONVERGED, "%d page eigensolves hit the sweep cap", words[STATUS_NOT_CONVERGED]);
    return PUZZLEKV_OK;
}

puzzlekv_status puzzlekv_factorize_counters(puzzlekv_store *s, void *stream, int64_t *page_jobs,
                                            int64_t *ql_rotations) {
    if (!s || !page_jobs || !ql_rotations) return fail(PUZZLEKV_ERR_INVALID_ARG, "NULL argument");
    unsigned long long c[2] = {0, 0};  // status words 2-3 and 4-5
    static_assert(STATUS_ROTATIONS == STATUS_JOBS + 2, "counter words are adjacent");
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess && s->conv_stream) e = cudaStreamSynchronize(s->conv_stream);
    if (e == cudaSuccess) e = cudaMemcpy(c, status_ptr(s) + STATUS_JOBS, sizeof(c), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(status_ptr(s) + STATUS_JOBS, 0, sizeof(c));
    if (e != cudaSuccess) return cuda_fail(e, "counter read");
    *page_jobs = (int64_t)c[0];
    *ql_rotations = (int64_t)c[1];
    return PUZZLEKV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode attention with split-K scratch in a static device array.
//
// Some callers cannot allocate device memory at the point where they decode:
// serving runtimes that forbid allocation once they have started (so that the
// memory footprint stays fixed and no request can fail on, or wait for, the
// allocator), and embedders whose device memory belongs to another framework's
// allocator that this layer cannot reach.  Such callers cannot set aside a
// per-call scratch buffer for the split-K partial softmax states, so this
// entry point takes that scratch from a file-scope array instead.
namespace {

constexpr size_t kStaticScratchBytes = (size_t)16 << 20;  // 16 MiB per device

// Held by every GPU that loads this library, until the process exits.  In
// host code this name is only a host-side stand-in: its device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {nullptr};

}  // namespace

extern "C" puzzlekv_status puzzlekv_decode_attention_static_scratch(puzzlekv_store *s, int32_t layer, const void *q,
                                                                    float *out, const int32_t *seq_ids, int32_t B,
                                                                    void *stream) {
    NvtxRange nvtx_range("puzzlekv_decode_attention_static_scratch");
    puzzlekv_status st = check_call(s, layer, seq_ids, B);
    if (st != PUZZLEKV_OK) return st;
    if (!q || !out || !aligned16(q) || !aligned16(out))
        return fail(PUZZLEKV_ERR_INVALID_ARG, "q and out must be non-NULL and 16-byte aligned");
    const Layout &y = s->y;
    // split tickets, then the partial states
    const size_t ticket_bytes = ((size_t)y.Bmax * y.H * 8 + 255) & ~(size_t)255;
    const size_t need = ticket_bytes + (size_t)y.Bmax * y.Hq * MAX_SPLITS * y.part_stride * 4;
    if (need > kStaticScratchBytes)
        return fail(PUZZLEKV_ERR_CAPACITY,
                    "static decode scratch holds %zu bytes; this store needs %zu (max_batch x num_q_heads too large)",
                    kStaticScratchBytes, need);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(PUZZLEKV_ERR_UNSUPPORTED, "device index %d too large", dev);
    void *base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!g_scratch_addr[dev]) {  // first call on this device: look up the array's device address
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_decode_scratch);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static decode scratch)");
            g_scratch_addr[dev] = p;
        }
        base = g_scratch_addr[dev];
    }
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    // split tickets must start at zero; the array keeps the previous call's contents
    e = cudaMemsetAsync(base, 0, ticket_bytes, strm);
    if (e != cudaSuccess) return cuda_fail(e, "static scratch ticket reset");
    DecodeParams dp;
    long total;
    int max_pages;
    fill_decode_params(s, layer, q, out, seq_ids, B, 0, dp, total, max_pages);
    dp.tickets = static_cast<int *>(base);
    dp.wait_first = 1;
    wait_conversions(s, strm, seq_ids, dp.lens, B);
    dp.partials = reinterpret_cast<float *>(static_cast<char *>(base) + ticket_bytes);
    e = launch_decode(dp, total, max_pages, s->num_sms, strm);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch (static scratch)");
    s->after_decode = true;
    return PUZZLEKV_OK;
}
