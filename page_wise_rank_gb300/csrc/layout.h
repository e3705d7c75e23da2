// Device-memory layout of the paged factor store (host and device code).
//
// Everything the library keeps in HBM lives in four caller-owned buffers:
//
//   factor pool  [layer][seq][kv_head][page] -> one factor record per page
//                (preallocated for every page a sequence can hold, so a page
//                converted during decoding never needs an allocation --
//                "PuzzleKV: Page-Wise Low-Rank Decomposition for KV Cache
//                Compression", §3.3 ⑤).
//   dense pool   [layer][seq][dense slot][kv_head][K|V][P][d]: sink pages
//                take slots 0..sink_pages-1, every other dense page takes
//                slot sink_pages + (page mod ring).  The ring is wide enough
//                for the window, the page being filled and the page being
//                converted, so a slot is "released" simply by the page
//                leaving the ring.
//   page table   int32 lengths[seq][layer], then int32 desc[seq][layer][page]
//                = kind << 30 | slot.
//   workspace    int32 status words, int32 split tickets [seq][kv_head][2] (one
//                counter, padded),
//                the batched-conversion job list (int2 per page), then
//                fp32 split-K partial states [seq][q_head][split][4 + d]
//                (m, l, two pad words, o[d]: 16-byte aligned rows).
//
// Factor record of one (layer, seq, kv head, page), element type e:
//   LK  [P][rkp]    key left factor,   row = token   (B operand of s = t L_K^T)
//   RK  [rkp][d]    key right factor,  row = rank    (B operand of t = q R_K^T)
//   LVt [rvp][P]    value left factor, transposed: row = rank
//   RVt [d][rvp]    value right factor, transposed: row = head dim
// rkp / rvp are the ranks rounded up to a multiple of 8 (zero padding).  Each
// row is a sequence of 16-byte chunks whose order is XOR-swizzled by row
// (swizzle_chunk below) so that eight consecutive rows read at the same
// logical chunk hit eight distinct bank groups; dense K/V rows use the same
// rule.  The record is contiguous, so one bulk copy brings a page into shared
// memory already in its conflict-free layout.
#pragma once
#include <stddef.h>
#include <stdint.h>

#if defined(__CUDACC__)
#define PKV_HD __host__ __device__ __forceinline__
#else
#define PKV_HD inline
#endif

namespace pkv {

constexpr int KIND_SHIFT = 30;
constexpr int32_t SLOT_MASK = (1 << KIND_SHIFT) - 1;
constexpr int KIND_FACTORED = 0;
constexpr int KIND_DENSE = 1;
constexpr int MAX_SPLITS = 128;     // split-K partials per (seq, q head)
constexpr int MAX_CHUNK_PAGES = 256; // pages per decode CTA
constexpr int MAX_CALL_BATCH = 64;  // sequences per append / attention call
constexpr int STATUS_WORDS = 16;    // int32 status words at the workspace start
constexpr int STATUS_NOT_CONVERGED = 0;
constexpr int STATUS_TIMEOUT = 1;
constexpr int STATUS_JOBS = 2;      // uint64 at words 2-3: page jobs factorized
constexpr int STATUS_ROTATIONS = 4; // uint64 at words 4-5: QL rotations those jobs applied (rank > P / 2)

PKV_HD int gcd8(int c) { return (c & 7) == 0 ? 8 : ((c & 3) == 0 ? 4 : ((c & 1) == 0 ? 2 : 1)); }

// Physical 16-byte chunk of logical chunk `c` in row `row` of a row made of
// `C` chunks.  Bijective within a row; conflict-free for 8 consecutive rows.
PKV_HD int swizzle_chunk(int row, int c, int C) {
    int g = gcd8(C);
    if (g == 1) return c;
    int period = 8 / g;
    return c ^ ((row / period) & (g - 1));
}

// Byte offset of byte `b` of row `row` in a swizzled tile whose rows are
// `pitch` bytes (a multiple of 16).
PKV_HD uint32_t swz_offset(int row, int b, int pitch) {
    int C = pitch >> 4;
    return (uint32_t)(row * pitch + (swizzle_chunk(row, b >> 4, C) << 4) + (b & 15));
}

PKV_HD int round_up8(int x) { return (x + 7) & ~7; }

// Page classification [PuzzleKV §3.3 ①②③, ⑤]: dense if the page holds one of
// the first sink_tokens tokens, one of the last W tokens, or is incomplete.
PKV_HD int page_kind(int p, int T, int P, int sink_tokens, int W) {
    int first = p * P;
    int end = first + P < T ? first + P : T;
    int sink_pages = (sink_tokens + P - 1) / P;
    bool dense = (p < sink_pages) || (end - first < P) || (end > T - W);
    return dense ? KIND_DENSE : KIND_FACTORED;
}

// Tokens in half `half` of page p (P/2 rows) of a sequence of T tokens.
PKV_HD int dense_half_valid(int T, int p, int P, int half) {
    int first = p * P + half * (P / 2);
    int v = T - first;
    return v < 0 ? 0 : (v > P / 2 ? P / 2 : v);
}

// Bytes a dense page streams in decode: a K and a V half page per non-empty half.
PKV_HD long long dense_page_bytes(int p, int T, int P, long long half_bytes) {
    return (dense_half_valid(T, p, P, 0) > 0 ? half_bytes : 0) + (dense_half_valid(T, p, P, 1) > 0 ? half_bytes : 0);
}

// Split of one sequence's pages over the n CTAs of a (sequence, KV head)
// decode group, balanced by the bytes each CTA streams: page p goes to the CTA
// whose equal share of the total holds the page's midpoint.  The kinds follow
// the classification rule -- dense sink pages [0, fs), factorized pages
// [fs, fw), dense window pages [fw, n_pages) -- so the factorized stretch is
// counted in closed form and only the few dense pages are walked.
struct PageSplit {
    int T, P, n_pages, fs, fw, n;
    long long rec, half, total;
    PKV_HD PageSplit(int T_, int P_, int sink_pages, int sink_tokens, int W, long long rec_bytes,
                     long long half_bytes, int n_)
        : T(T_), P(P_), n(n_), rec(rec_bytes), half(half_bytes) {
        n_pages = (T + P - 1) / P;
        fs = sink_pages < n_pages ? sink_pages : n_pages;
        fw = n_pages;
        while (fw > fs && page_kind(fw - 1, T, P, sink_tokens, W) == KIND_DENSE) --fw;
        total = (long long)(fw - fs) * rec;
        for (int p = 0; p < fs; ++p) total += dense_page_bytes(p, T, P, half);
        for (int p = fw; p < n_pages; ++p) total += dense_page_bytes(p, T, P, half);
    }
    // first page of CTA r: the pages whose midpoint lies below r / n of the
    // bytes, i.e. n (2 before + cost) < 2 total r
    PKV_HD int begin(int r) const {
        if (r <= 0) return 0;
        if (r >= n) return n_pages;
        const long long lim = 2 * total * r;
        long long before = 0;
        int cnt = 0;
        for (int p = 0; p < fs; ++p) {
            const long long c = dense_page_bytes(p, T, P, half);
            if (n * (2 * before + c) >= lim) return cnt;
            before += c;
            ++cnt;
        }
        // factorized pages j = 0, 1, ...: n (2 (before + j rec) + rec) < lim  <=>  j < rhs / step
        const long long rhs = lim - n * (2 * before + rec), step = 2 * (long long)n * rec;
        const long long k = rhs <= 0 ? 0 : (rhs + step - 1) / step;
        if (k < fw - fs) return cnt + (int)k;
        cnt += fw - fs;
        before += (long long)(fw - fs) * rec;
        for (int p = fw; p < n_pages; ++p) {
            const long long c = dense_page_bytes(p, T, P, half);
            if (n * (2 * before + c) >= lim) return cnt;
            before += c;
            ++cnt;
        }
        return cnt;
    }
};

// INT4 code streams [PuzzleKV §4.3].  Each factor enters the decode as the B
// operand (K x N, K the contraction) of m16n8k16 / m16n8k8 fp16 tensor-core
// products: R_K as B[k = head dim][n = rank], L_K as B[rank][token], L_V as
// B[token][rank], R_V as B[rank][head dim].  A factor's B operand is cut into
// k-steps (16-wide, then one 8-wide step if K is an odd multiple of 8), each
// k-step into n-tiles of 8, k-step outer; a 16-wide tile gives every lane
// (lane = 4 g + c) two registers b0 = (k0 + 2c, k0 + 2c + 1; n0 + g) and
// b1 = (k0 + 8 + 2c, k0 + 9 + 2c; n0 + g), an 8-wide tile one register b0.
// The key stream is R_K's registers then L_K's, the value stream L_V's then
// R_V's.  Register m of a lane sits in word m / 4 of the lane, nibbles
// (m % 4) and (m % 4) + 4 (the register's first and second element); words
// are laid out in 256-byte slabs of two words per lane: word w of lane l at
// byte ((w / 2) * 32 + l) * 8 + (w % 2) * 4.  Unused nibbles hold 8 (code 0).
PKV_HD int q4_operand_regs(int K, int N) { return K * N / 64; }  // registers per lane
PKV_HD int q4_stream_regs(int K0, int r, int K1) {  // B1 = K0 x r, then B2 = r x K1
    return q4_operand_regs(K0, r) + q4_operand_regs(r, K1);
}
// Element (k, n) of a K x N B operand held by register m (relative to the
// operand's first register) of lane `lane`, element `e` (0 or 1).
PKV_HD void q4_operand_elem(int K, int N, int m, int lane, int e, int &k, int &n) {
    const int g = lane >> 2, c = lane & 3, nt = N / 8, k16 = K / 16;
    if (m < k16 * 2 * nt) {
        const int ks = m / (2 * nt), rem = m % (2 * nt);
        k = 16 * ks + 8 * (rem & 1) + 2 * c + e;
        n = 8 * (rem >> 1) + g;
    } else {
        k = 16 * k16 + 2 * c + e;
        n = 8 * (m - k16 * 2 * nt) + g;
    }
}
// Position of element i of a scale vector of length K (a multiple of 8) in
// accumulator-column order: lane c's elements (8 t + 2c, 8 t + 2c + 1) for
// t = 0 .. K/8 - 1 are contiguous, lanes c = 0..3 one after another.
PKV_HD int q4_scale_index(int K, int i) { return ((i & 7) >> 1) * (K / 4) + (i >> 3) * 2 + (i & 1); }
// Position of element n of a head-dim scale vector (s_RK, s_RV; the length
// is a multiple of 16) in k-step order: per 16 columns, lane c's four
// elements 2c, 2c + 1, 8 + 2c, 9 + 2c contiguous, lanes c = 0..3 one after
// another, so the four lanes of a row read 32 contiguous bytes (one bank
// each) instead of quarters 64 bytes apart (two on each bank).
PKV_HD int q4_dscale_index(int n) { return (n >> 4) * 16 + ((n & 7) >> 1) * 4 + ((n >> 3) & 1) * 2 + (n & 1); }

struct Layout {
    int L, H, Hq, G, d, P, rk, rv, rkp, rvp, sink_tokens, W, Bmax, Tmax, esz, dtype;
    int n_pg_max, sink_pages, ring, dslots;
    size_t rec_bytes, off_RK, off_LV, off_RV;
    // INT4 factor records [PuzzleKV §4.3] (q4 = 1): a key stream and a value
    // stream of 4-bit codes (code + 8) in tensor-core operand order (Q4Stream
    // below), each a whole number of 256-byte slabs, then fp16 scales: s_RK
    // [d] (per head-dim column of R_K) and s_RV [d] (per head-dim column of
    // R_V) in k-step order (q4_dscale_index), s_LV [P] (per token row of L_V)
    // and s_LK [rkp] (per rank column of L_K) in accumulator-column order
    // (q4_scale_index).
    int q4;
    int q_kslabs, q_vslabs;  // 256-byte slabs of the key / value code streams
    // Keys stored before RoPE (rope = 1), turned at attention by
    // theta_i = rope_theta^(-2i/d): the workspace holds (cos, sin) float2
    // tables of the angles p P theta_i of every page's first position
    // ([n_pg_max][d/2] at rope_base_offset) and of the offsets delta theta_i
    // inside a page ([P][d/2] at rope_delta_offset).
    int rope;
    float rope_theta;
    size_t rope_base_offset, rope_delta_offset;
    size_t q_off_V, q_off_sRK, q_off_sRV, q_off_sLV, q_off_sLK;
    size_t dense_half_bytes;  // one K or V page: P * d * esz
    size_t factor_pool_bytes, dense_pool_bytes, page_table_bytes, workspace_bytes;
    size_t desc_offset;       // byte offset of desc[] in the page table
    size_t ticket_offset;     // byte offset of the per-(seq, kv head) split tickets in the workspace
    size_t jobs_offset;       // byte offset of the batched-conversion job list in the workspace
    int max_conv_jobs;        // entries of that list: one per (seq, layer, page) awaiting conversion
    size_t partial_offset;    // byte offset of split partials in the workspace
    int part_stride;          // floats per partial row: m, l, 2 pad, o[d]

    PKV_HD size_t record_index(int l, int b, int h, int p) const {
        return (((size_t)l * Bmax + b) * H + h) * (size_t)n_pg_max + p;
    }
    PKV_HD size_t record_offset(int l, int b, int h, int p) const { return record_index(l, b, h, p) * rec_bytes; }
    PKV_HD int dense_slot(int p) const { return p < sink_pages ? p : sink_pages + (p % ring); }
    // byte offset of the K (kv = 0) or V (kv = 1) half of a dense slot
    PKV_HD size_t dense_offset(int l, int b, int slot, int h, int kv) const {
        return (((((size_t)l * Bmax + b) * dslots + slot) * H + h) * 2 + kv) * dense_half_bytes;
    }
    PKV_HD size_t len_index(int b, int l) const { return (size_t)b * L + l; }
    PKV_HD size_t desc_index(int b, int l, int p) const { return ((size_t)b * L + l) * n_pg_max + p; }
    PKV_HD size_t partial_index(int b, int hq, int s) const { return ((size_t)b * Hq + hq) * MAX_SPLITS + s; }
    // one arrival counter per (seq, kv head), padded to two ints
    PKV_HD size_t ticket_index(int b, int h) const { return 2 * ((size_t)b * H + h); }
};

// Fill a Layout from a validated configuration.
inline void make_layout(Layout &y, int L, int H, int Hq, int d, int P, int rk, int rv, int sink, int W,
                        int Bmax, int Tmax, int dtype, int q4 = 0, float rope_theta = 0.f) {
    y.L = L; y.H = H; y.Hq = Hq; y.G = Hq / H; y.d = d; y.P = P; y.rk = rk; y.rv = rv;
    y.rkp = round_up8(rk); y.rvp = round_up8(rv);
    y.sink_tokens = sink; y.W = W; y.Bmax = Bmax; y.Tmax = Tmax; y.dtype = dtype;
    y.esz = dtype == 1 ? 2 : 4;
    y.n_pg_max = (Tmax + P - 1) / P;
    y.sink_pages = (sink + P - 1) / P;
    y.ring = (W + P - 1) / P + 2;
    y.dslots = y.sink_pages + y.ring;
    size_t e = (size_t)y.esz;
    y.off_RK = (size_t)P * y.rkp * e;
    y.off_LV = y.off_RK + (size_t)y.rkp * d * e;
    y.off_RV = y.off_LV + (size_t)y.rvp * P * e;
    y.rec_bytes = y.off_RV + (size_t)d * y.rvp * e;
    y.q4 = q4;
    {  // INT4 record: code streams, then scale vectors, each a multiple of 16 bytes
        y.q_kslabs = (q4_stream_regs(d, y.rkp, P) + 7) / 8;
        y.q_vslabs = (q4_stream_regs(P, y.rvp, d) + 7) / 8;
        size_t o = (size_t)y.q_kslabs * 256;
        y.q_off_V = o;
        o += (size_t)y.q_vslabs * 256;
        y.q_off_sRK = o;
        o += (size_t)d * 2;
        y.q_off_sRV = o;
        o += (size_t)d * 2;
        y.q_off_sLV = o;
        o += (size_t)P * 2;
        y.q_off_sLK = o;
        o += (size_t)y.rkp * 2;
        if (q4) y.rec_bytes = o;
    }
    y.dense_half_bytes = (size_t)P * d * e;
    y.factor_pool_bytes = (size_t)L * Bmax * H * y.n_pg_max * y.rec_bytes;
    y.dense_pool_bytes = (size_t)L * Bmax * y.dslots * H * 2 * y.dense_half_bytes;
    size_t len_bytes = ((size_t)Bmax * L * 4 + 255) & ~(size_t)255;
    y.desc_offset = len_bytes;
    y.page_table_bytes = len_bytes + (((size_t)Bmax * L * y.n_pg_max * 4 + 255) & ~(size_t)255);
    y.ticket_offset = 256;
    y.jobs_offset = y.ticket_offset + (((size_t)Bmax * H * 8 + 255) & ~(size_t)255);
    y.max_conv_jobs = Bmax * L * (y.ring + 1);
    y.partial_offset = y.jobs_offset + (((size_t)y.max_conv_jobs * 8 + 255) & ~(size_t)255);
    y.part_stride = d + 4;
    y.workspace_bytes = y.partial_offset + (size_t)Bmax * Hq * MAX_SPLITS * y.part_stride * 4;
    y.rope = rope_theta > 0.f;
    y.rope_theta = rope_theta;
    y.rope_base_offset = y.rope_delta_offset = 0;
    if (y.rope) {
        y.rope_base_offset = (y.workspace_bytes + 255) & ~(size_t)255;
        y.rope_delta_offset = y.rope_base_offset + (((size_t)y.n_pg_max * (d / 2) * 8 + 255) & ~(size_t)255);
        y.workspace_bytes = y.rope_delta_offset + (size_t)P * (d / 2) * 8;
    }
}

}  // namespace pkv
