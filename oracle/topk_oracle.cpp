// Oracle for the sparse-attention indexer's per-row top-k with its output
// transform. TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
// benchmark's CPU-baseline leg load it; the library's product path never does.
//
// Plain, slow, single-threaded C++17. It shares no code, header, table or
// helper with the CUDA library. Every step is the plain definition of the
// result, written out:
//
//   * The window of row b is the positions p = 0 .. L-1 of
//     scores[b * score_stride + row_start + p], with L = seq_lens[b] and
//     row_start = row_starts[b] (0 when row_starts is null).
//     (sglang PR #35175 page, "Implementation breakdown" item 2 and the
//     topk_ragged_kernel snippet: select top-k inside
//     [row_starts[b], row_starts[b] + seq_lens[b]).)
//   * When L <= k every position is emitted and no score is read (same
//     snippet, the "trivial path").
//   * Otherwise the window is sorted by (score descending, position ascending)
//     and the first k entries are kept. Scores are ordered by their fp32 bit
//     pattern mapped to an order-preserving unsigned 32-bit key, a total order
//     in which -0.0 sorts below +0.0. Equal scores go to the lowest position,
//     which is the deterministic reading of the tie rule (the PR #26788 page's
//     test snippet accepts any swap of equal scores; the PR #33006 report names
//     a deterministic tie-break flag without giving its value).
//   * RAGGED emit: p + out_offsets[b] (PR #35175 page, "Key source snippets",
//     TopKProblem::emit adds the bias to every selected index).
//   * PAGED emit: page_table[b * pt_stride + p / page_size] * page_size
//     + p % page_size (PR #35175 page, TopKProblem::transform_output through
//     page_to_indices; page_size = 1 << page_bits).
//   * Packed PAGED emit (oracle_topk_transform_packed): the score window
//     keeps its batch-global start row_starts[b], while the page-table lookup
//     uses the row's request table, row r = row_to_batch[b] (b when null), at
//     the request-local token t = page_table_row_starts[b] + p (p when null):
//     page_table[r * pt_stride + t / page_size] * page_size + t % page_size
//     (the PR #33006 report, "fix(dsa): use FlashInfer fused top-k for packed
//     PAGED rows": "功能与动机", and "实现拆解" item 2 with its snippet, where
//     page_table_row_starts = row_starts - cu_seqlens_k[row_to_batch]).
//     A negative page_table_row_starts[b] is a data error like a negative
//     row_start.
//   * Slots past the selected count hold -1, never biased or transformed
//     (PR #35175 page, "Review highlights": the trivial path cannot reuse a
//     helper whose -1 padding would pick up the bias).
//   * Selected positions are written in ascending position order (a canonical
//     form; the pages do not fix an output order).
//   * A row with seq_len < 0, or with row_start < 0, is a data error: it is
//     treated as an empty row (all -1) and counted in the return value (the
//     PR #35175 page states seq_lens must be non-negative).
//
//   * SWA combine (oracle_swa_combine; the PR #30255 page, "sparse_prefill_
//     utils.py": _combine_topk_swa_indices_kernel and combine_topk_swa_indices
//     merge the top-k indices with the sliding-window indices, topk_len =
//     min((pos + 1) // COMPRESS_RATIO, top_k); the page elides the kernel's
//     body, so this is the plainest reading of its signature): row b of width
//     `width` holds the row's selected entries (as the transform emitted them,
//     topk_len of them: with seq_len = (pos + 1) // COMPRESS_RATIO that is the
//     page's min((pos + 1) // COMPRESS_RATIO, top_k)), then the window's
//     tokens pos - w + 1 .. pos in ascending order, w = min(WINDOW_SIZE,
//     pos + 1) (none for pos < 0), each plus swa_offsets[b] (0 when null),
//     then -1 up to the width (the page's PADDED_TOP_K, at least top_k +
//     WINDOW_SIZE).
//
//   * Indexer logits (oracle_indexer_logits), the producer upstream of the
//     top-k. The pages name it without defining it: the PR #35175 page (the
//     PR body) says the DeepGEMM contiguous-KV indexer writes logit columns
//     at absolute positions of the batch-flattened KV, and the PR #36684
//     page ("Key source snippets", server_args.py) names an FP8 paged
//     MQA-logits kernel and ties the v2 path to tcgen05/TMEM. The plainest
//     reading of an FP8 multi-query logits producer, one key vector per KV
//     position shared by every head, is the lightning indexer's score:
//       logits[t][s] = kv_scale[s] * sum_h w[t][h] * max(0, q[t][h] . kv[s])
//     for ks[t] <= s < ke[t] (nothing is written elsewhere), with q and kv
//     in FP8 E4M3, w and kv_scale fp32. Row t of the logits is then the
//     RAGGED transform's window at row_start = ks[t], seq_len = ke[t] - ks[t].
//     E4M3 ("e4m3fn"): sign, 4 exponent bits with bias 7, 3 mantissa bits;
//     exponent field 0 holds the subnormals m/8 * 2^-6; S.1111.111 is NaN;
//     there is no infinity. Every product of two E4M3 values, and every sum
//     of up to 2^20 of them, is exact in fp64, so the dot products here are
//     exact; the weighted sum is fp64 and rounded to fp32 once.
//
// Parity pins (tests/test_oracle_pins.py): brute-force rank counting on tiny
// rows, an exhaustive sweep over short vectors with ties and signed zeros,
// invariants on every workload shape, numpy's partition on the tie-free
// special case, an independent page-table expansion, and hand-built examples
// under tests/golden/.
//
// ORACLE_MUTANT (compile-time, default 0) plants one deliberate mistake; it
// exists only so that a test can show each pin family catches that mistake.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

namespace {

// Order-preserving map from fp32 bits to uint32: a larger float gives a larger
// key. Negative values have every bit flipped, non-negative values only the
// sign bit set.
uint32_t order_key(float x) {
    uint32_t bits;
    std::memcpy(&bits, &x, sizeof(bits));
#if ORACLE_MUTANT == 3
    // mutant: order by float comparison only (loses -0.0 < +0.0)
    if (x == 0.0f) bits = 0u;
#endif
    if (bits & 0x80000000u) return ~bits;
    return bits | 0x80000000u;
}

struct Entry {
    uint32_t key;
    int32_t pos;
};

bool before(const Entry& a, const Entry& b) {
    if (a.key != b.key) return a.key > b.key;  // larger score first
#if ORACLE_MUTANT == 1
    return a.pos > b.pos;  // mutant: ties go to the highest position
#else
    return a.pos < b.pos;  // ties go to the lowest position
#endif
}

int32_t ragged_index(int32_t p, int32_t offset) { return p + offset; }

int32_t paged_index(const int32_t* pt_row, int32_t page_size, int32_t p) {
#if ORACLE_MUTANT == 2
    return pt_row[p / page_size] * page_size + (p + 1) % page_size;  // mutant
#else
    return pt_row[p / page_size] * page_size + p % page_size;
#endif
}

// The value of an FP8 E4M3 code (see the header).
double e4m3_value(uint8_t c) {
    const int e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
    const double mag = e == 0 ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
    return (c & 0x80u) ? -mag : mag;
}

// One head's weighted contribution w * max(0, dot) to a logit.
double head_term(double w, double dot) {
#if ORACLE_MUTANT == 10
    return w * dot;  // mutant: the ReLU is dropped
#elif ORACLE_MUTANT == 11
    return std::max(w * dot, 0.0);  // mutant: the ReLU taken after the head weight
#else
    return w * std::max(dot, 0.0);
#endif
}

}  // namespace

extern "C" {

// mode: 0 = RAGGED (out_offsets used), 1 = PAGED (page_table used).
// scores: host fp32; row b's window starts at scores + b*score_stride + row_start.
// page_table_row_starts, row_to_batch: PAGED only, may be null (packed PAGED).
// out, out_raw: [batch, k] int32 (out_raw may be null).
// Returns the number of rows with a data error (seq_len < 0, row_start < 0 or
// page_table_row_start < 0).
int64_t oracle_topk_transform_packed(int32_t mode, const float* scores, int64_t score_stride,
                                     const int32_t* row_starts, const int32_t* seq_lens,
                                     const int32_t* out_offsets, const int32_t* page_table,
                                     int64_t page_table_stride, int32_t page_size,
                                     const int32_t* page_table_row_starts, const int32_t* row_to_batch,
                                     int32_t batch, int32_t k, int32_t* out, int32_t* out_raw) {
    int64_t errors = 0;
    std::vector<Entry> window;
    std::vector<int32_t> selected;
    for (int32_t b = 0; b < batch; ++b) {
        int32_t L = seq_lens[b];
        const int32_t start = row_starts ? row_starts[b] : 0;
#if ORACLE_MUTANT == 7
        const int32_t token0 = 0;  // mutant: the packed page-table start is ignored
#else
        const int32_t token0 = (mode == 1 && page_table_row_starts) ? page_table_row_starts[b] : 0;
#endif
        const int64_t table_row = (mode == 1 && row_to_batch) ? row_to_batch[b] : b;
        if (L < 0 || start < 0 || token0 < 0) {
            ++errors;
            L = 0;
        }
#if ORACLE_MUTANT == 4
        const float* row = scores + (int64_t)b * score_stride;  // mutant: start ignored
#else
        const float* row = scores + (int64_t)b * score_stride + start;
#endif
        selected.clear();
        if (L <= k) {
            for (int32_t p = 0; p < L; ++p) selected.push_back(p);
        } else {
            window.clear();
#if ORACLE_MUTANT == 5
            for (int32_t p = 0; p < L - 1; ++p) window.push_back({order_key(row[p]), p});
#else
            for (int32_t p = 0; p < L; ++p) window.push_back({order_key(row[p]), p});
#endif
            std::sort(window.begin(), window.end(), before);
            for (int32_t t = 0; t < k && t < (int32_t)window.size(); ++t)
                selected.push_back(window[t].pos);
            std::sort(selected.begin(), selected.end());
        }
        int32_t* o = out + (int64_t)b * k;
        int32_t* r = out_raw ? out_raw + (int64_t)b * k : nullptr;
        for (int32_t t = 0; t < k; ++t) {
            int32_t value = -1;
            int32_t raw = -1;
            if (t < (int32_t)selected.size()) {
                raw = selected[t];
                if (mode == 1)
                    value = paged_index(page_table + table_row * page_table_stride, page_size, token0 + raw);
                else
                    value = ragged_index(raw, out_offsets[b]);
            }
#if ORACLE_MUTANT == 6
            else if (mode == 0) {
                value = -1 + out_offsets[b];  // mutant: padding picks up the bias
            }
#endif
            o[t] = value;
            if (r) r[t] = raw;
        }
    }
    return errors;
}

// The plain form: every page-table lookup in the row's own table from token 0.
int64_t oracle_topk_transform(int32_t mode, const float* scores, int64_t score_stride,
                              const int32_t* row_starts, const int32_t* seq_lens,
                              const int32_t* out_offsets, const int32_t* page_table,
                              int64_t page_table_stride, int32_t page_size, int32_t batch,
                              int32_t k, int32_t* out, int32_t* out_raw) {
    return oracle_topk_transform_packed(mode, scores, score_stride, row_starts, seq_lens, out_offsets,
                                        page_table, page_table_stride, page_size, nullptr, nullptr, batch, k,
                                        out, out_raw);
}

// SWA combine (see the header): out / out_raw are the transform's [batch, k]
// rows (out_raw's -1 padding marks where the selected entries end),
// positions[b] the row's query position, result [batch, width].
void oracle_swa_combine(int32_t batch, int32_t k, const int32_t* out, const int32_t* out_raw,
                        const int32_t* positions, int32_t window_size, const int32_t* swa_offsets,
                        int32_t width, int32_t* result) {
    for (int32_t b = 0; b < batch; ++b) {
        const int32_t* o = out + (int64_t)b * k;
        const int32_t* r = out_raw + (int64_t)b * k;
        int32_t* res = result + (int64_t)b * width;
        int32_t n = 0;
        while (n < k && r[n] >= 0) ++n;  // the selected entries lead the row
        int32_t t = 0;
        for (int32_t i = 0; i < n; ++i) res[t++] = o[i];
#if ORACLE_MUTANT == 9
        for (int32_t i = 0; i < n; ++i) res[i] = r[i];  // mutant: untransformed positions
#endif
        const int32_t pos = positions[b];
        const int32_t w = pos < 0 ? 0 : std::min(window_size, pos + 1);
        const int32_t off = swa_offsets ? swa_offsets[b] : 0;
        for (int32_t i = 0; i < w; ++i) {
#if ORACLE_MUTANT == 8
            res[t++] = pos - w + i + off;  // mutant: the window ends one token early
#else
            res[t++] = pos - w + 1 + i + off;
#endif
        }
        while (t < width) res[t++] = -1;
    }
}

double oracle_e4m3_value(uint8_t code) { return e4m3_value(code); }

// Indexer logits (see the header): q [n_q, heads, dim] and kv [n_kv, dim] E4M3
// codes, kv_scale [n_kv], weights [n_q, heads]; row t of `out` (stride
// out_stride) gets columns max(ks[t], 0) .. min(ke[t], n_kv) - 1 and nothing
// else.
void oracle_indexer_logits(const uint8_t* q, const uint8_t* kv, const float* kv_scale, const float* weights,
                           const int32_t* ks, const int32_t* ke, int32_t n_q, int32_t heads, int32_t dim,
                           int64_t n_kv, float* out, int64_t out_stride) {
    for (int32_t t = 0; t < n_q; ++t) {
        const int64_t lo = std::max<int64_t>(ks[t], 0), hi = std::min<int64_t>(ke[t], n_kv);
        for (int64_t s = lo; s < hi; ++s) {
            double acc = 0.0;
            for (int32_t h = 0; h < heads; ++h) {
                const uint8_t* qh = q + ((int64_t)t * heads + h) * dim;
                const uint8_t* ks_row = kv + s * dim;
                double dot = 0.0;
                for (int32_t d = 0; d < dim; ++d) dot += e4m3_value(qh[d]) * e4m3_value(ks_row[d]);
                acc += head_term(weights[(int64_t)t * heads + h], dot);
            }
#if ORACLE_MUTANT == 12
            out[(int64_t)t * out_stride + s] = (float)acc;  // mutant: the key's scale is dropped
#else
            out[(int64_t)t * out_stride + s] = (float)((double)kv_scale[s] * acc);
#endif
        }
    }
}

}  // extern "C"
