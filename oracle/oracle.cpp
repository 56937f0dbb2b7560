// Float64 CPU oracle for split-KV decode attention (flash-decoding).
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
// call this file: only tests/, the smoke check and bench.py's CPU-baseline
// leg do. It shares no code with the CUDA library.
//
// What it computes, and where the pages define it:
//
//  * oracle_attention: the plain definition, with no split. For query head h
//    of sequence b, whose KV head is kvh = h / (Hq / Hkv):
//        s_j = scale * sum_d q[b,h,d] * k_j[kvh,d]          j in [0, L_b)
//        p_j = exp(s_j - max s) / sum_i exp(s_i - max s)
//        out[b,h,:] = sum_j p_j * v_j[kvh,:]
//    (MiniInfer flash_decode_splitk.py, flash_decode_reference: softmax of
//    the scaled scores times V, here in float64 and without its cast of the
//    probabilities to the input dtype; the GQA head mapping is the
//    cur_kv_head rule of the TileLang decode_attention_splitkv.py split
//    segment.) It also reports lse = ln sum_j exp(s_j).
//
//  * oracle_split_partials: the per-split values of the flash-decoding
//    split step. Split s of a length-L sequence covers
//        [floor(L*s/S), floor(L*(s+1)/S))
//    (TileLang decode_attention_splitkv.py, split segment: proportional
//    split bounds; module docstring item 4 gives the reason). For it:
//        lse_s = ln sum_{j in s} exp(s_j)
//        o_s   = sum_{j in s} exp(s_j - lse_s) * v_j
//    (CS349E lecture 11, 04_flash_decoding.py, demo1_exact, first
//    observation). An empty split has lse_s = -inf and o_s = 0, the
//    convention of the MiniInfer reduce kernel (m = -inf, l = 0 gives the
//    split weight 0).
//
//  * Several new query tokens per sequence (the _mq functions): each sequence
//    has tq query tokens, stored [B, tq, Hq, D], whose keys and values are
//    already the last tq rows of its cache. Token t sits at position L - tq + t
//    and sees the keys before and at it, j < L - tq + t + 1 (causal decoding
//    of several tokens at once); a token that sees no key gets out = 0. The
//    splits still cut the whole range [0, L); a split holding no key a token
//    may see is empty for that token. With tq = 1 every function reduces to
//    the single-query one above.
//
//  * oracle_merge: the exact log-sum-exp combine of the same observation:
//        lse = ln sum_s exp(lse_s),   o = sum_s exp(lse_s - lse) * o_s,
//    with the maximum subtracted first, as the TileLang combine segment does.
//    Splits with lse_s = -inf get weight 0; if every split is empty the
//    output is 0 and lse = -inf.
//
// Inputs are binary16 or bfloat16 bit patterns, decoded here to double from
// the IEEE 754 binary16 and the bfloat16 encodings. All arithmetic is double.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

struct Problem {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const int32_t* cu;
    int32_t B, Hq, Hkv, D;
    int64_t kv_rows;
    int32_t dtype;   // 0 binary16, 1 bfloat16
    int32_t layout;  // 0 varlen [kv_rows, Hkv, D]; 1 bhsd [B, Hkv, kv_rows, D]
    double scale;
    int32_t tq;      // query tokens per sequence, q and out [B, tq, Hq, D]
};

const double kNegInf = -std::numeric_limits<double>::infinity();

double decode_f16(uint16_t h) {
    int sign = h >> 15, e = (h >> 10) & 0x1f, m = h & 0x3ff;
    double val;
    if (e == 0) val = std::ldexp((double)m, -24);
    else if (e == 31) val = m ? std::numeric_limits<double>::quiet_NaN() : std::numeric_limits<double>::infinity();
    else val = std::ldexp((double)(1024 + m), e - 25);
    return sign ? -val : val;
}

double decode_bf16(uint16_t h) {
    int sign = h >> 15, e = (h >> 7) & 0xff, m = h & 0x7f;
    double val;
    if (e == 0) val = std::ldexp((double)m, -133);
    else if (e == 255) val = m ? std::numeric_limits<double>::quiet_NaN() : std::numeric_limits<double>::infinity();
    else val = std::ldexp((double)(128 + m), e - 134);
    return sign ? -val : val;
}

inline double dec(const Problem& p, uint16_t bits) {
    return p.dtype == 0 ? decode_f16(bits) : decode_bf16(bits);
}

inline int64_t seq_len(const Problem& p, int b) { return (int64_t)p.cu[b + 1] - (int64_t)p.cu[b]; }

// Keys query token t of sequence b may see: [0, L - tq + t + 1), clamped to [0, L].
inline int64_t visible(const Problem& p, int b, int t) {
    int64_t v = seq_len(p, b) - p.tq + t + 1;
    return v < 0 ? 0 : v;
}

// Element offset of (sequence b, key j, KV head kvh, dim 0).
inline int64_t kv_offset(const Problem& p, int b, int64_t j, int kvh) {
    if (p.layout == 0) return (((int64_t)p.cu[b] + j) * p.Hkv + kvh) * (int64_t)p.D;
    return (((int64_t)b * p.Hkv + kvh) * p.kv_rows + j) * (int64_t)p.D;
}

bool valid(const Problem& p) {
    if (!p.q || !p.cu || p.B < 0 || p.Hq < 1 || p.Hkv < 1 || p.D < 1) return false;
    if (p.Hq % p.Hkv != 0) return false;
    if (p.dtype != 0 && p.dtype != 1) return false;
    if (p.layout != 0 && p.layout != 1) return false;
    for (int b = 0; b < p.B; ++b) {
        if (seq_len(p, b) < 0) return false;
        if (p.layout == 0 && (p.cu[b] < 0 || p.cu[b + 1] > p.kv_rows)) return false;
        if (p.layout == 1 && seq_len(p, b) > p.kv_rows) return false;
    }
    return true;
}

// s_j for one (b, h) over [lo, hi): scale * q . k_j, in double.
void scores(const Problem& p, int b, int t, int h, int64_t lo, int64_t hi, std::vector<double>& qd,
            double* s) {
    int kvh = h / (p.Hq / p.Hkv);
    const uint16_t* qrow = p.q + (((int64_t)b * p.tq + t) * p.Hq + h) * p.D;
    qd.resize(p.D);
    for (int d = 0; d < p.D; ++d) qd[d] = dec(p, qrow[d]);
    for (int64_t j = lo; j < hi; ++j) {
        const uint16_t* krow = p.k + kv_offset(p, b, j, kvh);
        double acc = 0.0;
        for (int d = 0; d < p.D; ++d) acc += qd[d] * dec(p, krow[d]);
        s[j - lo] = p.scale * acc;
    }
}

// The plain definition for one (b, t, h): out[D] and lse.
void attend_row(const Problem& p, int b, int t, int h, double* out, double* lse) {
    int64_t L = visible(p, b, t);
    int kvh = h / (p.Hq / p.Hkv);
    for (int d = 0; d < p.D; ++d) out[d] = 0.0;
    if (L == 0) {
        *lse = kNegInf;
        return;
    }
    std::vector<double> s((size_t)L), qd;
    scores(p, b, t, h, 0, L, qd, s.data());
    double m = kNegInf;
    for (int64_t j = 0; j < L; ++j) m = s[j] > m ? s[j] : m;
    double z = 0.0;
    for (int64_t j = 0; j < L; ++j) {
        s[j] = std::exp(s[j] - m);
        z += s[j];
    }
    for (int64_t j = 0; j < L; ++j) {
        double pj = s[j] / z;
        const uint16_t* vrow = p.v + kv_offset(p, b, j, kvh);
        for (int d = 0; d < p.D; ++d) out[d] += pj * dec(p, vrow[d]);
    }
    *lse = m + std::log(z);
}

void split_bounds(int64_t L, int64_t S, int64_t s, int64_t* lo, int64_t* hi) {
    *lo = L * s / S;
    *hi = L * (s + 1) / S;
}

// Per-split partials for one (b, t, h): o_part[S][D], lse[S].
void split_row(const Problem& p, int b, int t, int h, int S, double* o_part, double* lse) {
    int64_t L = seq_len(p, b), vis = visible(p, b, t);
    int kvh = h / (p.Hq / p.Hkv);
    std::vector<double> s, qd;
    for (int sp = 0; sp < S; ++sp) {
        double* o = o_part + (int64_t)sp * p.D;
        for (int d = 0; d < p.D; ++d) o[d] = 0.0;
        int64_t lo, hi;
        split_bounds(L, S, sp, &lo, &hi);
        if (hi > vis) hi = vis;   // keys this token may not see
        if (hi <= lo) {
            lse[sp] = kNegInf;
            continue;
        }
        s.resize((size_t)(hi - lo));
        scores(p, b, t, h, lo, hi, qd, s.data());
        double m = kNegInf;
        for (double x : s) m = x > m ? x : m;
        double z = 0.0;
        for (double x : s) z += std::exp(x - m);
        double l = m + std::log(z);
        lse[sp] = l;
        for (int64_t j = lo; j < hi; ++j) {
            double w = std::exp(s[j - lo] - l);
            const uint16_t* vrow = p.v + kv_offset(p, b, j, kvh);
            for (int d = 0; d < p.D; ++d) o[d] += w * dec(p, vrow[d]);
        }
    }
}

template <class F>
void parallel_rows(int64_t rows, int nthreads, F f) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if (nthreads > rows) nthreads = (int)(rows > 0 ? rows : 1);
    if (nthreads == 1) {
        for (int64_t r = 0; r < rows; ++r) f(r);
        return;
    }
    std::vector<std::thread> pool;
    pool.reserve(nthreads);
    for (int t = 0; t < nthreads; ++t) {
        pool.emplace_back([=]() {
            for (int64_t r = t; r < rows; r += nthreads) f(r);
        });
    }
    for (auto& th : pool) th.join();
}

Problem make(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B, int32_t Hq,
             int32_t Hkv, int32_t D, int64_t kv_rows, int32_t dtype, int32_t layout, double scale) {
    Problem p;
    p.q = (const uint16_t*)q;
    p.k = (const uint16_t*)k;
    p.v = (const uint16_t*)v;
    p.cu = cu;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.D = D;
    p.kv_rows = kv_rows;
    p.dtype = dtype;
    p.layout = layout;
    p.scale = scale;
    p.tq = 1;
    return p;
}

}  // namespace

extern "C" {

double oracle_f16_to_double(uint16_t h) { return decode_f16(h); }
double oracle_bf16_to_double(uint16_t h) { return decode_bf16(h); }

// Split s of S over a length-L sequence: [floor(L*s/S), floor(L*(s+1)/S)).
void oracle_split_range(int64_t L, int64_t S, int64_t s, int64_t* start, int64_t* end) {
    split_bounds(L, S, s, start, end);
}

// out[B, Hq, D] and lse[B, Hq] (natural log) from the plain definition.
// Returns 0, or -1 if the shapes or cu_seqlens are inconsistent.
int oracle_attention(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B,
                     int32_t Hq, int32_t Hkv, int32_t D, int64_t kv_rows, int32_t dtype,
                     int32_t layout, double scale, double* out, double* lse, int nthreads) {
    Problem p = make(q, k, v, cu, B, Hq, Hkv, D, kv_rows, dtype, layout, scale);
    if (!valid(p)) return -1;
    parallel_rows((int64_t)B * Hq, nthreads, [&](int64_t r) {
        int b = (int)(r / Hq), h = (int)(r % Hq);
        attend_row(p, b, 0, h, out + r * D, lse + r);
    });
    return 0;
}

// The plain definition on selected (b, h) pairs: out[n, D], lse[n].
int oracle_attention_rows(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B,
                          int32_t Hq, int32_t Hkv, int32_t D, int64_t kv_rows, int32_t dtype,
                          int32_t layout, double scale, const int32_t* rows_b,
                          const int32_t* rows_h, int32_t n, double* out, double* lse,
                          int nthreads) {
    Problem p = make(q, k, v, cu, B, Hq, Hkv, D, kv_rows, dtype, layout, scale);
    if (!valid(p)) return -1;
    for (int i = 0; i < n; ++i)
        if (rows_b[i] < 0 || rows_b[i] >= B || rows_h[i] < 0 || rows_h[i] >= Hq) return -1;
    parallel_rows(n, nthreads, [&](int64_t i) {
        attend_row(p, rows_b[i], 0, rows_h[i], out + i * D, lse + i);
    });
    return 0;
}

// Per-split partials: o_part[B, Hq, S, D], lse_part[B, Hq, S] (natural log).
int oracle_split_partials(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B,
                          int32_t Hq, int32_t Hkv, int32_t D, int64_t kv_rows, int32_t dtype,
                          int32_t layout, double scale, int32_t S, double* o_part,
                          double* lse_part, int nthreads) {
    Problem p = make(q, k, v, cu, B, Hq, Hkv, D, kv_rows, dtype, layout, scale);
    if (!valid(p) || S < 1) return -1;
    parallel_rows((int64_t)B * Hq, nthreads, [&](int64_t r) {
        int b = (int)(r / Hq), h = (int)(r % Hq);
        split_row(p, b, 0, h, S, o_part + r * S * D, lse_part + r * S);
    });
    return 0;
}

// Per-sequence split counts: sequence b is cut into
//     S_b = 1 if L_b = 0, else min(max_splits, ceil(L_b / split_len))
// Per-sequence split counts with tq query tokens per sequence (causal within
// them, as in oracle_split_partials_mq; oracle_split_partials_var below is tq = 1): o_part[B, tq, Hq, max_splits, D], lse_part[B, tq,
// Hq, max_splits]; a split holding no key that a token may see is empty for it.
int oracle_split_partials_var_mq(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B,
                                 int32_t Hq, int32_t Hkv, int32_t D, int64_t kv_rows, int32_t dtype,
                                 int32_t layout, double scale, int32_t tq, int32_t split_len,
                                 int32_t max_splits, double* o_part, double* lse_part, int32_t* s_count,
                                 int nthreads) {
    Problem p = make(q, k, v, cu, B, Hq, Hkv, D, kv_rows, dtype, layout, scale);
    if (!valid(p) || tq < 1 || split_len < 1 || max_splits < 1) return -1;
    p.tq = tq;
    for (int b = 0; b < B; ++b) {
        int64_t L = seq_len(p, b);
        int64_t sb = L == 0 ? 1 : (L + split_len - 1) / split_len;
        s_count[b] = (int32_t)(sb < max_splits ? sb : max_splits);
    }
    parallel_rows((int64_t)B * tq * Hq, nthreads, [&](int64_t r) {
        int h = (int)(r % Hq), t = (int)((r / Hq) % tq), b = (int)(r / ((int64_t)Hq * tq));
        double* o = o_part + r * max_splits * D;
        double* l = lse_part + r * max_splits;
        split_row(p, b, t, h, s_count[b], o, l);
        for (int sp = s_count[b]; sp < max_splits; ++sp) {
            l[sp] = kNegInf;
            for (int d = 0; d < D; ++d) o[(int64_t)sp * D + d] = 0.0;
        }
    });
    return 0;
}

// proportional splits (the same floor rule as above with S = S_b), so that long
// sequences get more splits than short ones. o_part[B, Hq, max_splits, D] and
// lse_part[B, Hq, max_splits]; entries s >= S_b hold lse = -inf, o = 0.
// Also returns S_b in s_count[B].
int oracle_split_partials_var(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B,
                              int32_t Hq, int32_t Hkv, int32_t D, int64_t kv_rows, int32_t dtype,
                              int32_t layout, double scale, int32_t split_len, int32_t max_splits,
                              double* o_part, double* lse_part, int32_t* s_count, int nthreads) {
    return oracle_split_partials_var_mq(q, k, v, cu, B, Hq, Hkv, D, kv_rows, dtype, layout, scale, 1, split_len,
                                        max_splits, o_part, lse_part, s_count, nthreads);
}

// Several query tokens per sequence: out[B, tq, Hq, D], lse[B, tq, Hq].
int oracle_attention_mq(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B,
                        int32_t Hq, int32_t Hkv, int32_t D, int64_t kv_rows, int32_t dtype,
                        int32_t layout, double scale, int32_t tq, double* out, double* lse,
                        int nthreads) {
    Problem p = make(q, k, v, cu, B, Hq, Hkv, D, kv_rows, dtype, layout, scale);
    if (!valid(p) || tq < 1) return -1;
    p.tq = tq;
    parallel_rows((int64_t)B * tq * Hq, nthreads, [&](int64_t r) {
        int h = (int)(r % Hq), t = (int)((r / Hq) % tq), b = (int)(r / ((int64_t)Hq * tq));
        attend_row(p, b, t, h, out + r * D, lse + r);
    });
    return 0;
}

// The same on selected (b, t, h) triples: out[n, D], lse[n].
int oracle_attention_rows_mq(const void* q, const void* k, const void* v, const int32_t* cu,
                             int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int64_t kv_rows,
                             int32_t dtype, int32_t layout, double scale, int32_t tq,
                             const int32_t* rows_b, const int32_t* rows_t, const int32_t* rows_h,
                             int32_t n, double* out, double* lse, int nthreads) {
    Problem p = make(q, k, v, cu, B, Hq, Hkv, D, kv_rows, dtype, layout, scale);
    if (!valid(p) || tq < 1) return -1;
    p.tq = tq;
    for (int i = 0; i < n; ++i)
        if (rows_b[i] < 0 || rows_b[i] >= B || rows_t[i] < 0 || rows_t[i] >= tq || rows_h[i] < 0 ||
            rows_h[i] >= Hq)
            return -1;
    parallel_rows(n, nthreads, [&](int64_t i) {
        attend_row(p, rows_b[i], rows_t[i], rows_h[i], out + i * D, lse + i);
    });
    return 0;
}

// Per-split partials with several query tokens: o_part[B, tq, Hq, S, D], lse_part[B, tq, Hq, S].
int oracle_split_partials_mq(const void* q, const void* k, const void* v, const int32_t* cu,
                             int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int64_t kv_rows,
                             int32_t dtype, int32_t layout, double scale, int32_t tq, int32_t S,
                             double* o_part, double* lse_part, int nthreads) {
    Problem p = make(q, k, v, cu, B, Hq, Hkv, D, kv_rows, dtype, layout, scale);
    if (!valid(p) || tq < 1 || S < 1) return -1;
    p.tq = tq;
    parallel_rows((int64_t)B * tq * Hq, nthreads, [&](int64_t r) {
        int h = (int)(r % Hq), t = (int)((r / Hq) % tq), b = (int)(r / ((int64_t)Hq * tq));
        split_row(p, b, t, h, S, o_part + r * S * D, lse_part + r * S);
    });
    return 0;
}

// Exact combine of per-split partials: out[rows, D], lse[rows].
int oracle_merge(const double* o_part, const double* lse_part, int64_t rows, int32_t S, int32_t D,
                 double* out, double* lse) {
    if (S < 1 || D < 1 || rows < 0) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const double* ls = lse_part + r * S;
        const double* os = o_part + r * S * D;
        double* o = out + r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        double m = kNegInf;
        for (int s = 0; s < S; ++s) m = ls[s] > m ? ls[s] : m;
        if (m == kNegInf) {
            lse[r] = kNegInf;
            continue;
        }
        double z = 0.0;
        for (int s = 0; s < S; ++s)
            if (ls[s] != kNegInf) z += std::exp(ls[s] - m);
        double tot = m + std::log(z);
        lse[r] = tot;
        for (int s = 0; s < S; ++s) {
            if (ls[s] == kNegInf) continue;
            double w = std::exp(ls[s] - tot);
            for (int d = 0; d < D; ++d) o[d] += w * os[(int64_t)s * D + d];
        }
    }
    return 0;
}

// Softmax weights p_j, j in [0, L_b), of one (b, h) under the plain definition.
int oracle_weights(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B,
                   int32_t Hq, int32_t Hkv, int32_t D, int64_t kv_rows, int32_t dtype,
                   int32_t layout, double scale, int32_t b, int32_t h, double* p_out) {
    Problem p = make(q, k, v, cu, B, Hq, Hkv, D, kv_rows, dtype, layout, scale);
    if (!valid(p) || b < 0 || b >= B || h < 0 || h >= Hq) return -1;
    int64_t L = seq_len(p, b);
    if (L == 0) return 0;
    std::vector<double> qd;
    scores(p, b, 0, h, 0, L, qd, p_out);
    double m = kNegInf;
    for (int64_t j = 0; j < L; ++j) m = p_out[j] > m ? p_out[j] : m;
    double z = 0.0;
    for (int64_t j = 0; j < L; ++j) {
        p_out[j] = std::exp(p_out[j] - m);
        z += p_out[j];
    }
    for (int64_t j = 0; j < L; ++j) p_out[j] /= z;
    return 0;
}

}  // extern "C"
