// GB300 time model of one decode call (host only; see decode_attn_splitkv_model_us
// in decode_attn_splitkv.h).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "decode_attn_splitkv.h"
#include "geometry.h"

using namespace da_impl;

extern "C" {

// A GB300 restatement of the lecture page's decode time model
// (04_flash_decoding.py: decode_attention_time / best_splits, whose A100/H100
// constants are not on the page): the call is modelled as
//   T = t0 + makespan + kappa * (largest item's bytes) / (bw / min(items, CTAs))
//         + [some S_b > 1] (t_comb + W_ws / bw_comb)
// where makespan is a processor-sharing run of the work items, in queue order,
// over the persistent CTAs: each CTA spends t_item before an item and then
// streams its bytes (each split's key count rounded up to the 16-key TMA box)
// at min(r_cta, bw / streaming CTAs), r_cta being one CTA's rate for 8-column
// items and r_cta2 for 16-column ones; kappa charges the last item for the
// CTAs' unequal rates, and W_ws is the workspace bytes the combine reads (the
// rows of sequences with more than one split). S_b = S with uniform splits,
// min(S, ceil(L_b / split_len)) with per-sequence counts.
// Fitted (least squares in log time) on one GB300 to the 311 calls, of 546
// measured (17 single-token workloads of the CodeLlama, Llama, Qwen and MHA
// shapes and 9 of them with 2 or 4 new tokens x split counts 1 to 256, L2
// flushed, CUDA-event median per call), that lie within 30 % of their
// workload's fastest split count: median error 2.6 %, 90th percentile 11.5 %.
// The fit puts t_item at zero: the ring, which keeps filling across items,
// hides the per-item work.
static const double kModelGb300[8] = {
    /* t0 us       */ 11.98,
    /* t_item us   */ 0.0,
    /* r_cta B/us  */ 76280,
    /* bw B/us     */ 7.757e+06,
    /* t_comb us   */ 3.209,
    /* bw_comb     */ 6.478e+05,
    /* kappa       */ 0.05065,
    /* r_cta2 B/us */ 46550};

}  // extern "C"

namespace {

// The model of one call: S splits per sequence (split_len = 0), or per-sequence
// counts S_b = min(S, ceil(L_b / split_len)) (1 for an empty sequence).
double model_call(const int32_t* kv_lens, int B, int Hq, int Hkv, int D, int T_q, int num_splits, int split_len,
                  int sm_count, const double* params) {
    if (!kv_lens || B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || (D != 64 && D != 128) || T_q < 1 ||
        num_splits < 1 || num_splits > DA_MAX_SPLITS || sm_count < 1 || split_len < 0)
        return -1.0;
    const double* m = params ? params : kModelGb300;
    const double t0 = m[0], t_item = m[1], bw = m[3], t_comb = m[4], bw_comb = m[5], kappa = m[6];
    // one CTA's streaming cap: 16-column items carry twice the products per key
    const bool wide = item_cols(static_cast<int64_t>(Hq / Hkv) * T_q) > kHeadsPerCta;
    const double r_cta = (wide ? m[7] : m[2]) / static_cast<double>(item_chunks(static_cast<int64_t>(Hq / Hkv) * T_q));
    if (!(r_cta > 0) || !(bw > 0) || !(bw_comb > 0) || !(t_item >= 0) || !(kappa >= 0)) return -1.0;
    const int S = num_splits;
    const int chunks = static_cast<int>(item_chunks(static_cast<int64_t>(Hq / Hkv) * T_q));
    const int slots = sm_count * (D == 128 ? 2 : 4);
    const double key_bytes = 4.0 * D;   // K and V rows of one key and KV head
    // the work items in queue order and the bytes each streams. With uniform
    // splits the split step hands out the sequences of a batch of at most 128
    // longest first (a varlen batch, which is what the model assumes), ties in
    // index order; per-sequence counts go out in index order.
    std::vector<int> order(static_cast<size_t>(B));
    for (int b = 0; b < B; ++b) order[b] = b;
    if (split_len == 0 && B > 1 && B <= kMaxSortedBatch)
        std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
            return std::max(kv_lens[x], 0) > std::max(kv_lens[y], 0);
        });
    std::vector<double> items;
    double biggest = 0.0, comb_rows = 0.0;   // rows the combine merges, times their split counts
    for (int b : order) {
        const int64_t L = kv_lens[b] < 0 ? 0 : kv_lens[b];
        int Sb = S;
        if (split_len > 0) Sb = L == 0 ? 1 : static_cast<int>(std::min<int64_t>(S, (L + split_len - 1) / split_len));
        if (Sb > 1) comb_rows += static_cast<double>(T_q) * Hq * Sb;
        for (int kvh = 0; kvh < Hkv; ++kvh)
            for (int s = 0; s < Sb; ++s) {
                const int64_t n = L * (s + 1) / Sb - L * s / Sb;
                const double bytes = static_cast<double>((n + kBoxKeys - 1) / kBoxKeys * kBoxKeys) * key_bytes;
                biggest = std::max(biggest, bytes / chunks);
                // the `chunks` items of a split run side by side and read its keys
                // once from HBM between them (the rest from L2): each item is charged
                // its share of the HBM bytes, at its share of one CTA's rate
                for (int c = 0; c < chunks; ++c) items.push_back(bytes / chunks);
            }
    }
    // Processor sharing: every CTA that is streaming gets min(r_cta, bw / streaming)
    // bytes per us; before each item a CTA spends t_item not streaming. All
    // streaming CTAs advance together, so their progress is one "virtual bytes"
    // clock V and a CTA's stream ends at a fixed V.
    using Ev = std::pair<double, int>;
    std::priority_queue<Ev, std::vector<Ev>, std::greater<Ev>> streams;    // (V at end, cta)
    std::priority_queue<Ev, std::vector<Ev>, std::greater<Ev>> overheads;  // (time at end, cta)
    size_t next = 0;
    double now = 0.0, V = 0.0;
    for (int c = 0; c < slots && next < items.size(); ++c) overheads.push({t_item, c}), ++next;
    std::vector<double> pending(static_cast<size_t>(slots), 0.0);   // bytes of the item a CTA prepares
    for (int c = 0; c < slots && c < static_cast<int>(items.size()); ++c) pending[c] = items[c];
    while (!streams.empty() || !overheads.empty()) {
        const double rate = streams.empty() ? 0.0 : std::min(r_cta, bw / static_cast<double>(streams.size()));
        const double t_stream = streams.empty() ? INFINITY : now + (streams.top().first - V) / rate;
        const double t_over = overheads.empty() ? INFINITY : overheads.top().first;
        if (t_stream <= t_over) {
            V = streams.top().first;
            now = t_stream;
            const int c = streams.top().second;
            streams.pop();
            if (next < items.size()) {
                pending[c] = items[next++];
                overheads.push({now + t_item, c});
            }
        } else {
            V += rate * (t_over - now);
            now = t_over;
            const int c = overheads.top().second;
            overheads.pop();
            streams.push({V + pending[c], c});
        }
    }
    const double makespan = now;
    // CTAs stream at unequal rates; the work queue evens them out except over
    // the last item, which costs a fraction kappa of its time at the fair share
    const double fair = bw / static_cast<double>(std::max<size_t>(1, std::min<size_t>(items.size(), slots)));
    double t = t0 + makespan + kappa * biggest / fair;
    if (comb_rows > 0) t += t_comb + comb_rows * (D + 1) * 4.0 / bw_comb;
    return t;
}

}  // namespace

extern "C" {

double decode_attn_splitkv_model_us(const int32_t* kv_lens, int B, int Hq, int Hkv, int D, int T_q, int num_splits,
                                    int sm_count, const double* params) {
    return model_call(kv_lens, B, Hq, Hkv, D, T_q, num_splits, 0, sm_count, params);
}

double decode_attn_splitkv_model_varsplit_us(const int32_t* kv_lens, int B, int Hq, int Hkv, int D, int T_q,
                                             int split_len, int max_splits, int sm_count, const double* params) {
    if (split_len < 1) return -1.0;
    return model_call(kv_lens, B, Hq, Hkv, D, T_q, max_splits, split_len, sm_count, params);
}

int decode_attn_splitkv_model_best_splits(const int32_t* kv_lens, int B, int Hq, int Hkv, int D, int T_q,
                                          int sm_count, double* predicted_us) {
    if (!kv_lens || B < 1) return 1;
    int min_kv = INT32_MAX;
    for (int b = 0; b < B; ++b) min_kv = std::min(min_kv, kv_lens[b] < 0 ? 0 : kv_lens[b]);
    const int s_max = std::max(1, std::min(min_kv, 256));
    int best = 1;
    double best_t = decode_attn_splitkv_model_us(kv_lens, B, Hq, Hkv, D, T_q, 1, sm_count, nullptr);
    for (int S = 2; S <= s_max; S += (S < 16 ? 1 : S < 64 ? 4 : 16)) {
        const double t = decode_attn_splitkv_model_us(kv_lens, B, Hq, Hkv, D, T_q, S, sm_count, nullptr);
        if (t > 0 && (best_t < 0 || t < best_t)) {
            best_t = t;
            best = S;
        }
    }
    if (predicted_us) *predicted_us = best_t;
    return best;
}

}  // extern "C"