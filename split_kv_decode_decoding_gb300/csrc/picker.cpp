// Host-side choices of the split step: the uniform split count and the
// per-sequence split plan, and the split bounds (decode_attn_splitkv.h). No
// kernel code: a change here leaves the kernels as they are.

#include <algorithm>
#include <cmath>
#include <cstdint>

#include <cuda_runtime.h>

#include "decode_attn_splitkv.h"
#include "geometry.h"

using namespace da_impl;

namespace {

constexpr double kLongStreamBytes = 1.5e9;   // K/V bytes above which even batches are split for balance

// SMs of the current device (148 if it cannot be queried).
int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return 148;
    return sms;
}

}  // namespace

extern "C" {

void decode_attn_splitkv_split_range(int64_t L, int num_splits, int s, int64_t* start, int64_t* end) {
    if (!start || !end) return;
    if (num_splits < 1 || L < 0) {
        *start = *end = 0;
        return;
    }
    *start = L * s / num_splits;
    *end = L * (s + 1) / num_splits;
}

int decode_attn_splitkv_num_splits(int B, int Hq, int Hkv, int D, int min_kv, int max_kv, int sm_count) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || (D != 64 && D != 128)) return 1;
    if (min_kv <= 0 || max_kv < min_kv) return 1;
    if (sm_count <= 0) sm_count = device_sm_count();
    const int64_t chunks = item_chunks(Hq / Hkv);
    const int64_t units = static_cast<int64_t>(B) * Hkv * chunks;   // (sequence, KV head, chunk)
    const int64_t slots = static_cast<int64_t>(sm_count) * (D == 128 ? 2 : 4);   // persistent CTAs
    int64_t S;
    if (2 * static_cast<int64_t>(min_kv) <= max_kv) {
        // Ragged lengths: about eight items per SM, so the work queue can even
        // out splits of unequal length; splits may be short ...
        // (16-column items carry twice the work per key and a two-round merge:
        // half as many of them, with longer splits, measured best)
        const bool wide = item_cols(Hq / Hkv) > kHeadsPerCta;
        const double total = static_cast<double>(max_kv) + static_cast<double>(B - 1) * min_kv;
        // A batch of up to kMaxSortedBatch sequences is handed out longest first,
        // so its short items come last and even out the end by themselves: fewer,
        // longer splits measure best (six items per SM, splits up to four CTA
        // shares), unless one sequence holds most of the keys. Its splits are then
        // the critical path whatever the width: at most two CTA shares each
        // (16-column items stream slower per CTA, and four shares took 153 against
        // 114 us on one 131072-key sequence among fifteen of 512 with four query
        // tokens).
        const bool dominant = 2.0 * max_kv > total;
        const bool sorted = B <= kMaxSortedBatch && !dominant;
        const int64_t per_sm = sorted ? (wide ? 3 : 6) : (wide ? 4 : 8);
        const double shares = sorted ? (wide ? 8.0 : 4.0) : (dominant || !wide ? 2.0 : 4.0);
        S = (per_sm * static_cast<int64_t>(sm_count) + units - 1) / units;
        S = std::min<int64_t>(S, std::max<int64_t>(1, min_kv / 64));
        // ... and the longest sequence's splits at most about `shares` times one
        // CTA's share of the keys (the share taken from a lower bound of the
        // total), so that no single split outlasts the rest of the batch.
        const double share = total * Hkv * chunks / static_cast<double>(slots);
        S = std::max<int64_t>(S, static_cast<int64_t>(std::ceil(max_kv / (shares * share))));
    } else if (5 * units >= 4 * static_cast<int64_t>(sm_count)) {
        // Even lengths, about one unit per SM or more: one split (no combine)
        // while the stream is short; for a long stream about 1.7 waves of items,
        // so the work queue evens out the SMs' unequal rates and the last wave
        // still keeps a third of the CTAs busy.
        const double kv_bytes = static_cast<double>(B) * Hkv * min_kv * 4.0 * D;
        S = kv_bytes <= kLongStreamBytes ? 1 : std::max<int64_t>(1, std::llround(1.68 * slots / units));
    } else {
        // Even lengths, fewer units than SMs: about one item per SM, each split
        // long enough (256 to 1024 keys) that its start-up and merge stay small
        // next to its stream.
        S = (static_cast<int64_t>(sm_count) + units - 1) / units;
        const int64_t min_len =
            std::min<int64_t>(1024, std::max<int64_t>(256, static_cast<int64_t>(min_kv) * units / sm_count));
        S = std::min<int64_t>(S, std::max<int64_t>(1, min_kv / min_len));
    }
    // never an empty split (the TileLang page's num_splits <= min_kv rule)
    S = std::min<int64_t>(S, min_kv);
    S = std::max<int64_t>(1, std::min<int64_t>(S, DA_MAX_SPLITS));
    return static_cast<int>(S);
}

int decode_attn_splitkv_varsplit_plan(int B, int Hq, int Hkv, int D, int64_t total_kv, int max_kv,
                                      int sm_count, int* split_len, int* max_splits) {
    if (!split_len || !max_splits) return -1;
    *split_len = 1;
    *max_splits = 1;
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || (D != 64 && D != 128) || total_kv < 0 || max_kv < 0)
        return -1;
    if (sm_count <= 0) sm_count = device_sm_count();
    const int64_t chunks = item_chunks(Hq / Hkv);
    const int64_t key_units = total_kv * Hkv * chunks;      // keys to stream, summed over (KV head, chunk)
    const int64_t slots = static_cast<int64_t>(sm_count) * (D == 128 ? 2 : 4);   // persistent CTAs
    // Items of about 0.4 of one CTA's share of the keys (two or three per CTA, so the
    // work queue evens out unequal lengths), but the longest sequence in no more
    // items than half the CTAs: its splits would otherwise multiply the combine's
    // work and the per-item costs without better balance. Measured on GB300 over
    // split lengths 512 .. 7680 on the Qwen-shaped ragged batch and on a batch of
    // one 131072-key sequence among fifteen of 512. Items of a whole share leave
    // the last ones of the queue, in sequence order, as long as any: 102.4 against
    // 96.7 us on the Qwen-shaped batch.
    int64_t len = (2 * key_units + 5 * slots - 1) / (5 * slots);
    len = std::max<int64_t>(len, (2 * static_cast<int64_t>(max_kv) * Hkv * chunks + slots - 1) / slots);
    len = std::max<int64_t>(256, (len + kStageKeys - 1) / kStageKeys * kStageKeys);   // whole stages
    int64_t ms = max_kv > 0 ? (max_kv + len - 1) / len : 1;
    ms = std::max<int64_t>(1, std::min<int64_t>(ms, DA_MAX_SPLITS));
    *split_len = static_cast<int>(std::min<int64_t>(len, 1 << 30));
    *max_splits = static_cast<int>(ms);
    return 0;
}

}  // extern "C"
