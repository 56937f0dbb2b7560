// Work-item geometry of the split step, shared by the kernels (device and host
// code), the host-side split choices and the host-only time model.
#ifndef DECODE_ATTN_SPLITKV_GEOMETRY_H
#define DECODE_ATTN_SPLITKV_GEOMETRY_H

#include <cstdint>

namespace da_impl {

constexpr int kBoxKeys = 16;        // keys per TMA box = rows of one mma m-tile
constexpr int kStageKeys = 64;      // keys per pipeline stage
constexpr int kHeadsPerCta = 8;     // mma N: packed (token, head) columns per n-tile
// Uniform splits over a varlen batch of at most this many sequences: the work
// queue hands out the sequences longest first.
constexpr int kMaxSortedBatch = 128;

// Columns (packed query token x head pairs) of one work item: one n-tile of 8,
// or two when a KV head serves more than 8 columns, so that K and V are read
// and multiplied once for up to 16 columns.
inline int item_cols(int64_t cols) { return cols > kHeadsPerCta ? 2 * kHeadsPerCta : kHeadsPerCta; }
inline int64_t item_chunks(int64_t cols) {
    const int c = item_cols(cols);
    return (cols + c - 1) / c;
}

}  // namespace da_impl

#endif
