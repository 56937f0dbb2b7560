// Split-KV decode attention (flash-decoding) for GB300 / sm_103a.
//
// Split step: a persistent kernel, two CTAs per SM (more at head_dim 64), that
// takes work items (sequence b, KV head, column chunk, split s) from a queue in
// the workspace. The columns of a KV head are its query heads times the query
// tokens (one token in plain decode). For each item it computes, for the up-to-8
// (or, when the KV head serves more than 8 columns, up-to-16) columns that the
// chunk holds, the normalised partial output o_s and
// lse_s = ln sum_{j in split} exp(s_j), and writes them to the workspace.
//   * The GQA group is packed into the N = 8 columns of m16n8k16 tensor-core
//     products (two such n-tiles for 16 columns), so every K/V byte is read
//     from HBM once per group (TileLang decode_attention_splitkv.py, split
//     segment, cur_kv_head; CS349E lecture 11 04_flash_decoding.py, demo1_exact
//     second observation). Keys are the M rows: S^T[key, col] = K_tile . Q^T, then
//     O^T[dim, col] += V_tile^T . P^T; the score fragment turns into the P^T
//     operand with one movmatrix transpose per 8x8 block, so P stays in
//     registers; with two n-tiles each K and V fragment feeds both.
//   * One producer warp runs ahead of four consumer warps: it takes the next
//     item from the queue, publishes its descriptor and bulk-copies its Q rows
//     into shared memory, and streams the item's K and V tiles with TMA
//     (cp.async.bulk.tensor, 128-byte swizzle; 64-key boxes for full stages,
//     16-key boxes for the ragged end of a split) into a three-stage ring
//     guarded by full/empty mbarriers. The ring keeps filling
//     across item boundaries, so one item's epilogue overlaps the next item's
//     loads. Each consumer warp owns 16 keys of every 64-key stage.
//   * Online softmax in the exp2 domain (scale * log2 e folded into the
//     scores), with running max, running sum and accumulator per consumer warp
//     in fp32 registers (TileLang page, split segment online softmax; MiniInfer
//     flash_decode_splitk.py, _splitk_stage1_kernel). The accumulator is
//     rescaled only when the running max moves; in 16-column items the
//     reference lags, moving only when a score passes it by more than 8 (log2
//     units) as one warp vote decides, so the weights stay below 2^8. At the
//     end of an item the producer hands the consumers one ring stage instead
//     of a tile, and the four warps merge their states through it in a fixed
//     order (the result does not depend on timing), one n-tile per round.
//   * Split bounds are proportional: [L*s/S, L*(s+1)/S) in 64-bit integers
//     (TileLang page, split segment). Keys of a stage past the split end are
//     masked to -inf before the max, and their V rows are cleared in shared
//     memory (0 * NaN is NaN); TMA reads past the K/V extent are zero-filled
//     by the hardware, so no load leaves the tensor.
// Combine step: one warp per (b, query head, slice of head_dim), reading the
// splits' lse and o from L2: lse = ln sum exp(lse_s), out = sum exp(lse_s -
// lse) * o_s, empty splits weighing 0 (TileLang page, combine segment, with
// the weight indexed by head row; MiniInfer _splitk_reduce_kernel).
// The two kernels are chained with programmatic dependent launch. With a single
// split the split kernel writes the output itself and no combine is launched.
// split_kernel_tc runs the same split step on the tcgen05 tensor cores with the
// accumulators in tensor memory, for items of 9 to 32 columns; it is a
// comparison arm (decode_attn_splitkv_multiquery_tmem) that the library's own
// calls never use.
//
// Every mbarrier wait is bounded in time; on expiry the kernel sets
// DA_DEVERR_TIMEOUT in the workspace error word and winds down instead of
// hanging.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <functional>
#include <vector>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <queue>

#include "decode_attn_splitkv.h"

namespace {

constexpr int kBoxKeys = 16;        // keys per TMA box = rows of one mma m-tile
constexpr int kStageKeys = 64;      // keys per pipeline stage
constexpr int kConsumerWarps = 4;   // each owns 16 keys of a stage
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kHeadsPerCta = 8;     // mma N: packed (token, head) columns per n-tile
constexpr int kStages = 3;          // pipeline depth (two CTAs per SM at head_dim 128)
constexpr int kPrefetchStages = 4;  // BHSD: first stages pulled into L2 while cu_seqlens_k is read
constexpr int kMinBlocksPerSm = 2;
constexpr int kItemSlots = 2;       // item descriptors the producer may run ahead
constexpr float kLazyRescale = 8.f; // 16-column items: headroom (log2) before the running max moves
constexpr size_t kHeaderBytes = 256;
constexpr size_t kWorkCounterOff = 64;   // header: uint32 work-queue head
constexpr size_t kDoneCounterOff = 128;  // header: uint32 count of CTAs finished
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr int kMaxStagedBatch = 1024;                          // B up to which cu_seqlens_k is staged in smem
constexpr int kStagedBytes = ((kMaxStagedBatch + 1) * 4 + 15) / 16 * 16;   // one [B + 1] int32 array

struct ItemSlot {          // one work item, as the producer decoded it
    int32_t b, kvh, h0, nh;            // h0: first query head of the KV head's group; nh columns
    int32_t s, nkeys, ntiles, valid;   // valid = 0 marks the end of the queue
    int64_t first_key;                 // varlen: K/V row of the split start; bhsd: position
    int32_t c0;                        // first packed (token, head) column of this item
    int32_t vis0;                      // keys of the split query token 0 may see (may be <= 0)
};
static_assert(sizeof(ItemSlot) == 48, "ItemSlot layout");

// Columns (packed query token x head pairs) of one work item: one n-tile of 8,
// or two when a KV head serves more than 8 columns, so that K and V are read
// and multiplied once for up to 16 columns.
inline int item_cols(int64_t cols) { return cols > kHeadsPerCta ? 2 * kHeadsPerCta : kHeadsPerCta; }
inline int64_t item_chunks(int64_t cols) {
    const int c = item_cols(cols);
    return (cols + c - 1) / c;
}

template <int D, int NT>
struct Shape {
    static constexpr int kHalves = D / 64;                         // 128-byte column slices
    static constexpr int kSliceBytes = kStageKeys * 128;           // one slice of a stage tile
    static constexpr int kTileBytes = kHalves * kSliceBytes;       // K (or V) bytes per stage
    static constexpr int kStageBytes = 2 * kTileBytes;             // K + V
    static constexpr int kBoxBytes = kBoxKeys * 128;               // one TMA box
    static constexpr int kRingBytes = kStages * kStageBytes;
    // Item merge, laid out in the ring stage the producer hands over at the end of
    // each item: per-warp accumulators [warp][head][D + 4] (the pad keeps both the
    // fragment stores and the row reads free of bank conflicts), then [warp][8]
    // maxima and [warp][8] sums.
    static constexpr int kMergeRow = D + 4;
    static constexpr int kMergeBytes = (kConsumerWarps * kHeadsPerCta * kMergeRow + 2 * kConsumerWarps * kHeadsPerCta) * 4;
    static_assert(kMergeBytes <= kStageBytes, "item merge must fit in one ring stage");
    static constexpr int kQBytes = NT * kHeadsPerCta * D * 2;      // Q rows of one item
    static constexpr int kQOff = kRingBytes;
    static constexpr int kSlotOff = kQOff + kItemSlots * kQBytes;
    static constexpr int kBarOff = kSlotOff + kItemSlots * (int)sizeof(ItemSlot);
    static constexpr int kNumBars = 2 * kStages + 2 * kItemSlots + 1 + (NT > 1 ? 1 : 0);
    static constexpr int kEnd = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = 1024 /* alignment slack */ + kEnd;
    static_assert(kQOff % 16 == 0 && kSlotOff % 16 == 0 && kBarOff % 8 == 0, "smem alignment");
};

struct SplitParams {
    const uint16_t* q;       // [B, Hq, D]
    const int32_t* cu;       // [B + 1]
    float* lse;              // [B, Hq, S]
    float* opart;            // [B, Hq, S, D]
    uint32_t* err;           // device error word
    uint32_t* work;          // work-queue head
    uint32_t* done;          // CTAs finished
    uint16_t* out;           // [B, Hq, D] when S == 1 (o_0 is the output), else nullptr
    int B, Hq, Hkv, G, S, kv_rows, layout, chunks, no_kv, n_items;
    int split_len;           // 0: every sequence has S splits; else S_b = min(S, ceil(L_b / split_len))
    int stage_cu;            // cu_seqlens_k staged in shared memory (B small enough)
    int tq;                  // query tokens per sequence; columns per KV head = G * tq
    float scale_log2;        // scale * log2(e)
    unsigned long long wait_limit_ns;
};

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity to complete, for at most
// limit_ns nanoseconds. Returns false on expiry.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// mbar_wait by every lane of a warp, with one verdict for the whole warp, so
// that the warp-synchronous instructions after it are never split by a
// time-out that only some lanes saw.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               unsigned long long limit_ns) {
    const bool ok = mbar_wait(bar, parity, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// Contiguous global -> shared copy (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// Pull one tile of a tensor into L2 (no shared-memory destination, no barrier).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

template <int DT>
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
    if constexpr (DT == DA_F16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
            " {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
            " {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// One 16-bit input element to fp32 (exact).
template <int DT>
__device__ __forceinline__ float bits_to_f32(uint32_t h) {
    if constexpr (DT == DA_F16) {
        float f;
        asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(static_cast<uint16_t>(h)));
        return f;
    } else {
        return __uint_as_float(h << 16);
    }
}

// Eight 16-bit elements (one 16-byte shared-memory chunk) to fp32.
template <int DT>
__device__ __forceinline__ void chunk_to_f32(uint32_t addr, float (&f)[8]) {
    uint32_t w[4];
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        f[2 * j] = bits_to_f32<DT>(w[j] & 0xffffu);
        f[2 * j + 1] = bits_to_f32<DT>(w[j] >> 16);
    }
}

// Pack two fp32 values into one register of two 16-bit values (lo = a), RN.
template <int DT>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    uint32_t r;
    if constexpr (DT == DA_F16) {
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    } else {
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    }
    return r;
}

template <int DT>
__device__ __forceinline__ uint16_t to_bits(float a) {
    uint16_t r;
    if constexpr (DT == DA_F16) {
        asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(a));
    } else {
        asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(a));
    }
    return r;
}

// 2^x on the SFU (ex2.approx; 2^-inf = +0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2(x) on the SFU (lg2.approx; relative error about 2^-22).
__device__ __forceinline__ float fast_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 1/x on the SFU (rcp.approx; within one ulp).
__device__ __forceinline__ float fast_rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ int ld_cg_s32(const int32_t* p) {
    int v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void flag_error(uint32_t* err, uint32_t bits) { atomicOr(err, bits); }

// Length of a sequence whose cu_seqlens_k entries are c0, c1, validated
// against the K/V extent: a range that cannot be read safely counts as empty
// (and *bad is set).
__device__ __forceinline__ int64_t checked_len_of(int64_t c0, int64_t c1, int layout, int kv_rows, int no_kv,
                                                  int64_t* base, bool* bad) {
    const int64_t L = c1 - c0;
    bool ok = L >= 0;
    if (layout == DA_LAYOUT_VARLEN) ok = ok && c0 >= 0 && c1 <= kv_rows;
    else ok = ok && L <= kv_rows;
    if (no_kv) ok = ok && L == 0;
    *base = layout == DA_LAYOUT_VARLEN ? c0 : 0;
    *bad = !ok;
    return ok ? L : 0;
}

__device__ __forceinline__ int64_t checked_len(const int32_t* cu, int b, int layout, int kv_rows, int no_kv,
                                               int64_t* base, bool* bad) {
    return checked_len_of(ld_cg_s32(cu + b), ld_cg_s32(cu + b + 1), layout, kv_rows, no_kv, base, bad);
}

// Split count of a sequence of length L (per-sequence mode): 1 for an empty
// sequence, else ceil(L / split_len) capped at max_splits; never an empty split.
__device__ __forceinline__ int seq_splits(int64_t L, int split_len, int max_splits) {
    if (L == 0) return 1;
    const int64_t sb = (L + split_len - 1) / split_len;
    return static_cast<int>(sb < max_splits ? sb : max_splits);
}

// Decode work item `idx` into its descriptor. Items run head-chunk fastest
// (the chunks of one split read the same K/V at the same time, the second
// read coming from L2), then split, then KV head, then sequence. `cus` is
// cu_seqlens_k staged in shared memory (nullptr: read it from global memory).
// With per-sequence split counts, `prefix` holds the running sum of S_b
// (prefix[b] splits before sequence b) and the sequence is found by binary
// search.
__device__ __forceinline__ ItemSlot decode_item_cols(const SplitParams& p, int idx, const int32_t* cus,
                                                     const int32_t* prefix, int kCols) {
    ItemSlot it;
    int chunk, Sb;
    const int hc_count = p.Hkv * p.chunks;
    if (p.split_len == 0) {
        int r = idx;
        chunk = r % p.chunks;
        r /= p.chunks;
        it.s = r % p.S;
        r /= p.S;
        it.kvh = r % p.Hkv;
        it.b = r / p.Hkv;
        Sb = p.S;
    } else {
        int lo = 0, hi = p.B - 1;   // last b with prefix[b] * hc_count <= idx
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (static_cast<int64_t>(prefix[mid]) * hc_count <= idx) lo = mid;
            else hi = mid - 1;
        }
        it.b = lo;
        Sb = prefix[lo + 1] - prefix[lo];
        int r = idx - prefix[lo] * hc_count;
        chunk = r % p.chunks;
        r /= p.chunks;
        it.s = r % Sb;
        it.kvh = r / Sb;
    }
    it.h0 = it.kvh * p.G;
    it.c0 = chunk * kCols;
    it.nh = min(kCols, p.G * p.tq - it.c0);
    int64_t base;
    bool bad;
    const int64_t L = cus != nullptr
                          ? checked_len_of(cus[it.b], cus[it.b + 1], p.layout, p.kv_rows, p.no_kv, &base, &bad)
                          : checked_len(p.cu, it.b, p.layout, p.kv_rows, p.no_kv, &base, &bad);
    if (bad && it.s == 0 && chunk == 0 && it.kvh == 0) flag_error(p.err, DA_DEVERR_SEQLENS);
    const int64_t lo = L * it.s / Sb, hi = L * (it.s + 1) / Sb;
    it.nkeys = static_cast<int>(hi - lo);
    it.ntiles = (it.nkeys + kStageKeys - 1) / kStageKeys;
    it.first_key = base + lo;
    // query token t sits at position L - tq + t and sees keys up to it
    const int64_t vis0 = L - p.tq + 1 - lo;
    it.vis0 = static_cast<int>(vis0 < -(1 << 30) ? -(1 << 30) : vis0);
    it.valid = 1;
    return it;
}

template <int kCols>
__device__ __forceinline__ ItemSlot decode_item(const SplitParams& p, int idx, const int32_t* cus,
                                                const int32_t* prefix) {
    return decode_item_cols(p, idx, cus, prefix, kCols);
}

// ------------------------------------------------------------ tensor-memory helpers (tcgen05)
// Shared-memory matrix descriptor of a 128-byte-swizzled operand tile: start
// address, leading and stride byte offsets (16-byte units), the tcgen05
// descriptor version and the swizzle mode.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = static_cast<uint64_t>((addr & 0x3FFFF) >> 4);
    d |= static_cast<uint64_t>((lbo & 0x3FFFF) >> 4) << 16;
    d |= static_cast<uint64_t>((sbo & 0x3FFFF) >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;   // descriptor version
    d |= static_cast<uint64_t>(2) << 61;   // 128-byte swizzle
    return d;
}

// Instruction descriptor of a kind::f16 MMA: fp32 accumulator, A and B both
// fp16 (DT = DA_F16) or both bf16, K-major A, B K-major or MN-major, M x N.
template <int DT>
constexpr uint32_t umma_idesc(int M, int N, bool b_mn_major) {
    return (1u << 4) | (DT == DA_BF16 ? (1u << 7) | (1u << 10) : 0u) | (b_mn_major ? (1u << 16) : 0u) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] . B[smem]^T
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(accumulate)));
}

// D[tmem] (+)= A[tmem] . B[smem]^T
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, bool accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(accumulate)));
}

// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// A warp reads its 32 lanes x N consecutive 32-bit columns (lane i: row i of its quarter)
// or writes them.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Workspace/output row of packed column c of an item: token t = c / G, head
// h = h0 + c % G, row = (b * tq + t) * Hq + h.
__device__ __forceinline__ int64_t column_row(const SplitParams& p, const ItemSlot& it, int c) {
    const int cg = it.c0 + c;
    if (p.tq == 1) return static_cast<int64_t>(it.b) * p.Hq + it.h0 + cg;   // token 0: cg < G
    return (static_cast<int64_t>(it.b) * p.tq + cg / p.G) * p.Hq + it.h0 + cg % p.G;
}

// ------------------------------------------------------------ split step
// MATH 0: tensor-core products (the library's path); 1: the same kernel with the
// products on CUDA-core fp32 FMAs, kept as the comparison arm for that choice.
template <int D, int DT, int NT, int MATH>
__global__ void __launch_bounds__(kThreads, kMinBlocksPerSm)
split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
             const __grid_constant__ CUtensorMap tmK16, const __grid_constant__ CUtensorMap tmV16,
             const SplitParams p) {
    using Sh = Shape<D, NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    ItemSlot* slots = reinterpret_cast<ItemSlot*>(smem + Sh::kSlotOff);
    const uint32_t ring = smem_addr(smem);
    const uint32_t qbuf = ring + Sh::kQOff;
    const uint32_t full0 = ring + Sh::kBarOff;          // [kStages]
    const uint32_t empty0 = full0 + 8 * kStages;        // [kStages]
    const uint32_t ifull0 = empty0 + 8 * kStages;       // [kItemSlots]
    const uint32_t iempty0 = ifull0 + 8 * kItemSlots;   // [kItemSlots]
    const uint32_t mfull = iempty0 + 8 * kItemSlots;    // an item's per-warp partials written
    const uint32_t mdone = mfull + 8;                   // two n-tiles: a merge round's rows all read
    // past the fixed layout: cu_seqlens_k [B + 1] (when staged), then prefix[B + 1] (per-sequence mode)
    int32_t* cus = p.stage_cu ? reinterpret_cast<int32_t*>(smem + Sh::kEnd) : nullptr;
    int32_t* prefix = reinterpret_cast<int32_t*>(smem + Sh::kEnd + (p.stage_cu ? kStagedBytes : 0));
    // CUDA-core math only: per consumer warp, softmax weights [16 keys][8 columns] and 8 rescale factors
    float* fma_p = reinterpret_cast<float*>(smem + Sh::kEnd + (p.stage_cu ? kStagedBytes : 0) +
                                            (p.split_len != 0 ? kStagedBytes : 0));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, kConsumerWarps);
        }
        for (int i = 0; i < kItemSlots; ++i) {
            mbar_init(ifull0 + 8 * i, 1);
            mbar_init(iempty0 + 8 * i, kConsumerWarps);
        }
        mbar_init(mfull, kConsumerWarps);
        if constexpr (NT > 1) mbar_init(mdone, kConsumerWarps);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kConsumerWarps && lane == 0 && p.no_kv == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        prefetch_tensormap(&tmK16);
        prefetch_tensormap(&tmV16);
    }
    __syncthreads();
    // Everything above overlaps the previous kernel in the stream; from here on
    // this grid touches global memory, so wait for that kernel to finish.
    grid_dependency_wait();
    if (threadIdx.x == 0) grid_dependents_launch();

    if (warp == kConsumerWarps) {
        // ---------------- producer: one lane takes items and issues every copy
        int n_items = p.n_items;
        if (lane == 0 && p.layout == DA_LAYOUT_BHSD && p.no_kv == 0 && p.split_len == 0 &&
            static_cast<int>(blockIdx.x) < n_items) {
            // This CTA's first item is its own index. When that is a sequence's first
            // split, its keys start at position 0 of its slab whatever the length:
            // start pulling its first stages into L2 while cu_seqlens_k is read.
            const int r = static_cast<int>(blockIdx.x) / p.chunks;   // (b * Hkv + kvh) * S + s
            if (r % p.S == 0) {
                const int slab = r / p.S;
                for (int t = 0; t < kPrefetchStages; ++t)
                    for (int hf = 0; hf < Sh::kHalves; ++hf) {
                        tma_prefetch_3d(&tmK, hf * 64, t * kStageKeys, slab);
                        tma_prefetch_3d(&tmV, hf * 64, t * kStageKeys, slab);
                    }
            }
        }
        if (cus != nullptr) {
            // one coalesced read of cu_seqlens_k per CTA; every item is then decoded from shared memory
            for (int i = lane; i <= p.B; i += 32) cus[i] = ld_cg_s32(p.cu + i);
            __syncwarp();
        }
        if (p.split_len != 0) {
            // per-sequence split counts: the whole warp builds prefix[] = running sum of S_b
            int carry = 0;
            for (int b0 = 0; b0 < p.B; b0 += 32) {
                const int b = b0 + lane;
                int sb = 0;
                if (b < p.B) {
                    int64_t base;
                    bool bad;
                    const int64_t L = cus != nullptr ? checked_len_of(cus[b], cus[b + 1], p.layout, p.kv_rows,
                                                                      p.no_kv, &base, &bad)
                                                     : checked_len(p.cu, b, p.layout, p.kv_rows, p.no_kv, &base, &bad);
                    sb = seq_splits(L, p.split_len, p.S);
                }
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, sb, off);
                    if (lane >= off) sb += y;
                }
                if (b < p.B) prefix[b + 1] = carry + sb;
                carry += __shfl_sync(0xffffffffu, sb, 31);
            }
            if (lane == 0) prefix[0] = 0;
            __syncwarp();
            n_items = carry * p.Hkv * p.chunks;
        }
        if (lane == 0) {
            int st = 0;          // ring position of the next tile
            uint32_t ph = 0;     // its phase parity
            // Put work item `idx` in descriptor slot `it % kItemSlots` and start the
            // copy of its Q rows. Returns 1 for an item, 0 at the end of the queue
            // (the slot then says so), -1 when the wait for a free slot timed out.
            auto publish = [&](uint32_t it, int idx, ItemSlot& item) -> int {
                const int slot = it % kItemSlots;
                const uint32_t iph = (it / kItemSlots) & 1;
                if (!mbar_wait(iempty0 + 8 * slot, iph ^ 1, p.wait_limit_ns)) {
                    flag_error(p.err, DA_DEVERR_TIMEOUT);
                    return -1;
                }
                if (idx >= n_items) {
                    slots[slot].valid = 0;
                    mbar_arrive(ifull0 + 8 * slot);
                    return 0;
                }
                item = decode_item<NT * kHeadsPerCta>(p, idx, cus, prefix);
                slots[slot] = item;
                const uint32_t ib = ifull0 + 8 * slot;
                mbar_arrive_expect_tx(ib, item.nh * D * 2);
                if (p.tq == 1) {
                    // one query token: the item's heads are contiguous rows of q
                    bulk_load(qbuf + slot * Sh::kQBytes, p.q + column_row(p, item, 0) * D, item.nh * D * 2, ib);
                } else {
                    for (int c = 0; c < item.nh; ++c)
                        bulk_load(qbuf + slot * Sh::kQBytes + c * D * 2, p.q + column_row(p, item, c) * D, D * 2, ib);
                }
                return 1;
            };
            ItemSlot item;
            // the first item of each CTA is its own index
            int state = publish(0, static_cast<int>(blockIdx.x), item);
            for (uint32_t it = 0; state == 1; ++it) {
                // The next item is taken from the queue a few stages before this one's
                // last tile: the atomic's round trip then overlaps the last copies, yet a
                // CTA never holds a reserved item for long (which would hurt the balance
                // at the end of the queue).
                const int fetch_at = max(0, item.ntiles - kStages);
                int next_idx = 0;
                if (item.ntiles == 0) next_idx = static_cast<int>(gridDim.x + atomicAdd(p.work, 1u));
                bool ok = true;
                for (int t = 0; t < item.ntiles; ++t) {
                    if (t == fetch_at) next_idx = static_cast<int>(gridDim.x + atomicAdd(p.work, 1u));
                    if (!mbar_wait(empty0 + 8 * st, ph ^ 1, p.wait_limit_ns)) {
                        flag_error(p.err, DA_DEVERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    const int keys_t = min(kStageKeys, item.nkeys - t * kStageKeys);
                    const uint32_t fb = full0 + 8 * st;
                    const uint32_t kdst = ring + st * Sh::kStageBytes;
                    const uint32_t vdst = kdst + Sh::kTileBytes;
                    const int key0 = static_cast<int>(item.first_key) + t * kStageKeys;
                    const int slab = item.b * p.Hkv + item.kvh;
                    if (keys_t == kStageKeys) {
                        // a full stage: one 64-key box per 128-byte column slice
                        mbar_arrive_expect_tx(fb, Sh::kHalves * 2 * Sh::kSliceBytes);
                        for (int hf = 0; hf < Sh::kHalves; ++hf) {
                            const uint32_t off = hf * Sh::kSliceBytes;
                            if (p.layout == DA_LAYOUT_VARLEN) {
                                tma_load_3d(kdst + off, &tmK, hf * 64, item.kvh, key0, fb);
                                tma_load_3d(vdst + off, &tmV, hf * 64, item.kvh, key0, fb);
                            } else {
                                tma_load_3d(kdst + off, &tmK, hf * 64, key0, slab, fb);
                                tma_load_3d(vdst + off, &tmV, hf * 64, key0, slab, fb);
                            }
                        }
                    } else {
                        // the ragged last stage of a split: 16-key boxes up to its end
                        const int nbox = (keys_t + kBoxKeys - 1) / kBoxKeys;
                        mbar_arrive_expect_tx(fb, nbox * Sh::kHalves * 2 * Sh::kBoxBytes);
                        for (int bx = 0; bx < nbox; ++bx) {
                            const int key = key0 + bx * kBoxKeys;
                            for (int hf = 0; hf < Sh::kHalves; ++hf) {
                                const uint32_t off = hf * Sh::kSliceBytes + bx * Sh::kBoxBytes;
                                if (p.layout == DA_LAYOUT_VARLEN) {
                                    tma_load_3d(kdst + off, &tmK16, hf * 64, item.kvh, key, fb);
                                    tma_load_3d(vdst + off, &tmV16, hf * 64, item.kvh, key, fb);
                                } else {
                                    tma_load_3d(kdst + off, &tmK16, hf * 64, key, slab, fb);
                                    tma_load_3d(vdst + off, &tmV16, hf * 64, key, slab, fb);
                                }
                            }
                        }
                    }
                    if (++st == kStages) {
                        st = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                // The next item's descriptor and Q copy go out before this item's merge
                // stage, so both are in place when the consumers finish the merge.
                ItemSlot next;
                const int next_state = publish(it + 1, next_idx, next);
                if (next_state < 0) break;
                // Hand the next stage to the consumers, empty, for this item's merge.
                if (!mbar_wait(empty0 + 8 * st, ph ^ 1, p.wait_limit_ns)) {
                    flag_error(p.err, DA_DEVERR_TIMEOUT);
                    break;
                }
                mbar_arrive(full0 + 8 * st);
                if (++st == kStages) {
                    st = 0;
                    ph ^= 1;
                }
                item = next;
                state = next_state;
            }
        }
        return;
    }

    // ---------------- consumers
    const int g = lane >> 2, t4 = lane & 3;
    const int mi = lane >> 3, r8 = lane & 7;
    const int krow = warp * kBoxKeys + (mi & 1) * 8 + r8;      // K: matrices (rows lo/hi) x (k lo/hi)
    const int kchunk_add = mi >> 1;
    const int vrow = warp * kBoxKeys + (mi >> 1) * 8 + r8;     // V^T: matrices (dims lo/hi) x (keys lo/hi)
    const int vchunk_add = mi & 1;
    bool ok = true;
    uint32_t bad_bar = 0, bad_ph = 0;
    int st = 0;          // ring position of the next tile
    uint32_t ph = 0;     // its phase parity

    uint32_t mz = 0, md = 0;   // two n-tiles: phases used of mfull and mdone
    uint32_t it = 0;
    for (;; ++it) {
        const int slot = it % kItemSlots;
        const uint32_t iph = (it / kItemSlots) & 1;
        if (!mbar_wait_warp(ifull0 + 8 * slot, iph, p.wait_limit_ns)) {
            if (lane == 0) flag_error(p.err, DA_DEVERR_TIMEOUT);
            ok = false;
            break;
        }
        const ItemSlot item = slots[slot];
        if constexpr (MATH == 1) {
        // ---- CUDA-core math (comparison arm): fp32 FMA dot products and PV for the
        // item's live columns, over the same pipeline and merge as the tensor-core path
            static_assert(NT == 1, "CUDA-core math handles items of up to 8 columns");
            constexpr int kDpl = D / 32;               // dims per lane in the PV product
            if (!item.valid) {
                __syncwarp();
                if (lane == 0) mbar_arrive(iempty0 + 8 * slot);
                break;
            }
            const uint32_t qrows = qbuf + slot * Sh::kQBytes;    // Q rows [column][D] of this item
            float* pw = fma_p + warp * 17 * 8;                   // [16 keys][8 columns], then [8]
            const int c0 = 2 * t4, c1 = 2 * t4 + 1;              // this thread's score columns
            const bool live0 = c0 < item.nh, live1 = c1 < item.nh;
            int visA = item.nkeys, visB = item.nkeys;
            if (p.tq > 1) {
                visA = min(item.nkeys, item.vis0 + (item.c0 + c0) / p.G);
                visB = min(item.nkeys, item.vis0 + (item.c0 + c1) / p.G);
            }
            float acc[8][kDpl];                                  // [column][dim kDpl * lane + j]
#pragma unroll
            for (int c = 0; c < 8; ++c)
#pragma unroll
                for (int j = 0; j < kDpl; ++j) acc[c][j] = 0.f;
            float m_run[2] = {-INFINITY, -INFINITY};
            float l_run[2] = {0.f, 0.f};
            for (int t = 0; t < item.ntiles; ++t) {
                const uint32_t fb = full0 + 8 * st;
                if (ok && !mbar_wait_warp(fb, ph, p.wait_limit_ns)) {
                    ok = false;
                    bad_bar = fb;
                    bad_ph = ph;
                    if (lane == 0) flag_error(p.err, DA_DEVERR_TIMEOUT);
                }
                const int keys_t = min(kStageKeys, item.nkeys - t * kStageKeys);
                bool zeroed = false;
                if (ok && warp * kBoxKeys < keys_t) {
                    const uint32_t kbase = ring + st * Sh::kStageBytes;
                    const uint32_t vbase = kbase + Sh::kTileBytes;
                    const int valid_rows = keys_t - warp * kBoxKeys;
                    if (valid_rows < kBoxKeys) {
                        const int per_row = Sh::kHalves * 8;
                        for (int c = lane; c < (kBoxKeys - valid_rows) * per_row; c += 32) {
                            const int r = valid_rows + c / per_row;
                            const int hf = (c % per_row) >> 3, ch = c & 7;
                            const uint32_t addr = vbase + hf * Sh::kSliceBytes + (warp * kBoxKeys + r) * 128 + ch * 16;
                            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
                        }
                        zeroed = true;
                        __syncwarp();
                    }
                    // scores of keys g and g + 8 of this warp's 16 against columns c0, c1
                    const int r0 = warp * kBoxKeys + g, r1 = r0 + 8;
                    float s00 = 0.f, s01 = 0.f, s10 = 0.f, s11 = 0.f;
#pragma unroll 4
                    for (int ch = 0; ch < D / 8; ++ch) {
                        const int hf = ch >> 3, cc = ch & 7;
                        float k0[8], k1[8];
                        chunk_to_f32<DT>(kbase + hf * Sh::kSliceBytes + r0 * 128 + ((cc ^ (r0 & 7)) << 4), k0);
                        chunk_to_f32<DT>(kbase + hf * Sh::kSliceBytes + r1 * 128 + ((cc ^ (r1 & 7)) << 4), k1);
                        if (live0) {
                            float q[8];
                            chunk_to_f32<DT>(qrows + c0 * D * 2 + ch * 16, q);
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                s00 = fmaf(q[j], k0[j], s00);
                                s10 = fmaf(q[j], k1[j], s10);
                            }
                        }
                        if (live1) {
                            float q[8];
                            chunk_to_f32<DT>(qrows + c1 * D * 2 + ch * 16, q);
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                s01 = fmaf(q[j], k0[j], s01);
                                s11 = fmaf(q[j], k1[j], s11);
                            }
                        }
                    }
                    const int key_lo = t * kStageKeys + warp * kBoxKeys + g;
                    const float x0 = key_lo < visA ? s00 * p.scale_log2 : -INFINITY;
                    const float x1 = key_lo < visB ? s01 * p.scale_log2 : -INFINITY;
                    const float x2 = key_lo + 8 < visA ? s10 * p.scale_log2 : -INFINITY;
                    const float x3 = key_lo + 8 < visB ? s11 * p.scale_log2 : -INFINITY;
                    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                    }
                    const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
                    const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
                    const float p0 = fast_exp2(x0 - ms0), p1 = fast_exp2(x1 - ms1);
                    const float p2 = fast_exp2(x2 - ms0), p3 = fast_exp2(x3 - ms1);
                    const bool moved = mn0 != m_run[0] || mn1 != m_run[1];
                    const float al0 = moved ? fast_exp2(m_run[0] - ms0) : 1.f;
                    const float al1 = moved ? fast_exp2(m_run[1] - ms1) : 1.f;
                    l_run[0] = l_run[0] * al0 + p0 + p2;
                    l_run[1] = l_run[1] * al1 + p1 + p3;
                    m_run[0] = mn0;
                    m_run[1] = mn1;
                    // every lane's PV needs the weights of all 16 keys and 8 columns: through shared memory
                    pw[g * 8 + c0] = p0;
                    pw[g * 8 + c1] = p1;
                    pw[(g + 8) * 8 + c0] = p2;
                    pw[(g + 8) * 8 + c1] = p3;
                    if (g == 0) {
                        pw[16 * 8 + c0] = al0;
                        pw[16 * 8 + c1] = al1;
                    }
                    __syncwarp();
                    if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const float a = pw[16 * 8 + c];
#pragma unroll
                            for (int j = 0; j < kDpl; ++j) acc[c][j] *= a;
                        }
                    }
                    // O[column, dims kDpl * lane ..] += p[key, column] * V[key, dims], one key at a time
                    const int nk = min(kBoxKeys, valid_rows);
                    const int d0 = kDpl * lane;
                    const int ch = d0 >> 3;                                // 16-byte chunk of the row
                    for (int kk = 0; kk < nk; ++kk) {
                        const int r = warp * kBoxKeys + kk;
                        const uint32_t vaddr = vbase + (ch >> 3) * Sh::kSliceBytes + r * 128 +
                                               (((ch & 7) ^ (r & 7)) << 4) + (d0 & 7) * 2;
                        float v[kDpl];
                        if constexpr (kDpl == 4) {
                            uint32_t w0, w1;
                            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(vaddr));
                            v[0] = bits_to_f32<DT>(w0 & 0xffffu);
                            v[1] = bits_to_f32<DT>(w0 >> 16);
                            v[2] = bits_to_f32<DT>(w1 & 0xffffu);
                            v[3] = bits_to_f32<DT>(w1 >> 16);
                        } else {
                            uint32_t w0;
                            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(vaddr));
                            v[0] = bits_to_f32<DT>(w0 & 0xffffu);
                            v[1] = bits_to_f32<DT>(w0 >> 16);
                        }
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            if (c < item.nh) {
                                const float pc = pw[kk * 8 + c];
#pragma unroll
                                for (int j = 0; j < kDpl; ++j) acc[c][j] = fmaf(pc, v[j], acc[c][j]);
                            }
                        }
                    }
                    __syncwarp();   // the weights are read before the next stage rewrites them
                }
                if (zeroed) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8 * st);
                if (++st == kStages) {
                    st = 0;
                    ph ^= 1;
                }
            }
            // the item's Q rows are no longer read: release its descriptor slot
            __syncwarp();
            if (lane == 0) mbar_arrive(iempty0 + 8 * slot);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], off);
                l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], off);
            }
            if (ok && !mbar_wait_warp(full0 + 8 * st, ph, p.wait_limit_ns)) {
                ok = false;
                if (lane == 0) flag_error(p.err, DA_DEVERR_TIMEOUT);
            }
            float* red_acc = reinterpret_cast<float*>(smem + st * Sh::kStageBytes);   // [warp][8][D+4]
            float* red_m = red_acc + kConsumerWarps * 8 * Sh::kMergeRow;               // [warp][8]
            float* red_l = red_m + kConsumerWarps * 8;                                  // [warp][8]
            if (g == 0) {
                red_m[warp * 8 + c0] = m_run[0];
                red_m[warp * 8 + c1] = m_run[1];
                red_l[warp * 8 + c0] = l_run[0];
                red_l[warp * 8 + c1] = l_run[1];
            }
#pragma unroll
            for (int c = 0; c < 8; ++c)
#pragma unroll
                for (int j = 0; j < kDpl; ++j) red_acc[(warp * 8 + c) * Sh::kMergeRow + kDpl * lane + j] = acc[c][j];
            __syncwarp();
            if (lane == 0) mbar_arrive(mfull);
            if (ok && !mbar_wait_warp(mfull, it & 1, p.wait_limit_ns)) {
                ok = false;
                if (lane == 0) flag_error(p.err, DA_DEVERR_TIMEOUT);
            }
            constexpr int kLanesPerHead = D / 4;
            constexpr int kHeadsPerPass = 32 / kLanesPerHead;
            constexpr int kPasses = (8 / kConsumerWarps) / kHeadsPerPass;
            const int d4 = (lane % kLanesPerHead) * 4;
#pragma unroll
            for (int pass = 0; pass < kPasses; ++pass) {
                const int hh = warp + kConsumerWarps * (pass * kHeadsPerPass + lane / kLanesPerHead);
                const bool live = hh < item.nh;
                float mw[kConsumerWarps];
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    mw[w] = red_m[w * 8 + hh];
                    M = fmaxf(M, mw[w]);
                }
                const float Ms = M == -INFINITY ? 0.f : M;
                float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                float lsum = 0.f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float wt = fast_exp2(mw[w] - Ms);
                    lsum = fmaf(wt, red_l[w * 8 + hh], lsum);
                    const float4 a = *reinterpret_cast<const float4*>(red_acc + (w * 8 + hh) * Sh::kMergeRow + d4);
                    o.x = fmaf(wt, a.x, o.x);
                    o.y = fmaf(wt, a.y, o.y);
                    o.z = fmaf(wt, a.z, o.z);
                    o.w = fmaf(wt, a.w, o.w);
                }
                const float inv = M == -INFINITY ? 0.f : fast_rcp(lsum);
                o.x *= inv;
                o.y *= inv;
                o.z *= inv;
                o.w *= inv;
                if (live) {
                    const int64_t qrow = column_row(p, item, hh);
                    const int64_t row = qrow * p.S + item.s;
                    *reinterpret_cast<float4*>(p.opart + row * D + d4) = o;
                    if (d4 == 0) p.lse[row] = M == -INFINITY ? -INFINITY : (M + fast_log2(lsum)) * kLn2;
                    if (p.out != nullptr)
                        *reinterpret_cast<uint2*>(p.out + qrow * D + d4) =
                            make_uint2(pack2<DT>(o.x, o.y), pack2<DT>(o.z, o.w));
                }
            }
        } else if constexpr (NT == 1) {
        // ---- one n-tile (up to 8 columns per item)
            // Q^T fragments (B operand, k16 x n8): head g, dims ks*16 + 2*t4 (+1) and +8 (+9).
            uint32_t qf[D / 16][2];
            {
                const bool hv = g < item.nh;
                const uint32_t qrow = qbuf + slot * Sh::kQBytes + (hv ? g : 0) * D * 2;
    #pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    uint32_t a0, a1;
                    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a0) : "r"(qrow + (ks * 16 + 2 * t4) * 2));
                    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a1) : "r"(qrow + (ks * 16 + 8 + 2 * t4) * 2));
                    qf[ks][0] = hv ? a0 : 0u;
                    qf[ks][1] = hv ? a1 : 0u;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(iempty0 + 8 * slot);
            if (!item.valid) break;

            // keys (relative to the split start) visible to this thread's two columns
            int visA = item.nkeys, visB = item.nkeys;
            if (p.tq > 1) {
                visA = min(item.nkeys, item.vis0 + (item.c0 + 2 * t4) / p.G);
                visB = min(item.nkeys, item.vis0 + (item.c0 + 2 * t4 + 1) / p.G);
            }
            float acc[D / 16][4];
    #pragma unroll
            for (int i = 0; i < D / 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
            float m_run[2] = {-INFINITY, -INFINITY};   // heads 2*t4, 2*t4+1 (log2 domain)
            float l_run[2] = {0.f, 0.f};               // this thread's share of the running sum

            for (int t = 0; t < item.ntiles; ++t) {
                const uint32_t fb = full0 + 8 * st;
                if (ok && !mbar_wait_warp(fb, ph, p.wait_limit_ns)) {
                    ok = false;
                    bad_bar = fb;
                    bad_ph = ph;
                    if (lane == 0) flag_error(p.err, DA_DEVERR_TIMEOUT);
                }
                const int keys_t = min(kStageKeys, item.nkeys - t * kStageKeys);
                bool zeroed = false;
                if (ok && warp * kBoxKeys < keys_t) {
                    const uint32_t kbase = ring + st * Sh::kStageBytes;
                    const uint32_t vbase = kbase + Sh::kTileBytes;
                    const int valid_rows = keys_t - warp * kBoxKeys;
                    if (valid_rows < kBoxKeys) {
                        // The box's rows past the split end hold other keys (or, in a
                        // padded cache, anything): their P is 0, but 0 * NaN is not, so
                        // clear those V rows before the PV product.
                        const int per_row = Sh::kHalves * 8;   // 16-byte chunks per row
                        for (int c = lane; c < (kBoxKeys - valid_rows) * per_row; c += 32) {
                            const int r = valid_rows + c / per_row;
                            const int hf = (c % per_row) >> 3, ch = c & 7;
                            const uint32_t addr = vbase + hf * Sh::kSliceBytes + (warp * kBoxKeys + r) * 128 + ch * 16;
                            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
                        }
                        zeroed = true;
                        __syncwarp();
                    }
                    // S^T[16 keys, 8 heads] = K_tile . Q^T, two independent accumulator chains
                    float sc[4] = {0.f, 0.f, 0.f, 0.f};
                    float sd[4] = {0.f, 0.f, 0.f, 0.f};
    #pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const int chunk16 = ks * 2 + kchunk_add;          // 16-byte chunk along D
                        const uint32_t addr = kbase + (chunk16 >> 3) * Sh::kSliceBytes + krow * 128 +
                                              (((chunk16 & 7) ^ (krow & 7)) << 4);
                        uint32_t a[4];
                        ldsm_x4(addr, a);
                        if (ks & 1) mma_16816<DT>(sd, a, qf[ks][0], qf[ks][1]);
                        else mma_16816<DT>(sc, a, qf[ks][0], qf[ks][1]);
                    }
                    // scores -> exp2 domain, mask keys past the split end
                    const int key_lo = t * kStageKeys + warp * kBoxKeys + g;   // relative to split start
                    const float x0 = key_lo < visA ? (sc[0] + sd[0]) * p.scale_log2 : -INFINITY;
                    const float x1 = key_lo < visB ? (sc[1] + sd[1]) * p.scale_log2 : -INFINITY;
                    const float x2 = key_lo + 8 < visA ? (sc[2] + sd[2]) * p.scale_log2 : -INFINITY;
                    const float x3 = key_lo + 8 < visB ? (sc[3] + sd[3]) * p.scale_log2 : -INFINITY;
                    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
    #pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                    }
                    const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
                    // a column that has seen no key yet (several query tokens) keeps -inf: use 0 as
                    // its reference so that every weight below is 0 rather than NaN
                    const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
                    const float p0 = fast_exp2(x0 - ms0), p1 = fast_exp2(x1 - ms1);
                    const float p2 = fast_exp2(x2 - ms0), p3 = fast_exp2(x3 - ms1);
                    if (mn0 != m_run[0] || mn1 != m_run[1]) {
                        const float al0 = fast_exp2(m_run[0] - ms0), al1 = fast_exp2(m_run[1] - ms1);
                        l_run[0] *= al0;
                        l_run[1] *= al1;
    #pragma unroll
                        for (int i = 0; i < D / 16; ++i) {
                            acc[i][0] *= al0;
                            acc[i][1] *= al1;
                            acc[i][2] *= al0;
                            acc[i][3] *= al1;
                        }
                        m_run[0] = mn0;
                        m_run[1] = mn1;
                    }
                    l_run[0] += p0 + p2;
                    l_run[1] += p1 + p3;
                    // P^T operand (k16 keys x n8 heads) via 8x8 transposes of the score fragment
                    const uint32_t pb0 = movmatrix_trans(pack2<DT>(p0, p1));
                    const uint32_t pb1 = movmatrix_trans(pack2<DT>(p2, p3));
                    // O^T[D, 8] += V_tile^T . P^T
    #pragma unroll
                    for (int i = 0; i < D / 16; ++i) {
                        const int chunk16 = i * 2 + vchunk_add;
                        const uint32_t addr = vbase + (chunk16 >> 3) * Sh::kSliceBytes + vrow * 128 +
                                              (((chunk16 & 7) ^ (vrow & 7)) << 4);
                        uint32_t a[4];
                        ldsm_x4_trans(addr, a);
                        mma_16816<DT>(acc[i], a, pb0, pb1);
                    }
                }
                if (zeroed) {
                    // order the generic-proxy stores above before the next TMA write to this stage
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8 * st);
                if (++st == kStages) {
                    st = 0;
                    ph ^= 1;
                }
            }

            // per-thread partial sums -> per-warp sums (over the 8 key rows g)
    #pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], off);
                l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], off);
            }

            // ---------------- merge the four warps' states for this item, in the
            // ring stage the producer handed over (it loads nothing into it)
            if (ok && !mbar_wait_warp(full0 + 8 * st, ph, p.wait_limit_ns)) {
                ok = false;
                if (lane == 0) flag_error(p.err, DA_DEVERR_TIMEOUT);
            }
            float* red_acc = reinterpret_cast<float*>(smem + st * Sh::kStageBytes);   // [warp][8][D+4]
            float* red_m = red_acc + kConsumerWarps * kHeadsPerCta * Sh::kMergeRow;    // [warp][8]
            float* red_l = red_m + kConsumerWarps * kHeadsPerCta;                       // [warp][8]
            if (g == 0) {
                red_m[warp * kHeadsPerCta + 2 * t4] = m_run[0];
                red_m[warp * kHeadsPerCta + 2 * t4 + 1] = m_run[1];
                red_l[warp * kHeadsPerCta + 2 * t4] = l_run[0];
                red_l[warp * kHeadsPerCta + 2 * t4 + 1] = l_run[1];
            }
            {
                float* h0row = red_acc + (warp * kHeadsPerCta + 2 * t4) * Sh::kMergeRow;
                float* h1row = h0row + Sh::kMergeRow;
    #pragma unroll
                for (int i = 0; i < D / 16; ++i) {
                    h0row[i * 16 + g] = acc[i][0];
                    h1row[i * 16 + g] = acc[i][1];
                    h0row[i * 16 + g + 8] = acc[i][2];
                    h1row[i * 16 + g + 8] = acc[i][3];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(mfull);
            if (ok && !mbar_wait_warp(mfull, it & 1, p.wait_limit_ns)) {
                ok = false;
                if (lane == 0) flag_error(p.err, DA_DEVERR_TIMEOUT);
            }
            // Warp w writes heads w and w + 4; a lane owns four consecutive dims, read
            // from each warp's row as one 16-byte load and stored as one vector. The
            // passes are predicated rather than skipped, so their latencies overlap.
            {
                constexpr int kLanesPerHead = D / 4;
                constexpr int kHeadsPerPass = 32 / kLanesPerHead;   // 1 at head_dim 128, 2 at 64
                constexpr int kPasses = (kHeadsPerCta / kConsumerWarps) / kHeadsPerPass;
                const int d0 = (lane % kLanesPerHead) * 4;
    #pragma unroll
                for (int pass = 0; pass < kPasses; ++pass) {
                    const int hh = warp + kConsumerWarps * (pass * kHeadsPerPass + lane / kLanesPerHead);
                    const bool live = hh < item.nh;
                    float mw[kConsumerWarps];
                    float M = -INFINITY;
    #pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) {
                        mw[w] = red_m[w * kHeadsPerCta + hh];
                        M = fmaxf(M, mw[w]);
                    }
                    // a head that saw no key keeps M = -inf: weights 0, output 0, lse -inf
                    const float Ms = M == -INFINITY ? 0.f : M;
                    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                    float lsum = 0.f;
    #pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) {
                        const float wt = fast_exp2(mw[w] - Ms);
                        lsum = fmaf(wt, red_l[w * kHeadsPerCta + hh], lsum);
                        const float4 a = *reinterpret_cast<const float4*>(
                            red_acc + (w * kHeadsPerCta + hh) * Sh::kMergeRow + d0);
                        o.x = fmaf(wt, a.x, o.x);
                        o.y = fmaf(wt, a.y, o.y);
                        o.z = fmaf(wt, a.z, o.z);
                        o.w = fmaf(wt, a.w, o.w);
                    }
                    // lsum >= 1 whenever M is finite (the largest score weighs 1)
                    const float inv = M == -INFINITY ? 0.f : fast_rcp(lsum);
                    o.x *= inv;
                    o.y *= inv;
                    o.z *= inv;
                    o.w *= inv;
                    if (live) {
                        const int64_t qrow = column_row(p, item, hh);
                        const int64_t row = qrow * p.S + item.s;
                        *reinterpret_cast<float4*>(p.opart + row * D + d0) = o;
                        if (d0 == 0) p.lse[row] = M == -INFINITY ? -INFINITY : (M + fast_log2(lsum)) * kLn2;
                        // one split: its weight exp(lse_0 - lse) is 1, so o_0 is the answer
                        if (p.out != nullptr)
                            *reinterpret_cast<uint2*>(p.out + qrow * D + d0) =
                                make_uint2(pack2<DT>(o.x, o.y), pack2<DT>(o.z, o.w));
                    }
                }
            }
        } else {
        // ---- two n-tiles (up to 16 columns per item): each K and V fragment feeds both
            // Q^T fragments (B operand, k16 x n8) of n-tile n: column 8n + g, dims ks*16 + 2*t4 (+1)
            // and +8 (+9).
            uint32_t qf[D / 16][NT][2];
    #pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int col = 8 * n + g;
                const bool hv = col < item.nh;
                const uint32_t qrow = qbuf + slot * Sh::kQBytes + (hv ? col : 0) * D * 2;
    #pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    uint32_t a0, a1;
                    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a0) : "r"(qrow + (ks * 16 + 2 * t4) * 2));
                    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a1) : "r"(qrow + (ks * 16 + 8 + 2 * t4) * 2));
                    qf[ks][n][0] = hv ? a0 : 0u;
                    qf[ks][n][1] = hv ? a1 : 0u;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(iempty0 + 8 * slot);
            if (!item.valid) break;

            // keys (relative to the split start) visible to this thread's two columns of each n-tile
            int visA[NT], visB[NT];
    #pragma unroll
            for (int n = 0; n < NT; ++n) {
                visA[n] = visB[n] = item.nkeys;
                if (p.tq > 1) {
                    visA[n] = min(item.nkeys, item.vis0 + (item.c0 + 8 * n + 2 * t4) / p.G);
                    visB[n] = min(item.nkeys, item.vis0 + (item.c0 + 8 * n + 2 * t4 + 1) / p.G);
                }
            }
            float acc[D / 16][NT][4];
    #pragma unroll
            for (int i = 0; i < D / 16; ++i)
    #pragma unroll
                for (int n = 0; n < NT; ++n) acc[i][n][0] = acc[i][n][1] = acc[i][n][2] = acc[i][n][3] = 0.f;
            float m_run[NT][2], l_run[NT][2];   // columns 8n + 2*t4 (+1): running max (log2 domain), sum share
    #pragma unroll
            for (int n = 0; n < NT; ++n) {
                m_run[n][0] = m_run[n][1] = -INFINITY;
                l_run[n][0] = l_run[n][1] = 0.f;
            }

            for (int t = 0; t < item.ntiles; ++t) {
                const uint32_t fb = full0 + 8 * st;
                if (ok && !mbar_wait_warp(fb, ph, p.wait_limit_ns)) {
                    ok = false;
                    bad_bar = fb;
                    bad_ph = ph;
                    if (lane == 0) flag_error(p.err, DA_DEVERR_TIMEOUT);
                }
                const int keys_t = min(kStageKeys, item.nkeys - t * kStageKeys);
                bool zeroed = false;
                if (ok && warp * kBoxKeys < keys_t) {
                    const uint32_t kbase = ring + st * Sh::kStageBytes;
                    const uint32_t vbase = kbase + Sh::kTileBytes;
                    const int valid_rows = keys_t - warp * kBoxKeys;
                    if (valid_rows < kBoxKeys) {
                        // The box's rows past the split end hold other keys (or, in a
                        // padded cache, anything): their P is 0, but 0 * NaN is not, so
                        // clear those V rows before the PV product.
                        const int per_row = Sh::kHalves * 8;   // 16-byte chunks per row
                        for (int c = lane; c < (kBoxKeys - valid_rows) * per_row; c += 32) {
                            const int r = valid_rows + c / per_row;
                            const int hf = (c % per_row) >> 3, ch = c & 7;
                            const uint32_t addr = vbase + hf * Sh::kSliceBytes + (warp * kBoxKeys + r) * 128 + ch * 16;
                            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
                        }
                        zeroed = true;
                        __syncwarp();
                    }
                    // S^T[16 keys, 8 columns] = K_tile . Q^T per n-tile, two independent accumulator
                    // chains each; one K fragment feeds every n-tile
                    float sc[NT][4], sd[NT][4];
    #pragma unroll
                    for (int n = 0; n < NT; ++n)
    #pragma unroll
                        for (int j = 0; j < 4; ++j) sc[n][j] = sd[n][j] = 0.f;
    #pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const int chunk16 = ks * 2 + kchunk_add;          // 16-byte chunk along D
                        const uint32_t addr = kbase + (chunk16 >> 3) * Sh::kSliceBytes + krow * 128 +
                                              (((chunk16 & 7) ^ (krow & 7)) << 4);
                        uint32_t a[4];
                        ldsm_x4(addr, a);
    #pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            if (ks & 1) mma_16816<DT>(sd[n], a, qf[ks][n][0], qf[ks][n][1]);
                            else mma_16816<DT>(sc[n], a, qf[ks][n][0], qf[ks][n][1]);
                        }
                    }
                    const int key_lo = t * kStageKeys + warp * kBoxKeys + g;   // relative to split start
                    uint32_t pb0[NT], pb1[NT];
    #pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        // scores -> exp2 domain, mask keys past the split end
                        const float x0 = key_lo < visA[n] ? (sc[n][0] + sd[n][0]) * p.scale_log2 : -INFINITY;
                        const float x1 = key_lo < visB[n] ? (sc[n][1] + sd[n][1]) * p.scale_log2 : -INFINITY;
                        const float x2 = key_lo + 8 < visA[n] ? (sc[n][2] + sd[n][2]) * p.scale_log2 : -INFINITY;
                        const float x3 = key_lo + 8 < visB[n] ? (sc[n][3] + sd[n][3]) * p.scale_log2 : -INFINITY;
                        // Lazy reference: a column's running max m_run moves only when some score
                        // of the warp's box exceeds it by more than kLazyRescale (log2 units), so
                        // the shuffle reduction and the accumulator rescale run on a few boxes
                        // per item; the weights stay below 2^kLazyRescale, well inside the fp16
                        // and bf16 range, and every sum below shares the same reference.
                        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
                        if (__any_sync(0xffffffffu, mx0 > m_run[n][0] + kLazyRescale ||
                                                        mx1 > m_run[n][1] + kLazyRescale)) {
    #pragma unroll
                            for (int off = 4; off < 32; off <<= 1) {
                                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                            }
                            const float mn0 = fmaxf(m_run[n][0], mx0), mn1 = fmaxf(m_run[n][1], mx1);
                            // a column that has seen no key yet (several query tokens) keeps -inf:
                            // 0 stands in as its reference so that no weight below is NaN
                            const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
                            const float al0 = fast_exp2(m_run[n][0] - ms0), al1 = fast_exp2(m_run[n][1] - ms1);
                            l_run[n][0] *= al0;
                            l_run[n][1] *= al1;
    #pragma unroll
                            for (int i = 0; i < D / 16; ++i) {
                                acc[i][n][0] *= al0;
                                acc[i][n][1] *= al1;
                                acc[i][n][2] *= al0;
                                acc[i][n][3] *= al1;
                            }
                            m_run[n][0] = mn0;
                            m_run[n][1] = mn1;
                        }
                        const float ms0 = m_run[n][0] == -INFINITY ? 0.f : m_run[n][0];
                        const float ms1 = m_run[n][1] == -INFINITY ? 0.f : m_run[n][1];
                        const float p0 = fast_exp2(x0 - ms0), p1 = fast_exp2(x1 - ms1);
                        const float p2 = fast_exp2(x2 - ms0), p3 = fast_exp2(x3 - ms1);
                        l_run[n][0] += p0 + p2;
                        l_run[n][1] += p1 + p3;
                        // P^T operand (k16 keys x n8 columns) via 8x8 transposes of the score fragment
                        pb0[n] = movmatrix_trans(pack2<DT>(p0, p1));
                        pb1[n] = movmatrix_trans(pack2<DT>(p2, p3));
                    }
                    // O^T[D, 8 per n-tile] += V_tile^T . P^T; one V fragment feeds every n-tile
    #pragma unroll
                    for (int i = 0; i < D / 16; ++i) {
                        const int chunk16 = i * 2 + vchunk_add;
                        const uint32_t addr = vbase + (chunk16 >> 3) * Sh::kSliceBytes + vrow * 128 +
                                              (((chunk16 & 7) ^ (vrow & 7)) << 4);
                        uint32_t a[4];
                        ldsm_x4_trans(addr, a);
    #pragma unroll
                        for (int n = 0; n < NT; ++n) mma_16816<DT>(acc[i][n], a, pb0[n], pb1[n]);
                    }
                }
                if (zeroed) {
                    // order the generic-proxy stores above before the next TMA write to this stage
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8 * st);
                if (++st == kStages) {
                    st = 0;
                    ph ^= 1;
                }
            }

            // per-thread partial sums -> per-warp sums (over the 8 key rows g)
    #pragma unroll
            for (int n = 0; n < NT; ++n)
    #pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    l_run[n][0] += __shfl_xor_sync(0xffffffffu, l_run[n][0], off);
                    l_run[n][1] += __shfl_xor_sync(0xffffffffu, l_run[n][1], off);
                }

            // ---------------- merge the four warps' states for this item, in the
            // ring stage the producer handed over (it loads nothing into it), one
            // n-tile (8 columns) per round
            if (ok && !mbar_wait_warp(full0 + 8 * st, ph, p.wait_limit_ns)) {
                ok = false;
                if (lane == 0) flag_error(p.err, DA_DEVERR_TIMEOUT);
            }
            float* red_acc = reinterpret_cast<float*>(smem + st * Sh::kStageBytes);   // [warp][8][D+4]
            float* red_m = red_acc + kConsumerWarps * 8 * Sh::kMergeRow;               // [warp][8]
            float* red_l = red_m + kConsumerWarps * 8;                                  // [warp][8]
    #pragma unroll
            for (int n = 0; n < NT; ++n) {
                if (n > 0) {
                    // every warp has read the previous round's rows before they are overwritten
                    __syncwarp();
                    if (lane == 0) mbar_arrive(mdone);
                    if (ok && !mbar_wait_warp(mdone, md & 1, p.wait_limit_ns)) {
                        ok = false;
                        if (lane == 0) flag_error(p.err, DA_DEVERR_TIMEOUT);
                    }
                    ++md;
                }
                if (g == 0) {
                    red_m[warp * 8 + 2 * t4] = m_run[n][0];
                    red_m[warp * 8 + 2 * t4 + 1] = m_run[n][1];
                    red_l[warp * 8 + 2 * t4] = l_run[n][0];
                    red_l[warp * 8 + 2 * t4 + 1] = l_run[n][1];
                }
                {
                    float* h0row = red_acc + (warp * 8 + 2 * t4) * Sh::kMergeRow;
                    float* h1row = h0row + Sh::kMergeRow;
    #pragma unroll
                    for (int i = 0; i < D / 16; ++i) {
                        h0row[i * 16 + g] = acc[i][n][0];
                        h1row[i * 16 + g] = acc[i][n][1];
                        h0row[i * 16 + g + 8] = acc[i][n][2];
                        h1row[i * 16 + g + 8] = acc[i][n][3];
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(mfull);
                if (ok && !mbar_wait_warp(mfull, mz & 1, p.wait_limit_ns)) {
                    ok = false;
                    if (lane == 0) flag_error(p.err, DA_DEVERR_TIMEOUT);
                }
                ++mz;
                // Warp w writes columns w and w + 4 of the round; a lane owns four consecutive
                // dims, read from each warp's row as one 16-byte load and stored as one vector.
                // The passes are predicated rather than skipped, so their latencies overlap.
                constexpr int kLanesPerHead = D / 4;
                constexpr int kHeadsPerPass = 32 / kLanesPerHead;   // 1 at head_dim 128, 2 at 64
                constexpr int kPasses = (8 / kConsumerWarps) / kHeadsPerPass;
                const int d0 = (lane % kLanesPerHead) * 4;
    #pragma unroll
                for (int pass = 0; pass < kPasses; ++pass) {
                    const int hh = warp + kConsumerWarps * (pass * kHeadsPerPass + lane / kLanesPerHead);
                    const bool live = 8 * n + hh < item.nh;
                    float mw[kConsumerWarps];
                    float M = -INFINITY;
    #pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) {
                        mw[w] = red_m[w * 8 + hh];
                        M = fmaxf(M, mw[w]);
                    }
                    // a column that saw no key keeps M = -inf: weights 0, output 0, lse -inf
                    const float Ms = M == -INFINITY ? 0.f : M;
                    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                    float lsum = 0.f;
    #pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) {
                        const float wt = fast_exp2(mw[w] - Ms);
                        lsum = fmaf(wt, red_l[w * 8 + hh], lsum);
                        const float4 a = *reinterpret_cast<const float4*>(red_acc + (w * 8 + hh) * Sh::kMergeRow + d0);
                        o.x = fmaf(wt, a.x, o.x);
                        o.y = fmaf(wt, a.y, o.y);
                        o.z = fmaf(wt, a.z, o.z);
                        o.w = fmaf(wt, a.w, o.w);
                    }
                    // lsum >= 1 whenever M is finite (the largest score weighs 1)
                    const float inv = M == -INFINITY ? 0.f : fast_rcp(lsum);
                    o.x *= inv;
                    o.y *= inv;
                    o.z *= inv;
                    o.w *= inv;
                    if (live) {
                        const int64_t qrow = column_row(p, item, 8 * n + hh);
                        const int64_t row = qrow * p.S + item.s;
                        *reinterpret_cast<float4*>(p.opart + row * D + d0) = o;
                        if (d0 == 0) p.lse[row] = M == -INFINITY ? -INFINITY : (M + fast_log2(lsum)) * kLn2;
                        // one split: its weight exp(lse_0 - lse) is 1, so o_0 is the answer
                        if (p.out != nullptr)
                            *reinterpret_cast<uint2*>(p.out + qrow * D + d0) =
                                make_uint2(pack2<DT>(o.x, o.y), pack2<DT>(o.z, o.w));
                    }
                }
            }
        }
        // release the stage: order these generic-proxy stores before the TMA writes that refill it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * st);
        if (++st == kStages) {
            st = 0;
            ph ^= 1;
        }
        if (!ok) break;
    }
    if (!ok) {
        // a copy may still be landing: give it one more bounded wait before the CTA exits
        if (bad_bar != 0) mbar_wait(bad_bar, bad_ph, p.wait_limit_ns);
        return;
    }
    // The last CTA to finish re-arms the work queue for the next call. No fence:
    // the counters order no data (the outputs are read only after this grid
    // completes), and every CTA's last queue atomic has returned before its
    // producer published the end of the queue, which precedes this increment.
    if (threadIdx.x == 0) {
        const uint32_t prev = atomicAdd(p.done, 1u);
        if (prev == gridDim.x - 1) {
            atomicExch(p.work, 0u);
            atomicExch(p.done, 0u);
        }
    }
}

// ------------------------------------------------------------ split step on tensor memory
// Items of more than 8 packed (query token, head) columns, up to 32 per item:
// the products run on the tcgen05 tensor cores with S, P and O held in tensor
// memory. Per 64-key stage,
//   S[row, key] = Q[row, :] . K[key, :]     (A = Q rows, M = 128; B = K tile, N = 64)
//   O[row, :]  += P[row, key] . V[key, :]   (A = P in tensor memory; B = V tile, MN-major)
// The 128 MMA rows cost the same whatever they hold, so the item's columns are
// laid into all four 32-row quarters: warp k (k = 0..3, one per SM
// sub-partition, each reading its own quarter of tensor memory) takes keys
// 16k .. 16k + 15 of every stage for every column, with its own running
// reference, sum and O rows (the P entries of the other keys of its rows stay
// 0). The four partial states of a column are merged through shared memory at
// the end of the item. Warps: 0-3 softmax and epilogue, 4 producer (TMA and the
// work queue, as in split_kernel), 5 MMA issue (one lane) and the tensor-memory
// allocation.
constexpr int kTcSoftmaxWarps = 4;
constexpr int kTcProducerWarp = 4;
constexpr int kTcMmaWarp = 5;
constexpr int kTcThreads = 6 * 32;
constexpr int kTcCols = 32;                                 // packed columns per item at most
constexpr int kTcM = 128;                                   // MMA M: four copies of the item's rows
constexpr int kTcKeysPerWarp = kStageKeys / kTcSoftmaxWarps;   // 16
constexpr int kTcMergeRow = 32 + 4;                         // floats per row of a merge chunk (padded)

struct TcParams {
    SplitParams sp;
    int item_cols;     // packed columns per item: G * item_tokens
    int item_tokens;   // query tokens per item
};

template <int D>
struct TcShape {
    static constexpr int kHalves = D / 64;
    static constexpr int kSliceBytes = kStageKeys * 128;
    static constexpr int kTileBytes = kHalves * kSliceBytes;
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kBoxBytes = kBoxKeys * 128;
    static constexpr int kStages = D == 128 ? 4 : 8;
    static constexpr int kQSliceBytes = kTcM * 128;             // one 64-dim slice of the A operand
    static constexpr int kQBytes = kHalves * kQSliceBytes;
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = kItemSlots * kQBytes;
    // item merge: [warp][column][32 dims + pad] of one 32-dim chunk of O, then [warp][column] m and l
    static constexpr int kMergeOff = kRingOff + kStages * kStageBytes;
    static constexpr int kMergeBytes = (kTcSoftmaxWarps * kTcCols * kTcMergeRow + 2 * kTcSoftmaxWarps * kTcCols) * 4;
    static constexpr int kSlotOff = kMergeOff + kMergeBytes;
    static constexpr int kBarOff = kSlotOff + kItemSlots * (int)sizeof(ItemSlot);
    // full/empty [kStages], ifull/iempty [kItemSlots], s_full/s_free/p_full/p_free [2], o_full, o_free, fin, merge
    static constexpr int kNumBars = 2 * kStages + 2 * kItemSlots + 8 + 4;
    static constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
    static constexpr int kEnd = kTmemSlotOff + 16;
    static constexpr int kSmemBytes = 1024 + kEnd;
    static_assert(kRingOff % 1024 == 0 && kQSliceBytes % 1024 == 0, "swizzled tiles need 1024-byte alignment");
    static_assert(kSlotOff % 16 == 0 && kBarOff % 8 == 0, "smem alignment");
    // tensor-memory columns: S[2] (64 fp32 each), P[2] (32 columns of fp16 pairs each), O (D fp32)
    static constexpr uint32_t kTmemS = 0;
    static constexpr uint32_t kTmemP = 128;
    static constexpr uint32_t kTmemO = D == 128 ? 256 : 192;
    static constexpr uint32_t kTmemCols = D == 128 ? 512 : 256;
};

template <int D, int DT>
__global__ void __launch_bounds__(kTcThreads, 1)
split_kernel_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const __grid_constant__ CUtensorMap tmK16, const __grid_constant__ CUtensorMap tmV16,
                const __grid_constant__ CUtensorMap tmQ, const TcParams tp) {
    const SplitParams& p = tp.sp;
    using Sh = TcShape<D>;
    constexpr int kSt = Sh::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    ItemSlot* slots = reinterpret_cast<ItemSlot*>(smem + Sh::kSlotOff);
    const uint32_t base = smem_addr(smem);
    const uint32_t qbuf = base + Sh::kQOff;
    const uint32_t ring = base + Sh::kRingOff;
    const uint32_t full0 = base + Sh::kBarOff;        // [kSt]   K/V stage landed
    const uint32_t empty0 = full0 + 8 * kSt;          // [kSt]   its PV product done
    const uint32_t ifull0 = empty0 + 8 * kSt;         // [slots] item descriptor and Q rows in place
    const uint32_t iempty0 = ifull0 + 8 * kItemSlots; // [slots] item slot free again
    const uint32_t sfull0 = iempty0 + 8 * kItemSlots; // [2]     S product done
    const uint32_t sfree0 = sfull0 + 16;              // [2]     S read by the softmax warps
    const uint32_t pfull0 = sfree0 + 16;              // [2]     P written (and O rescaled)
    const uint32_t pfree0 = pfull0 + 16;              // [2]     PV product done
    const uint32_t ofull = pfree0 + 16;               // item's last PV product done
    const uint32_t ofree = ofull + 8;                 // item's O read by the epilogue
    const uint32_t fin = ofree + 8;                   // every MMA done (before the free)
    const uint32_t mrg = fin + 8;                     // one round of the item merge
    const uint32_t tmem_slot = base + Sh::kTmemSlotOff;
    int32_t* cus = p.stage_cu ? reinterpret_cast<int32_t*>(smem + Sh::kEnd) : nullptr;
    int32_t* prefix = reinterpret_cast<int32_t*>(smem + Sh::kEnd + (p.stage_cu ? kStagedBytes : 0));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSt; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
        }
        for (int i = 0; i < kItemSlots; ++i) {
            mbar_init(ifull0 + 8 * i, 1);
            mbar_init(iempty0 + 8 * i, kTcSoftmaxWarps + 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(sfull0 + 8 * i, 1);
            mbar_init(sfree0 + 8 * i, kTcSoftmaxWarps);
            mbar_init(pfull0 + 8 * i, kTcSoftmaxWarps);
            mbar_init(pfree0 + 8 * i, 1);
        }
        mbar_init(ofull, 1);
        mbar_init(ofree, kTcSoftmaxWarps);
        mbar_init(fin, 1);
        mbar_init(mrg, kTcSoftmaxWarps);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_slot),
                     "r"(Sh::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == kTcProducerWarp && lane == 0 && p.no_kv == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        prefetch_tensormap(&tmK16);
        prefetch_tensormap(&tmV16);
        prefetch_tensormap(&tmQ);
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    uint32_t tmem;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(tmem_slot) : "memory");
    grid_dependency_wait();
    if (threadIdx.x == 0) grid_dependents_launch();

    bool ok = true;
    if (warp == kTcProducerWarp) {
        // ---------------- producer: the work queue, Q rows and the K/V ring
        int n_items = p.n_items;
        if (cus != nullptr) {
            for (int i = lane; i <= p.B; i += 32) cus[i] = ld_cg_s32(p.cu + i);
            __syncwarp();
        }
        if (p.split_len != 0) {
            int carry = 0;
            for (int b0 = 0; b0 < p.B; b0 += 32) {
                const int b = b0 + lane;
                int sb = 0;
                if (b < p.B) {
                    int64_t kv_base;
                    bool bad;
                    const int64_t L = cus != nullptr ? checked_len_of(cus[b], cus[b + 1], p.layout, p.kv_rows,
                                                                      p.no_kv, &kv_base, &bad)
                                                     : checked_len(p.cu, b, p.layout, p.kv_rows, p.no_kv, &kv_base, &bad);
                    sb = seq_splits(L, p.split_len, p.S);
                }
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, sb, off);
                    if (lane >= off) sb += y;
                }
                if (b < p.B) prefix[b + 1] = carry + sb;
                carry += __shfl_sync(0xffffffffu, sb, 31);
            }
            if (lane == 0) prefix[0] = 0;
            __syncwarp();
            n_items = carry * p.Hkv * p.chunks;
        }
        if (lane == 0) {
            int st = 0;
            uint32_t ph = 0;
            // Item `idx` into slot `it % kItemSlots`, with its Q rows: a TMA box
            // [tokens][G heads][64 dims] lands as rows c - c0 of each 32-row quarter
            // of a 64-dim slice, in the 128-byte-swizzled layout the MMA reads.
            auto publish = [&](uint32_t it, int idx, ItemSlot& item) -> int {
                const int slot = it % kItemSlots;
                const uint32_t iph = (it / kItemSlots) & 1;
                if (!mbar_wait(iempty0 + 8 * slot, iph ^ 1, p.wait_limit_ns)) {
                    flag_error(p.err, DA_DEVERR_TIMEOUT);
                    return -1;
                }
                if (idx >= n_items) {
                    slots[slot].valid = 0;
                    mbar_arrive(ifull0 + 8 * slot);
                    return 0;
                }
                item = decode_item_cols(p, idx, cus, prefix, tp.item_cols);
                slots[slot] = item;
                const uint32_t ib = ifull0 + 8 * slot;
                mbar_arrive_expect_tx(ib, Sh::kHalves * kTcSoftmaxWarps * 64 * p.G * tp.item_tokens * 2);
                const int row0 = item.b * p.tq + item.c0 / p.G;   // token coordinate of the box
                for (int hf = 0; hf < Sh::kHalves; ++hf)
                    for (int k = 0; k < kTcSoftmaxWarps; ++k)
                        tma_load_3d(qbuf + slot * Sh::kQBytes + hf * Sh::kQSliceBytes + k * 32 * 128, &tmQ, hf * 64,
                                    item.h0, row0, ib);
                return 1;
            };
            ItemSlot item;
            int state = publish(0, static_cast<int>(blockIdx.x), item);
            for (uint32_t it = 0; state == 1; ++it) {
                const int fetch_at = max(0, item.ntiles - kSt);
                int next_idx = 0;
                if (item.ntiles == 0) next_idx = static_cast<int>(gridDim.x + atomicAdd(p.work, 1u));
                for (int t = 0; t < item.ntiles; ++t) {
                    if (t == fetch_at) next_idx = static_cast<int>(gridDim.x + atomicAdd(p.work, 1u));
                    if (!mbar_wait(empty0 + 8 * st, ph ^ 1, p.wait_limit_ns)) {
                        flag_error(p.err, DA_DEVERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    const int keys_t = min(kStageKeys, item.nkeys - t * kStageKeys);
                    const uint32_t fb = full0 + 8 * st;
                    const uint32_t kdst = ring + st * Sh::kStageBytes;
                    const uint32_t vdst = kdst + Sh::kTileBytes;
                    const int key0 = static_cast<int>(item.first_key) + t * kStageKeys;
                    const int slab = item.b * p.Hkv + item.kvh;
                    if (keys_t == kStageKeys) {
                        mbar_arrive_expect_tx(fb, Sh::kHalves * 2 * Sh::kSliceBytes);
                        for (int hf = 0; hf < Sh::kHalves; ++hf) {
                            const uint32_t off = hf * Sh::kSliceBytes;
                            if (p.layout == DA_LAYOUT_VARLEN) {
                                tma_load_3d(kdst + off, &tmK, hf * 64, item.kvh, key0, fb);
                                tma_load_3d(vdst + off, &tmV, hf * 64, item.kvh, key0, fb);
                            } else {
                                tma_load_3d(kdst + off, &tmK, hf * 64, key0, slab, fb);
                                tma_load_3d(vdst + off, &tmV, hf * 64, key0, slab, fb);
                            }
                        }
                    } else {
                        const int nbox = (keys_t + kBoxKeys - 1) / kBoxKeys;
                        mbar_arrive_expect_tx(fb, nbox * Sh::kHalves * 2 * Sh::kBoxBytes);
                        for (int bx = 0; bx < nbox; ++bx) {
                            const int key = key0 + bx * kBoxKeys;
                            for (int hf = 0; hf < Sh::kHalves; ++hf) {
                                const uint32_t off = hf * Sh::kSliceBytes + bx * Sh::kBoxBytes;
                                if (p.layout == DA_LAYOUT_VARLEN) {
                                    tma_load_3d(kdst + off, &tmK16, hf * 64, item.kvh, key, fb);
                                    tma_load_3d(vdst + off, &tmV16, hf * 64, item.kvh, key, fb);
                                } else {
                                    tma_load_3d(kdst + off, &tmK16, hf * 64, key, slab, fb);
                                    tma_load_3d(vdst + off, &tmV16, hf * 64, key, slab, fb);
                                }
                            }
                        }
                    }
                    if (++st == kSt) {
                        st = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                ItemSlot next;
                const int next_state = publish(it + 1, next_idx, next);
                if (next_state < 0) {
                    ok = false;
                    break;
                }
                item = next;
                state = next_state;
            }
        }
    } else if (warp == kTcMmaWarp) {
        // ---------------- MMA issue: S(g) for the next stage goes out before PV(g - 1)
        if (lane == 0) {
            constexpr uint32_t kIdS = umma_idesc<DT>(kTcM, kStageKeys, false);
            constexpr uint32_t kIdPV = umma_idesc<DT>(kTcM, 64, true);
            uint32_t g = 0;          // stages consumed by this CTA so far (S and P buffer = g & 1)
            int st = 0;
            uint32_t ph = 0;
            uint32_t nitem = 0;
            // O += P(u) . V(stage): two 64-dim halves, four 16-key steps
            auto pv = [&](uint32_t u, int stage, bool first) -> bool {
                if (!mbar_wait(pfull0 + 8 * (u & 1), (u >> 1) & 1, p.wait_limit_ns)) return false;
                if (first && nitem > 0 && !mbar_wait(ofree, (nitem - 1) & 1, p.wait_limit_ns)) return false;
                tmem_fence_after_sync();
                const uint64_t vdesc = umma_desc_sw128(ring + stage * Sh::kStageBytes + Sh::kTileBytes, 1024, 1024);
                const uint32_t pa = tmem + Sh::kTmemP + (u & 1) * 32;
#pragma unroll
                for (int hf = 0; hf < Sh::kHalves; ++hf)
#pragma unroll
                    for (int k16 = 0; k16 < kStageKeys / 16; ++k16)
                        umma_ts(tmem + Sh::kTmemO + hf * 64, pa + k16 * 8,
                                vdesc + ((hf * Sh::kSliceBytes + k16 * 16 * 128) >> 4), kIdPV, !(first && k16 == 0));
                umma_commit(empty0 + 8 * stage);
                umma_commit(pfree0 + 8 * (u & 1));
                return true;
            };
            for (uint32_t it = 0; ok; ++it) {
                const int slot = it % kItemSlots;
                if (!mbar_wait(ifull0 + 8 * slot, (it / kItemSlots) & 1, p.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                const ItemSlot item = slots[slot];
                if (!item.valid) {
                    mbar_arrive(iempty0 + 8 * slot);
                    break;
                }
                const uint64_t qdesc = umma_desc_sw128(qbuf + slot * Sh::kQBytes, 16, 1024);
                int st_prev = 0;
                for (int t = 0; t < item.ntiles; ++t) {
                    if (!mbar_wait(full0 + 8 * st, ph, p.wait_limit_ns) ||
                        (g >= 2 && !mbar_wait(sfree0 + 8 * (g & 1), ((g - 2) >> 1) & 1, p.wait_limit_ns))) {
                        ok = false;
                        break;
                    }
                    tmem_fence_after_sync();
                    const uint64_t kdesc = umma_desc_sw128(ring + st * Sh::kStageBytes, 16, 1024);
#pragma unroll
                    for (int k16 = 0; k16 < D / 16; ++k16) {
                        const uint32_t off = (k16 & 3) * 32;   // 16-dim step inside the 128-byte row
                        umma_ss(tmem + Sh::kTmemS + (g & 1) * 64, qdesc + (((k16 >> 2) * Sh::kQSliceBytes + off) >> 4),
                                kdesc + (((k16 >> 2) * Sh::kSliceBytes + off) >> 4), kIdS, k16 > 0);
                    }
                    umma_commit(sfull0 + 8 * (g & 1));
                    if (t > 0 && !pv(g - 1, st_prev, t == 1)) {
                        ok = false;
                        break;
                    }
                    st_prev = st;
                    if (++st == kSt) {
                        st = 0;
                        ph ^= 1;
                    }
                    ++g;
                }
                if (!ok) break;
                if (item.ntiles > 0 && !pv(g - 1, st_prev, item.ntiles == 1)) {
                    ok = false;
                    break;
                }
                umma_commit(iempty0 + 8 * slot);   // the slot's Q rows are free once these MMAs are done
                umma_commit(ofull);
                ++nitem;
            }
            // every MMA issued has completed before the tensor memory is freed
            umma_commit(fin);
            mbar_wait(fin, 0, p.wait_limit_ns);
        }
        __syncwarp();
    } else {
        // ---------------- softmax and epilogue: warp k = keys 16k..16k+15 of every stage, lane = column
        const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
        const int col = lane;
        float* red_o = reinterpret_cast<float*>(smem + Sh::kMergeOff);       // [warp][column][kTcMergeRow]
        float* red_m = red_o + kTcSoftmaxWarps * kTcCols * kTcMergeRow;       // [warp][column]
        float* red_l = red_m + kTcSoftmaxWarps * kTcCols;                     // [warp][column]
        {
            // the P entries of the other warps' keys stay 0 in this warp's rows
            uint32_t z[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) z[j] = 0u;
            tmem_st32(tmem + lane_base + Sh::kTmemP, z);
            tmem_st32(tmem + lane_base + Sh::kTmemP + 32, z);
        }
        uint32_t g = 0;
        int st = 0;
        uint32_t nitem = 0;
        uint32_t mq = 0;   // rounds of the merge barrier used
        // all four softmax warps meet (a bounded wait, so that a warp that gave up
        // elsewhere cannot hold the others)
        auto merge_round = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(mrg);
            const bool r = mbar_wait_warp(mrg, mq & 1, p.wait_limit_ns);
            ++mq;
            return r;
        };
        for (uint32_t it = 0;; ++it) {
            const int slot = it % kItemSlots;
            if (!mbar_wait_warp(ifull0 + 8 * slot, (it / kItemSlots) & 1, p.wait_limit_ns)) {
                if (lane == 0) flag_error(p.err, DA_DEVERR_TIMEOUT);
                ok = false;
                break;
            }
            const ItemSlot item = slots[slot];
            if (!item.valid) {
                __syncwarp();
                if (lane == 0) mbar_arrive(iempty0 + 8 * slot);
                break;
            }
            const bool live = col < item.nh;
            int vis = item.nkeys;
            if (p.tq > 1) vis = min(item.nkeys, item.vis0 + (item.c0 + col) / p.G);
            float m_ref = -INFINITY, l_sum = 0.f;
            for (int t = 0; t < item.ntiles; ++t) {
                const uint32_t b = g & 1;
                if (!mbar_wait_warp(sfull0 + 8 * b, (g >> 1) & 1, p.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                tmem_fence_after_sync();
                uint32_t x[kTcKeysPerWarp];
                tmem_ld16(tmem + lane_base + Sh::kTmemS + b * 64 + warp * kTcKeysPerWarp, x);
                tmem_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(sfree0 + 8 * b);
                // keys of this warp's range the column sees
                const int lim = live ? vis - t * kStageKeys - warp * kTcKeysPerWarp : 0;
                float mx = -INFINITY;
#pragma unroll
                for (int j = 0; j < kTcKeysPerWarp; ++j) {
                    const float sc = j < lim ? __uint_as_float(x[j]) * p.scale_log2 : -INFINITY;
                    x[j] = __float_as_uint(sc);
                    mx = fmaxf(mx, sc);
                }
                // lagging reference: it moves only when a score passes it by more than
                // kLazyRescale (log2 units); this warp's O rows are rescaled then
                if (__any_sync(0xffffffffu, mx > m_ref + kLazyRescale)) {
                    const float mn = fmaxf(m_ref, mx);
                    const float ms = mn == -INFINITY ? 0.f : mn;
                    const float al = fast_exp2(m_ref - ms);   // 0 while the column has seen nothing
                    l_sum *= al;
                    if (t > 0) {
                        // O holds this item's sums up to the previous stage: wait for that PV
                        if (!mbar_wait_warp(pfree0 + 8 * ((g - 1) & 1), ((g - 1) >> 1) & 1, p.wait_limit_ns)) {
                            ok = false;
                            break;
                        }
                        tmem_fence_after_sync();
#pragma unroll 1
                        for (int q32 = 0; q32 < D / 32; ++q32) {
                            uint32_t o[32];
                            tmem_ld32(tmem + lane_base + Sh::kTmemO + q32 * 32, o);
#pragma unroll
                            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * al);
                            tmem_st32(tmem + lane_base + Sh::kTmemO + q32 * 32, o);
                        }
                    }
                    m_ref = mn;
                }
                const float ms = m_ref == -INFINITY ? 0.f : m_ref;
                uint32_t pk[kTcKeysPerWarp / 2];
                float sum = 0.f;
#pragma unroll
                for (int j = 0; j < kTcKeysPerWarp / 2; ++j) {
                    const float p0 = fast_exp2(__uint_as_float(x[2 * j]) - ms);
                    const float p1 = fast_exp2(__uint_as_float(x[2 * j + 1]) - ms);
                    sum += p0 + p1;
                    pk[j] = pack2<DT>(p0, p1);
                }
                l_sum += sum;
                // P buffer b was last read by PV(g - 2)
                if (g >= 2 && !mbar_wait_warp(pfree0 + 8 * b, ((g - 2) >> 1) & 1, p.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                tmem_st8(tmem + lane_base + Sh::kTmemP + b * 32 + warp * (kTcKeysPerWarp / 2), pk);
                const int keys_t = min(kStageKeys, item.nkeys - t * kStageKeys);
                if (keys_t < kStageKeys) {
                    // V rows past the split end hold other keys (or anything, in a padded
                    // cache): their P is 0, but 0 * NaN is not, so clear them before PV
                    const uint32_t vb = ring + st * Sh::kStageBytes + Sh::kTileBytes;
                    const int nchunks = (kStageKeys - keys_t) * 8 * Sh::kHalves;
                    for (int c = 32 * warp + lane; c < nchunks; c += 32 * kTcSoftmaxWarps) {
                        const int r = keys_t + c / (8 * Sh::kHalves);
                        const int rem = c % (8 * Sh::kHalves);
                        const uint32_t addr = vb + (rem >> 3) * Sh::kSliceBytes + r * 128 + (rem & 7) * 16;
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                tmem_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(pfull0 + 8 * b);
                ++g;
                if (++st == kSt) st = 0;
            }
            if (!ok) break;
            // ---- epilogue: merge the four warps' partial states of each column,
            // o_s = sum_k 2^(m_k - M) O_k / sum_k 2^(m_k - M) l_k, lse_s = ln of the sum + M
            if (!mbar_wait_warp(ofull, nitem & 1, p.wait_limit_ns)) {
                ok = false;
                break;
            }
            tmem_fence_after_sync();
            red_m[warp * kTcCols + col] = m_ref;
            red_l[warp * kTcCols + col] = l_sum;
            if (!merge_round()) {
                ok = false;
                break;
            }
            float M = -INFINITY;
#pragma unroll
            for (int k = 0; k < kTcSoftmaxWarps; ++k) M = fmaxf(M, red_m[k * kTcCols + col]);
            const float Ms = M == -INFINITY ? 0.f : M;
            float L = 0.f;
#pragma unroll
            for (int k = 0; k < kTcSoftmaxWarps; ++k) L += fast_exp2(red_m[k * kTcCols + col] - Ms) * red_l[k * kTcCols + col];
            // L >= 1 once the column has seen a key (its largest score weighs at least 1)
            const float wk = M == -INFINITY ? 0.f : fast_exp2(m_ref - Ms) * fast_rcp(L);
            if (warp == 0 && live) {
                const int64_t row = column_row(p, item, col) * p.S + item.s;
                p.lse[row] = M == -INFINITY ? -INFINITY : (M + fast_log2(L)) * kLn2;
            }
            // the chunk's rows out: warp k writes columns 8k..8k+7, 8 dims per lane
            const int oc = 8 * warp + (lane >> 2);
            const int od = (lane & 3) * 8;
            const bool olive = oc < item.nh;
            int64_t oqrow = 0, orow = 0;
            if (olive) {
                oqrow = column_row(p, item, oc);
                orow = oqrow * p.S + item.s;
            }
#pragma unroll 1
            for (int q32 = 0; q32 < D / 32; ++q32) {
                uint32_t o[32];
                if (item.ntiles > 0) tmem_ld32(tmem + lane_base + Sh::kTmemO + q32 * 32, o);
                float* mine = red_o + (warp * kTcCols + col) * kTcMergeRow;
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4*>(mine + j) =
                        item.ntiles > 0 ? make_float4(__uint_as_float(o[j]) * wk, __uint_as_float(o[j + 1]) * wk,
                                                      __uint_as_float(o[j + 2]) * wk, __uint_as_float(o[j + 3]) * wk)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                if (!merge_round()) {
                    ok = false;
                    break;
                }
                float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
#pragma unroll
                for (int k = 0; k < kTcSoftmaxWarps; ++k) {
                    const float* src = red_o + (k * kTcCols + oc) * kTcMergeRow + od;
                    const float4 u0 = *reinterpret_cast<const float4*>(src);
                    const float4 u1 = *reinterpret_cast<const float4*>(src + 4);
                    a0.x += u0.x; a0.y += u0.y; a0.z += u0.z; a0.w += u0.w;
                    a1.x += u1.x; a1.y += u1.y; a1.z += u1.z; a1.w += u1.w;
                }
                if (olive) {
                    float* dst = p.opart + orow * D + q32 * 32 + od;
                    *reinterpret_cast<float4*>(dst) = a0;
                    *reinterpret_cast<float4*>(dst + 4) = a1;
                    if (p.out != nullptr)
                        *reinterpret_cast<uint4*>(p.out + oqrow * D + q32 * 32 + od) =
                            make_uint4(pack2<DT>(a0.x, a0.y), pack2<DT>(a0.z, a0.w), pack2<DT>(a1.x, a1.y),
                                       pack2<DT>(a1.z, a1.w));
                }
                // every warp has read the chunk before the next one overwrites it
                if (!merge_round()) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            tmem_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(ofree);
                mbar_arrive(iempty0 + 8 * slot);
            }
            ++nitem;
        }
    }

    // every warp gets here, also after a timed-out wait (each wait is bounded)
    tmem_fence_before_sync();
    const int all_ok = __syncthreads_and(ok ? 1 : 0);
    if (warp == kTcMmaWarp) {
        tmem_fence_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Sh::kTmemCols)
                     : "memory");
    }
    if (!all_ok) {
        if (threadIdx.x == 0) flag_error(p.err, DA_DEVERR_TIMEOUT);
        return;
    }
    // the last CTA to finish re-arms the work queue (as in split_kernel)
    if (threadIdx.x == 0) {
        const uint32_t prev = atomicAdd(p.done, 1u);
        if (prev == gridDim.x - 1) {
            atomicExch(p.work, 0u);
            atomicExch(p.done, 0u);
        }
    }
}

// ------------------------------------------------------------ combine step
// Fold one split (its lse and four dims of its o) into a lane's running
// (max, sum, weighted accumulator); the max moves up as larger lse arrive, so a
// single pass over the splits suffices. Empty splits (lse = -inf) weigh 0.
__device__ __forceinline__ void combine_fold(float lv, float4 ov, float& m, float& z, float4& acc) {
    if (lv == -INFINITY) return;
    if (lv > m) {
        const float sc = fast_exp2((m - lv) * kLog2e);   // 0 when m is still -inf
        acc.x *= sc;
        acc.y *= sc;
        acc.z *= sc;
        acc.w *= sc;
        z *= sc;
        m = lv;
    }
    const float w = fast_exp2((lv - m) * kLog2e);
    acc.x = fmaf(w, ov.x, acc.x);
    acc.y = fmaf(w, ov.y, acc.y);
    acc.z = fmaf(w, ov.z, acc.z);
    acc.w = fmaf(w, ov.w, acc.w);
    z += w;
}

// One warp per (row = (b, query head), slice of DC = D / dchunks dims). Each
// lane owns four dims of one split at a time; 32 / (DC / 4) splits are read per
// iteration, four iterations' loads are issued together, and the lanes' partial
// states are merged with shuffles at the end (a fixed order: deterministic).
struct CombineParams {
    const float* lse;        // [rows, S]
    const float* opart;      // [rows, S, D]
    uint16_t* out;           // [rows, D]
    const int32_t* cu;       // per-sequence mode: row r's split count comes from sequence r / Hq
    int rows, S, dchunks, Hq, split_len, layout, kv_rows, no_kv;
};

template <int D, int DT>
__global__ void __launch_bounds__(128) combine_kernel(const CombineParams cp) {
    grid_dependency_wait();
    if (threadIdx.x == 0) grid_dependents_launch();
    const int warp_id = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (warp_id >= cp.rows * cp.dchunks) return;
    const int dchunks = cp.dchunks, S = cp.S;
    const int row = warp_id / dchunks, dc = warp_id % dchunks;
    int Srow = S;   // splits present in this row
    if (cp.split_len != 0) {
        int64_t base;
        bool bad;
        Srow = seq_splits(checked_len(cp.cu, row / cp.Hq, cp.layout, cp.kv_rows, cp.no_kv, &base, &bad),
                          cp.split_len, S);
    }
    const int DC = D / dchunks;
    const int lps = DC / 4;               // lanes per split row
    const int spi = 32 / lps;             // splits per iteration
    const int sub = lane / lps, dv = lane % lps;
    const int d0 = dc * DC + dv * 4;
    const float* l = cp.lse + static_cast<int64_t>(row) * S;
    const float* po = cp.opart + static_cast<int64_t>(row) * S * D + d0;

    float m = -INFINITY, z = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // four iterations' loads are issued before any is folded (a missing one reads
    // as an empty split), so a row of up to 4 * spi splits costs one L2 round trip
    for (int s0 = sub; s0 < Srow; s0 += 4 * spi) {
        float lv[4];
        float4 ov[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int s = s0 + u * spi;
            if (s < Srow) {
                lv[u] = __ldcg(l + s);
                ov[u] = __ldcg(reinterpret_cast<const float4*>(po + static_cast<int64_t>(s) * D));
            } else {
                lv[u] = -INFINITY;
                ov[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) combine_fold(lv[u], ov[u], m, z, acc);
    }
    // merge the lanes that hold the same dims
    for (int off = lps; off < 32; off <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float z2 = __shfl_xor_sync(0xffffffffu, z, off);
        float4 a2;
        a2.x = __shfl_xor_sync(0xffffffffu, acc.x, off);
        a2.y = __shfl_xor_sync(0xffffffffu, acc.y, off);
        a2.z = __shfl_xor_sync(0xffffffffu, acc.z, off);
        a2.w = __shfl_xor_sync(0xffffffffu, acc.w, off);
        const float M = fmaxf(m, m2);
        if (M != -INFINITY) {
            const float a = m == -INFINITY ? 0.f : fast_exp2((m - M) * kLog2e);
            const float b = m2 == -INFINITY ? 0.f : fast_exp2((m2 - M) * kLog2e);
            acc.x = a * acc.x + b * a2.x;
            acc.y = a * acc.y + b * a2.y;
            acc.z = a * acc.z + b * a2.z;
            acc.w = a * acc.w + b * a2.w;
            z = a * z + b * z2;
            m = M;
        }
    }
    if (sub == 0) {
        uint16_t* o = cp.out + static_cast<int64_t>(row) * D + d0;
        if (m == -INFINITY) {
            *reinterpret_cast<uint2*>(o) = make_uint2(0u, 0u);
        } else {
            const float inv = 1.f / z;
            const uint32_t lo = pack2<DT>(acc.x * inv, acc.y * inv);
            const uint32_t hi = pack2<DT>(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2*>(o) = make_uint2(lo, hi);
        }
    }
}

// ------------------------------------------------------------ diagnostics
__global__ void selftest_timeout_kernel(uint32_t* err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t a = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(a, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // Nothing arrives on `bar`: phase 0 never completes.
    if (threadIdx.x == 0 && !mbar_wait(a, 0, limit_ns)) flag_error(err, DA_DEVERR_TIMEOUT);
}

// ------------------------------------------------------------ host side
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

bool make_kv_map(CUtensorMap* map, const void* base, da_dtype dt, da_layout lay, int B, int Hkv,
                 int D, int kv_rows, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3], estr[3] = {1, 1, 1};
    if (lay == DA_LAYOUT_VARLEN) {
        dims[0] = D; dims[1] = Hkv; dims[2] = kv_rows;
        strides[0] = static_cast<cuuint64_t>(D) * 2;
        strides[1] = static_cast<cuuint64_t>(Hkv) * D * 2;
        box[0] = 64; box[1] = 1; box[2] = box_rows;
    } else {
        dims[0] = D; dims[1] = kv_rows; dims[2] = static_cast<cuuint64_t>(B) * Hkv;
        strides[0] = static_cast<cuuint64_t>(D) * 2;
        strides[1] = static_cast<cuuint64_t>(kv_rows) * D * 2;
        box[0] = 64; box[1] = box_rows; box[2] = 1;
    }
    CUresult r = fn(map, dt == DA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Per-kernel, per-device launch facts: the dynamic shared-memory limit is
// raised once per device and the persistent grid size is cached.
struct DeviceCache {
    std::atomic<uint64_t> attr_done{0};
    std::atomic<int> grid[64] = {};
};

template <class K>
cudaError_t persistent_grid(K kernel, int threads, int smem, DeviceCache& cache, int* grid) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << dev;
    if (!(cache.attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        cache.grid[dev].store(sms * per_sm, std::memory_order_relaxed);
        cache.attr_done.fetch_or(bit, std::memory_order_acq_rel);
    }
    *grid = cache.grid[dev].load(std::memory_order_relaxed);
    return cudaSuccess;
}

da_status check_common(const void* q, const void* k, const void* v, const int32_t* cu, int B, int Hq,
                       int Hkv, int D, int kv_rows, int dt, int lay, float scale, int S,
                       const void* ws, size_t ws_bytes) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || kv_rows < 0) return DA_ERR_INVALID_ARG;
    if (S < 1 || S > DA_MAX_SPLITS) return DA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return DA_ERR_INVALID_ARG;
    if (dt != DA_F16 && dt != DA_BF16) return DA_ERR_INVALID_ARG;
    if (lay != DA_LAYOUT_VARLEN && lay != DA_LAYOUT_BHSD) return DA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return DA_ERR_UNSUPPORTED;
    if (!q || !cu || !ws) return DA_ERR_INVALID_ARG;
    if (kv_rows > 0 && (!k || !v)) return DA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(cu, 4) || !aligned(ws, 256)) return DA_ERR_ALIGNMENT;
    if (kv_rows > 0 && (!aligned(k, 16) || !aligned(v, 16))) return DA_ERR_ALIGNMENT;
    const size_t need = decode_attn_splitkv_workspace_size(B, Hq, D, S);
    if (need == 0) return DA_ERR_INVALID_ARG;
    if (ws_bytes < need) return DA_ERR_WORKSPACE_TOO_SMALL;
    const int64_t chunks = item_chunks(Hq / Hkv);
    if (static_cast<int64_t>(B) * Hkv * chunks * S > 0x7fffffffll) return DA_ERR_INVALID_ARG;
    return DA_OK;
}

cudaLaunchAttribute pdl_attr() {
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

// One decode call's arguments, after the host checks.
struct Call {
    const void *q, *k, *v;
    const int32_t* cu;
    int B, Hq, Hkv, D, kv_rows;
    da_dtype dt;
    da_layout lay;
    float scale;
    int S;           // splits per sequence, or the cap of S_b in per-sequence mode
    int split_len;   // 0: S splits for every sequence; else per-sequence S_b
    int tq;          // query tokens per sequence
    int math;        // 0: mma.sync products; 1: CUDA-core FMAs; 2: tcgen05 with tensor memory (comparison arms)
    void* ws;
};

constexpr int kMaxVarsplitBatch = 1024;                                   // sequences, per-sequence mode
constexpr double kLongStreamBytes = 1.5e9;   // K/V bytes above which even batches are split for balance

// `out` is written by the split kernel itself only with one uniform split.
template <int D, int DT, int NT, int MATH>
da_status launch_split(const Call& c, void* out, cudaStream_t stream) {
    // 64-key boxes for full stages, 16-key boxes for the ragged end of a split
    alignas(64) CUtensorMap mk, mv, mk16, mv16;
    std::memset(&mk, 0, sizeof(mk));
    std::memset(&mv, 0, sizeof(mv));
    std::memset(&mk16, 0, sizeof(mk16));
    std::memset(&mv16, 0, sizeof(mv16));
    if (c.kv_rows > 0) {
        const da_dtype dt = static_cast<da_dtype>(DT);
        if (!make_kv_map(&mk, c.k, dt, c.lay, c.B, c.Hkv, D, c.kv_rows, kStageKeys) ||
            !make_kv_map(&mv, c.v, dt, c.lay, c.B, c.Hkv, D, c.kv_rows, kStageKeys) ||
            !make_kv_map(&mk16, c.k, dt, c.lay, c.B, c.Hkv, D, c.kv_rows, kBoxKeys) ||
            !make_kv_map(&mv16, c.v, dt, c.lay, c.B, c.Hkv, D, c.kv_rows, kBoxKeys))
            return DA_ERR_CUDA;
    }
    SplitParams p;
    uint8_t* wsb = static_cast<uint8_t*>(c.ws);
    p.q = static_cast<const uint16_t*>(c.q);
    p.cu = c.cu;
    p.err = reinterpret_cast<uint32_t*>(wsb);
    p.work = reinterpret_cast<uint32_t*>(wsb + kWorkCounterOff);
    p.done = reinterpret_cast<uint32_t*>(wsb + kDoneCounterOff);
    p.out = (c.S == 1 && c.split_len == 0) ? static_cast<uint16_t*>(out) : nullptr;
    p.lse = reinterpret_cast<float*>(wsb + decode_attn_splitkv_lse_offset());
    p.opart = reinterpret_cast<float*>(wsb + decode_attn_splitkv_opart_offset(c.B * c.tq, c.Hq, c.S));
    p.B = c.B;
    p.Hq = c.Hq;
    p.Hkv = c.Hkv;
    p.G = c.Hq / c.Hkv;
    p.S = c.S;
    p.kv_rows = c.kv_rows;
    p.layout = c.lay;
    p.tq = c.tq;
    p.chunks = (p.G * c.tq + NT * kHeadsPerCta - 1) / (NT * kHeadsPerCta);
    p.no_kv = c.kv_rows == 0;
    p.n_items = c.B * c.Hkv * p.chunks * c.S;   // per-sequence mode: an upper bound (the kernel counts)
    p.split_len = c.split_len;
    p.stage_cu = c.B <= kMaxStagedBatch;
    p.scale_log2 = c.scale * kLog2e;
    p.wait_limit_ns = kWaitLimitNs;

    const bool var = c.split_len != 0;
    const int smem = Shape<D, NT>::kSmemBytes + (p.stage_cu ? kStagedBytes : 0) + (var ? kStagedBytes : 0) +
                     (MATH == 1 ? kConsumerWarps * 17 * 8 * 4 : 0);
    auto kern = split_kernel<D, DT, NT, MATH>;
    static DeviceCache caches[3];   // by the number of staged [B + 1] arrays
    int grid = 0;
    if (persistent_grid(kern, kThreads, smem, caches[(p.stage_cu ? 1 : 0) + (var ? 1 : 0)], &grid) != cudaSuccess)
        return DA_ERR_CUDA;
    grid = std::min(grid, p.n_items);
    cudaLaunchAttribute attrs[1] = {pdl_attr()};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, mk, mv, mk16, mv16, p) == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

// Q viewed as [B * tq][Hq][D]: one box holds `tokens` query tokens x the G heads
// of one KV head x 64 dims, i.e. the packed columns of one tensor-memory item.
bool make_q_map(CUtensorMap* map, const void* q, da_dtype dt, int rows, int Hq, int D, int G, int tokens) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hq) * D * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(tokens)}, estr[3] = {1, 1, 1};
    CUresult r = fn(map, dt == DA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    3, const_cast<void*>(q), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Items of more than 8 columns with G <= 32 on the tensor-memory split kernel (the
// tcgen05 comparison arm): one CTA per SM, up to 32 columns (whole query tokens of
// one KV head's group) per item.
template <int D, int DT>
da_status launch_split_tc(const Call& c, void* out, cudaStream_t stream) {
    alignas(64) CUtensorMap mk, mv, mk16, mv16, mq;
    std::memset(&mk, 0, sizeof(mk));
    std::memset(&mv, 0, sizeof(mv));
    std::memset(&mk16, 0, sizeof(mk16));
    std::memset(&mv16, 0, sizeof(mv16));
    std::memset(&mq, 0, sizeof(mq));
    const da_dtype dt = static_cast<da_dtype>(DT);
    const int G = c.Hq / c.Hkv;
    const int tokens = std::min(c.tq, kTcCols / G);
    if (c.kv_rows > 0) {
        if (!make_kv_map(&mk, c.k, dt, c.lay, c.B, c.Hkv, D, c.kv_rows, kStageKeys) ||
            !make_kv_map(&mv, c.v, dt, c.lay, c.B, c.Hkv, D, c.kv_rows, kStageKeys) ||
            !make_kv_map(&mk16, c.k, dt, c.lay, c.B, c.Hkv, D, c.kv_rows, kBoxKeys) ||
            !make_kv_map(&mv16, c.v, dt, c.lay, c.B, c.Hkv, D, c.kv_rows, kBoxKeys))
            return DA_ERR_CUDA;
    }
    if (!make_q_map(&mq, c.q, dt, c.B * c.tq, c.Hq, D, G, tokens)) return DA_ERR_CUDA;
    TcParams tp;
    SplitParams& p = tp.sp;
    uint8_t* wsb = static_cast<uint8_t*>(c.ws);
    p.q = static_cast<const uint16_t*>(c.q);
    p.cu = c.cu;
    p.err = reinterpret_cast<uint32_t*>(wsb);
    p.work = reinterpret_cast<uint32_t*>(wsb + kWorkCounterOff);
    p.done = reinterpret_cast<uint32_t*>(wsb + kDoneCounterOff);
    p.out = (c.S == 1 && c.split_len == 0) ? static_cast<uint16_t*>(out) : nullptr;
    p.lse = reinterpret_cast<float*>(wsb + decode_attn_splitkv_lse_offset());
    p.opart = reinterpret_cast<float*>(wsb + decode_attn_splitkv_opart_offset(c.B * c.tq, c.Hq, c.S));
    p.B = c.B;
    p.Hq = c.Hq;
    p.Hkv = c.Hkv;
    p.G = G;
    p.S = c.S;
    p.kv_rows = c.kv_rows;
    p.layout = c.lay;
    p.tq = c.tq;
    tp.item_tokens = tokens;
    tp.item_cols = G * tokens;
    p.chunks = (c.tq + tokens - 1) / tokens;
    p.no_kv = c.kv_rows == 0;
    p.n_items = c.B * c.Hkv * p.chunks * c.S;   // per-sequence mode: an upper bound (the kernel counts)
    p.split_len = c.split_len;
    p.stage_cu = c.B <= kMaxStagedBatch;
    p.scale_log2 = c.scale * kLog2e;
    p.wait_limit_ns = kWaitLimitNs;

    const bool var = c.split_len != 0;
    const int smem = TcShape<D>::kSmemBytes + (p.stage_cu ? kStagedBytes : 0) + (var ? kStagedBytes : 0);
    auto kern = split_kernel_tc<D, DT>;
    static DeviceCache caches[3];
    int grid = 0;
    if (persistent_grid(kern, kTcThreads, smem, caches[(p.stage_cu ? 1 : 0) + (var ? 1 : 0)], &grid) !=
        cudaSuccess)
        return DA_ERR_CUDA;
    grid = std::min(grid, p.n_items);
    cudaLaunchAttribute attrs[1] = {pdl_attr()};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, mk, mv, mk16, mv16, mq, tp) == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

// dims per combine warp: enough warps to cover the GPU, at least 8 dims each
int combine_dchunks(int rows, int D, int S) {
    int dchunks = 1;
    while (D / dchunks > 8 && static_cast<int64_t>(rows) * dchunks < 2048 && S > 4 * dchunks) dchunks *= 2;
    return dchunks;
}

template <int D, int DT>
da_status launch_combine(const Call& c, void* out, cudaStream_t stream) {
    CombineParams cp;
    const uint8_t* wsb = static_cast<const uint8_t*>(c.ws);
    cp.lse = reinterpret_cast<const float*>(wsb + decode_attn_splitkv_lse_offset());
    cp.opart = reinterpret_cast<const float*>(wsb + decode_attn_splitkv_opart_offset(c.B * c.tq, c.Hq, c.S));
    cp.out = static_cast<uint16_t*>(out);
    cp.cu = c.cu;
    cp.rows = c.B * c.tq * c.Hq;
    cp.S = c.S;
    cp.dchunks = combine_dchunks(cp.rows, D, c.S);
    cp.Hq = c.Hq * c.tq;   // rows per sequence
    cp.split_len = c.split_len;
    cp.layout = c.lay;
    cp.kv_rows = c.kv_rows;
    cp.no_kv = c.kv_rows == 0;
    const int64_t warps = static_cast<int64_t>(cp.rows) * cp.dchunks;
    cudaLaunchAttribute attrs[1] = {pdl_attr()};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((warps + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel<D, DT>, cp) == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

template <int D, int DT>
da_status launch_split_cols(const Call& c, void* out, cudaStream_t st) {
    const bool wide = item_cols(static_cast<int64_t>(c.Hq / c.Hkv) * c.tq) > kHeadsPerCta;
    if (c.math == 1) return wide ? DA_ERR_UNSUPPORTED : launch_split<D, DT, 1, 1>(c, out, st);
    if (c.math == 2) return wide && c.Hq / c.Hkv <= kTcCols ? launch_split_tc<D, DT>(c, out, st) : DA_ERR_UNSUPPORTED;
    if (wide) return launch_split<D, DT, 2, 0>(c, out, st);
    return launch_split<D, DT, 1, 0>(c, out, st);
}

da_status dispatch_split(const Call& c, void* out, cudaStream_t st) {
    if (c.D == 128)
        return c.dt == DA_F16 ? launch_split_cols<128, DA_F16>(c, out, st) : launch_split_cols<128, DA_BF16>(c, out, st);
    return c.dt == DA_F16 ? launch_split_cols<64, DA_F16>(c, out, st) : launch_split_cols<64, DA_BF16>(c, out, st);
}

da_status dispatch_combine(const Call& c, void* out, cudaStream_t st) {
    if (c.D == 128)
        return c.dt == DA_F16 ? launch_combine<128, DA_F16>(c, out, st) : launch_combine<128, DA_BF16>(c, out, st);
    return c.dt == DA_F16 ? launch_combine<64, DA_F16>(c, out, st) : launch_combine<64, DA_BF16>(c, out, st);
}

// Split step, then the combine step unless a single uniform split already wrote `out`.
da_status run_decode(const Call& c, void* out, cudaStream_t st) {
    da_status r = dispatch_split(c, out, st);
    if (r != DA_OK || (c.S == 1 && c.split_len == 0)) return r;
    return dispatch_combine(c, out, st);
}

Call make_call(const void* q, const void* k, const void* v, const int32_t* cu, int B, int Hq, int Hkv, int D,
               int kv_rows, da_dtype dt, da_layout lay, float scale, int S, int split_len, void* ws, int tq = 1) {
    Call c;
    c.tq = tq;
    c.math = 0;
    c.q = q;
    c.k = k;
    c.v = v;
    c.cu = cu;
    c.B = B;
    c.Hq = Hq;
    c.Hkv = Hkv;
    c.D = D;
    c.kv_rows = kv_rows;
    c.dt = dt;
    c.lay = lay;
    c.scale = scale;
    c.S = S;
    c.split_len = split_len;
    c.ws = ws;
    return c;
}

}  // namespace

// ================================================================ C ABI
extern "C" {

size_t decode_attn_splitkv_lse_offset(void) { return kHeaderBytes; }

size_t decode_attn_splitkv_opart_offset(int B, int Hq, int num_splits) {
    return kHeaderBytes + round_up(static_cast<size_t>(B) * Hq * num_splits * 4, 256);
}

size_t decode_attn_splitkv_workspace_size(int B, int Hq, int D, int num_splits) {
    if (B < 1 || Hq < 1 || D < 1 || num_splits < 1 || num_splits > DA_MAX_SPLITS) return 0;
    return decode_attn_splitkv_opart_offset(B, Hq, num_splits) +
           static_cast<size_t>(B) * Hq * num_splits * D * 4;
}

da_status decode_attn_splitkv_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace || workspace_bytes < kHeaderBytes) return DA_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return DA_ERR_ALIGNMENT;
    return cudaMemsetAsync(workspace, 0, kHeaderBytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DA_OK
               : DA_ERR_CUDA;
}

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
    if (sm_count <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sm_count <= 0)
            sm_count = 148;
    }
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
        const int64_t per_sm = wide ? 4 : 8;
        const double shares = wide ? 4.0 : 2.0;
        S = (per_sm * static_cast<int64_t>(sm_count) + units - 1) / units;
        S = std::min<int64_t>(S, std::max<int64_t>(1, min_kv / 64));
        // ... and the longest sequence's splits at most about twice (wide items:
        // four times) one CTA's share of the keys (the share taken from a lower
        // bound of the total), so that no single split outlasts the rest of the batch.
        const double total = static_cast<double>(max_kv) + static_cast<double>(B - 1) * min_kv;
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

da_status decode_attn_splitkv_partial(const void* q, const void* k, const void* v,
                                      const int32_t* cu_seqlens_k, int B, int Hq, int Hkv, int D,
                                      int kv_rows, da_dtype dtype, da_layout layout, float scale,
                                      int num_splits, void* workspace, size_t workspace_bytes,
                                      void* stream) {
    da_status st = check_common(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale,
                                num_splits, workspace, workspace_bytes);
    if (st != DA_OK) return st;
    return dispatch_split(make_call(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale,
                                    num_splits, 0, workspace),
                          nullptr, static_cast<cudaStream_t>(stream));
}

da_status decode_attn_splitkv_partial_cuda_core(const void* q, const void* k, const void* v,
                                                const int32_t* cu_seqlens_k, int B, int Hq, int Hkv, int D,
                                                int kv_rows, da_dtype dtype, da_layout layout, float scale,
                                                int num_splits, void* workspace, size_t workspace_bytes,
                                                void* stream) {
    da_status st = check_common(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale,
                                num_splits, workspace, workspace_bytes);
    if (st != DA_OK) return st;
    if (Hq / Hkv > kHeadsPerCta) return DA_ERR_UNSUPPORTED;
    Call c = make_call(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale, num_splits, 0,
                       workspace);
    c.math = 1;
    return dispatch_split(c, nullptr, static_cast<cudaStream_t>(stream));
}

da_status decode_attn_splitkv_combine(int B, int Hq, int D, int num_splits, da_dtype dtype, void* out,
                                      const void* workspace, size_t workspace_bytes, void* stream) {
    if (B < 1 || Hq < 1 || num_splits < 1 || num_splits > DA_MAX_SPLITS) return DA_ERR_INVALID_ARG;
    if (dtype != DA_F16 && dtype != DA_BF16) return DA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return DA_ERR_UNSUPPORTED;
    if (!out || !workspace) return DA_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(workspace, 256)) return DA_ERR_ALIGNMENT;
    if (workspace_bytes < decode_attn_splitkv_workspace_size(B, Hq, D, num_splits))
        return DA_ERR_WORKSPACE_TOO_SMALL;
    if (static_cast<int64_t>(B) * Hq * D > 0x7fffffffll) return DA_ERR_INVALID_ARG;
    return dispatch_combine(make_call(nullptr, nullptr, nullptr, nullptr, B, Hq, 1, D, 0, dtype,
                                      DA_LAYOUT_VARLEN, 1.f, num_splits, 0, const_cast<void*>(workspace)),
                            out, static_cast<cudaStream_t>(stream));
}

da_status decode_attn_splitkv(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_k,
                              int B, int Hq, int Hkv, int D, int kv_rows, da_dtype dtype,
                              da_layout layout, float scale, int num_splits, void* out,
                              void* workspace, size_t workspace_bytes, void* stream) {
    da_status st = check_common(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale,
                                num_splits, workspace, workspace_bytes);
    if (st != DA_OK) return st;
    if (!out) return DA_ERR_INVALID_ARG;
    if (!aligned(out, 16)) return DA_ERR_ALIGNMENT;
    if (static_cast<int64_t>(B) * Hq * D > 0x7fffffffll) return DA_ERR_INVALID_ARG;
    return run_decode(make_call(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale, num_splits, 0,
                                workspace),
                      out, static_cast<cudaStream_t>(stream));
}

int decode_attn_splitkv_varsplit_plan(int B, int Hq, int Hkv, int D, int64_t total_kv, int max_kv,
                                      int sm_count, int* split_len, int* max_splits) {
    if (!split_len || !max_splits) return -1;
    *split_len = 1;
    *max_splits = 1;
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || (D != 64 && D != 128) || total_kv < 0 || max_kv < 0)
        return -1;
    if (sm_count <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sm_count <= 0)
            sm_count = 148;
    }
    const int64_t chunks = item_chunks(Hq / Hkv);
    const int64_t key_units = total_kv * Hkv * chunks;      // keys to stream, summed over (KV head, chunk)
    const int64_t target = 8 * static_cast<int64_t>(sm_count);   // about four items per resident CTA
    int64_t len = (key_units + target - 1) / std::max<int64_t>(1, target);
    len = std::max<int64_t>(256, (len + kStageKeys - 1) / kStageKeys * kStageKeys);   // whole stages
    int64_t ms = max_kv > 0 ? (max_kv + len - 1) / len : 1;
    ms = std::max<int64_t>(1, std::min<int64_t>(ms, DA_MAX_SPLITS));
    *split_len = static_cast<int>(std::min<int64_t>(len, 1 << 30));
    *max_splits = static_cast<int>(ms);
    return 0;
}

da_status decode_attn_splitkv_varsplit(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_k,
                                       int B, int Hq, int Hkv, int D, int kv_rows, da_dtype dtype,
                                       da_layout layout, float scale, int split_len, int max_splits, void* out,
                                       void* workspace, size_t workspace_bytes, void* stream) {
    if (split_len < 1) return DA_ERR_INVALID_ARG;
    if (B > kMaxVarsplitBatch) return DA_ERR_UNSUPPORTED;
    da_status st = check_common(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale, max_splits,
                                workspace, workspace_bytes);
    if (st != DA_OK) return st;
    if (!out) return DA_ERR_INVALID_ARG;
    if (!aligned(out, 16)) return DA_ERR_ALIGNMENT;
    if (static_cast<int64_t>(B) * Hq * D > 0x7fffffffll) return DA_ERR_INVALID_ARG;
    return run_decode(make_call(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale, max_splits,
                                split_len, workspace),
                      out, static_cast<cudaStream_t>(stream));
}

da_status decode_attn_splitkv_multiquery(const void* q, const void* k, const void* v,
                                         const int32_t* cu_seqlens_k, int B, int T_q, int Hq, int Hkv,
                                         int D, int kv_rows, da_dtype dtype, da_layout layout, float scale,
                                         int num_splits, void* out, void* workspace, size_t workspace_bytes,
                                         void* stream) {
    if (T_q < 1 || T_q > DA_MAX_QUERY_TOKENS) return DA_ERR_INVALID_ARG;
    if (B < 1 || static_cast<int64_t>(B) * T_q > 0x7fffffffll) return DA_ERR_INVALID_ARG;
    // the workspace holds B * T_q rows of Hq heads
    const size_t need = decode_attn_splitkv_workspace_size(B * T_q, Hq, D, num_splits);
    da_status st = check_common(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale, num_splits,
                                workspace, need == 0 ? workspace_bytes : std::max(workspace_bytes, need));
    if (st != DA_OK) return st;
    if (workspace_bytes < need) return DA_ERR_WORKSPACE_TOO_SMALL;
    if (!out) return DA_ERR_INVALID_ARG;
    if (!aligned(out, 16)) return DA_ERR_ALIGNMENT;
    const int64_t chunks = item_chunks(static_cast<int64_t>(Hq / Hkv) * T_q);
    if (static_cast<int64_t>(B) * Hkv * chunks * num_splits > 0x7fffffffll) return DA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(B) * T_q * Hq * D > 0x7fffffffll) return DA_ERR_INVALID_ARG;
    return run_decode(make_call(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale, num_splits, 0,
                                workspace, T_q),
                      out, static_cast<cudaStream_t>(stream));
}

da_status decode_attn_splitkv_multiquery_tmem(const void* q, const void* k, const void* v,
                                              const int32_t* cu_seqlens_k, int B, int T_q, int Hq, int Hkv,
                                              int D, int kv_rows, da_dtype dtype, da_layout layout, float scale,
                                              int num_splits, void* out, void* workspace, size_t workspace_bytes,
                                              void* stream) {
    if (T_q < 1 || T_q > DA_MAX_QUERY_TOKENS) return DA_ERR_INVALID_ARG;
    if (B < 1 || static_cast<int64_t>(B) * T_q > 0x7fffffffll) return DA_ERR_INVALID_ARG;
    const size_t need = decode_attn_splitkv_workspace_size(B * T_q, Hq, D, num_splits);
    da_status st = check_common(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale, num_splits,
                                workspace, need == 0 ? workspace_bytes : std::max(workspace_bytes, need));
    if (st != DA_OK) return st;
    if (workspace_bytes < need) return DA_ERR_WORKSPACE_TOO_SMALL;
    if (!out) return DA_ERR_INVALID_ARG;
    if (!aligned(out, 16)) return DA_ERR_ALIGNMENT;
    const int G = Hq / Hkv;
    if (static_cast<int64_t>(G) * T_q <= kHeadsPerCta || G > kTcCols) return DA_ERR_UNSUPPORTED;
    const int64_t chunks = (T_q + kTcCols / G - 1) / (kTcCols / G);
    if (static_cast<int64_t>(B) * Hkv * chunks * num_splits > 0x7fffffffll) return DA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(B) * T_q * Hq * D > 0x7fffffffll) return DA_ERR_INVALID_ARG;
    Call c = make_call(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale, num_splits, 0, workspace,
                       T_q);
    c.math = 2;
    return run_decode(c, out, static_cast<cudaStream_t>(stream));
}

da_status decode_attn_splitkv_get_error(void* workspace, uint32_t* device_error_bits, void* stream) {
    if (!workspace || !device_error_bits) return DA_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return DA_ERR_ALIGNMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t bits = 0;
    if (cudaMemcpyAsync(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return DA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DA_ERR_CUDA;
    *device_error_bits = bits;
    if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return DA_ERR_CUDA;
    return DA_OK;
}

da_status decode_attn_splitkv_selftest_timeout(void* workspace, size_t workspace_bytes,
                                               unsigned timeout_us, void* stream) {
    if (!workspace || workspace_bytes < kHeaderBytes || timeout_us == 0 || timeout_us > 10000000u)
        return DA_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return DA_ERR_ALIGNMENT;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(32);
    cfg.stream = static_cast<cudaStream_t>(stream);
    return cudaLaunchKernelEx(&cfg, selftest_timeout_kernel, static_cast<uint32_t*>(workspace),
                              static_cast<unsigned long long>(timeout_us) * 1000ull) == cudaSuccess
               ? DA_OK
               : DA_ERR_CUDA;
}

const char* decode_attn_splitkv_status_string(da_status status) {
    switch (status) {
        case DA_OK: return "DA_OK";
        case DA_ERR_INVALID_ARG: return "DA_ERR_INVALID_ARG: an argument is out of range or NULL";
        case DA_ERR_UNSUPPORTED: return "DA_ERR_UNSUPPORTED: head_dim must be 64 or 128";
        case DA_ERR_ALIGNMENT: return "DA_ERR_ALIGNMENT: a pointer is not aligned as documented";
        case DA_ERR_WORKSPACE_TOO_SMALL: return "DA_ERR_WORKSPACE_TOO_SMALL";
        case DA_ERR_CUDA: return "DA_ERR_CUDA: a CUDA runtime or driver call failed";
        case DA_ERR_SCRATCH_LIMIT:
            return "DA_ERR_SCRATCH_LIMIT: the problem needs more scratch than the library's "
                   "8 MiB built-in array (use decode_attn_splitkv with a workspace)";
    }
    return "unknown da_status";
}

// ---------------------------------------------------------------- time model
// A GB300 restatement of the lecture page's decode time model
// (04_flash_decoding.py: decode_attention_time / best_splits, whose A100/H100
// constants are not on the page): the call is modelled as
//   T = t0 + makespan + kappa * (largest item's bytes) / (bw / min(items, CTAs))
//         + [S > 1] (t_comb + W_ws / bw_comb)
// where makespan is a processor-sharing run of the work items, in queue order,
// over the persistent CTAs: each CTA spends t_item before an item and then
// streams its bytes (each split's key count rounded up to the 16-key TMA box)
// at min(r_cta, bw / streaming CTAs), r_cta being one CTA's rate for 8-column
// items and r_cta2 for 16-column ones; kappa charges the last item for the
// CTAs' unequal rates, and W_ws is the workspace bytes the combine reads.
// Fitted (least squares in log time) on one GB300 to the 310 calls, of 546
// measured (17 single-token workloads of the CodeLlama, Llama, Qwen and MHA
// shapes and 9 of them with 2 or 4 new tokens x split counts 1 to 256, L2
// flushed, CUDA-event median per call), that lie within 30 % of their
// workload's fastest split count: median error 2.9 %, 90th percentile 10.8 %.
static const double kModelGb300[8] = {
    /* t0 us       */ 12.24,
    /* t_item us   */ 0.1241,
    /* r_cta B/us  */ 76340,
    /* bw B/us     */ 7.592e+06,
    /* t_comb us   */ 2.462,
    /* bw_comb     */ 8.561e+05,
    /* kappa       */ 0.05135,
    /* r_cta2 B/us */ 52610};

double decode_attn_splitkv_model_us(const int32_t* kv_lens, int B, int Hq, int Hkv, int D, int T_q, int num_splits,
                                    int sm_count, const double* params) {
    if (!kv_lens || B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || (D != 64 && D != 128) || T_q < 1 ||
        num_splits < 1 || num_splits > DA_MAX_SPLITS || sm_count < 1)
        return -1.0;
    const double* m = params ? params : kModelGb300;
    const double t0 = m[0], t_item = m[1], bw = m[3], t_comb = m[4], bw_comb = m[5], kappa = m[6];
    // one CTA's streaming cap: 16-column items carry twice the products per key
    const bool wide = item_cols(static_cast<int64_t>(Hq / Hkv) * T_q) > kHeadsPerCta;
    const double r_cta = wide ? m[7] : m[2];
    if (!(r_cta > 0) || !(bw > 0) || !(bw_comb > 0) || !(t_item >= 0) || !(kappa >= 0)) return -1.0;
    const int S = num_splits;
    const int chunks = static_cast<int>(item_chunks(static_cast<int64_t>(Hq / Hkv) * T_q));
    const int slots = sm_count * (D == 128 ? 2 : 4);
    const double key_bytes = 4.0 * D;   // K and V rows of one key and KV head
    // the work items in queue order: the bytes each streams (later chunks of a
    // split re-read its keys from L2 and are not counted in W)
    std::vector<double> items;
    double W = 0.0, biggest = 0.0;
    for (int b = 0; b < B; ++b) {
        const int64_t L = kv_lens[b] < 0 ? 0 : kv_lens[b];
        for (int kvh = 0; kvh < Hkv; ++kvh)
            for (int s = 0; s < S; ++s) {
                const int64_t n = L * (s + 1) / S - L * s / S;
                const double bytes = static_cast<double>((n + kBoxKeys - 1) / kBoxKeys * kBoxKeys) * key_bytes;
                biggest = std::max(biggest, bytes);
                W += bytes;
                for (int c = 0; c < chunks; ++c) items.push_back(bytes);
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
    if (S > 1) t += t_comb + static_cast<double>(B) * T_q * Hq * S * (D + 1) * 4.0 / bw_comb;
    (void)W;
    return t;
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

// ================================================================ no-allocation variant
// For callers that may not allocate device memory: the workspace is a scratch
// array compiled into this library instead of a caller buffer.
namespace {

__device__ __align__(256) uint8_t g_noalloc_scratch[DA_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[128] = {};   // device address of g_noalloc_scratch, per device ordinal

// In host code g_noalloc_scratch names a host-side shadow, not device memory:
// the device address comes from cudaGetSymbolAddress, looked up once per
// device with that device current.
da_status noalloc_scratch(void** addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return DA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return DA_ERR_CUDA;
        g_noalloc_addr[dev] = p;
    }
    *addr = g_noalloc_addr[dev];
    return DA_OK;
}

}  // namespace

extern "C" da_status decode_attn_splitkv_noalloc(const void* q, const void* k, const void* v,
                                                 const int32_t* cu_seqlens_k, int B, int Hq, int Hkv,
                                                 int D, int kv_rows, da_dtype dtype, da_layout layout,
                                                 float scale, int num_splits, void* out, void* stream) {
    const size_t need = decode_attn_splitkv_workspace_size(B, Hq, D, num_splits);
    if (need > DA_NOALLOC_SCRATCH_BYTES) return DA_ERR_SCRATCH_LIMIT;
    void* ws = nullptr;
    if (need > 0) {
        // only sizes that pass the workspace arithmetic reach the device lookup
        da_status st = noalloc_scratch(&ws);
        if (st != DA_OK) return st;
    }
    da_status st = check_common(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale,
                                num_splits, ws, DA_NOALLOC_SCRATCH_BYTES);
    if (st != DA_OK) return st;
    if (!out) return DA_ERR_INVALID_ARG;
    if (!aligned(out, 16)) return DA_ERR_ALIGNMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, kHeaderBytes, s) != cudaSuccess) return DA_ERR_CUDA;
    return run_decode(make_call(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale, num_splits, 0,
                                ws),
                      out, s);
}
