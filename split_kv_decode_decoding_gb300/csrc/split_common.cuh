// Pieces of the split step shared by the library's split kernel
// (decode_attn_splitkv.cu) and the comparison arms (comparison_arms.cu):
// work-item decoding, PTX wrappers, the producer warp that feeds the K/V ring,
// the write-out of a merged item, and the host-side helpers (tensor maps,
// argument checks, launch facts). Included by exactly those two translation
// units; it defines no kernel.
#ifndef DECODE_ATTN_SPLITKV_SPLIT_COMMON_CUH
#define DECODE_ATTN_SPLITKV_SPLIT_COMMON_CUH

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "decode_attn_splitkv.h"
#include "geometry.h"

namespace da_impl {

constexpr int kConsumerWarps = 4;   // each owns 16 keys of a stage
constexpr int kThreads = (kConsumerWarps + 1) * 32;
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
// Uniform splits over a varlen batch of at most kMaxSortedBatch sequences: the work
// queue hands out the sequences longest first, so that the last items to start are
// the short ones. The order (perm[rank] = sequence) lives in the staged
// cu_seqlens_k area, past the B + 1 entries it uses.
constexpr int kLenOff = 384;    // int32 entries into the staged cu_seqlens_k area: lengths [B]
constexpr int kPermOff = 512;   // and the order [B] (the area holds 1025 + 3 entries)
static_assert(kLenOff >= kMaxSortedBatch + 1 && kPermOff >= kLenOff + kMaxSortedBatch &&
                  kPermOff + kMaxSortedBatch <= kStagedBytes / 4,
              "the sorted order fits the staged cu_seqlens_k area past its entries");

struct ItemSlot {          // one work item, as the producer decoded it
    int32_t b, kvh, h0, nh;            // h0: first query head of the KV head's group; nh columns
    int32_t s, nkeys, ntiles, valid;   // valid: 0 end of the queue, 1 an item, 2 the only split of its sequence
    int64_t first_key;                 // varlen: K/V row of the split start; bhsd: position
    int32_t c0;                        // first packed (token, head) column of this item
    int32_t vis0;                      // keys of the split query token 0 may see (may be <= 0)
};
static_assert(sizeof(ItemSlot) == 48, "ItemSlot layout");

template <int D, int NT, int ST = kStages>
struct Shape {
    static constexpr int kStages = ST;                             // ring depth
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
    uint32_t* done;          // CTAs finished (the tcgen05 comparison arm's queue reset)
    uint16_t* out;           // [B, Hq, D]: rows of sequences with one split are written here (nullptr: none)
    int B, Hq, Hkv, G, S, kv_rows, layout, chunks, no_kv, n_items;
    int split_len;           // 0: every sequence has S splits; else S_b = min(S, ceil(L_b / split_len))
    int stage_cu;            // cu_seqlens_k staged in shared memory (B small enough)
    int sorted;              // the producer hands out sequences longest first (see kMaxSortedBatch)
    int keep_partials;       // store the partials that the combine reads back with an L2 evict-last
                             // hint (the K/V stream is larger than the L2 and would evict them)
    int prefix_off;          // per-sequence mode: prefix[] at this int32 offset in the staged
                             // cu_seqlens_k area, or -1: in an area of its own past it
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
// Whether the work queue hands out sequences longest first (see kMaxSortedBatch):
// set by the host for launches whose producer builds the order.
__device__ __forceinline__ bool longest_first(const SplitParams& p, const int32_t* cus) {
    return p.sorted != 0 && cus != nullptr;
}

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
        if (longest_first(p, cus)) it.b = cus[kPermOff + it.b];
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
    // the only split of its sequence: its weight in the combine is exactly 1, so the
    // split step writes the output row itself
    it.valid = Sb == 1 ? 2 : 1;
    return it;
}

template <int kCols>
__device__ __forceinline__ ItemSlot decode_item(const SplitParams& p, int idx, const int32_t* cus,
                                                const int32_t* prefix) {
    return decode_item_cols(p, idx, cus, prefix, kCols);
}

// Workspace/output row of packed column c of an item: token t = c / G, head
// h = h0 + c % G, row = (b * tq + t) * Hq + h.
__device__ __forceinline__ int64_t column_row(const SplitParams& p, const ItemSlot& it, int c) {
    const int cg = it.c0 + c;
    if (p.tq == 1) return static_cast<int64_t>(it.b) * p.Hq + it.h0 + cg;   // token 0: cg < G
    return (static_cast<int64_t>(it.b) * p.tq + cg / p.G) * p.Hq + it.h0 + cg % p.G;
}

// ------------------------------------------------------------ split-kernel skeleton
// Shared-memory layout of one split-kernel CTA (Shape<D, NT> plus the staged
// per-sequence arrays past its end).
struct SplitLayout {
    uint8_t* smem;          // 1024-byte aligned base: the K/V ring
    ItemSlot* slots;        // [kItemSlots] item descriptors
    uint32_t ring, qbuf;    // shared addresses of the ring and the Q rows [kItemSlots][columns][D]
    uint32_t full0, empty0; // [stages] stage landed / stage released
    uint32_t ifull0, iempty0;   // [kItemSlots] descriptor published / slot released
    uint32_t mfull, mdone;  // an item's per-warp partials written; (two n-tiles) a merge round read
    int32_t* cus;           // cu_seqlens_k [B + 1] staged in shared memory, or nullptr
    int32_t* prefix;        // per-sequence mode: running sum of S_b [B + 1]
    uint8_t* extra;         // past the staged arrays (free for the kernel's own use)
};

template <int D, int NT, int ST>
__device__ __forceinline__ SplitLayout split_layout(uint8_t* smem_raw, const SplitParams& p) {
    using Sh = Shape<D, NT, ST>;
    SplitLayout s;
    s.smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    s.slots = reinterpret_cast<ItemSlot*>(s.smem + Sh::kSlotOff);
    s.ring = smem_addr(s.smem);
    s.qbuf = s.ring + Sh::kQOff;
    s.full0 = s.ring + Sh::kBarOff;
    s.empty0 = s.full0 + 8 * ST;
    s.ifull0 = s.empty0 + 8 * ST;
    s.iempty0 = s.ifull0 + 8 * kItemSlots;
    s.mfull = s.iempty0 + 8 * kItemSlots;
    s.mdone = s.mfull + 8;
    s.cus = p.stage_cu ? reinterpret_cast<int32_t*>(s.smem + Sh::kEnd) : nullptr;
    const bool own_prefix = p.split_len != 0 && p.prefix_off < 0;
    s.prefix = p.prefix_off >= 0 && s.cus != nullptr
                   ? s.cus + p.prefix_off
                   : reinterpret_cast<int32_t*>(s.smem + Sh::kEnd + (p.stage_cu ? kStagedBytes : 0));
    s.extra = s.smem + Sh::kEnd + (p.stage_cu ? kStagedBytes : 0) + (own_prefix ? kStagedBytes : 0);
    return s;
}

// Barrier set-up and tensor-map prefetch; everything before the grid-dependency
// wait overlaps the previous kernel in the stream.
template <int D, int NT, int ST>
__device__ __forceinline__ void split_setup(const SplitLayout& sl, const SplitParams& p, const CUtensorMap* tmK,
                                            const CUtensorMap* tmV, const CUtensorMap* tmK16,
                                            const CUtensorMap* tmV16) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(sl.full0 + 8 * i, 1);
            mbar_init(sl.empty0 + 8 * i, kConsumerWarps);
        }
        for (int i = 0; i < kItemSlots; ++i) {
            mbar_init(sl.ifull0 + 8 * i, 1);
            mbar_init(sl.iempty0 + 8 * i, kConsumerWarps);
        }
        mbar_init(sl.mfull, kConsumerWarps);
        if constexpr (NT > 1) mbar_init(sl.mdone, kConsumerWarps);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kConsumerWarps && lane == 0 && p.no_kv == 0) {
        prefetch_tensormap(tmK);
        prefetch_tensormap(tmV);
        prefetch_tensormap(tmK16);
        prefetch_tensormap(tmV16);
    }
    __syncthreads();
    // From here on this grid touches global memory: wait for the previous kernel.
    grid_dependency_wait();
    if (threadIdx.x == 0) grid_dependents_launch();
    if (warp == kConsumerWarps && lane == 0 && p.layout == DA_LAYOUT_BHSD && p.no_kv == 0 && p.split_len == 0 &&
        static_cast<int>(blockIdx.x) < p.n_items) {
        // This CTA's first item is its own index. When that is a sequence's first
        // split, its keys start at position 0 of its slab whatever the length:
        // start pulling its first stages into L2 while cu_seqlens_k is read.
        const int r = static_cast<int>(blockIdx.x) / p.chunks;   // (b * Hkv + kvh) * S + s
        if (r % p.S == 0) {
            const int slab = r / p.S;
            for (int t = 0; t < kPrefetchStages; ++t)
                for (int hf = 0; hf < D / 64; ++hf) {
                    tma_prefetch_3d(tmK, hf * 64, t * kStageKeys, slab);
                    tma_prefetch_3d(tmV, hf * 64, t * kStageKeys, slab);
                }
        }
    }
    if (sl.cus != nullptr) {
        // one coalesced read of cu_seqlens_k per CTA; every item is then decoded from shared memory
        for (int i = threadIdx.x; i <= p.B; i += kThreads) sl.cus[i] = ld_cg_s32(p.cu + i);
        __syncthreads();
        if (longest_first(p, sl.cus)) {
            // the order in which the work queue hands out sequences, longest first (ties
            // by index): thread t ranks sequence t; an even batch keeps the index order
            const int t = threadIdx.x;
            int32_t* len = sl.cus + kLenOff;
            const int Lt = t < p.B ? sl.cus[t + 1] - sl.cus[t] : 0;
            if (t < p.B) len[t] = Lt;
            const bool uneven = __syncthreads_or(t < p.B && Lt != sl.cus[1] - sl.cus[0]);
            if (t < p.B) {
                int rank = t;
                if (uneven) {
                    rank = 0;
#pragma unroll 8
                    for (int b2 = 0; b2 < p.B; ++b2) {
                        const int l2 = len[b2];
                        rank += (l2 > Lt) || (l2 == Lt && b2 < t);
                    }
                }
                sl.cus[kPermOff + rank] = t;
            }
            __syncthreads();
        }
    }
}

// The producer warp: one lane takes items from the work queue, publishes each
// item's descriptor and bulk-copies its Q rows, and streams its K/V tiles into
// the ring; after an item's tiles it hands the consumers one ring stage, empty,
// for the item's merge.
template <int D, int NT, int ST>
__device__ __forceinline__ void split_producer(const SplitLayout& sl, const SplitParams& p, const CUtensorMap* ptmK,
                                               const CUtensorMap* ptmV, const CUtensorMap* ptmK16,
                                               const CUtensorMap* ptmV16) {
    using Sh = Shape<D, NT, ST>;
    const int lane = threadIdx.x & 31;
    const CUtensorMap& tmK = *ptmK;
    const CUtensorMap& tmV = *ptmV;
    const CUtensorMap& tmK16 = *ptmK16;
    const CUtensorMap& tmV16 = *ptmV16;
    int32_t* cus = sl.cus;
    int32_t* prefix = sl.prefix;
    ItemSlot* slots = sl.slots;
    const uint32_t ring = sl.ring, qbuf = sl.qbuf, full0 = sl.full0, empty0 = sl.empty0;
    const uint32_t ifull0 = sl.ifull0, iempty0 = sl.iempty0;
    // ---------------- producer: one lane takes items and issues every copy
    int n_items = p.n_items;
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
        // Take the next item index from the queue. A call takes exactly n_items
        // indices from it (one per item after each CTA's first, one past the end
        // per CTA that had a first item), so the take that returns the last of them
        // resets the counter for the next call on this workspace: no CTA counts
        // itself out at the end.
        auto take_next = [&]() -> int {
            const uint32_t raw = atomicAdd(p.work, 1u);
            if (raw + 1u == static_cast<uint32_t>(n_items)) atomicExch(p.work, 0u);
            return static_cast<int>(gridDim.x + raw);
        };
        ItemSlot item;
        // the first item of each CTA is its own index
        int state = publish(0, static_cast<int>(blockIdx.x), item);
        for (uint32_t it = 0; state == 1; ++it) {
            // The next item is taken from the queue a few stages before this one's
            // last tile: the atomic's round trip then overlaps the last copies, yet a
            // CTA never holds a reserved item for long (which would hurt the balance
            // at the end of the queue).
            const int fetch_at = max(0, item.ntiles - Sh::kStages);
            int next_idx = 0;
            if (item.ntiles == 0) next_idx = take_next();
            bool ok = true;
            for (int t = 0; t < item.ntiles; ++t) {
                if (t == fetch_at) next_idx = take_next();
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
                if (++st == Sh::kStages) {
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
            if (++st == Sh::kStages) {
                st = 0;
                ph ^= 1;
            }
            item = next;
            state = next_state;
        }
    }
}

// Write column block n (columns 8n .. 8n + 7) of one item from the four consumer
// warps' states in the merge stage: red_acc [warp][8][D + 4], red_m and red_l
// [warp][8]. Warp w writes columns w and w + 4; a lane owns four consecutive
// dims, read from each warp's row as one 16-byte load and stored as one vector.
// The passes are predicated rather than skipped, so their latencies overlap.
template <int D, int DT>
__device__ __forceinline__ void merge_write(const SplitParams& p, const ItemSlot& item, const float* red_acc,
                                            const float* red_m, const float* red_l, int n) {
    using Sh = Shape<D, 1>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kLanesPerHead = D / 4;
    constexpr int kHeadsPerPass = 32 / kLanesPerHead;   // 1 at head_dim 128, 2 at 64
    constexpr int kPasses = (kHeadsPerCta / kConsumerWarps) / kHeadsPerPass;
    const int d0 = (lane % kLanesPerHead) * 4;
#pragma unroll
    for (int pass = 0; pass < kPasses; ++pass) {
        const int hh = warp + kConsumerWarps * (pass * kHeadsPerPass + lane / kLanesPerHead);
        const bool live = kHeadsPerCta * n + hh < item.nh;
        float mw[kConsumerWarps];
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            mw[w] = red_m[w * kHeadsPerCta + hh];
            M = fmaxf(M, mw[w]);
        }
        // a column that saw no key keeps M = -inf: weights 0, output 0, lse -inf
        const float Ms = M == -INFINITY ? 0.f : M;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        float lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float wt = fast_exp2(mw[w] - Ms);
            lsum = fmaf(wt, red_l[w * kHeadsPerCta + hh], lsum);
            const float4 a = *reinterpret_cast<const float4*>(red_acc + (w * kHeadsPerCta + hh) * Sh::kMergeRow + d0);
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
            const int64_t qrow = column_row(p, item, kHeadsPerCta * n + hh);
            const int64_t row = qrow * p.S + item.s;
            const float lse = M == -INFINITY ? -INFINITY : (M + fast_log2(lsum)) * kLn2;
            // the sequence's only split: its weight exp(lse_0 - lse) is 1, so o_0 is the answer
            const bool direct = p.out != nullptr && item.valid == 2;
            if (p.keep_partials) {
                // A K/V stream larger than the L2: the item's writes go to the L2 with an
                // evict-last policy, so that they are not written back to DRAM in the middle
                // of the stream (and the combine finds the partials it reads back there)
                uint64_t keep;
                asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
                asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p.opart + row * D + d0),
                             "f"(o.x), "f"(o.y), "f"(o.z), "f"(o.w), "l"(keep)
                             : "memory");
                if (d0 == 0)
                    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p.lse + row), "f"(lse), "l"(keep)
                                 : "memory");
                if (direct)
                    asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;" ::"l"(p.out + qrow * D + d0),
                                 "r"(pack2<DT>(o.x, o.y)), "r"(pack2<DT>(o.z, o.w)), "l"(keep)
                                 : "memory");
            } else {
                *reinterpret_cast<float4*>(p.opart + row * D + d0) = o;
                if (d0 == 0) p.lse[row] = lse;
                if (direct)
                    *reinterpret_cast<uint2*>(p.out + qrow * D + d0) =
                        make_uint2(pack2<DT>(o.x, o.y), pack2<DT>(o.z, o.w));
            }
        }
    }
}

// End of a consumer warp's run. The work queue needs nothing here: its last take
// reset it (split_producer).
__device__ __forceinline__ void split_finish(const SplitParams& p, bool ok, uint32_t bad_bar, uint32_t bad_ph) {
    // after a timed-out wait, a copy still in flight into this CTA's shared memory
    // gets one more bounded wait before the CTA exits
    if (!ok && bad_bar != 0) mbar_wait(bad_bar, bad_ph, p.wait_limit_ns);
}

// ------------------------------------------------------------ host side
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

inline bool make_kv_map(CUtensorMap* map, const void* base, da_dtype dt, da_layout lay, int B, int Hkv,
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
// L2 size of the current device (bytes; 0 if it cannot be queried).
inline int device_l2_bytes() {
    int dev = 0, l2 = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
        return 0;
    return l2;
}

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
        // The limit is the kernel's, shared by every configuration of it (each with
        // its own cache): raise it once to what the device allows, never to one
        // configuration's size, which a smaller one set later would undercut.
        int optin = 0;
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return e;
        const int limit = optin - static_cast<int>(fa.sharedSizeBytes);
        if (smem > limit) return cudaErrorInvalidValue;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
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

// Host checks of a decode call's arguments other than the workspace.
inline da_status check_args(const void* q, const void* k, const void* v, const int32_t* cu, int B, int Hq,
                            int Hkv, int D, int kv_rows, int dt, int lay, float scale, int S) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || kv_rows < 0) return DA_ERR_INVALID_ARG;
    if (S < 1 || S > DA_MAX_SPLITS) return DA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return DA_ERR_INVALID_ARG;
    if (dt != DA_F16 && dt != DA_BF16) return DA_ERR_INVALID_ARG;
    if (lay != DA_LAYOUT_VARLEN && lay != DA_LAYOUT_BHSD) return DA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return DA_ERR_UNSUPPORTED;
    if (!q || !cu) return DA_ERR_INVALID_ARG;
    if (kv_rows > 0 && (!k || !v)) return DA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(cu, 4)) return DA_ERR_ALIGNMENT;
    if (kv_rows > 0 && (!aligned(k, 16) || !aligned(v, 16))) return DA_ERR_ALIGNMENT;
    if (decode_attn_splitkv_workspace_size(B, Hq, D, S) == 0) return DA_ERR_INVALID_ARG;
    const int64_t chunks = item_chunks(Hq / Hkv);
    if (static_cast<int64_t>(B) * Hkv * chunks * S > 0x7fffffffll) return DA_ERR_INVALID_ARG;
    return DA_OK;
}

// check_args, then the caller's workspace: present, 256-byte aligned, large enough.
inline da_status check_common(const void* q, const void* k, const void* v, const int32_t* cu, int B, int Hq,
                              int Hkv, int D, int kv_rows, int dt, int lay, float scale, int S,
                              const void* ws, size_t ws_bytes) {
    const da_status st = check_args(q, k, v, cu, B, Hq, Hkv, D, kv_rows, dt, lay, scale, S);
    if (st != DA_OK) return st;
    if (!ws) return DA_ERR_INVALID_ARG;
    if (!aligned(ws, 256)) return DA_ERR_ALIGNMENT;
    if (ws_bytes < decode_attn_splitkv_workspace_size(B, Hq, D, S)) return DA_ERR_WORKSPACE_TOO_SMALL;
    return DA_OK;
}

inline cudaLaunchAttribute pdl_attr() {
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
    void* ws;
};


inline Call make_call(const void* q, const void* k, const void* v, const int32_t* cu, int B, int Hq, int Hkv, int D,
               int kv_rows, da_dtype dt, da_layout lay, float scale, int S, int split_len, void* ws, int tq = 1) {
    Call c;
    c.tq = tq;
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

// Tensor maps and kernel parameters of one launch of a split kernel
// (split_kernel or a comparison arm that shares its skeleton): 64-key boxes for
// full stages, 16-key boxes for the ragged end of a split, and NT n-tiles of 8
// packed columns per work item.
struct SplitLaunch {
    CUtensorMap mk;
    CUtensorMap mv;
    CUtensorMap mk16;
    CUtensorMap mv16;
    SplitParams p;
    int smem;        // dynamic shared memory, bytes
    int cache_idx;   // which DeviceCache: the number of [B + 1] arrays staged in shared memory
};

// `out` (nullptr for the split step alone) gets the rows of every sequence that has
// a single split, whose o_0 is already the answer.
template <int D, int NT, int ST = kStages>
inline bool prepare_split(const Call& c, void* out, SplitLaunch& a) {
    std::memset(&a.mk, 0, sizeof(a.mk));
    std::memset(&a.mv, 0, sizeof(a.mv));
    std::memset(&a.mk16, 0, sizeof(a.mk16));
    std::memset(&a.mv16, 0, sizeof(a.mv16));
    if (c.kv_rows > 0) {
        if (!make_kv_map(&a.mk, c.k, c.dt, c.lay, c.B, c.Hkv, D, c.kv_rows, kStageKeys) ||
            !make_kv_map(&a.mv, c.v, c.dt, c.lay, c.B, c.Hkv, D, c.kv_rows, kStageKeys) ||
            !make_kv_map(&a.mk16, c.k, c.dt, c.lay, c.B, c.Hkv, D, c.kv_rows, kBoxKeys) ||
            !make_kv_map(&a.mv16, c.v, c.dt, c.lay, c.B, c.Hkv, D, c.kv_rows, kBoxKeys))
            return false;
    }
    SplitParams& p = a.p;
    uint8_t* wsb = static_cast<uint8_t*>(c.ws);
    p.q = static_cast<const uint16_t*>(c.q);
    p.cu = c.cu;
    p.err = reinterpret_cast<uint32_t*>(wsb);
    p.work = reinterpret_cast<uint32_t*>(wsb + kWorkCounterOff);
    p.done = reinterpret_cast<uint32_t*>(wsb + kDoneCounterOff);
    p.out = static_cast<uint16_t*>(out);
    p.lse = reinterpret_cast<float*>(wsb + kHeaderBytes);
    p.opart = reinterpret_cast<float*>(wsb + kHeaderBytes +
                                       round_up(static_cast<size_t>(c.B) * c.tq * c.Hq * c.S * 4, 256));
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
    {
        // K/V bytes the call may stream (BHSD: the slabs' capacity) against the L2
        const double kv = 4.0 * c.D * c.Hkv * (c.lay == DA_LAYOUT_VARLEN ? 1.0 : static_cast<double>(c.B)) * c.kv_rows;
        p.keep_partials = kv > static_cast<double>(device_l2_bytes());
    }
    p.sorted = c.split_len == 0 && c.lay == DA_LAYOUT_VARLEN && c.B > 1 && c.B <= kMaxSortedBatch && p.stage_cu;
    p.scale_log2 = c.scale * kLog2e;
    p.wait_limit_ns = kWaitLimitNs;
    const bool var = c.split_len != 0;
    // per-sequence mode: prefix[] shares the staged cu_seqlens_k area, past its B + 1
    // entries, when it fits there, so that the 16-column kernel still runs two CTAs
    // per SM
    p.prefix_off = -1;
    if (var && p.stage_cu && 2 * (c.B + 1) + 3 <= kStagedBytes / 4) p.prefix_off = (c.B + 1 + 3) / 4 * 4;
    const bool own_prefix = var && p.prefix_off < 0;
    a.smem = Shape<D, NT, ST>::kSmemBytes + (p.stage_cu ? kStagedBytes : 0) + (own_prefix ? kStagedBytes : 0);
    a.cache_idx = (p.stage_cu ? 1 : 0) + (own_prefix ? 1 : 0);
    return true;
}

// Launch a persistent split kernel: as many CTAs as fit on the device at once,
// at most one per work item, with programmatic dependent launch.
template <class K>
inline da_status launch_persistent(K kern, const SplitLaunch& a, DeviceCache& cache, cudaStream_t stream) {
    int grid = 0;
    if (persistent_grid(kern, kThreads, a.smem, cache, &grid) != cudaSuccess) return DA_ERR_CUDA;
    grid = std::min(grid, a.p.n_items);
    cudaLaunchAttribute attrs[1] = {pdl_attr()};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = a.smem;
    cfg.stream = stream;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a.mk, a.mv, a.mk16, a.mv16, a.p) == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

// The combine step over a call's workspace (decode_attn_splitkv.cu).
da_status dispatch_combine(const Call& c, void* out, cudaStream_t st);

}  // namespace da_impl

#endif
