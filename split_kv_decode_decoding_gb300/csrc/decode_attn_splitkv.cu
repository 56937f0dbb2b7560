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
// The work-item decoding, the producer warp and the write-out of a merged item
// live in split_common.cuh, shared with the comparison arms (CUDA-core products
// and tcgen05 with tensor memory) of comparison_arms.cu, which the library's own
// calls never use; the split-count picker and the per-sequence planner are in
// picker.cpp, the host-only time model in time_model.cpp.
//
// Every mbarrier wait is bounded in time; on expiry the kernel sets
// DA_DEVERR_TIMEOUT in the workspace error word and winds down instead of
// hanging.

#include "split_common.cuh"

namespace da_impl {

constexpr int kMaxVarsplitBatch = 1024;       // sequences, per-sequence mode

// ------------------------------------------------------------ split step
template <int D, int DT, int NT, int ST>
__global__ void __launch_bounds__(kThreads, kMinBlocksPerSm)
split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
             const __grid_constant__ CUtensorMap tmK16, const __grid_constant__ CUtensorMap tmV16,
             const SplitParams p) {
    using Sh = Shape<D, NT, ST>;
    extern __shared__ uint8_t smem_raw[];
    const SplitLayout sl = split_layout<D, NT, ST>(smem_raw, p);
    uint8_t* smem = sl.smem;
    ItemSlot* slots = sl.slots;
    const uint32_t ring = sl.ring, qbuf = sl.qbuf, full0 = sl.full0, empty0 = sl.empty0;
    const uint32_t ifull0 = sl.ifull0, iempty0 = sl.iempty0, mfull = sl.mfull, mdone = sl.mdone;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    split_setup<D, NT, ST>(sl, p, &tmK, &tmV, &tmK16, &tmV16);
    if (warp == kConsumerWarps) {
        split_producer<D, NT, ST>(sl, p, &tmK, &tmV, &tmK16, &tmV16);
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
        if constexpr (NT == 1) {
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
                if (++st == Sh::kStages) {
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
            merge_write<D, DT>(p, item, red_acc, red_m, red_l, 0);
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
            // columns 8n + 2*t4 (+1): running max (log2 domain), sum share. A column that has
            // seen no key holds kNoKey, a finite stand-in for -inf: it is the reference of its
            // weights as it is (exp2(-inf - kNoKey) = 0, and the first key's rescale weighs
            // the empty state exp2(kNoKey - m) = 0), and it becomes -inf again at the merge.
            constexpr float kNoKey = -1e30f;
            float m_run[NT][2], l_run[NT][2];
    #pragma unroll
            for (int n = 0; n < NT; ++n) {
                m_run[n][0] = m_run[n][1] = kNoKey;
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
                    // scores -> exp2 domain, mask keys past the split end
                    float x[NT][4], mx0[NT], mx1[NT];
                    bool move = false;
    #pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        x[n][0] = key_lo < visA[n] ? (sc[n][0] + sd[n][0]) * p.scale_log2 : -INFINITY;
                        x[n][1] = key_lo < visB[n] ? (sc[n][1] + sd[n][1]) * p.scale_log2 : -INFINITY;
                        x[n][2] = key_lo + 8 < visA[n] ? (sc[n][2] + sd[n][2]) * p.scale_log2 : -INFINITY;
                        x[n][3] = key_lo + 8 < visB[n] ? (sc[n][3] + sd[n][3]) * p.scale_log2 : -INFINITY;
                        mx0[n] = fmaxf(x[n][0], x[n][2]);
                        mx1[n] = fmaxf(x[n][1], x[n][3]);
                        move = move || mx0[n] > m_run[n][0] + kLazyRescale || mx1[n] > m_run[n][1] + kLazyRescale;
                    }
                    // Lazy reference: a column's running max m_run moves only when some score
                    // of the warp's box exceeds it by more than kLazyRescale (log2 units), so
                    // the shuffle reduction and the accumulator rescale run on a few boxes per
                    // item; one vote covers every n-tile, and all of them move together (a
                    // column whose max did not rise keeps its reference: al = 1). The weights
                    // stay below 2^kLazyRescale, well inside the fp16 and bf16 range, and every
                    // sum below shares the same reference.
                    if (__any_sync(0xffffffffu, move)) {
    #pragma unroll
                        for (int n = 0; n < NT; ++n) {
    #pragma unroll
                            for (int off = 4; off < 32; off <<= 1) {
                                mx0[n] = fmaxf(mx0[n], __shfl_xor_sync(0xffffffffu, mx0[n], off));
                                mx1[n] = fmaxf(mx1[n], __shfl_xor_sync(0xffffffffu, mx1[n], off));
                            }
                            // a column that has still seen no key keeps kNoKey (al = 1 on zeros)
                            const float mn0 = fmaxf(m_run[n][0], mx0[n]), mn1 = fmaxf(m_run[n][1], mx1[n]);
                            const float al0 = fast_exp2(m_run[n][0] - mn0), al1 = fast_exp2(m_run[n][1] - mn1);
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
                    }
    #pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        const float p0 = fast_exp2(x[n][0] - m_run[n][0]), p1 = fast_exp2(x[n][1] - m_run[n][1]);
                        const float p2 = fast_exp2(x[n][2] - m_run[n][0]), p3 = fast_exp2(x[n][3] - m_run[n][1]);
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
                if (++st == Sh::kStages) {
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
                    red_m[warp * 8 + 2 * t4] = m_run[n][0] == kNoKey ? -INFINITY : m_run[n][0];
                    red_m[warp * 8 + 2 * t4 + 1] = m_run[n][1] == kNoKey ? -INFINITY : m_run[n][1];
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
                merge_write<D, DT>(p, item, red_acc, red_m, red_l, n);
            }
        }
        // release the stage: order these generic-proxy stores before the TMA writes that refill it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * st);
        if (++st == Sh::kStages) {
            st = 0;
            ph ^= 1;
        }
        if (!ok) break;
    }
    split_finish(p, ok, bad_bar, bad_ph);
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

// Merge the running states of lanes `first` apart, 2 * first apart, ... up to 16
// apart: afterwards the lanes that hold the same dims share the merged state
// (fixed order, deterministic).
__device__ __forceinline__ void merge_lanes(float& m, float& z, float4& acc, int first) {
    for (int off = first; off < 32; off <<= 1) {
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
}

// Four merged dims of an output row: acc / z rounded to the output dtype, or 0 when
// every split was empty.
template <int DT>
__device__ __forceinline__ void store_quad(uint16_t* o, float m, float z, const float4& acc) {
    if (m == -INFINITY) {
        *reinterpret_cast<uint2*>(o) = make_uint2(0u, 0u);
    } else {
        const float inv = 1.f / z;
        *reinterpret_cast<uint2*>(o) =
            make_uint2(pack2<DT>(acc.x * inv, acc.y * inv), pack2<DT>(acc.z * inv, acc.w * inv));
    }
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
        // a sequence with one split: the split step wrote its rows
        if (Srow == 1) return;
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
    merge_lanes(m, z, acc, lps);
    if (sub == 0) store_quad<DT>(cp.out + static_cast<int64_t>(row) * D + d0, m, z, acc);
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
template <int D, int DT, int NT, int ST>
da_status launch_split(const Call& c, void* out, cudaStream_t stream) {
    SplitLaunch a;
    if (!prepare_split<D, NT, ST>(c, out, a)) return DA_ERR_CUDA;
    static DeviceCache caches[3];
    return launch_persistent(split_kernel<D, DT, NT, ST>, a, caches[a.cache_idx], stream);
}


// dims per combine warp: enough warps to cover the GPU, at least 8 dims each. With
// per-sequence split counts the rows of one-split sequences return at once and the
// others may hold up to S splits, so the slices narrow with S alone: a lane then
// keeps every split of its slice in flight in a few loads.
int combine_dchunks(int rows, int D, int S, bool per_sequence) {
    int dchunks = 1;
    while (D / dchunks > 8 && (per_sequence || static_cast<int64_t>(rows) * dchunks < 2048) && S > 4 * dchunks)
        dchunks *= 2;
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
    cp.dchunks = combine_dchunks(cp.rows, D, c.S, c.split_len != 0);
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
    if (wide) return launch_split<D, DT, 2, kStages>(c, out, st);
    return launch_split<D, DT, 1, kStages>(c, out, st);
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

// Split step, then the combine step unless every sequence has a single split
// (S = 1, or a per-sequence cap of 1): the split step then wrote all of `out`.
da_status run_decode(const Call& c, void* out, cudaStream_t st) {
    da_status r = dispatch_split(c, out, st);
    if (r != DA_OK || c.S == 1) return r;
    return dispatch_combine(c, out, st);
}

}  // namespace da_impl

using namespace da_impl;

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


da_status decode_attn_splitkv_multiquery_varsplit(const void* q, const void* k, const void* v,
                                                  const int32_t* cu_seqlens_k, int B, int T_q, int Hq, int Hkv,
                                                  int D, int kv_rows, da_dtype dtype, da_layout layout,
                                                  float scale, int split_len, int max_splits, void* out,
                                                  void* workspace, size_t workspace_bytes, void* stream) {
    if (split_len < 1) return DA_ERR_INVALID_ARG;
    if (T_q < 1 || T_q > DA_MAX_QUERY_TOKENS) return DA_ERR_INVALID_ARG;
    if (B < 1 || static_cast<int64_t>(B) * T_q > 0x7fffffffll) return DA_ERR_INVALID_ARG;
    if (B > kMaxVarsplitBatch) return DA_ERR_UNSUPPORTED;
    // the workspace holds B * T_q rows of Hq heads, max_splits splits each
    const size_t need = decode_attn_splitkv_workspace_size(B * T_q, Hq, D, max_splits);
    da_status st = check_common(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale, max_splits,
                                workspace, need == 0 ? workspace_bytes : std::max(workspace_bytes, need));
    if (st != DA_OK) return st;
    if (workspace_bytes < need) return DA_ERR_WORKSPACE_TOO_SMALL;
    if (!out) return DA_ERR_INVALID_ARG;
    if (!aligned(out, 16)) return DA_ERR_ALIGNMENT;
    const int64_t chunks = item_chunks(static_cast<int64_t>(Hq / Hkv) * T_q);
    if (static_cast<int64_t>(B) * Hkv * chunks * max_splits > 0x7fffffffll) return DA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(B) * T_q * Hq * D > 0x7fffffffll) return DA_ERR_INVALID_ARG;
    return run_decode(make_call(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale, max_splits,
                                split_len, workspace, T_q),
                      out, static_cast<cudaStream_t>(stream));
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
    return (bits & DA_DEVERR_TIMEOUT) ? DA_ERR_DEVICE_TIMEOUT : DA_OK;
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
        case DA_ERR_DEVICE_TIMEOUT:
            return "DA_ERR_DEVICE_TIMEOUT: a pipeline wait on the device timed out; that call's "
                   "outputs are invalid";
    }
    return "unknown da_status";
}

}  // extern "C"

// ================================================================ no-allocation variant
// For callers that may not allocate device memory: the workspace is a scratch
// array compiled into this library instead of a caller buffer.
namespace da_impl {

__device__ __align__(256) uint8_t g_noalloc_scratch[DA_NOALLOC_SCRATCH_BYTES];
static_assert(static_cast<uint64_t>(DA_NOALLOC_SCRATCH_BYTES) / 4 <= 0x7fffffffull,
              "every o_part index of a problem that fits the scratch stays within int32");

constexpr int kMaxDevices = 128;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};                 // device address of the array, per device ordinal
unsigned long long g_noalloc_ctx[kMaxDevices] = {};     // id of the context that address belongs to

// Id of the calling thread's current CUDA context (0 if none is current yet).
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// In host code g_noalloc_scratch names a host-side shadow, not device memory:
// the device address comes from cudaGetSymbolAddress, looked up with the device
// current, once per device and context (a context made after cudaDeviceReset
// holds a fresh copy of the array at a possibly different address).
da_status noalloc_scratch(void** addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    const unsigned long long ctx = current_context_id();
    if (g_noalloc_addr[dev] == nullptr || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return DA_ERR_CUDA;
        g_noalloc_addr[dev] = p;
        // the lookup made the context current if none was: record the one it used
        g_noalloc_ctx[dev] = current_context_id();
    }
    *addr = g_noalloc_addr[dev];
    return DA_OK;
}

}  // namespace da_impl

extern "C" da_status decode_attn_splitkv_noalloc(const void* q, const void* k, const void* v,
                                                 const int32_t* cu_seqlens_k, int B, int Hq, int Hkv,
                                                 int D, int kv_rows, da_dtype dtype, da_layout layout,
                                                 float scale, int num_splits, void* out, void* stream) {
    // every host check first: a refused call makes no CUDA call
    const size_t need = decode_attn_splitkv_workspace_size(B, Hq, D, num_splits);
    if (need > DA_NOALLOC_SCRATCH_BYTES) return DA_ERR_SCRATCH_LIMIT;
    da_status st = check_args(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale, num_splits);
    if (st != DA_OK) return st;
    if (!out) return DA_ERR_INVALID_ARG;
    if (!aligned(out, 16)) return DA_ERR_ALIGNMENT;
    if (static_cast<int64_t>(B) * Hq * D > 0x7fffffffll) return DA_ERR_INVALID_ARG;
    void* ws = nullptr;
    st = noalloc_scratch(&ws);
    if (st != DA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, kHeaderBytes, s) != cudaSuccess) return DA_ERR_CUDA;
    return run_decode(make_call(q, k, v, cu_seqlens_k, B, Hq, Hkv, D, kv_rows, dtype, layout, scale, num_splits, 0,
                                ws),
                      out, s);
}

extern "C" da_status decode_attn_splitkv_noalloc_get_error(uint32_t* device_error_bits, void* stream) {
    if (!device_error_bits) return DA_ERR_INVALID_ARG;
    void* ws = nullptr;
    const da_status st = noalloc_scratch(&ws);
    if (st != DA_OK) return st;
    return decode_attn_splitkv_get_error(ws, device_error_bits, stream);
}
