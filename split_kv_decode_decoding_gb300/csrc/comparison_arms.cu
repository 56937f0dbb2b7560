// Comparison arms of the split step, for the design choices of the library's
// split kernel (decode_attn_splitkv.cu). The library's own calls never use them;
// they are exported for the benchmark and the tests.
//   * split_kernel_fma: the same persistent kernel, producer warp, ring and item
//     merge, with the two products (q.k and p.v) on CUDA-core fp32 FMAs instead
//     of mma.sync tensor-core instructions; the pages' kernels put a packed GQA
//     group's products on tensor cores, and this measures what plain FMAs reach
//     on the same pipeline (decode_attn_splitkv_partial_cuda_core).
//   * split_kernel_tc: the split step for items of 9 to 32 packed columns on the
//     Blackwell tcgen05 tensor cores, with S, P and O in tensor memory
//     (decode_attn_splitkv_multiquery_tmem).

#include "split_common.cuh"

namespace da_impl {

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

// ------------------------------------------------------------ split step on CUDA-core FMAs
// The library's split kernel with both products (q.k and p.v) on fp32 FMAs
// instead of tensor cores, over the same producer, ring and item merge: the
// comparison arm for the tensor-core choice. Items of up to 8 columns.
template <int D, int DT>
__global__ void __launch_bounds__(kThreads, kMinBlocksPerSm)
split_kernel_fma(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmK16, const __grid_constant__ CUtensorMap tmV16,
                 const SplitParams p) {
    constexpr int NT = 1;
    using Sh = Shape<D, NT>;
    extern __shared__ uint8_t smem_raw[];
    const SplitLayout sl = split_layout<D, NT, kStages>(smem_raw, p);
    uint8_t* smem = sl.smem;
    ItemSlot* slots = sl.slots;
    const uint32_t ring = sl.ring, qbuf = sl.qbuf, full0 = sl.full0, empty0 = sl.empty0;
    const uint32_t iempty0 = sl.iempty0, mfull = sl.mfull, ifull0 = sl.ifull0;
    // per consumer warp: softmax weights [16 keys][8 columns] and 8 rescale factors
    float* fma_p = reinterpret_cast<float*>(sl.extra);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    split_setup<D, NT, kStages>(sl, p, &tmK, &tmV, &tmK16, &tmV16);
    if (warp == kConsumerWarps) {
        split_producer<D, NT, kStages>(sl, p, &tmK, &tmV, &tmK16, &tmV16);
        return;
    }

    // ---------------- consumers
    const int g = lane >> 2, t4 = lane & 3;
    bool ok = true;
    uint32_t bad_bar = 0, bad_ph = 0;
    int st = 0;          // ring position of the next tile
    uint32_t ph = 0;     // its phase parity

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
        {
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
            merge_write<D, DT>(p, item, red_acc, red_m, red_l, 0);
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
    split_finish(p, ok, bad_bar, bad_ph);
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
    // the last CTA to finish re-arms the work queue (this kernel counts its CTAs out;
    // split_kernel resets the queue at its last take instead)
    if (threadIdx.x == 0) {
        const uint32_t prev = atomicAdd(p.done, 1u);
        if (prev == gridDim.x - 1) {
            atomicExch(p.work, 0u);
            atomicExch(p.done, 0u);
        }
    }
}

// ------------------------------------------------------------ host side
template <int D, int DT>
da_status launch_split_fma(const Call& c, cudaStream_t stream) {
    SplitLaunch a;
    if (!prepare_split<D, 1>(c, nullptr, a)) return DA_ERR_CUDA;
    a.smem += kConsumerWarps * 17 * 8 * 4;   // the per-warp weights of the FMA products
    static DeviceCache caches[3];
    return launch_persistent(split_kernel_fma<D, DT>, a, caches[a.cache_idx], stream);
}

da_status dispatch_split_fma(const Call& c, cudaStream_t st) {
    if (c.D == 128)
        return c.dt == DA_F16 ? launch_split_fma<128, DA_F16>(c, st) : launch_split_fma<128, DA_BF16>(c, st);
    return c.dt == DA_F16 ? launch_split_fma<64, DA_F16>(c, st) : launch_split_fma<64, DA_BF16>(c, st);
}

// Q viewed as [B * tq][Hq][D]: one box holds `tokens` query tokens x the G heads
// of one KV head x 64 dims, i.e. the packed columns of one tensor-memory item.
inline bool make_q_map(CUtensorMap* map, const void* q, da_dtype dt, int rows, int Hq, int D, int G, int tokens) {
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
    p.sorted = 0;   // this kernel's producer hands out items in index order
    p.prefix_off = -1;   // and keeps prefix[] in an area of its own
    p.keep_partials = 0;
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

da_status dispatch_split_tc(const Call& c, void* out, cudaStream_t st) {
    if (c.D == 128)
        return c.dt == DA_F16 ? launch_split_tc<128, DA_F16>(c, out, st) : launch_split_tc<128, DA_BF16>(c, out, st);
    return c.dt == DA_F16 ? launch_split_tc<64, DA_F16>(c, out, st) : launch_split_tc<64, DA_BF16>(c, out, st);
}

}  // namespace da_impl

using namespace da_impl;

extern "C" {

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
    return dispatch_split_fma(c, static_cast<cudaStream_t>(stream));
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
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const da_status r = dispatch_split_tc(c, out, s);
    if (r != DA_OK || num_splits == 1) return r;   // one split: the split kernel wrote `out`
    return dispatch_combine(c, out, s);
}

}  // extern "C"
