// Read-ceiling probe: the bare HBM read rate a persistent kernel reaches on this
// GPU when each CTA streams one contiguous range through shared memory with bulk
// copies and consumes nothing. It is the measured floor against which the split
// kernel's small-workload times are judged (same flush, same event pair); it is
// not part of the decode path and the decode library does not use it.
//
// Each CTA takes bytes / grid of the buffer (in 16-byte units, the last CTA the
// remainder) and copies it chunk by chunk with cp.async.bulk into a ring of
// shared-memory stages, one thread issuing and waiting on the stages' mbarriers.
// Every wait is bounded in time (2 s); on expiry the kernel sets the error word
// and returns.

#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr int kProbeThreads = 32;
constexpr unsigned long long kProbeWaitNs = 2000000000ull;

__device__ __forceinline__ uint32_t probe_smem(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool probe_wait(uint32_t bar, uint32_t parity) {
    unsigned long long t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    while (true) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > kProbeWaitNs) return false;
    }
}

// stages x chunk bytes of dynamic shared memory, then stages mbarriers
__global__ void __launch_bounds__(kProbeThreads) read_probe_kernel(const uint8_t* buf, uint64_t bytes, int stages,
                                                                    int chunk, uint32_t* err) {
    extern __shared__ __align__(128) uint8_t sm[];
    const uint32_t ring = probe_smem(sm);
    const uint32_t bars = ring + static_cast<uint32_t>(stages) * chunk;
    if (threadIdx.x != 0) return;
    for (int i = 0; i < stages; ++i)
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bars + 8 * i) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const uint64_t units = bytes / 16;
    const uint64_t per = units / gridDim.x;
    const uint64_t lo = per * blockIdx.x * 16;
    const uint64_t hi = (blockIdx.x + 1 == gridDim.x ? units : per * (blockIdx.x + 1)) * 16;
    uint64_t issued = 0, done = 0;
    const uint64_t n = (hi - lo + chunk - 1) / chunk;
    while (done < n) {
        while (issued < n && issued - done < static_cast<uint64_t>(stages)) {
            const int slot = static_cast<int>(issued % stages);
            const uint64_t off = lo + issued * chunk;
            const uint32_t len = static_cast<uint32_t>(hi - off < static_cast<uint64_t>(chunk) ? hi - off : chunk);
            const uint32_t bar = bars + 8 * slot;
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(len) : "memory");
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    ring + slot * chunk),
                "l"(reinterpret_cast<uint64_t>(buf + off)), "r"(len), "r"(bar)
                : "memory");
            ++issued;
        }
        const int slot = static_cast<int>(done % stages);
        if (!probe_wait(bars + 8 * slot, static_cast<uint32_t>((done / stages) & 1))) {
            atomicOr(err, 1u);
            // give each copy still in flight one more bounded wait before the CTA exits
            for (uint64_t d = done; d < issued; ++d)
                probe_wait(bars + 8 * static_cast<int>(d % stages), static_cast<uint32_t>((d / stages) & 1));
            return;
        }
        ++done;
    }
}

}  // namespace

extern "C" {

// Stream `bytes` (a multiple of 16, buffer 16-byte aligned) of device memory
// through shared memory: grid = SMs x ctas_per_sm, each CTA a contiguous range
// in chunks of chunk_bytes (a multiple of 16) over `stages` shared-memory stages.
// `err` (device, uint32) gets bit 0 if a wait timed out. Returns 0, or -1 on a
// bad argument, -2 if the launch failed.
int read_probe(const void* buf, unsigned long long bytes, int ctas_per_sm, int chunk_bytes, int stages,
               unsigned int* err, void* stream) {
    if (!buf || !err || bytes == 0 || bytes % 16 || ctas_per_sm < 1 || chunk_bytes < 16 || chunk_bytes % 16 ||
        stages < 1 || reinterpret_cast<uintptr_t>(buf) % 16)
        return -1;
    const size_t smem = static_cast<size_t>(stages) * chunk_bytes + 8 * stages;
    if (smem > 227 * 1024) return -1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -2;
    if (cudaFuncSetAttribute(read_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return -2;
    uint64_t grid = static_cast<uint64_t>(sms) * ctas_per_sm;
    if (grid > bytes / 16) grid = bytes / 16;
    read_probe_kernel<<<static_cast<unsigned>(grid), kProbeThreads, smem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(buf), bytes, stages, chunk_bytes, err);
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

}  // extern "C"
