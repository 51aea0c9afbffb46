// selftest.cu -- self-test of the bounded mbarrier wait that every pipeline
// barrier of the library relies on, and the two calibrations of the expert
// GEMM's roofline (the block-scaled MMA alone, and the MMA fed by the GEMM's
// own operand stream).  A time-out here (or anywhere) is a status the host
// reads, never a trap or a fault: the waiting thread gives up at a
// global-timer deadline and the kernel returns normally.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

// One CTA of 64 threads.  Thread 0 waits on a fresh barrier (one expected
// arrival); if `arrive`, thread 32 arrives after about 20 us.
__global__ void __launch_bounds__(64) bounded_wait_kernel(int arrive, uint64_t timeout_ns, int32_t* out) {
#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 1000)
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = ptx::smem_addr(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    const uint64_t t0 = ptx::globaltimer();
    if (threadIdx.x == 32 && arrive) {
        while (ptx::globaltimer() < t0 + 20000ull) __nanosleep(1000);  // ends: a fixed 20 us
        ptx::mbar_arrive(b);
    } else if (threadIdx.x == 0) {
        const bool ok = ptx::mbar_wait(b, 0, t0 + timeout_ns);
        out[0] = ok ? MOE_OK : MOE_ERR_TIMEOUT;
        out[1] = static_cast<int32_t>((ptx::globaltimer() - t0) / 1000ull);
    }
#else
    if (threadIdx.x == 0) out[0] = MOE_ERR_NO_KERNEL;
#endif
}

// Tensor-pipe ceiling of the block-scaled MMA the expert GEMMs issue: one CTA
// per SM (the shared-memory request keeps a second one off the SM), one
// thread issuing `kblocks` x 4 tcgen05.mma.kind::mxf8f6f4.block_scale (M = 128,
// N = 256, K = 32, E4M3 x E2M1, UE8M0 scales) back to back on fixed
// shared-memory operands into one tensor-memory accumulator, then waiting
// (bounded) for them to complete.  The operands are a fixed pseudo-random
// pattern; nothing is read from or written to global memory except the
// status word.
constexpr int kRateABytes = 16384, kRateBBytes = 32768, kRateSfBytes = 1536;
constexpr int kRateSmem = 120 * 1024;  // above half of the SM's shared memory: one CTA per SM

__global__ void __launch_bounds__(64, 1) mma_rate_kernel(int kblocks, int32_t* status) {
#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 1000)
    extern __shared__ uint8_t raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tbase;
    // operands: a fixed pseudo-random byte pattern (finite E4M3 codes: bit 3 of
    // every byte cleared, so no byte is 0x7F or 0xFF), so that the tensor pipe
    // switches as it does on real data; scale bytes 127 (2^0)
    for (int i = threadIdx.x; i < (kRateABytes + kRateBBytes) / 4; i += blockDim.x) {
        uint32_t h = static_cast<uint32_t>(i) * 2654435761u + blockIdx.x * 40503u;
        h ^= h >> 15;
        h *= 2246822519u;
        h ^= h >> 13;
        reinterpret_cast<uint32_t*>(smem)[i] = h & 0xF7F7F7F7u;
    }
    for (int i = threadIdx.x; i < kRateSfBytes; i += blockDim.x) smem[kRateABytes + kRateBBytes + i] = 127;
    ptx::fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_addr(&bar), 1);
        ptx::fence_mbar_init();
    }
    if (threadIdx.x < 32) {
        ptx::tmem_alloc(ptx::smem_addr(&tbase), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&tbase);
    if (threadIdx.x == 32) {
        const uint32_t s0 = ptx::smem_addr(smem);
        const uint64_t sf = ptx::desc_sf_32x16(s0 + kRateABytes + kRateBBytes);
        ptx::tc_cp_32x128b_warpx4(tmem + 256, sf);
        ptx::tc_cp_32x128b_warpx4(tmem + 260, sf + (512 >> 4));
        ptx::tc_cp_32x128b_warpx4(tmem + 264, sf + (1024 >> 4));
        const uint64_t a = ptx::desc_kmajor_sw128(s0), b = ptx::desc_kmajor_sw128(s0 + kRateABytes);
        constexpr uint32_t idesc = ptx::idesc_e4m3_e2m1(128, 256);
        for (int kb = 0; kb < kblocks; ++kb) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                ptx::mma_mxf8f6f4(tmem, a + 2 * kk, b + 2 * kk, ptx::idesc_with_sf_id(idesc, kk), tmem + 256,
                                  tmem + 260, (kb | kk) != 0);
        }
        ptx::tc_commit(ptx::smem_addr(&bar));
        if (!ptx::mbar_wait(ptx::smem_addr(&bar), 0, ptx::globaltimer() + 2000000000ull)) {
            atomicExch(status, MOE_ERR_TIMEOUT);
            // the accumulator must not be freed under running MMAs: wait once more, bounded
            ptx::mbar_wait(ptx::smem_addr(&bar), 0, ptx::globaltimer() + 2000000000ull);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
#else
    if (threadIdx.x == 0 && blockIdx.x == 0) *status = MOE_ERR_NO_KERNEL;
#endif
}

// Operand-stream ceiling of the expert GEMM's layer-1 tile: the same MMAs as
// mma_rate_kernel, but fed the way the expert kernel feeds them -- a 4-stage
// ring of 50 KB stages (the 128-row E4M3 A box, the 256-row two-plane E2M1 B
// box expanded to one byte per element, the A scale chunk and the B scale
// pair), a producer thread, a scale thread copying each stage's scales into
// tensor memory, and the MMA thread -- with no epilogue.  One CTA per SM;
// CTA c streams row block (c / 16) % 16 of A against weight rows of N tile
// c % 16 (so about ten A blocks and sixteen B tiles are live at once, as in
// the expert kernel's row-block-major order), cycling through the 56 k-blocks
// of K = 7168.  Every wait is bounded (2 s); on a time-out the kernel records
// MOE_ERR_TIMEOUT, lets its own copies in flight land and returns.
constexpr int kStrK = 7168, kStrRows = 2048, kStrKb = kStrK / kBlockK, kStrTiles = 16;
constexpr int kStrStages = 4, kStrStride = 51200;
constexpr int kStrA = kBlockM * kBlockK, kStrB = 256 * kBlockK;  // shared bytes per stage
constexpr int kStrSfOff = kStrA + kStrB;
constexpr uint32_t kStrTx = kStrA + kStrB / 2 + 3 * kSfChunkBytes;  // an E2M1 box counts its packed bytes
constexpr int kStrSmem = kStrStages * kStrStride + 1024;
constexpr uint64_t kStrWaitNs = 2000000000ull;
static_assert(kStrSfOff + 3 * kSfChunkBytes <= kStrStride && kStrStride % 1024 == 0, "stream stage");

struct StreamMaps {
    CUtensorMap a, b;
};

__global__ void __launch_bounds__(96, 1) stream_rate_kernel(const __grid_constant__ StreamMaps m,
                                                             const uint8_t* __restrict__ sfa,
                                                             const uint8_t* __restrict__ sfb, int kblocks,
                                                             int32_t* status) {
#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 1000)
    extern __shared__ uint8_t raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t done_bar, drain, full[kStrStages], ready[kStrStages], empty[kStrStages];
    __shared__ uint32_t tbase;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_addr(&done_bar), 1);
        ptx::mbar_init(ptx::smem_addr(&drain), 1);
        for (int s = 0; s < kStrStages; ++s) {
            ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&ready[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&empty[s]), 1);
        }
        ptx::fence_mbar_init();
    }
    if (threadIdx.x >= 32 && threadIdx.x < 64) {
        ptx::tmem_alloc(ptx::smem_addr(&tbase), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&tbase);
    const int rb = (blockIdx.x / kStrTiles) % kStrTiles, j = blockIdx.x % kStrTiles;
    if (threadIdx.x == 0) {
        // ------------------------------------------------ producer
        uint32_t issued = 0, parity = 0;
        for (int kb = 0; kb < kblocks; ++kb) {
            const int s = kb % kStrStages;
            if (kb >= kStrStages &&
                !ptx::mbar_wait(ptx::smem_addr(&empty[s]), ((kb / kStrStages) - 1) & 1,
                                ptx::globaltimer() + kStrWaitNs)) {
                atomicExch(status, MOE_ERR_TIMEOUT);
                break;
            }
            const int kx = kb % kStrKb;
            uint8_t* st = ring + s * kStrStride;
            const uint32_t f = ptx::smem_addr(&full[s]);
            ptx::mbar_arrive_expect_tx(f, kStrTx);
            ptx::tma_load_2d(ptx::smem_addr(st), &m.a, kx * kBlockK, rb * kBlockM, f);
            ptx::tma_load_3d(ptx::smem_addr(st + kStrA), &m.b, kx * kBlockK, j * 128, 0, f);
            ptx::bulk_load(ptx::smem_addr(st + kStrSfOff), sfa + (static_cast<size_t>(rb) * kStrKb + kx) * kSfChunkBytes,
                           kSfChunkBytes, f);
            ptx::bulk_load(ptx::smem_addr(st + kStrSfOff + kSfChunkBytes),
                           sfb + (static_cast<size_t>(j) * kStrKb + kx) * 2 * kSfChunkBytes, 2 * kSfChunkBytes, f);
            issued |= 1u << s;
            parity = (parity & ~(1u << s)) | (static_cast<uint32_t>((kb / kStrStages) & 1) << s);
        }
        // the last copies land before the CTA may exit (the scale thread
        // normally saw them all; after a time-out this is what waits)
        for (int s = 0; s < kStrStages; ++s)
            if (issued & (1u << s))
                ptx::mbar_wait(ptx::smem_addr(&full[s]), (parity >> s) & 1u, ptx::globaltimer() + kStrWaitNs);
    } else if (threadIdx.x == 64) {
        // ------------------------------------------------ scale copies
        for (int kb = 0; kb < kblocks; ++kb) {
            const int s = kb % kStrStages;
            if (!ptx::mbar_wait(ptx::smem_addr(&full[s]), (kb / kStrStages) & 1, ptx::globaltimer() + kStrWaitNs)) {
                atomicExch(status, MOE_ERR_TIMEOUT);
                break;
            }
            ptx::tc_fence_after();
            const uint64_t sf = ptx::desc_sf_32x16(ptx::smem_addr(ring + s * kStrStride + kStrSfOff));
            const uint32_t tsf = tmem + 256 + 16 * s;
            ptx::tc_cp_32x128b_warpx4(tsf + 0, sf);
            ptx::tc_cp_32x128b_warpx4(tsf + 4, sf + (kSfChunkBytes >> 4));
            ptx::tc_cp_32x128b_warpx4(tsf + 8, sf + (2 * kSfChunkBytes >> 4));
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_addr(&ready[s]));
        }
        ptx::tc_commit(ptx::smem_addr(&drain));
        if (!ptx::mbar_wait(ptx::smem_addr(&drain), 0, ptx::globaltimer() + kStrWaitNs))
            atomicExch(status, MOE_ERR_TIMEOUT);
    } else if (threadIdx.x == 32) {
        // ------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = ptx::idesc_e4m3_e2m1(kBlockM, 256);
        const uint64_t a0 = ptx::desc_kmajor_sw128(ptx::smem_addr(ring));
        const uint64_t b0 = ptx::desc_kmajor_sw128(ptx::smem_addr(ring + kStrA));
        for (int kb = 0; kb < kblocks; ++kb) {
            const int s = kb % kStrStages;
            if (!ptx::mbar_wait(ptx::smem_addr(&ready[s]), (kb / kStrStages) & 1, ptx::globaltimer() + kStrWaitNs)) {
                atomicExch(status, MOE_ERR_TIMEOUT);
                break;
            }
            ptx::tc_fence_after();
            const uint64_t so = static_cast<uint64_t>(s * (kStrStride >> 4));
            const uint32_t tsf = tmem + 256 + 16 * s;
#pragma unroll
            for (int kk = 0; kk < kBlockK / 32; ++kk)
                ptx::mma_mxf8f6f4(tmem, a0 + so + 2 * kk, b0 + so + 2 * kk, ptx::idesc_with_sf_id(idesc, kk), tsf + 0,
                                  tsf + 4, (kb | kk) != 0);
            ptx::tc_commit(ptx::smem_addr(&empty[s]));
        }
        ptx::tc_commit(ptx::smem_addr(&done_bar));
        if (!ptx::mbar_wait(ptx::smem_addr(&done_bar), 0, ptx::globaltimer() + kStrWaitNs)) {
            atomicExch(status, MOE_ERR_TIMEOUT);
            // the accumulator must not be freed under running MMAs: wait once more, bounded
            ptx::mbar_wait(ptx::smem_addr(&done_bar), 0, ptx::globaltimer() + kStrWaitNs);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (threadIdx.x >= 32 && threadIdx.x < 64) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
#else
    if (threadIdx.x == 0 && blockIdx.x == 0) *status = MOE_ERR_NO_KERNEL;
#endif
}

}  // namespace

cudaError_t launch_stream_rate_selftest(const void* a, const void* b, const void* sfa, const void* sfb, int kblocks,
                                        int ctas, int32_t* status, cudaStream_t s) {
    static std::atomic<int> attr_done[64] = {};
    int dev = 0;
    cudaError_t st = cudaGetDevice(&dev);
    if (st != cudaSuccess) return st;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev].load(std::memory_order_acquire)) {
        st = cudaFuncSetAttribute(stream_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStrSmem);
        if (st != cudaSuccess) return st;
        attr_done[dev].store(1, std::memory_order_release);
    }
    StreamMaps m;
    if (!make_layer1_operand_maps(&m.a, a, &m.b, b, kStrK, kStrRows)) return cudaErrorInvalidValue;
    if ((st = cudaMemsetAsync(status, 0, sizeof(int32_t), s)) != cudaSuccess) return st;
    stream_rate_kernel<<<ctas, 96, kStrSmem, s>>>(m, static_cast<const uint8_t*>(sfa), static_cast<const uint8_t*>(sfb),
                                                  kblocks, status);
    return cudaGetLastError();
}

cudaError_t launch_mma_rate_selftest(int kblocks, int ctas, int32_t* status, cudaStream_t s) {
    static std::atomic<int> attr_done[64] = {};
    int dev = 0;
    cudaError_t st = cudaGetDevice(&dev);
    if (st != cudaSuccess) return st;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev].load(std::memory_order_acquire)) {
        st = cudaFuncSetAttribute(mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRateSmem);
        if (st != cudaSuccess) return st;
        attr_done[dev].store(1, std::memory_order_release);
    }
    if ((st = cudaMemsetAsync(status, 0, sizeof(int32_t), s)) != cudaSuccess) return st;
    mma_rate_kernel<<<ctas, 64, kRateSmem, s>>>(kblocks, status);
    return cudaGetLastError();
}

cudaError_t launch_bounded_wait_selftest(int arrive, uint64_t timeout_ns, int32_t* out, cudaStream_t s) {
    bounded_wait_kernel<<<1, 64, 0, s>>>(arrive, timeout_ns, out);
    return cudaGetLastError();
}

}  // namespace moe
