// Tensor-core throughput probe for the roofline's compute term: the dense
// block-scaled MXFP4 rate (tcgen05.mma .kind::mxf4, scale_vec::2X) that one CTA
// per SM reaches with operands resident in shared memory and nothing else to
// do.  It also shows the cost of the scale-factor copies the GEMM kernel issues
// beside its MMAs: with copies_per_mma > 0 each MMA is preceded by that many
// tcgen05.cp .32x128b.warpx4 copies, as the GEMM's stages interleave them.
//
// Variants (bits of `variant`): bit 0, the copies are tcgen05.cp .128x256b
// (4 KB source, 128 lanes x 8 columns) instead of .32x128b.warpx4 (512 B source
// replicated to four lane quadrants, 4 columns); bit 1, the copies are issued by
// a second warp (into columns the MMAs do not read) instead of the MMA thread;
// bits 2-3, the MMAs rotate over 2^(bits) independent accumulators (n columns
// each, at most 256 columns in all) instead of accumulating into one, so that
// consecutive MMAs do not depend on each other; bits 4-5, the MMA thread
// commits its tensor operations to an mbarrier (which nothing waits on) after
// every 1, 4 or 8 MMAs (bits 1, 2, 3), as a pipeline releases its stages.
//
// Operand values do not matter for the timing: shared memory is zero-filled,
// so every product is zero.  One thread per CTA issues every MMA; the tensor
// pipe's queue paces it.  The final waits for the issued work are bounded and
// record a status bit if they run out.
#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kProbeThreads = 128;
constexpr uint32_t kProbeAOff = 0;            // A: 128 rows x 128 B (128-byte swizzle)
constexpr uint32_t kProbeBOff = 16384;        // B: up to 256 rows x 128 B
constexpr uint32_t kProbeSfOff = 16384 + 32768;  // zeroed scale-factor source (4 KB)
constexpr uint32_t kProbeBarOff = kProbeSfOff + 4096;
constexpr uint32_t kProbeSmem = kProbeBarOff + 64 + 1024;  // + alignment slack (barriers: 3 x 8 B, slot)

__global__ void __launch_bounds__(kProbeThreads, 1)
    moe_mxf4_probe_kernel(int n, int iters, int copies_per_mma, int variant, uint32_t* status) {
    extern __shared__ uint8_t probe_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(probe_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* done = reinterpret_cast<uint64_t*>(smem + kProbeBarOff);
    uint64_t* done2 = done + 1;
    uint64_t* tick = done + 2;  // periodic commits (never waited on)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kProbeBarOff + 24);
    for (uint32_t i = threadIdx.x * 16u; i < kProbeBarOff; i += kProbeThreads * 16u)
        *reinterpret_cast<uint4*>(smem + i) = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        mbar_init(done, 1);
        mbar_init(done2, 1);
        mbar_init(tick, 1);
        fence_barrier_init();
    }
    fence_proxy_async_smem();  // the zeros are read by the tensor core (async proxy)
    if (threadIdx.x < 32) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const bool wide = (variant & 1) != 0, other_warp = (variant & 2) != 0;
    // 32x128b source: 32 rows x 16 B, 8-row core matrices 128 B apart;
    // 128x256b source: 128 rows x 32 B as 16 groups of 8 rows, each two 128-byte
    // core matrices (the row's two 16-byte halves) 128 B apart, groups 256 B apart
    const uint64_t dsf = smem_desc(smem_u32(smem + kProbeSfOff), 0, 128, 0);
    const uint64_t dsf_wide = smem_desc(smem_u32(smem + kProbeSfOff), 128, 256, 0);
    // accumulator in columns [0, n); scale factors the MMAs read at 256 (A) and
    // 264 (B); copies of the second warp go to columns 384.. (never read)
    const uint32_t sfa = tmem + 256u, sfb = tmem + 264u;
    auto copy = [&](uint32_t col) {
        if (wide)
            tmem_cp_128x256b(col, dsf_wide);
        else
            tmem_cp_sf(col, dsf);
    };
    auto wait_done = [&](uint64_t* bar) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(bar), 0)) {
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                atomicOr(status, kErrTimeoutDrain);
                break;
            }
        }
    };
    if (threadIdx.x == 0) {
        tmem_cp_sf(sfa, dsf);
        tmem_cp_sf(sfb, dsf);
        tmem_cp_sf(sfb + 4u, dsf);
        const uint64_t ad = smem_desc(smem_u32(smem + kProbeAOff), 16, 1024, 2);
        const uint64_t bd = smem_desc(smem_u32(smem + kProbeBOff), 16, 1024, 2);
        const uint32_t idesc = mxf4_idesc(128, (uint32_t)n, 0, 0);
        const uint32_t amask = (1u << ((variant >> 2) & 3)) - 1u;  // accumulators - 1
        const int cbits = (variant >> 4) & 3;
        const int cper = cbits == 1 ? 1 : cbits == 2 ? 4 : cbits == 3 ? 8 : 0;  // MMAs per commit
        for (int it = 0; it < iters; ++it) {
            if (!other_warp)
                for (int c = 0; c < copies_per_mma; ++c) copy(sfa + 8u * (uint32_t)(c & 1));
            const uint32_t acc = (uint32_t)it & amask;
            mma_mxf4(tmem + acc * (uint32_t)n, ad, bd, idesc, sfa, sfb, (uint32_t)it > amask ? 1u : 0u);
            if (cper && (it % cper) == cper - 1) tc_commit(tick);
        }
        tc_commit(done);
        wait_done(done);
    } else if (threadIdx.x == 32 && other_warp) {
        for (int it = 0; it < iters; ++it)
            for (int c = 0; c < copies_per_mma; ++c) copy(tmem + 384u + 8u * (uint32_t)(c & 1));
        tc_commit(done2);
        wait_done(done2);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x < 32) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_mxf4_probe(int n, int iters, int copies_per_mma, int variant, int grid,
                              uint32_t* status, cudaStream_t stream) {
    static bool limit_set[64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!limit_set[dev]) {
        err = cudaFuncSetAttribute(moe_mxf4_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)kProbeSmem);
        if (err != cudaSuccess) return err;
        limit_set[dev] = true;
    }
    moe_mxf4_probe_kernel<<<grid, kProbeThreads, kProbeSmem, stream>>>(n, iters, copies_per_mma, variant,
                                                                        status);
    return cudaGetLastError();
}

}  // namespace moe
