// Grouped GEMMs of the MoE forward with bf16 activations and MXFP4 weights
// (W4A16: b12x moe/fused/w4a16/kernel.py, W4A16GemmKernel, which dequantises
// the e2m1 weights and their e8m0 scales in registers and runs bf16 MMAs; the
// bf16-activation path of flower_moe.py, custom_kernel, taken when ksplit > 1;
// solution.py, _reference_forward, is the same arithmetic without kernels).
//
// tcgen05 has no bf16 x e2m1 MMA, so the weights are dequantised to bf16 in
// shared memory and multiplied with tcgen05.mma .kind::f16.  Everything else
// follows the MXFP4 GEMM kernel (gemm.cu): weights on the M = 128 side, route
// tiles on N, both stages in one persistent launch, stage-2 route tiles copied
// once their stage-1 feature tiles are counted, every wait bounded.
//
//   stage 1: acc[m, j] = sum_k W13[row m, k] * x[slot j, k]   (x: bf16 hidden row)
//            h = bf16(silu(g) * u), written in bf16 (no requantisation)
//   stage 2: acc[m, j] = sum_k W2[row m, k] * h[slot j, k];  P[route] = w * acc
// with W = e2m1 * 2^(s - 127), exact in bf16, and fp32 accumulation.
//
// Pipeline (one CTA per SM, 512 threads):
//   warp 0     TMA producer: per stage (128 K elements) the raw weight tile
//              (128 rows x 64 bytes of e2m1) and the bf16 route tile
//              (tile_rows x 256 bytes, 128-byte swizzle) -> ring slot
//   warp 1     MMA: 8 x tcgen05.mma.kind::f16 (K = 16) per stage
//   warp 2     allocates / frees TMEM
//   warps 4-7  epilogue (TMEM lane quadrant = warp % 4)
//   warps 8-15 dequantisation: two threads per weight row expand its 64-element
//              halves of a stage into one of two bf16 tiles (K-major, 128-byte
//              swizzle)
// A ring slot is released when both its consumers are done (the dequantisers
// with the raw weights, the MMAs with the route tile): its `empty` barrier
// counts two arrivals.  Two or three dequantised tiles (three where shared
// memory leaves the ring at least four slots) let the expansion run ahead of
// the MMAs.
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

struct W4Item {
    int e, row0, nrows, f, tile;
};

// bf16 bits of an e8m0 scale byte's 2^(s - 127), twice: exact for every byte
// (s = 0: the subnormal 2^-127), 255 gives NaN.
__device__ __forceinline__ uint32_t w4_scale2(uint32_t s) {
    const uint32_t b = s == 255u ? 0x7fc0u : (s == 0u ? 0x0040u : (s << 7));
    return b | (b << 16);
}

// Four e2m1 codes (16 bits, element i in bits 4i..4i+3) -> four bf16 (two
// bf16x2 words), times the block scale.  The magnitude (3 bits) picks the low
// and the high byte of the bf16 pattern from two 8-byte tables with a byte
// permute (0, 0.5, 1, 1.5, 2, 3, 4, 6 = 0x0000 0x3F00 0x3F80 0x3FC0 0x4000
// 0x4040 0x4080 0x40C0), the sign bit moves to bit 15, and the product with a
// power of two is exact in bf16.
__device__ __forceinline__ void w4_expand4(uint32_t w16, uint32_t sc2, uint32_t& o01, uint32_t& o23) {
    const uint32_t mag = w16 & 0x7777u;
    const uint32_t lo = __byte_perm(0xC0800000u, 0xC0804000u, mag);
    const uint32_t hi = __byte_perm(0x3F3F3F00u, 0x40404040u, mag);
    uint32_t a = __byte_perm(lo, hi, 0x5140u);
    uint32_t b = __byte_perm(lo, hi, 0x7362u);
    a |= ((w16 << 12) & 0x8000u) | ((w16 << 24) & 0x80000000u);
    b |= ((w16 << 4) & 0x8000u) | ((w16 << 16) & 0x80000000u);
    const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162*>(&sc2);
    const __nv_bfloat162 ra = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&a), s2);
    const __nv_bfloat162 rb = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&b), s2);
    o01 = *reinterpret_cast<const uint32_t*>(&ra);
    o23 = *reinterpret_cast<const uint32_t*>(&rb);
}

// Dequantise half hf (64 elements, K-box hf) of weight row m of one stage: 32
// bytes of e2m1 (byte j: element 2j in the low nibble) with 2 scale bytes ->
// 64 bf16 in the K-major 128-byte-swizzled tile [2 K-boxes][128 rows][128 bytes],
// 16-byte chunk c of a row at chunk c ^ (row % 8).
__device__ __forceinline__ void w4_dequant_half(const uint8_t* raw, uint32_t sc_pair, uint8_t* deq_box,
                                                int m) {
    const uint4* src = reinterpret_cast<const uint4*>(raw);
#pragma unroll
    for (int q = 0; q < 2; ++q) {  // 16 bytes = 32 elements = one scale block
        const uint4 r = src[q];
        const uint32_t sc2 = w4_scale2((sc_pair >> (8 * q)) & 0xffu);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {  // 4 bytes = 8 elements = one 16-byte output chunk
            uint32_t o[4];
            w4_expand4(w[h] & 0xffffu, sc2, o[0], o[1]);
            w4_expand4(w[h] >> 16, sc2, o[2], o[3]);
            const int c8 = q * 4 + h;
            *reinterpret_cast<uint4*>(deq_box + m * 128 + ((c8 ^ (m & 7)) * 16)) =
                make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

}  // namespace

// ============================================================== gather
//
// One thread per (token, 16 bytes of its bf16 row): the chunk is loaded once and
// stored to the sorted slot of every valid route of the token.  Launched after
// the routing kernel (dependent launch: the load overlaps it).
constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads)
    moe_gather_bf16_kernel(const uint4* __restrict__ hidden, int T, int K, int D, WsPtrs ws) {
    grid_dep_launch();
    const int nch = D / 8;  // 16-byte chunks per row
    const long gid = (long)blockIdx.x * kGatherThreads + threadIdx.x;
    const bool active = gid < (long)T * nch;
    const int t = active ? (int)(gid / nch) : 0;
    const int c = active ? (int)(gid - (long)t * nch) : 0;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (active) v = __ldg(hidden + (size_t)t * nch + c);
    grid_dep_wait();  // route_pos comes from the routing kernel
    if (!active) return;
    for (int k = 0; k < K; ++k) {
        const int pos = ws.route_pos[t * K + k];
        if (pos >= 0) reinterpret_cast<uint4*>(ws.a1b + (size_t)pos * D)[c] = v;
    }
}

cudaError_t launch_gather_bf16(const void* hidden, int T, int K, int D, const WsPtrs& ws,
                               cudaStream_t stream) {
    const long total = (long)T * (D / 8);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((total + kGatherThreads - 1) / kGatherThreads));
    cfg.blockDim = dim3(kGatherThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_gather_bf16_kernel, static_cast<const uint4*>(hidden), T, K,
                              D, ws);
}

// ============================================================== GEMM kernel

__global__ void __launch_bounds__(kW4Threads, 1)
    moe_w4a16_gemm_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                          const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                          const W4Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const int NS = p.num_stages;
    const int NB = p.deq_bufs;  // dequantised weight tiles (2 or 3)

    // full: raw weights + route tile landed; empty: dequantisers and MMAs done with a
    // slot (2 arrivals); dfull / dempty: a dequantised tile written / consumed;
    // tfull / tempty: an accumulator written / drained.
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    uint64_t* empty = full + kMaxStages;
    uint64_t* dfull = empty + kMaxStages;
    uint64_t* dempty = dfull + kW4MaxDeq;
    uint64_t* tfull = dempty + kW4MaxDeq;
    uint64_t* tempty = tfull + kMaxAccBufs;
    uint64_t* drain = tempty + kMaxAccBufs;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* xg = reinterpret_cast<float*>(smem + p.off_xchg);
    uint8_t* deq = smem + p.off_deq;
    uint32_t* status = p.ws.status;

    grid_dep_launch();
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 2);
        }
        for (int b = 0; b < NB; ++b) {
            mbar_init(&dfull[b], 1);
            mbar_init(&dempty[b], 1);
        }
        for (int a = 0; a < p.acc_bufs; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA1);
        tma_prefetch_desc(&tmB1);
        tma_prefetch_desc(&tmA2);
        tma_prefetch_desc(&tmB2);
    }
    grid_dep_wait();  // routing, gathered rows (and TMEM of earlier kernels) are ready
    const int num_tiles = __ldcg(p.ws.num_valid + 2);
    const int nitems[2] = {num_tiles * p.n_ftiles1, num_tiles * p.n_ftiles2};
    const int G = (int)gridDim.x;
    const int b0 = (int)blockIdx.x;
    if (b0 >= nitems[0] && b0 >= nitems[1]) return;
    int4* tcache = reinterpret_cast<int4*>(smem + p.off_tiles);
    for (int i = (int)threadIdx.x; i < num_tiles && i < kTileCache; i += kW4Threads)
        tcache[i] = __ldcg(p.ws.tiles + i);
    if (warp == 2) {
        tmem_alloc(tmem_slot, p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // item it of stage phs (round-robin over the CTAs): route tile, feature tile
    auto item = [&](int phs, int it) -> W4Item {
        const int nft = phs ? p.n_ftiles2 : p.n_ftiles1;
        W4Item x;
        x.tile = it / nft;
        x.f = it - x.tile * nft;
        const int4 t = x.tile < kTileCache ? tcache[x.tile] : __ldcg(p.ws.tiles + x.tile);
        x.e = t.x;
        x.row0 = t.y;
        x.nrows = t.z;
        return x;
    };
    const uint32_t b_box = (uint32_t)p.tile_rows * 128u;  // bytes per K-box of a route tile

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            uint32_t issued = 0, last_ph = 0;
            int ready_tile = -1;
            for (int phs = 0; phs < 2 && ok; ++phs) {
                const int kst = phs ? p.kstages2 : p.kstages1;
                for (int it = b0; it < nitems[phs] && ok; it += G) {
                    const W4Item x = item(phs, it);
                    for (int ks = 0; ks < kst; ++ks) {
                        if (!mbar_wait(&empty[s], ph ^ 1u, status, kErrTimeoutEmpty, abort_flag)) {
                            ok = false;
                            break;
                        }
                        uint8_t* st = smem + (size_t)s * p.slot_bytes;
                        mbar_arrive_expect_tx(&full[s], kW4RawBytes + (uint32_t)p.tile_rows * 256u);
                        if (phs == 0) {
                            // 64 gate rows, then the 64 matching up rows (I rows further)
                            const int rg = x.e * 2 * p.I + x.f * 64;
                            tma_load_2d_hint(st, &tmA1, ks * 64, rg, &full[s], pol_w);
                            tma_load_2d_hint(st + kW4RawBytes / 2, &tmA1, ks * 64, rg + p.I, &full[s], pol_w);
                        } else {
                            tma_load_2d_hint(st, &tmA2, ks * 64, x.e * p.D + x.f * 128, &full[s], pol_w);
                            if (x.tile != ready_tile) {
                                // every stage-1 feature tile of this route tile written
                                const uint32_t need = (uint32_t)p.n_ftiles1;
                                const uint64_t t0 = globaltimer_ns();
                                bool got = false;
                                for (uint32_t n = 0;; ++n) {
                                    if (ld_relaxed_gpu(p.ws.tile_done + x.tile) >= need &&
                                        ld_acquire_gpu(p.ws.tile_done + x.tile) >= need) {
                                        got = true;
                                        break;
                                    }
                                    if ((n & 63u) == 63u) {
                                        if (*abort_flag) break;
                                        if (globaltimer_ns() - t0 > kWaitLimitNs) {
                                            atomicOr(status, kErrTimeoutTile);
                                            *abort_flag = 1;
                                            break;
                                        }
                                    }
                                }
                                // the copy below is issued either way so that the stage completes
                                if (got) {
                                    fence_proxy_async_global();
                                    ready_tile = x.tile;
                                } else {
                                    ok = false;
                                }
                            }
                        }
                        // route tile: tile_rows sorted slots x 2 K-boxes of 64 bf16
                        tma_load_3d(st + kW4RawBytes, phs ? &tmB2 : &tmB1, 0, x.row0, ks * 2, &full[s]);
                        issued |= 1u << s;
                        last_ph = (last_ph & ~(1u << s)) | (ph << s);
                        if (++s == NS) {
                            s = 0;
                            ph ^= 1u;
                        }
                        if (!ok) break;
                    }
                }
            }
            if (!ok) {
                for (int i = 0; i < NS; ++i) {
                    if (!((issued >> i) & 1u)) continue;
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(smem_u32(&full[i]), (last_ph >> i) & 1u)) {
                        if (globaltimer_ns() - t0 > kWaitLimitNs) {
                            atomicOr(status, kErrTimeoutDrain);
                            break;
                        }
                    }
                }
            }
        }
    }
    if (warp == 1) {
        // ------------------------------------------------------------ MMA
        int s = 0, b = 0, a = 0;
        uint32_t ph = 0, bph = 0, aph = 0;
        bool ok = true;
        bool any = false;  // this thread issued MMAs (drained on abort)
        for (int phs = 0; phs < 2 && ok; ++phs) {
            const int kst = phs ? p.kstages2 : p.kstages1;
            for (int it = b0; it < nitems[phs] && ok; it += G) {
                const W4Item x = item(phs, it);
                if (!mbar_wait_warp(&tempty[a], aph ^ 1u, status, kErrTimeoutTmemEmpty, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(a * p.tile_rows);
                const uint32_t idesc = bf16_idesc(128, (uint32_t)x.nrows);
                for (int ks = 0; ks < kst; ++ks) {
                    if (!mbar_wait_warp(&full[s], ph, status, kErrTimeoutFull, abort_flag) ||
                        !mbar_wait_warp(&dfull[b], bph, status, kErrTimeoutFull, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        tc_fence_after();
                        const uint64_t ad0 = smem_desc(smem_u32(deq + (size_t)b * kW4DeqBytes), 16, 1024, 2);
                        const uint64_t bd0 =
                            smem_desc(smem_u32(smem + (size_t)s * p.slot_bytes + kW4RawBytes), 16, 1024, 2);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {  // K = 16 per MMA, 4 per 128-byte K-box
                            const uint32_t kbox = (uint32_t)i >> 2, kk = (uint32_t)i & 3u;
                            mma_bf16(d, ad0 + (uint64_t)(kbox * ((128u * 128u) >> 4) + kk * 2u),
                                     bd0 + (uint64_t)(kbox * (b_box >> 4) + kk * 2u), idesc,
                                     (ks > 0 || i > 0) ? 1u : 0u);
                        }
                        tc_commit(&empty[s]);
                        tc_commit(&dempty[b]);
                        any = true;
                    }
                    __syncwarp();
                    if (++s == NS) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (++b == NB) {
                        b = 0;
                        bph ^= 1u;
                    }
                }
                if (!ok) break;
                if (lane == 0) tc_commit(&tfull[a]);
                __syncwarp();
                if (++a == p.acc_bufs) {
                    a = 0;
                    aph ^= 1u;
                }
            }
        }
        if (!ok && lane == 0 && any) {
            tc_commit(drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(drain), 0)) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    atomicOr(status, kErrTimeoutDrain);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp >= 8) {
        // ------------------------------------------------------------ dequantisation
        const int dt = (int)threadIdx.x - 256;
        const int m = dt & 127;   // weight row of the tile
        const int hf = dt >> 7;   // which 64 elements (K-box) of the stage
        int s = 0, b = 0;
        uint32_t ph = 0, bph = 0;
        bool ok = true;
        for (int phs = 0; phs < 2 && ok; ++phs) {
            const int kst = phs ? p.kstages2 : p.kstages1;
            const int srow = phs ? p.I / 32 : p.D / 32;  // scale bytes per weight row
            for (int it = b0; it < nitems[phs] && ok; it += G) {
                const W4Item x = item(phs, it);
                const size_t rowg = phs ? (size_t)x.e * p.D + (size_t)x.f * 128 + m
                                        : (size_t)x.e * 2 * p.I + (size_t)(m < 64 ? 0 : p.I) +
                                              (size_t)x.f * 64 + (m & 63);
                const uint32_t* srow_p =
                    reinterpret_cast<const uint32_t*>((phs ? p.w2_scale : p.w13_scale) + rowg * srow);
                for (int ks = 0; ks < kst; ++ks) {
                    const uint32_t sc_pair = __ldg(srow_p + ks) >> (16 * hf);  // this half's 2 scales
                    if (!mbar_wait_warp(&full[s], ph, status, kErrTimeoutFull, abort_flag) ||
                        !mbar_wait_warp(&dempty[b], bph ^ 1u, status, kErrTimeoutFull, abort_flag)) {
                        ok = false;
                        break;
                    }
                    w4_dequant_half(smem + (size_t)s * p.slot_bytes + m * 64 + hf * 32, sc_pair,
                                    deq + (size_t)b * kW4DeqBytes + hf * (128 * 128), m);
                    fence_proxy_async_smem();  // the MMAs read the tile through the async proxy
                    named_bar_sync(5, 256);
                    if (dt == 0) {
                        mbar_arrive(&dfull[b]);
                        mbar_arrive(&empty[s]);
                    }
                    if (++s == NS) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (++b == NB) {
                        b = 0;
                        bph ^= 1u;
                    }
                }
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const uint32_t q4 = warp & 3u;
        const int R = p.R;
        int a = 0;
        uint32_t aph = 0;
        bool ok = true;
        const int tq = (int)(q4 * 32u + lane);
        const int ri = tq >> 4, bb = (tq >> 3) & 1, sub = tq & 7;
        for (int phs = 0; phs < 2 && ok; ++phs) {
            for (int it = b0; it < nitems[phs] && ok; it += G) {
                const W4Item x = item(phs, it);
                const int slot0 = x.row0 + (int)(lane & 15);
                const int rid_pre = __ldg(p.ws.sorted_ids + slot0);
                const float w_pre = phs == 1 ? __ldg(p.ws.sorted_w + slot0) : 0.0f;
                if (!mbar_wait_warp(&tfull[a], aph, status, kErrTimeoutTmemFull, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tacc = tmem_base + ((q4 * 32u) << 16) + (uint32_t)(a * p.tile_rows);
                const int nchunks = x.nrows / 16;
                auto release = [&]() {
                    tc_fence_before();
                    mbar_arrive(&tempty[a]);
                };
                bool released = false;
                if (phs == 0) {
                    // rows 0-63 gate, 64-127 up of features x.f*64 + 0..63; per chunk of
                    // 16 routes in two halves of 8 through the exchange buffer, thread t
                    // takes route t / 16, feature block (t / 8) % 2 and its 4 features
                    const int feat0 = x.f * 64 + 32 * bb;
                    for (int c = 0; c < nchunks; ++c) {
                        float v[16];
                        tmem_ld16(tacc + 16u * c, v);
                        tmem_ld_wait();
                        if (c + 1 == nchunks) {
                            release();
                            released = true;
                        }
                        const int rid_l = c == 0 ? rid_pre : __ldg(p.ws.sorted_ids + x.row0 + 16 * c + (int)(lane & 15));
                        const uint32_t valid = __ballot_sync(0xffffffffu, rid_l < R);
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            if (((valid >> (8 * hh)) & 0xffu) == 0u) continue;  // all padding
#pragma unroll
                            for (int i = 0; i < 8; ++i) xg[(q4 * 8 + i) * 32 + lane] = v[8 * hh + i];
                            named_bar_sync(1, 128);
                            const float4 g4 = *reinterpret_cast<const float4*>(xg + (bb * 8 + ri) * 32 + sub * 4);
                            const float4 u4 = *reinterpret_cast<const float4*>(xg + ((2 + bb) * 8 + ri) * 32 + sub * 4);
                            const float gs[4] = {g4.x, g4.y, g4.z, g4.w};
                            const float us[4] = {u4.x, u4.y, u4.z, u4.w};
                            float hv[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j) hv[j] = (gs[j] / (1.0f + expf(-gs[j]))) * us[j];
                            const __nv_bfloat162 h01 = __floats2bfloat162_rn(hv[0], hv[1]);
                            const __nv_bfloat162 h23 = __floats2bfloat162_rn(hv[2], hv[3]);
                            const int rid = __shfl_sync(0xffffffffu, rid_l, 8 * hh + ri);
                            const int slot = x.row0 + 16 * c + 8 * hh + ri;
                            if (rid < R)
                                *reinterpret_cast<uint2*>(p.ws.a2b + (size_t)slot * p.I + feat0 + sub * 4) =
                                    make_uint2(*reinterpret_cast<const uint32_t*>(&h01),
                                               *reinterpret_cast<const uint32_t*>(&h23));
                            named_bar_sync(1, 128);  // the buffer is refilled next
                        }
                    }
                    // the feature tile is written: count it for the stage-2 route-tile copies
                    fence_proxy_async_global();
                    named_bar_sync(1, 128);
                    if (q4 == 0 && lane == 0) {
                        __threadfence();
                        if (atomicAdd(p.ws.tile_done + x.tile, 1u) >= (uint32_t)p.n_ftiles1)
                            atomicOr(status, kErrCounterState);
                    }
                } else {
                    const int n = x.f * 128 + 32 * (int)q4 + (int)lane;  // output feature of this lane
                    for (int c = 0; c < nchunks; ++c) {
                        float v[16];
                        tmem_ld16(tacc + 16u * c, v);
                        tmem_ld_wait();
                        if (c + 1 == nchunks) {
                            release();
                            released = true;
                        }
                        int rid_l = rid_pre;
                        float w_l = w_pre;
                        if (c > 0) {
                            const int sl = x.row0 + 16 * c + (int)(lane & 15);
                            rid_l = __ldg(p.ws.sorted_ids + sl);
                            w_l = __ldg(p.ws.sorted_w + sl);
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int rid = __shfl_sync(0xffffffffu, rid_l, i);
                            const float wv = __shfl_sync(0xffffffffu, w_l, i);
                            if (rid < R) p.ws.P[(size_t)rid * p.D + n] = wv * v[i];
                        }
                    }
                }
                if (!released) release();
                if (++a == p.acc_bufs) {
                    a = 0;
                    aph ^= 1u;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tmem_base, p.tmem_cols);
}

cudaError_t launch_w4a16_gemm(const CUtensorMap* maps, const W4Params& p, int grid,
                              cudaStream_t stream) {
    static bool limit_set[64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!limit_set[dev]) {
        err = cudaFuncSetAttribute(moe_w4a16_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kGemmSmemLimit);
        if (err != cudaSuccess) return err;
        limit_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kW4Threads);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_w4a16_gemm_kernel, maps[0], maps[1], maps[2], maps[3], p);
}

}  // namespace moe
