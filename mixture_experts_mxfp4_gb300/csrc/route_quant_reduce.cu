// Routing (counting sort of routes by expert), dynamic MXFP4 quantisation of
// the hidden states with the scatter into sorted order, and the per-token
// deterministic top-k sum.
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {

// ============================================================== routing
//
// One CTA of 1024 threads.  Structure from kernelbot-amd-moe-mxfp4-723815
// (solution.py: kernel_count_tokens -> kernel_prefix_sum -> kernel_scatter_tokens)
// with block_m padding per expert and per-block expert ids as in
// kernelbot-amd-moe-mxfp4-754773 (flower_moe.py: moe_sorting_fwd buffers), the
// route id t*topk+k and sentinel T*topk of b12x moe/fused/w4a16/kernel.py
// (_read_moe_block_data).  Deterministic: each warp owns a contiguous chunk of
// routes; a per-warp, per-expert histogram and its prefix over warps give every
// route its rank, so routes appear in ascending route id within an expert.

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;

// Inclusive scan over the 1024 threads of two values at once.
__device__ __forceinline__ void block_scan2(int& a, int& b, int* wsum_a, int* wsum_b) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int ta = __shfl_up_sync(0xffffffffu, a, o);
        const int tb = __shfl_up_sync(0xffffffffu, b, o);
        if (lane >= o) {
            a += ta;
            b += tb;
        }
    }
    if (lane == 31) {
        wsum_a[warp] = a;
        wsum_b[warp] = b;
    }
    __syncthreads();
    if (warp == 0) {
        int xa = wsum_a[lane], xb = wsum_b[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ta = __shfl_up_sync(0xffffffffu, xa, o);
            const int tb = __shfl_up_sync(0xffffffffu, xb, o);
            if (lane >= o) {
                xa += ta;
                xb += tb;
            }
        }
        wsum_a[lane] = xa;
        wsum_b[lane] = xb;
    }
    __syncthreads();
    if (warp > 0) {
        a += wsum_a[warp - 1];
        b += wsum_b[warp - 1];
    }
}

__global__ void __launch_bounds__(kRouteThreads, 1)
    moe_route_kernel(const int32_t* __restrict__ topk_ids, const float* __restrict__ topk_w,
                     int T, int K, int E, int tile_rows, int cap, int n_counters, WsPtrs ws) {
    extern __shared__ int route_smem[];
    int* hist = route_smem;                 // [32][E]: per-warp counts, then prefixes
    int* seg = hist + kRouteWarps * E;      // [E + 1]
    int* wsum = seg + (E + 1);              // [64]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int R = T * K;
    const int bm = kBlockM;
    grid_dep_launch();

    for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) hist[i] = 0;
    for (int i = tid; i < n_counters; i += kRouteThreads) ws.counters[i] = 0;
    if (tid < 16) ws.status[tid] = 0;
    __syncthreads();

    const int chunk = (R + kRouteWarps - 1) / kRouteWarps;
    const int r_begin = min(warp * chunk, R);
    const int r_end = min(r_begin + chunk, R);

    // Pass 1: per-warp histogram (one leader per distinct expert in a batch).
    for (int base = r_begin; base < r_end; base += 32) {
        const int r = base + lane;
        const int e = (r < r_end) ? topk_ids[r] : -1;
        const bool valid = (r < r_end) && e >= 0 && e < E;
        const int key = valid ? e : -1;
        const uint32_t m = __match_any_sync(0xffffffffu, key);
        if (valid && lane == __ffs(m) - 1) hist[warp * E + e] += __popc(m);
        __syncwarp();
    }
    __syncthreads();

    // Per expert: prefix over warps, padded length, tiles.
    int cnt = 0, padded = 0, ntiles = 0;
    if (tid < E) {
        int run = 0;
        for (int w = 0; w < kRouteWarps; ++w) {
            const int c = hist[w * E + tid];
            hist[w * E + tid] = run;
            run += c;
        }
        cnt = run;
        padded = (cnt + bm - 1) / bm * bm;
        ntiles = (padded + tile_rows - 1) / tile_rows;
    }
    int seg_incl = padded, tile_incl = ntiles;
    block_scan2(seg_incl, tile_incl, wsum, wsum + 32);
    const int seg_e = seg_incl - padded, tile_e = tile_incl - ntiles;
    if (tid < E) seg[tid] = seg_e;
    if (tid == kRouteThreads - 1) seg[E] = seg_incl;  // total padded length
    __shared__ int s_totals[2];
    if (tid == kRouteThreads - 1) {
        s_totals[0] = seg_incl;
        s_totals[1] = tile_incl;
    }
    int valid_incl = cnt, dummy = 0;
    __syncthreads();
    block_scan2(valid_incl, dummy, wsum, wsum + 32);
    const int total_padded = s_totals[0], total_tiles = s_totals[1];

    if (tid < E) ws.seg_start[tid] = seg[tid];
    if (tid == 0) ws.seg_start[E] = seg[E];  // (E may equal the thread count)
    if (tid < E && cnt > 0 && moe_check(tile_e + ntiles <= n_counters && seg_e + padded <= cap, ws.status)) {
        for (int j = 0; j < ntiles; ++j) {
            const int rows = min(tile_rows, padded - j * tile_rows);
            ws.tiles[tile_e + j] = make_int4(tid, seg_e + j * tile_rows, rows, 0);
        }
        for (int b = seg_e / bm; b < (seg_e + padded) / bm; ++b) ws.block_expert[b] = tid;
        for (int p = seg_e + cnt; p < seg_e + padded; ++p) {
            ws.sorted_ids[p] = R;
            ws.sorted_w[p] = 0.0f;
        }
    }
    for (int p = total_padded + tid; p < cap; p += kRouteThreads) {
        ws.sorted_ids[p] = R;
        ws.sorted_w[p] = 0.0f;
    }
    for (int b = total_padded / bm + tid; b < cap / bm; b += kRouteThreads) ws.block_expert[b] = -1;
    if (tid == kRouteThreads - 1) {
        ws.num_valid[0] = total_padded;
        ws.num_valid[1] = valid_incl;
        ws.num_valid[2] = total_tiles;
        ws.num_valid[3] = 0;
    }

    // Pass 2: scatter in the same order; rank = warp prefix + rank in batch.
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int base = r_begin; base < r_end; base += 32) {
        const int r = base + lane;
        const int e = (r < r_end) ? topk_ids[r] : -1;
        const bool valid = (r < r_end) && e >= 0 && e < E;
        const int key = valid ? e : -1;
        const uint32_t m = __match_any_sync(0xffffffffu, key);
        if (valid) {
            const int pos = seg[e] + hist[warp * E + e] + __popc(m & lt_mask);
            if (moe_check(pos >= 0 && pos < cap, ws.status)) {
                ws.sorted_ids[pos] = r;
                ws.sorted_w[pos] = topk_w[r];
                ws.route_pos[r] = pos;
            }
        } else if (r < r_end) {
            ws.route_pos[r] = -1;
        }
        __syncwarp();
        if (valid && lane == __ffs(m) - 1) hist[warp * E + e] += __popc(m);
        __syncwarp();
    }
}

// ============================================================== routing over many CTAs
//
// For large batches the same layout in three launches: per-CTA expert counts
// of contiguous route chunks, one CTA that turns them into segment and per-chunk
// offsets (and writes everything the one-CTA kernel writes except the routes'
// own slots), then every CTA scatters its chunk.  The order is the one-CTA
// kernel's: a chunk's routes precede the next chunk's, and inside a chunk the
// per-warp ranks are as there.  The per-chunk counts live in the P region,
// which the stage-2 GEMM overwrites later.

constexpr int kRouteMaxChunks = 144;
constexpr int kChunkThreads = 256;
constexpr int kChunkWarps = kChunkThreads / 32;
constexpr int kScanBatch = 12;  // per-chunk counts a scan thread loads at once

// Per-warp expert histogram of routes [c0, c1) (contiguous sub-chunk per warp)
// into hist[kChunkWarps][E] (zeroed by the caller); whole CTA.
__device__ __forceinline__ void chunk_histogram(const int32_t* __restrict__ topk_ids, int c0, int c1,
                                                int E, int* hist, int& r_begin, int& r_end) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int wchunk = (c1 - c0 + kChunkWarps - 1) / kChunkWarps;
    r_begin = min(c0 + warp * wchunk, c1);
    r_end = min(r_begin + wchunk, c1);
    for (int base = r_begin; base < r_end; base += 32) {
        const int r = base + lane;
        const int e = (r < r_end) ? topk_ids[r] : -1;
        const bool valid = (r < r_end) && e >= 0 && e < E;
        const uint32_t m = __match_any_sync(0xffffffffu, valid ? e : -1);
        if (valid && lane == __ffs(m) - 1) hist[warp * E + e] += __popc(m);
        __syncwarp();
    }
}

__global__ void __launch_bounds__(kChunkThreads)
    moe_route_count_kernel(const int32_t* __restrict__ topk_ids, int R, int E, int chunk,
                           int* __restrict__ ccount) {
    extern __shared__ int cs_smem[];
    int* hist = cs_smem;  // [kChunkWarps][E]
    grid_dep_launch();
    for (int i = threadIdx.x; i < kChunkWarps * E; i += kChunkThreads) hist[i] = 0;
    __syncthreads();
    const int c0 = min((int)blockIdx.x * chunk, R), c1 = min(c0 + chunk, R);
    int rb, re;
    chunk_histogram(topk_ids, c0, c1, E, hist, rb, re);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kChunkThreads) {
        int sum = 0;
        for (int w = 0; w < kChunkWarps; ++w) sum += hist[w * E + e];
        ccount[(size_t)blockIdx.x * E + e] = sum;
    }
}

// One CTA of kRouteThreads: expert totals over the C chunks, the padded segment
// layout (as moe_route_kernel), and ccount[c][e] replaced by the first slot of
// chunk c's routes of expert e.
__global__ void __launch_bounds__(kRouteThreads, 1)
    moe_route_scan_kernel(int C, int T, int K, int E, int tile_rows, int cap, int n_counters,
                          int* __restrict__ ccount, WsPtrs ws) {
    __shared__ int seg[1025];
    __shared__ int wsum[64];
    __shared__ int s_totals[2];
    const int tid = threadIdx.x;
    const int R = T * K;
    const int bm = kBlockM;
    grid_dep_launch();
    grid_dep_wait();  // the chunk counts
    for (int i = tid; i < n_counters; i += kRouteThreads) ws.counters[i] = 0;
    if (tid < 16) ws.status[tid] = 0;

    int cnt = 0, padded = 0, ntiles = 0;
    if (tid < E) {
        for (int c0 = 0; c0 < C; c0 += kScanBatch) {
            int v[kScanBatch];
#pragma unroll
            for (int i = 0; i < kScanBatch; ++i) v[i] = (c0 + i < C) ? ccount[(size_t)(c0 + i) * E + tid] : 0;
#pragma unroll
            for (int i = 0; i < kScanBatch; ++i) cnt += v[i];
        }
        padded = (cnt + bm - 1) / bm * bm;
        ntiles = (padded + tile_rows - 1) / tile_rows;
    }
    int seg_incl = padded, tile_incl = ntiles;
    block_scan2(seg_incl, tile_incl, wsum, wsum + 32);
    const int seg_e = seg_incl - padded, tile_e = tile_incl - ntiles;
    if (tid < E) seg[tid] = seg_e;
    if (tid == kRouteThreads - 1) {
        seg[E] = seg_incl;
        s_totals[0] = seg_incl;
        s_totals[1] = tile_incl;
    }
    int valid_incl = cnt, dummy = 0;
    __syncthreads();
    block_scan2(valid_incl, dummy, wsum, wsum + 32);
    const int total_padded = s_totals[0], total_tiles = s_totals[1];

    if (tid < E) ws.seg_start[tid] = seg[tid];
    if (tid == 0) ws.seg_start[E] = seg[E];  // (E may equal the thread count)
    if (tid < E) {
        // chunk c's routes of this expert start after the earlier chunks' ones
        int run = seg_e;
        for (int c0 = 0; c0 < C; c0 += kScanBatch) {
            int v[kScanBatch];
#pragma unroll
            for (int i = 0; i < kScanBatch; ++i) v[i] = (c0 + i < C) ? ccount[(size_t)(c0 + i) * E + tid] : 0;
#pragma unroll
            for (int i = 0; i < kScanBatch; ++i) {
                if (c0 + i < C) ccount[(size_t)(c0 + i) * E + tid] = run;
                run += v[i];
            }
        }
    }
    if (tid < E && cnt > 0 && moe_check(tile_e + ntiles <= n_counters && seg_e + padded <= cap, ws.status)) {
        for (int j = 0; j < ntiles; ++j) {
            const int rows = min(tile_rows, padded - j * tile_rows);
            ws.tiles[tile_e + j] = make_int4(tid, seg_e + j * tile_rows, rows, 0);
        }
        for (int b = seg_e / bm; b < (seg_e + padded) / bm; ++b) ws.block_expert[b] = tid;
        for (int p = seg_e + cnt; p < seg_e + padded; ++p) {
            ws.sorted_ids[p] = R;
            ws.sorted_w[p] = 0.0f;
        }
    }
    for (int p = total_padded + tid; p < cap; p += kRouteThreads) {
        ws.sorted_ids[p] = R;
        ws.sorted_w[p] = 0.0f;
    }
    for (int b = total_padded / bm + tid; b < cap / bm; b += kRouteThreads) ws.block_expert[b] = -1;
    if (tid == kRouteThreads - 1) {
        ws.num_valid[0] = total_padded;
        ws.num_valid[1] = valid_incl;
        ws.num_valid[2] = total_tiles;
        ws.num_valid[3] = 0;
    }
}

// Every CTA: its chunk's routes to their slots (ids, weights, route_pos).
__global__ void __launch_bounds__(kChunkThreads)
    moe_route_scatter_kernel(const int32_t* __restrict__ topk_ids, const float* __restrict__ topk_w,
                             int R, int E, int chunk, int cap, const int* __restrict__ ccount, WsPtrs ws) {
    extern __shared__ int cs_smem[];
    int* hist = cs_smem;  // [kChunkWarps][E]: counts, then first slots per warp
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    grid_dep_launch();
    for (int i = threadIdx.x; i < kChunkWarps * E; i += kChunkThreads) hist[i] = 0;
    __syncthreads();
    const int c0 = min((int)blockIdx.x * chunk, R), c1 = min(c0 + chunk, R);
    int r_begin, r_end;
    chunk_histogram(topk_ids, c0, c1, E, hist, r_begin, r_end);
    grid_dep_wait();  // the per-chunk first slots from the scan kernel
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kChunkThreads) {
        int run = ccount[(size_t)blockIdx.x * E + e];
        for (int w = 0; w < kChunkWarps; ++w) {
            const int c = hist[w * E + e];
            hist[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int base = r_begin; base < r_end; base += 32) {
        const int r = base + lane;
        const int e = (r < r_end) ? topk_ids[r] : -1;
        const bool valid = (r < r_end) && e >= 0 && e < E;
        const uint32_t m = __match_any_sync(0xffffffffu, valid ? e : -1);
        if (valid) {
            const int pos = hist[warp * E + e] + __popc(m & lt_mask);
            if (moe_check(pos >= 0 && pos < cap, ws.status)) {
                ws.sorted_ids[pos] = r;
                ws.sorted_w[pos] = topk_w[r];
                ws.route_pos[r] = pos;
            }
        } else if (r < r_end) {
            ws.route_pos[r] = -1;
        }
        __syncwarp();
        if (valid && lane == __ffs(m) - 1) hist[warp * E + e] += __popc(m);
        __syncwarp();
    }
}

cudaError_t launch_route(const int32_t* topk_ids, const float* topk_w, int T, int K, int E,
                         int tile_rows, int cap, int n_counters, const WsPtrs& ws,
                         cudaStream_t stream) {
    const int R = T * K;
    if (R >= kRouteMultiMin) {
        // count -> scan -> scatter; the per-chunk counts go to the P region
        // (R * D floats >= C * E ints: R >= 4096, D >= 128, C <= 144, E <= 1024)
        const int C = min(kRouteMaxChunks, (R + 1023) / 1024);
        const int chunk = (R + C - 1) / C;
        int* ccount = reinterpret_cast<int*>(ws.P);
        const size_t csmem = sizeof(int) * (size_t)kChunkWarps * E;
        moe_route_count_kernel<<<C, kChunkThreads, csmem, stream>>>(topk_ids, R, E, chunk, ccount);
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.stream = stream;
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(kRouteThreads);
        cfg.dynamicSmemBytes = 0;
        err = cudaLaunchKernelEx(&cfg, moe_route_scan_kernel, C, T, K, E, tile_rows, cap, n_counters,
                                 ccount, ws);
        if (err != cudaSuccess) return err;
        cfg.gridDim = dim3((unsigned)C);
        cfg.blockDim = dim3(kChunkThreads);
        cfg.dynamicSmemBytes = csmem;
        return cudaLaunchKernelEx(&cfg, moe_route_scatter_kernel, topk_ids, topk_w, R, E, chunk, cap,
                                  static_cast<const int*>(ccount), ws);
    }
    const size_t smem = sizeof(int) * ((size_t)kRouteWarps * E + (E + 1) + 64);
    // limit raised once per device to what E <= 1024 can need
    static bool limit_set[64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!limit_set[dev]) {
        const int max_smem = (int)(sizeof(int) * ((size_t)kRouteWarps * 1024 + 1025 + 64));
        err = cudaFuncSetAttribute(moe_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   max_smem);
        if (err != cudaSuccess) return err;
        limit_set[dev] = true;
    }
    moe_route_kernel<<<1, kRouteThreads, smem, stream>>>(topk_ids, topk_w, T, K, E, tile_rows,
                                                         cap, n_counters, ws);
    return cudaGetLastError();
}

// ============================================================== quant + scatter
//
// One thread per (token, 32-element block): the block (64 bytes of bf16, four
// 16-byte loads) is quantised once, then its 16 code bytes and scale byte are
// written to the sorted slot of every valid route of the token (the token's
// activation is quantised once per token, as flower_moe.py does with topk=1
// for the hidden states).  The loads and the quantisation run before the
// routing kernel has finished (dependent launch); only the scatter waits.

constexpr int kQuantThreads = 256;

// e2m1 codes of two values already divided by the block scale, packed as one
// byte (lo in the low nibble): the conversion instruction rounds to nearest,
// ties to even, and saturates at +-6, which is the quantiser's rule (checked on
// the GPU against that rule for every finite bf16 value, exact ties and signed
// zeros included).
__device__ __forceinline__ uint32_t e2m1x2_rn(float hi, float lo) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

__global__ void __launch_bounds__(kQuantThreads)
    moe_quant_kernel(const __nv_bfloat16* __restrict__ hidden, int T, int K, int D, int Dl,
                     int a1s_stride, int cap, WsPtrs ws) {
    grid_dep_launch();
    const int nblk = D / 32;
    const long gid = (long)blockIdx.x * kQuantThreads + threadIdx.x;
    const bool active = gid < (long)T * nblk;
    const int t = active ? (int)(gid / nblk) : 0;
    const int g = active ? (int)(gid - (long)t * nblk) : 0;
    uint4 codes = make_uint4(0, 0, 0, 0);  // (padding blocks past Dl stay zero, scale 0)
    uint32_t s = 0;
    if (active && g < Dl / 32) {
        const uint4* src = reinterpret_cast<const uint4*>(hidden + (size_t)t * Dl) + g * 4;
        uint4 raw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) raw[i] = __ldg(src + i);
        const uint32_t* w = reinterpret_cast<const uint32_t*>(raw);
        float v[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
        uint32_t amax = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = max(amax, __float_as_uint(v[i]) & 0x7fffffffu);
        s = mx_scale_byte(amax);
        uint32_t packed[4] = {0, 0, 0, 0};
        if (s == 255u) {  // a NaN/Inf in the block: signed zeros
#pragma unroll
            for (int i = 0; i < 32; ++i)
                packed[i / 8] |= ((__float_as_uint(v[i]) >> 31) << 3) << (4 * (i % 8));
        } else {
            const float inv = mx_inv_scale(s);
#pragma unroll
            for (int j = 0; j < 16; ++j)  // elements 2j, 2j+1: byte j % 4 of word j / 4
                packed[j / 4] |= e2m1x2_rn(v[2 * j + 1] * inv, v[2 * j] * inv) << (8 * (j % 4));
        }
        codes = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
    grid_dep_wait();  // route_pos comes from the routing kernel
    if (!active) return;
    for (int k = 0; k < K; ++k) {
        const int pos = ws.route_pos[t * K + k];
        if (pos >= 0 && moe_check(pos < cap, ws.status)) {
            *reinterpret_cast<uint4*>(ws.a1q + (size_t)pos * (D / 2) + g * 16) = codes;
            ws.a1s[(size_t)pos * a1s_stride + g] = (uint8_t)s;
        }
    }
}

cudaError_t launch_quant(const void* hidden, int T, int K, int D, int Dl, int a1s_stride, int cap,
                         const WsPtrs& ws, cudaStream_t stream) {
    const long total = (long)T * (D / 32);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((total + kQuantThreads - 1) / kQuantThreads));
    cfg.blockDim = dim3(kQuantThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_quant_kernel,
                              reinterpret_cast<const __nv_bfloat16*>(hidden), T, K, D, Dl,
                              a1s_stride, cap, ws);
}

// ============================================================== top-k sum
//
// out[t, n] = bf16( sum over k ascending of P[t*K + k, n] ) over the routes of
// token t whose expert id is in [0, E) (route_pos >= 0: the routing kernel's map,
// so the ids are not read again), for the Dl logical columns (P rows hold D).
// P already holds w[t,k] * y (stage-2 epilogue).  Deterministic: one thread owns
// four outputs and adds the routes' values in k order in fp32 from zero, rounded
// once.  A token without a valid route gets a zero row.

__global__ void __launch_bounds__(256)
    moe_reduce_kernel(const int32_t* __restrict__ route_pos, int T, int K, int D, int Dl,
                      const float* __restrict__ P, __nv_bfloat16* __restrict__ out) {
    grid_dep_launch();
    grid_dep_wait();  // P comes from the stage-2 GEMM, route_pos from routing
    const int n4 = Dl / 4;
    const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long)T * n4) return;
    const int t = (int)(idx / n4);
    const int c = (int)(idx - (long)t * n4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < K; ++k) {
        if (__ldg(route_pos + t * K + k) < 0) continue;
        const float4 v = __ldcs(reinterpret_cast<const float4*>(P + ((size_t)t * K + k) * D) + c);
        acc.x = acc.x + v.x;
        acc.y = acc.y + v.y;
        acc.z = acc.z + v.z;
        acc.w = acc.w + v.w;
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + (size_t)t * Dl + 4 * c) = pk;
}

cudaError_t launch_reduce(int T, int K, int D, int Dl, void* out, const WsPtrs& ws,
                          cudaStream_t stream) {
    const long total = (long)T * (Dl / 4);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((total + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_reduce_kernel, static_cast<const int32_t*>(ws.route_pos), T, K,
                              D, Dl, static_cast<const float*>(ws.P), reinterpret_cast<__nv_bfloat16*>(out));
}

// ============================================================== run-width copies
//
// A call whose weight widths the GEMM kernels do not run at as they are (they
// run d_model, d_inter at the next width of 128, 256 or a multiple of 512): one
// warp per row copies each weight-scale row of S bytes into a row of Sp bytes (a
// multiple of 16, as the tensor-memory-access copies need), the extra bytes 127
// (a scale of 1: the matching weight columns read as zeros), and sets to zero
// the quantised intermediate's columns that the gate_up GEMM does not write
// (codes from byte q_from and scale bytes from s_from, in every slot's row),
// which the down GEMM multiplies by those zero weight columns.

__global__ void __launch_bounds__(256) moe_widen_kernel(const uint8_t* __restrict__ s13, uint8_t* __restrict__ d13,
                                                        long rows13, int S13, int Sp13,
                                                        const uint8_t* __restrict__ s2, uint8_t* __restrict__ d2,
                                                        long rows2, int S2, int Sp2, uint8_t* __restrict__ a2q,
                                                        int q_row, int q_from, uint8_t* __restrict__ a2s,
                                                        int s_row, int s_from, long cap) {
    const int lane = threadIdx.x & 31;
    const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
    const long nrows = rows13 + rows2 + 2 * cap;
    for (long r = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < nrows; r += nwarps) {
        if (r < rows13) {
            for (int c = lane; c < Sp13; c += 32) d13[r * Sp13 + c] = c < S13 ? s13[r * S13 + c] : (uint8_t)127;
        } else if (r < rows13 + rows2) {
            const long k = r - rows13;
            for (int c = lane; c < Sp2; c += 32) d2[k * Sp2 + c] = c < S2 ? s2[k * S2 + c] : (uint8_t)127;
        } else if (r < rows13 + rows2 + cap) {
            const long k = r - rows13 - rows2;
            for (int c = q_from + lane; c < q_row; c += 32) a2q[k * q_row + c] = 0;
        } else {
            const long k = r - rows13 - rows2 - cap;
            for (int c = s_from + lane; c < s_row; c += 32) a2s[k * s_row + c] = 0;
        }
    }
}

cudaError_t launch_widen(const void* w13_scale, void* d13, long rows13, int S13, int Sp13, const void* w2_scale,
                         void* d2, long rows2, int S2, int Sp2, const WsPtrs& ws, int q_row, int q_from,
                         int s_row, int s_from, long cap, int grid, cudaStream_t stream) {
    moe_widen_kernel<<<grid, 256, 0, stream>>>(
        static_cast<const uint8_t*>(w13_scale), static_cast<uint8_t*>(d13), rows13, S13, Sp13,
        static_cast<const uint8_t*>(w2_scale), static_cast<uint8_t*>(d2), rows2, S2, Sp2, ws.a2q, q_row, q_from,
        ws.a2s, s_row, s_from, cap);
    return cudaGetLastError();
}

// ============================================================== wait self-check
//
// One thread waits on an mbarrier that nothing arrives on, through the same
// bounded wait the GEMM kernels use, with a short limit: the wait runs out,
// records kErrSelfCheck in the status word and the kernel returns normally.

__global__ void moe_check_wait_kernel(uint32_t* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    status[0] = 0;
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_barrier_init();
    const bool ok = mbar_wait(&bar, 0, status, kErrSelfCheck, &abort_flag, limit_ns);
    if (ok) status[1] = 1;  // cannot happen: nothing arrives
    mbar_inval(&bar);
}

cudaError_t launch_check_wait(uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
    moe_check_wait_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace moe

extern "C" moe_status_t moe_mxfp4_topk_sum(const float* P, const int32_t* route_pos, void* out, int T,
                                           int d_model, int topk, cudaStream_t stream) {
    if (T < 0 || topk < 1 || topk > 16 || d_model <= 0) return MOE_ERR_INVALID_ARG;
    if (d_model % 128 != 0 || (long long)T * topk > (1LL << 24)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    if (!P || !route_pos || !out) return MOE_ERR_INVALID_ARG;
    if (((reinterpret_cast<uintptr_t>(P) | reinterpret_cast<uintptr_t>(route_pos) |
          reinterpret_cast<uintptr_t>(out)) & 15u) != 0)
        return MOE_ERR_MISALIGNED;
    moe::WsPtrs ws = {};
    ws.route_pos = const_cast<int32_t*>(route_pos);
    ws.P = const_cast<float*>(P);
    return moe::launch_reduce(T, topk, d_model, d_model, out, ws, stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
