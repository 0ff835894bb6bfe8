// Grouped block-scaled MXFP4 GEMMs of the MoE forward on tcgen05 tensor cores,
// both stages in one persistent kernel.
//
// Operand roles (weights on the MMA M side, routes on the N side): for one work
// item the CTA computes
//     acc[m, j] = sum_k (Wtile[m, k] * sW) * (Act[slot_j, k] * sA)      (fp32, TMEM)
// with Wtile 128 weight rows and j over up to `tile_rows` sorted route slots of
// one expert.  M = 128 fixed, N = rows of the route tile (16..128).
//
// Stage 1 (kernelbot-amd-moe-mxfp4-723815, solution.py, kernel_stage1 and
// _reference_forward: gate rows [0, I), up rows [I, 2I) of w13; SwiGLU
// silu(g) * u; bf16 intermediate as in kernelbot-amd-moe-mxfp4-754773,
// flower_moe.py, custom_kernel): the 128 A rows are 64 gate rows followed by
// the 64 matching up rows, so TMEM lanes 0..63 hold gate and 64..127 up
// accumulators of 64 features.  The epilogue forms bf16(silu(g) * u) and
// requantises each 32-feature block to MXFP4 in place of the bf16 a2 buffer.
//
// Stage 2 (solution.py, kernel_stage2: down projection, weight applied to the
// output; flower_moe.py passes sorted_weights to stage 2): A = 128 rows of w2,
// the epilogue writes w[route] * y into P[route, :] (fp32) for the per-token sum.
//
// One launch runs both stages: every CTA takes its stage-1 items, then its
// stage-2 items, through the same shared-memory ring, so stage-2 weight tiles
// stream in while other CTAs finish stage 1.  Stage-1 items go round-robin, so
// the CTAs from n1 % G on have one item fewer; the first stage-2 items go
// round-robin over those CTAs only (as many as one stage-1 item is worth), the
// rest round-robin over all CTAs, which evens out the CTAs' work.  A stage-2 item's route tile (the
// stage-1 output of one route tile) is loaded once every stage-1 feature tile of
// that route tile has been written: the epilogue that completes a feature tile
// counts it in tile_done (release), the producer polls the count (acquire,
// bounded) before it issues the route-tile copy.  Stage-1 work never waits on
// stage 2 and the grid is one CTA per SM, so every dependency is on work that
// is already resident.
//
// Pipeline (one CTA per SM, persistent over work items):
//   warp 0  TMA producer: one box each for the weight tile, the route tile and
//           the two raw scale tiles per stage -> smem ring
//   warp 1  MMA warp: issues tcgen05.mma (and, in copy scheme 0, copies its
//           stages' scale factors to TMEM with tcgen05.cp).  With two MMA warps
//           (schemes 0 and 3) warp 2 is the second: the CTA's stages alternate
//           between the two, each into its own accumulator, so two threads issue
//           MMAs (one issuing thread serialises them)
//   warp 2  also allocates / frees TMEM
//   warp 3  rearranges each stage's raw scale tiles into the tcgen05
//           scale-factor layout ahead of the MMA warps (schemes 1-3: it also
//           copies them to TMEM and signals when the copies have run)
//   warps 4-11 (4-15)  epilogue: two (three) groups of four warps take items in
//           turn; with two MMA warps their partial accumulators are summed in a
//           fixed order
// Single-launch mode (few routes): the CTAs also route (in shared memory) and
// quantise the hidden states before the first route-tile copies (front_route,
// front_quant), so no routing or quantisation kernel runs before this one.
// All waits are bounded (ptx.cuh).
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {

struct Item {
    int e, row0, nrows, f, ks0, ks1, tile;
};

// Item `it` of a stage: route tile it / n_ftiles, then feature tile; it runs
// over the whole K extent.  The first kTileCache route tiles come from the
// shared-memory copy.
__device__ __forceinline__ Item decode_item(const StageGeom& q, const int4* gtiles, int it,
                                            const int4* tcache) {
    Item x;
    const int tile = it / q.n_ftiles;
    x.f = it - tile * q.n_ftiles;
    const int4 t = tile < kTileCache ? tcache[tile] : __ldcg(gtiles + tile);
    x.e = t.x;
    x.row0 = t.y;
    x.nrows = t.z;
    x.ks0 = 0;
    x.ks1 = q.kstages;
    x.tile = tile;
    return x;
}

// Checked build: an item's route-tile fields lie in range (expert id, slots
// inside the sorted arrays, rows a positive multiple of 16 within the tile
// width, tile index below the call's tile count).  Every weight row, route row
// and accumulator column an item touches follows from these.
__device__ __forceinline__ bool item_in_range(const GemmParams& p, const Item& x, int num_tiles) {
    return x.e >= 0 && x.e < p.E && x.row0 >= 0 && x.nrows > 0 && x.nrows <= p.tile_rows &&
           (x.nrows & 15) == 0 && x.row0 + x.nrows <= p.cap && x.tile >= 0 && x.tile < num_tiles;
}

// ---------------------------------------------------------------- front end
//
// Single-launch path (few routes): every CTA routes all routes in shared memory
// with the routing kernel's deterministic order (routes of an expert in
// ascending route id, block_m padding, sentinel slots; route_quant_reduce.cu),
// so it knows its route tiles without waiting for another kernel.  scr (ring
// slot 0, not yet in use): hist [NW][E], seg [E + 1], wsum [2 NW], totals [4].
// pos [R] receives every route's slot (-1 for ids outside [0, E)); the tiles go
// to tcache.  CTA 0 (write_global) also clears the call's error bits, writes
// the workspace routing arrays and then stores kFrontReady to status[15] (the
// last CTA of the same kernel sets it back to 0, front_exit).  Returns the number of
// route tiles.  Whole CTA; E <= kFrontMaxExperts.
__device__ int front_route(const GemmParams& p, int* scr, int* pos, int4* tcache, bool write_global) {
    constexpr int NW = kGemmThreads / 32;
    const int E = p.E, R = p.T * p.K, bm = kBlockM, tr = p.tile_rows;
    int* hist = scr;
    int* seg = hist + NW * E;
    int* wsum = seg + (E + 1);
    int* totals = wsum + 2 * NW;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < NW * E; i += kGemmThreads) hist[i] = 0;
    if (tid < 4) totals[tid] = 0;
    if (write_global && tid < 15) p.ws.status[tid] = 0;  // this call's error bits
    __syncthreads();

    const int chunk = (R + NW - 1) / NW;
    const int r_begin = min(warp * chunk, R);
    const int r_end = min(r_begin + chunk, R);
    // pass 1: per-warp histogram (one leader per distinct expert in a batch of 32)
    for (int base = r_begin; base < r_end; base += 32) {
        const int r = base + lane;
        const int e = (r < r_end) ? __ldg(p.topk_ids + r) : -1;
        const bool valid = (r < r_end) && e >= 0 && e < E;
        const uint32_t m = __match_any_sync(0xffffffffu, valid ? e : -1);
        if (valid && lane == __ffs(m) - 1) hist[warp * E + e] += __popc(m);
        __syncwarp();
    }
    __syncthreads();

    // per expert: prefix over warps, padded length, tiles; then exclusive scans
    int cnt = 0, padded = 0, ntiles = 0;
    if (tid < E) {
        int run = 0;
        for (int w = 0; w < NW; ++w) {
            const int c = hist[w * E + tid];
            hist[w * E + tid] = run;
            run += c;
        }
        cnt = run;
        padded = (cnt + bm - 1) / bm * bm;
        ntiles = (padded + tr - 1) / tr;
    }
    int a = padded, b = ntiles;
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
        wsum[warp] = a;
        wsum[NW + warp] = b;
    }
    __syncthreads();
    if (warp == 0) {
        int xa = lane < NW ? wsum[lane] : 0, xb = lane < NW ? wsum[NW + lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ta = __shfl_up_sync(0xffffffffu, xa, o);
            const int tb = __shfl_up_sync(0xffffffffu, xb, o);
            if (lane >= o) {
                xa += ta;
                xb += tb;
            }
        }
        if (lane < NW) {
            wsum[lane] = xa;
            wsum[NW + lane] = xb;
        }
    }
    __syncthreads();
    if (warp > 0) {
        a += wsum[warp - 1];
        b += wsum[NW + warp - 1];
    }
    const int seg_e = a - padded, tile_e = b - ntiles;
    if (tid < E) seg[tid] = seg_e;
    if (tid == kGemmThreads - 1) {
        seg[E] = a;
        totals[0] = a;  // padded length
        totals[1] = b;  // route tiles
    }
    if (tid < E && cnt > 0) atomicAdd(&totals[2], cnt);  // valid routes
    __syncthreads();
    const int total_padded = totals[0], total_tiles = totals[1];

    if (tid < E && cnt > 0) {
        for (int j = 0; j < ntiles; ++j) {
            const int4 t4 = make_int4(tid, seg_e + j * tr, min(tr, padded - j * tr), 0);
            if (tile_e + j < kTileCache) tcache[tile_e + j] = t4;
            if (write_global) p.ws.tiles[tile_e + j] = t4;
        }
    }
    if (write_global) {
        if (tid < E) p.ws.seg_start[tid] = seg[tid];
        if (tid == 0) p.ws.seg_start[E] = seg[E];  // (E may equal the thread count)
        if (tid < E && cnt > 0) {
            for (int blk = seg_e / bm; blk < (seg_e + padded) / bm; ++blk) p.ws.block_expert[blk] = tid;
            for (int q = seg_e + cnt; q < seg_e + padded; ++q) {
                p.ws.sorted_ids[q] = R;
                p.ws.sorted_w[q] = 0.0f;
            }
        }
        for (int q = total_padded + tid; q < p.cap; q += kGemmThreads) {
            p.ws.sorted_ids[q] = R;
            p.ws.sorted_w[q] = 0.0f;
        }
        for (int blk = total_padded / bm + tid; blk < p.cap / bm; blk += kGemmThreads)
            p.ws.block_expert[blk] = -1;
        if (tid == 0) {
            p.ws.num_valid[0] = total_padded;
            p.ws.num_valid[1] = totals[2];
            p.ws.num_valid[2] = total_tiles;
            p.ws.num_valid[3] = 0;
        }
    }
    // pass 2: slots in the same order; rank = warp prefix + rank in the batch
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int base = r_begin; base < r_end; base += 32) {
        const int r = base + lane;
        const int e = (r < r_end) ? __ldg(p.topk_ids + r) : -1;
        const bool valid = (r < r_end) && e >= 0 && e < E;
        const uint32_t m = __match_any_sync(0xffffffffu, valid ? e : -1);
        if (valid) {
            int slot = seg[e] + hist[warp * E + e] + __popc(m & lt_mask);
            if (!moe_check(slot >= 0 && slot < p.cap, p.ws.status)) slot = -1;  // (skipped below)
            pos[r] = slot;
            if (write_global && slot >= 0) {
                p.ws.sorted_ids[slot] = r;
                p.ws.sorted_w[slot] = __ldg(p.topk_w + r);
                p.ws.route_pos[r] = slot;
            }
        } else if (r < r_end) {
            pos[r] = -1;
            if (write_global) p.ws.route_pos[r] = -1;
        }
        __syncwarp();
        if (valid && lane == __ffs(m) - 1) hist[warp * E + e] += __popc(m);
        __syncwarp();
    }
    fence_proxy_async_smem();  // the scratch is ring memory that TMA copies fill next
    __syncthreads();
    if (write_global && tid == 0) {
        // publish the routing arrays (the epilogues read the slots' route ids and weights)
        __threadfence();
        st_release_gpu(p.ws.status + 15, kFrontReady);
    }
    return total_tiles;
}

// MX quantisation of a 32-element block of bf16 by four lanes (lane % 4 = qd
// holds elements 8qd .. 8qd+7 as one 16-byte load): the lanes share the block's
// amax, and each returns its 4 code bytes (low nibble = even element); sc is the
// block's e8m0 scale byte.  All 32 lanes of the warp call it (inactive lanes
// with zeros: their group's result is not used).
__device__ __forceinline__ uint32_t front_quant8(const uint4 raw, uint32_t& sc) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
    uint32_t amax = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = max(amax, __float_as_uint(v[i]) & 0x7fffffffu);
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    sc = mx_scale_byte(amax);
    const float inv = mx_inv_scale(sc == 255u ? 0u : sc);
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) word |= e2m1_code(v[i], sc, inv) << (4 * i);
    return word;
}

// Blocks of 32 elements that one CTA quantises per pass (four epilogue threads each).
constexpr int kFrontQuantBlocks = 64;
// Stages whose weight copies a CTA issues before the quantisation is complete.
constexpr int kFrontPreStages = 2;

// First 16-byte load of an epilogue thread's quantisation share, issued before
// the routing and before any weight copy (the copies of the first stages fill
// the memory system's queues for microseconds), and an L2 prefetch of the
// CTA's later passes; zeros past the end and for padding blocks (columns past
// the logical d_model).  Block j = (token t, block gb) of the D/32 blocks per
// row reads 64 bytes at t * 2 Dl + 64 gb; without padding, at 64 j.
__device__ __forceinline__ uint4 front_quant_first_load(const GemmParams& p) {
    const int et = (int)threadIdx.x - 128;
    const int nblk = p.D / 32;
    const long total = (long)p.T * nblk;
    const uint8_t* hid = static_cast<const uint8_t*>(p.hidden);
    constexpr int kLines = kFrontQuantBlocks * 64 / 128;  // 128-byte lines per pass
    if (et < kLines && p.Dl == p.D) {
        for (long jb = (long)(blockIdx.x + gridDim.x) * kFrontQuantBlocks; jb < total;
             jb += (long)gridDim.x * kFrontQuantBlocks)
            if (jb * 64 + et * 128 < total * 64) prefetch_l2(hid + jb * 64 + et * 128);
    }
    const long j = (long)blockIdx.x * kFrontQuantBlocks + (et >> 2);
    if (j >= total) return make_uint4(0, 0, 0, 0);
    const int t = (int)(j / nblk);
    const int gb = (int)(j - (long)t * nblk);
    if (gb >= p.Dl / 32) return make_uint4(0, 0, 0, 0);
    return ld_nc_v4_now(hid + (size_t)t * p.Dl * 2 + (size_t)gb * 64 + (et & 3) * 16);
}

// Bounded wait (one thread) until a global word equals `want` (equal) or
// reaches it; returns after an acquire load that saw it.  False, with the
// status bit and the CTA's abort flag set, when the limit passes; false when
// the CTA has already aborted.
__device__ __forceinline__ bool poll_word(const uint32_t* word, uint32_t want, bool equal,
                                          uint32_t* status, uint32_t err_bit,
                                          volatile int* abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 0;; ++n) {
        const uint32_t v = ld_relaxed_gpu(word);
        if (equal ? v == want : v >= want) {
            const uint32_t va = ld_acquire_gpu(word);
            if (equal ? va == want : va >= want) return true;
        }
        if ((n & 63u) == 63u) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                atomicOr(status, err_bit);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// The epilogue warps' part of the single-launch front end: quantise this CTA's
// share of the hidden states (passes of kFrontQuantBlocks consecutive blocks of
// 32 elements, spread over the CTAs; first16: the thread's first load) and
// write each block to the sorted slot of every valid route of its token; then
// count the CTA in quant_done (zero at the start of the call: the last CTA of
// the previous single-launch call cleared it, or it was never used).
// Warps 4..11 (named barrier 3).
__device__ void front_quant(const GemmParams& p, const int* pos, uint4 first16) {
    const int et = (int)threadIdx.x - 128;
    const int D = p.D, K = p.K, nblk = D / 32;
    const long total = (long)p.T * nblk;
    const __nv_bfloat16* hidden = static_cast<const __nv_bfloat16*>(p.hidden);
    const int qd = et & 3;
    bool first = true;
    for (long jb = (long)blockIdx.x * kFrontQuantBlocks; jb < total;
         jb += (long)gridDim.x * kFrontQuantBlocks) {
        const long j = jb + (et >> 2);
        const bool active = j < total;
        const int t = active ? (int)(j / nblk) : 0;
        const int gb = active ? (int)(j - (long)t * nblk) : 0;
        uint4 raw = first16;
        if (!first) {
            raw = make_uint4(0, 0, 0, 0);  // padding blocks (past the logical d_model): zero
            if (active && gb < p.Dl / 32)
                raw = __ldg(reinterpret_cast<const uint4*>(hidden + (size_t)t * p.Dl) + gb * 4 + qd);
        }
        first = false;
        uint32_t sc;
        const uint32_t word = front_quant8(raw, sc);  // whole warp
        if (active) {
            for (int k = 0; k < K; ++k) {
                const int ps = pos[t * K + k];
                if (ps >= 0 && moe_check(ps < p.cap && gb < nblk, p.ws.status)) {
                    *reinterpret_cast<uint32_t*>(p.ws.a1q + (size_t)ps * (D / 2) + gb * 16 + qd * 4) = word;
                    if (qd == 0) p.ws.a1s[(size_t)ps * p.a1s_stride + gb] = (uint8_t)sc;
                }
            }
        }
    }
    // the stage-1 route-tile copies (async proxy) read these bytes
    fence_proxy_async_global();
    named_bar_sync(3, 256);
    if (et == 0) {
        __threadfence();
        if (atomicAdd(p.ws.quant_done, 1u) >= gridDim.x) atomicOr(p.ws.status, kErrCounterState);
    }
}

// Routing-array read in the epilogue: through the read-only cache when an
// earlier kernel wrote the arrays, from L2 when CTA 0 of this kernel did.
template <typename V>
__device__ __forceinline__ V ld_route(bool written_here, const V* ptr) {
    return written_here ? __ldcg(ptr) : __ldg(ptr);
}

// Scale factors in TMEM: tcgen05.cp .32x128b.warpx4 copies 32 rows x 16 bytes
// and replicates them into the four 32-lane quadrants; one 128-element chunk of
// 128 rows occupies an "atom" of 4 columns, and the MMA's scale-factor address
// must be the first (4-aligned) column of an atom.
//
// Rearrange a raw scale tile (row m at src + m*sr bytes, 4-byte chunk c =
// scales of K elements [128c, 128c+128)) into natoms scale-factor atoms at dst:
// atom c holds 128 rows as [m % 32][m / 32][4 bytes], the layout tcgen05.cp
// .32x128b.warpx4 expects.  dst may overlap src (every row is read before any
// write).  Whole warp; rows >= 128 are not touched.
__device__ __forceinline__ void sf_to_atoms(const uint8_t* src, int sr, int natoms, uint8_t* dst,
                                            uint32_t lane) {
    uint32_t v[4][4];
    if (sr == 16 && natoms == 4) {  // whole 16-byte rows: conflict-free vector loads
#pragma unroll
        for (int m1 = 0; m1 < 4; ++m1) {
            const uint4 r = *reinterpret_cast<const uint4*>(src + (m1 * 32 + lane) * 16);
            v[m1][0] = r.x;
            v[m1][1] = r.y;
            v[m1][2] = r.z;
            v[m1][3] = r.w;
        }
    } else {
#pragma unroll
        for (int m1 = 0; m1 < 4; ++m1) {
            const uint32_t* row = reinterpret_cast<const uint32_t*>(src + (m1 * 32 + lane) * sr);
#pragma unroll
            for (int c = 0; c < 4; ++c) v[m1][c] = (c < natoms) ? row[c] : 0u;
        }
    }
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (c < natoms) {
            uint4 w = make_uint4(v[0][c], v[1][c], v[2][c], v[3][c]);
            *reinterpret_cast<uint4*>(dst + c * 512 + lane * 16) = w;
        }
    }
}

// Two-atom scale-factor copies (tcgen05.cp .128x256b: 128 source rows of 32
// bytes -> TMEM lanes 0..127, 8 columns).  Atom c's layout above repeats in each
// 32-lane quadrant, so source row L = 32q + r (q = 0..3) holds atom c's row r
// then atom c+1's row r; one copy fills atoms c and c+1.  The source is stored as
// 16 groups of 8 rows, each group two 128-byte core matrices (the rows' first
// and second 16 bytes): row L, half j at (L / 8) * 256 + j * 128 + (L % 8) * 16.
// wide_sf_rows: read raw rows lane, lane+32, lane+64, lane+96 (sr bytes each:
// 4 scale bytes per 128-element chunk) and write the natoms / 2 atom pairs of
// this 128-row block, 4 KB each, from dst.  Whole warp.
__device__ __forceinline__ uint32_t wide_sf_off(uint32_t L, uint32_t half) {
    return (L >> 3) * 256u + half * 128u + (L & 7u) * 16u;
}

__device__ __forceinline__ void wide_sf_rows(const uint8_t* raw, int sr, int natoms, uint8_t* dst,
                                             uint32_t lane) {
    uint32_t v[4][4];
#pragma unroll
    for (int m1 = 0; m1 < 4; ++m1) {
        const uint8_t* row = raw + (m1 * 32 + lane) * sr;
        if (sr == 16 && natoms == 4) {
            const uint4 r = *reinterpret_cast<const uint4*>(row);
            v[m1][0] = r.x;
            v[m1][1] = r.y;
            v[m1][2] = r.z;
            v[m1][3] = r.w;
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) v[m1][c] = (c < natoms) ? reinterpret_cast<const uint32_t*>(row)[c] : 0u;
        }
    }
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
        if (2 * pp + 1 >= natoms) break;
        uint8_t* d = dst + pp * 4096;
        const uint4 lo = make_uint4(v[0][2 * pp], v[1][2 * pp], v[2][2 * pp], v[3][2 * pp]);
        const uint4 hi = make_uint4(v[0][2 * pp + 1], v[1][2 * pp + 1], v[2][2 * pp + 1], v[3][2 * pp + 1]);
#pragma unroll
        for (uint32_t q = 0; q < 4; ++q) {
            const uint32_t L = 32u * q + lane;
            *reinterpret_cast<uint4*>(d + wide_sf_off(L, 0)) = lo;
            *reinterpret_cast<uint4*>(d + wide_sf_off(L, 1)) = hi;
        }
    }
}

// Issue KSTEPS of a stage's K-steps of 64, starting at K-step j0 (one thread).
// SPB = K-steps per TMA box row (4 for 128-byte rows, 2 for 64-byte rows).
// Descriptors advance by constant offsets: +32 bytes per K-step inside a
// swizzled row, + one box per SPB steps; K-step j uses scale-factor atom j / 2
// and the even/odd scale-factor selector j % 2.
template <int KSTEPS, int SPB>
__device__ __forceinline__ void issue_stage_mmas(uint32_t d, uint64_t adesc0, uint64_t bdesc0,
                                                 uint32_t a_box, uint32_t b_box, uint32_t idesc_even,
                                                 uint32_t idesc_odd, uint32_t sfa, uint32_t sfb,
                                                 int j0, bool accumulate) {
#pragma unroll
    for (int i = 0; i < KSTEPS; ++i) {
        const uint32_t j = (uint32_t)(j0 + i);
        const uint32_t kt = j / SPB, kk = j % SPB;
        const uint64_t ad = adesc0 + (uint64_t)(kt * a_box + kk * 2u);
        const uint64_t bd = bdesc0 + (uint64_t)(kt * b_box + kk * 2u);
        mma_mxf4(d, ad, bd, (j & 1u) ? idesc_odd : idesc_even, sfa + 4u * (j >> 1),
                 sfb + 4u * (j >> 1), (accumulate || i > 0) ? 1u : 0u);
    }
}


// Single-launch path, once per CTA after all its work: count the CTA out; the
// last CTA clears the words the path shares across CTAs (ready word,
// quantisation count, exit count, route-tile counters) for the next call.
// Every other CTA has finished reading them when it counted itself out.  One
// thread.
__device__ __forceinline__ void front_exit(const GemmParams& p, int num_tiles) {
    uint32_t* st = p.ws.status;
    __threadfence();
    if (atomicAdd(st + kFrontExitWord, 1u) == gridDim.x - 1u) {
        __threadfence();
        for (int i = 0; i < num_tiles && i < kStatusWords - kFrontTileWord; ++i) st[kFrontTileWord + i] = 0u;
        st[15] = 0u;
        st[kFrontQuantWord] = 0u;
        st[kFrontExitWord] = 0u;
    }
}

// kSfMode: who copies the scale factors to TMEM: 0 the two MMA warps, each for
// its own stages; 1 warp 3 (one MMA warp), one 128-element chunk per copy;
// 2 warp 3 (one MMA warp), two chunks per copy where the stage holds an even
// number of chunks (p.wide_sf; staging buffers outside the ring); 3 warp 3, one
// chunk per copy, with two MMA warps taking alternate stages (a single issuing
// thread serialises its MMAs at ~190 cycles each whatever N, two issue in
// parallel: the probe measured N = 16 434 -> 1974 TFLOP/s);
// kFront: single launch (routing and quantisation in this kernel; p.fused_front).
// kKs1, kKs2: K-steps per stage of stage 1 / stage 2, kMb2: weight blocks per
// stage-2 item (0: read from the geometry at run time).
// Template parameters so that each configuration's kernel carries only its code.
template <int kSfMode, bool kFront, int kKs1, int kKs2, int kMb2, int kEpi>
__global__ void __launch_bounds__(128 + 128 * kEpi, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmSA1,
                    const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmSB1,
                    const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmSA2,
                    const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmSB2,
                    const GemmParams p) {
    constexpr bool kSfByLayoutWarp = kSfMode != 0;
    constexpr bool kWide = kSfMode == 2;
    // MMA-issuing warps: two when they copy their own scale factors (mode 0) or in
    // mode 3, else one (the host geometry ties them; launch_gemm checks it)
    constexpr int kMW = (kSfMode == 0 || kSfMode == 3) ? 2 : 1;
    constexpr int kThreads = 128 + 128 * kEpi;  // kEpi epilogue groups
    static_assert(!kFront || kThreads == kGemmThreads, "the front end assumes the 12-warp layout");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const int NS = p.num_stages;

    // full: weight + route tiles landed; sfull: raw scale tiles landed (they are
    // small and arrive first, so their rearrangement overlaps the weight load);
    // sfready: scale tiles rearranged; empty: stage consumed by the MMAs.
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    uint64_t* empty = full + kMaxStages;
    uint64_t* sfready = empty + kMaxStages;
    uint64_t* sfull = sfready + kMaxStages;
    uint64_t* tfull = sfull + kMaxStages;
    uint64_t* tempty = tfull + kMaxAccBufs;
    uint64_t* drain = tempty + kMaxAccBufs;  // one per MMA warp
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 3);  // drain[2]: scale-layout warp
    // sbuf[b]: the scale-factor copies from staging buffer b have run (wide copies)
    uint64_t* sbuf = reinterpret_cast<uint64_t*>(smem + p.off_bar + kSbufBarOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // per epilogue group: a 4 KB exchange buffer (kXchgBytes apart)
    float* xchg = reinterpret_cast<float*>(smem + p.off_xchg);
    uint32_t* status = p.ws.status;

    grid_dep_launch();
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sfready[s], 1);
            mbar_init(&sfull[s], 1);
        }
        for (int a = 0; a < p.acc_bufs; ++a) {
            mbar_init(&tfull[a], (uint32_t)kMW);  // every MMA warp commits once per item
            mbar_init(&tempty[a], 128);
        }
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        mbar_init(&drain[2], 1);
        mbar_init(&sbuf[0], 1);
        mbar_init(&sbuf[1], 1);
        // checked build: accumulators and per-slot scale-factor columns inside the allocation
        bool geo = (uint32_t)p.acc_bufs * p.acc_cols <= p.sf_col0 &&
                   p.sf_col0 + (uint32_t)NS * p.sf_cols <= p.tmem_cols && p.acc_bufs <= kMaxAccBufs && NS <= kMaxStages &&
                   p.acc_bufs >= kEpi &&  // (see gemm_geometry: buffers >= epilogue groups)
                   (kKs1 == 0 || !p.kt_boxes);  // per-K-box weight copies: generic kernels only
        for (int ph2 = 0; ph2 < 2; ++ph2)
            geo = geo && (uint32_t)((p.g[ph2].mblocks + 1) * 4 * p.g[ph2].natoms) <= p.sf_cols;
        *abort_flag = moe_check(geo, p.ws.status) ? 0 : 1;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA1);
        tma_prefetch_desc(&tmSA1);
        tma_prefetch_desc(&tmB1);
        tma_prefetch_desc(&tmSB1);
        tma_prefetch_desc(&tmA2);
        tma_prefetch_desc(&tmSA2);
        tma_prefetch_desc(&tmB2);
        tma_prefetch_desc(&tmSB2);
    }
    // Everything above overlaps the previous kernel; from here on the kernel
    // reads what earlier kernels wrote, and TMEM is free once they have exited.
    grid_dep_wait();
    // Single-launch path: route in shared memory (the ring is not in use yet);
    // otherwise the routing kernel's tile count.
    constexpr bool front = kFront;
    // the generic instantiation keeps one copy of each phase loop: its shapes
    // are small, where cold code after launch costs more than the loop
    constexpr int kPhaseUnroll = kKs1 ? 2 : 1;
    // per-phase K-steps per stage and weight blocks per item (constants where the
    // instantiation fixes them; the phase loops below are unrolled)
    auto ks_of = [&](int phs) -> int {
        const int c = phs == 0 ? kKs1 : kKs2;
        return c ? c : p.g[phs].kstage_elems / 64;
    };
    auto mb_of = [&](int phs) -> int { return phs == 0 ? 1 : (kMb2 ? kMb2 : p.g[1].mblocks); };
    auto na_of = [&](int phs) -> int {  // scale atoms per 128-row block and stage
        return (phs == 0 ? kKs1 : kKs2) ? ks_of(phs) / 2 : p.g[phs].natoms;
    };
    int4* tcache = reinterpret_cast<int4*>(smem + p.off_tiles);
    int* fpos = reinterpret_cast<int*>(smem + p.off_xchg);  // route -> slot (front end only)
    uint4 qfirst = make_uint4(0, 0, 0, 0);  // epilogue threads: first hidden-state load
    if (front && warp >= 4) qfirst = front_quant_first_load(p);
    const int num_tiles = front ? front_route(p, reinterpret_cast<int*>(smem), fpos, tcache, blockIdx.x == 0)
                                : __ldcg(p.ws.num_valid + 2);
    const int nitems[2] = {num_tiles * p.g[0].n_ftiles, num_tiles * p.g[1].n_ftiles};
    const int G = (int)gridDim.x;
    const int b0 = (int)blockIdx.x;
    // stage-2 schedule: items [0, X) round-robin over the L CTAs with one stage-1
    // item fewer (r1 = n1 % G on), items [X, n2) round-robin over all CTAs.  A
    // stage-2 item (per2 stages) costs about 1.5 stage-1 stages (measured: its
    // narrower MMAs and P epilogue), so one stage-1 item is worth 2*per1/(3*per2)
    // stage-2 items.
    const int per1 = p.g[0].kstages, per2 = p.g[1].kstages;
    const int r1 = nitems[0] % G;
    const int L = r1 > 0 ? G - r1 : 0;
    const int X = min(L * ((2 * per1) / (3 * per2)), nitems[1]);
    const int seg1 = (L > 0 && b0 >= r1 && X > b0 - r1) ? (X - (b0 - r1) + L - 1) / L : 0;
    const int my_items0 = b0 < nitems[0] ? (nitems[0] - b0 + G - 1) / G : 0;
    const int my_items1 = seg1 + (X + b0 < nitems[1] ? (nitems[1] - X - b0 + G - 1) / G : 0);
    // m-th item of this CTA in stage phs, or -1
    auto item_of = [&](int phs, int m) -> int {
        if (phs == 0) {
            const int j = b0 + m * G;
            return j < nitems[0] ? j : -1;
        }
        if (m < seg1) return (b0 - r1) + m * L;
        const int j = X + b0 + (m - seg1) * G;
        return j < nitems[1] ? j : -1;
    };
    if (my_items0 == 0 && my_items1 == 0) {
        // an idle CTA still quantises its share of the hidden states
        if (front && warp >= 4) {
            front_quant(p, fpos, qfirst);
            if (threadIdx.x == 128) front_exit(p, num_tiles);
        }
        return;
    }
    if (!front) {
        for (int i = (int)threadIdx.x; i < num_tiles && i < kTileCache; i += kThreads)
            tcache[i] = __ldcg(p.ws.tiles + i);
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // stages of this CTA in both phases
    const long g_total = (long)my_items0 * per1 + (long)my_items1 * per2;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            uint32_t issued = 0;   // bit s: stage s has been filled at least once
            uint32_t last_ph = 0;  // bit s: parity of the last fill of stage s
            // route tiles seen complete by stage 1 (bit per tile, the first kTileCache)
            uint32_t* tready = reinterpret_cast<uint32_t*>(smem + p.off_bar + kReadyBitsOff);
            for (int i = 0; i < kTileCache / 32; ++i) tready[i] = 0u;
            const uint32_t need = (uint32_t)p.g[0].n_ftiles;
            // Single-launch path: the CTA's first kFrontPreStages stages (stage i in
            // slot i) get their weight copies at once and their route-tile copies
            // once every CTA has quantised its share of the hidden states; later
            // stages wait for that too.  (More early weight copies would fill the
            // memory system's queues and slow the front end's own loads, stores and
            // instruction fetches.)
            const int defer_n = front ? min(kFrontPreStages, my_items0 * per1) : 0;
            int n_st = 0;  // stages issued so far
            int drow[kMaxStages], dks[kMaxStages];
            bool resolved = !front;
            auto resolve = [&]() {
                const bool got =
                    poll_word(p.ws.quant_done, (uint32_t)G, false, status, kErrTimeoutFront, abort_flag);
                if (got)
                    fence_proxy_async_global();
                else
                    ok = false;
                // issued either way so that the deferred stages' barriers complete
                const StageGeom& q0 = p.g[0];
                for (int i = 0; i < min(n_st, defer_n); ++i) {
                    uint8_t* st = smem + (size_t)i * p.slot_bytes;
                    tma_load_2d(st + q0.off_sb, &tmSB1, q0.b_scale_x ? dks[i] * 16 : 0, drow[i], &sfull[i]);
                    tma_load_3d(st + q0.off_b, &tmB1, 0, drow[i], dks[i] * q0.nkt, &full[i]);
                }
                resolved = true;
            };
#pragma unroll kPhaseUnroll
            for (int phs = 0; phs < 2; ++phs) {
                if (!ok) break;
                if (phs == 1 && !resolved) resolve();
                if (!ok) break;
                const StageGeom& q = p.g[phs];
                const CUtensorMap* mA = phs ? &tmA2 : &tmA1;
                const CUtensorMap* mSA = phs ? &tmSA2 : &tmSA1;
                const CUtensorMap* mB = phs ? &tmB2 : &tmB1;
                const CUtensorMap* mSB = phs ? &tmSB2 : &tmSB1;
                const int kbytes_stage = ks_of(phs) * 32;  // bytes of one row per stage
                const int MBp = mb_of(phs);
                const uint32_t arows = 128u * (uint32_t)MBp;
                for (int m = 0, it = item_of(phs, 0); it >= 0 && ok; it = item_of(phs, ++m)) {
                    const Item x = decode_item(q, p.ws.tiles, it, tcache);
                    if (!moe_check(item_in_range(p, x, num_tiles), status) || *abort_flag) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    for (int ks = x.ks0; ks < x.ks1; ++ks) {
                        if (!resolved && n_st == defer_n) {
                            resolve();
                            if (!ok) break;
                        }
                        if (!mbar_wait(&empty[s], ph ^ 1u, status, kErrTimeoutEmpty, abort_flag)) {
                            ok = false;
                            break;
                        }
                        uint8_t* st = smem + (size_t)s * p.slot_bytes;
                        const int kt0 = ks * q.nkt;  // first K box of the stage
                        // first weight row (rows of the weight tensors: 2 Iw per expert
                        // in w13, Dw in w2)
                        const int rg = phs == 0 ? x.e * 2 * p.Iw + x.f * 64
                                                : x.e * p.Dw + x.f * 128 * MBp;
                        // weight scales, then the weight tile: they do not depend on stage 1
                        mbar_arrive_expect_tx(&sfull[s], arows * q.sr_a + (uint32_t)p.tile_rows * 16u);
                        mbar_arrive_expect_tx(&full[s], (arows + (uint32_t)p.tile_rows) * kbytes_stage);
                        if (phs == 0) {
                            // the 64 gate rows and the 64 matching up rows (I rows further)
                            if (q.a_scale_small)
                                tma_load_3d(st + q.off_sa, mSA, 0, rg / (16 / q.sr_a), 0, &sfull[s]);
                            else
                                tma_load_3d(st + q.off_sa, mSA, ks * 16, rg, 0, &sfull[s]);
                            if (kKs1 == 0 && p.kt_boxes) {
                                // weights narrower than D (generic instantiations only):
                                // one copy per K box (each box 128 rows, gate then up),
                                // zeros past the row
                                for (int kt = 0; kt < q.nkt; ++kt)
                                    tma_load_3d_hint(st + (size_t)kt * 128u * q.kb, mA, (kt0 + kt) * q.kb, rg, 0,
                                                     &full[s], pol_w);
                            } else {
                                tma_load_4d_hint(st, mA, 0, rg, 0, kt0, &full[s], pol_w);
                            }
                        } else {
                            if (q.a_scale_small)
                                tma_load_2d(st + q.off_sa, mSA, 0, rg / (16 / q.sr_a), &sfull[s]);
                            else
                                tma_load_2d(st + q.off_sa, mSA, ks * 16, rg, &sfull[s]);
                            if (kKs1 == 0 && p.kt_boxes) {
                                // weights narrower than I (generic instantiations only): one
                                // copy per K box of arows rows
                                for (int kt = 0; kt < q.nkt; ++kt)
                                    tma_load_2d_hint(st + (size_t)kt * arows * q.kb, mA, (kt0 + kt) * q.kb, rg,
                                                     &full[s], pol_w);
                            } else {
                                tma_load_3d_hint(st, mA, 0, rg, kt0, &full[s], pol_w);
                            }
                            const bool cached = x.tile < kTileCache;
                            if (!cached || !((tready[x.tile >> 5] >> (x.tile & 31)) & 1u)) {
                                // the route tile's stage-1 output: every feature tile written
                                const uint64_t t0 = globaltimer_ns();
                                bool got = ld_acquire_gpu(p.ws.tile_done + x.tile) >= need;
                                for (uint32_t n = 0; !got; ++n) {
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
                                // the route-tile copies below are issued either way so that
                                // this stage's barriers complete (on abort they carry stale
                                // data that is never used)
                                if (got) {
                                    fence_proxy_async_global();
                                    if (cached) tready[x.tile >> 5] |= 1u << (x.tile & 31);
                                } else {
                                    ok = false;
                                }
                            }
                        }
                        // route tile: tile_rows sorted slots from row0 (rows past the tile's
                        // own are read but never used; past the end they are zero-filled)
                        if (n_st < defer_n) {
                            drow[n_st] = x.row0;
                            dks[n_st] = ks;
                        } else {
                            tma_load_2d(st + q.off_sb, mSB, q.b_scale_x ? ks * 16 : 0, x.row0, &sfull[s]);
                            tma_load_3d(st + q.off_b, mB, 0, x.row0, kt0, &full[s]);
                        }
                        ++n_st;
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
            if (!resolved) resolve();  // (after an abort: completes the deferred stages)
            if (!ok) {
                // Let every copy already issued land before the CTA exits: the
                // last fill of stage i completes the phase with parity last_ph[i].
                for (int i = 0; i < NS; ++i) {
                    if (!((issued >> i) & 1u)) continue;
                    const uint32_t par = (last_ph >> i) & 1u;
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(smem_u32(&full[i]), par) ||
                           !mbar_try_wait(smem_u32(&sfull[i]), par)) {
                        if (globaltimer_ns() - t0 > kWaitLimitNs) {
                            atomicOr(status, kErrTimeoutDrain);
                            break;
                        }
                    }
                }
            }
        }
    }
    if (warp == 1 || (warp == 2 && kMW == 2)) {
        // ------------------------------------------------------------ MMA
        // The CTA's stages are numbered g = 0, 1, ... in (stage, item, k-stage)
        // order; MMA warp w issues the stages with g % mma_warps == w into its
        // own accumulator (two instruction streams keep the tensor pipe busy with
        // narrow MMAs; the epilogue adds the accumulators in a fixed order).  When
        // this warp's next stage is already resident, its scale factors are
        // copied before this stage's MMAs are issued.  Slot and phase indices
        // advance incrementally (no division on the per-stage path).
        const int w = (int)warp - 1;
        constexpr int MW = kMW;
        auto advance = [&](int& ss, uint32_t& pp) {
            ss += MW;
            while (ss >= NS) {
                ss -= NS;
                pp ^= 1u;
            }
        };
        auto sf_base = [&](int ss) { return tmem_base + p.sf_col0 + (uint32_t)ss * p.sf_cols; };
        long g = 0;          // index of the current stage in the CTA's sequence
        int s = w % NS;      // slot of this warp's next stage
        uint32_t ph = (uint32_t)(w / NS) & 1u;
        bool pre = false;    // that stage's scale factors are already in TMEM
        int a = 0;           // accumulator buffer of the current item
        uint32_t aph = 0;    // and its use parity
        bool ok = true;
#pragma unroll kPhaseUnroll
        for (int phs = 0; phs < 2; ++phs) {
            if (!ok) break;
            const StageGeom& q = p.g[phs];
            const uint32_t layout = (q.kb == 128) ? 2u : 4u;  // 128-byte / 64-byte swizzle
            const uint32_t sbo = 8u * q.kb;
            const int ksteps = ks_of(phs);
            const int MB = mb_of(phs);
            const uint32_t a_box = (128u * MB * q.kb) >> 4;  // descriptor units (16 B)
            const uint32_t a_blk = (128u * q.kb) >> 4;       // next 128-row block
            const uint32_t b_box = ((uint32_t)p.tile_rows * q.kb) >> 4;
            // scale copies of slot ss for this stage's layout (lane 0 only); a
            // look-ahead copy may reach into the next stage's layout
            auto copy_scales = [&](int ss, const StageGeom& qq, int qmb, int qna) {
                uint8_t* st = smem + (size_t)ss * p.slot_bytes;
                const uint32_t sfa = sf_base(ss), sfb = sfa + 4u * qmb * qna;
                const uint64_t da = smem_desc(smem_u32(st + qq.off_sa), 0, 128, 0);
                const uint64_t db = smem_desc(smem_u32(st + qq.off_sb), 0, 128, 0);
                for (int c = 0; c < qmb * qna; ++c)
                    tmem_cp_sf(sfa + 4u * c, da + (uint64_t)(32 * c));
                for (int c = 0; c < qna; ++c) tmem_cp_sf(sfb + 4u * c, db + (uint64_t)(32 * c));
            };
            const long g_phase_end = g + (long)(phs == 0 ? my_items0 : my_items1) * q.kstages;
            for (int m = 0, it = item_of(phs, 0); it >= 0 && ok; it = item_of(phs, ++m)) {
                const Item x = decode_item(q, p.ws.tiles, it, tcache);
                if (!moe_check(item_in_range(p, x, num_tiles), status)) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                if (!mbar_wait_warp(&tempty[a], aph ^ 1u, status, kErrTimeoutTmemEmpty, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)a * p.acc_cols + (uint32_t)(w * MB * p.tile_rows);
                const uint32_t idesc_even = mxf4_idesc(128, (uint32_t)x.nrows, 0, 0);
                const uint32_t idesc_odd = mxf4_idesc(128, (uint32_t)x.nrows, 2, 2);
                bool first = true;
                for (int ks = x.ks0; ks < x.ks1; ++ks, ++g) {
                    if ((int)(g & (MW - 1)) != w) continue;  // MW is 1 or 2
                    if (!pre) {
                        if (!mbar_wait_warp(&full[s], ph, status, kErrTimeoutFull, abort_flag) ||
                            !mbar_wait_warp(&sfready[s], ph, status, kErrTimeoutFull, abort_flag)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0) {
                            tc_fence_after();
                            if (!kSfByLayoutWarp) copy_scales(s, q, MB, na_of(phs));  // else warp 3 did
                        }
                    }
                    // this warp's next stage g + MW (its slot's previous fill, stage
                    // g + MW - NS, was this warp's when NS % MW == 0)
                    int sn = s;
                    uint32_t pn = ph;
                    advance(sn, pn);
                    int rd = 0;
                    if (lane == 0 && p.lookahead && !kSfByLayoutWarp && g + MW < g_total)
                        rd = (mbar_test(&full[sn], pn) && mbar_test(&sfready[sn], pn)) ? 1 : 0;
                    rd = __shfl_sync(0xffffffffu, rd, 0);
                    if (rd && lane == 0) {
                        tc_fence_after();
                        if constexpr (kKs1 == 0) {
                            const StageGeom& qn = g + MW < g_phase_end ? q : p.g[1];
                            copy_scales(sn, qn, qn.mblocks, qn.natoms);
                        } else if (g + MW < g_phase_end) {
                            copy_scales(sn, q, MB, na_of(phs));
                        } else {
                            copy_scales(sn, p.g[1], mb_of(1), na_of(1));
                        }
                    }
                    if (lane == 0) {
                        uint8_t* st = smem + (size_t)s * p.slot_bytes;
                        const uint64_t ad0 = smem_desc(smem_u32(st), 16, sbo, layout);
                        const uint64_t bd0 = smem_desc(smem_u32(st + q.off_b), 16, sbo, layout);
                        const uint32_t sfa = sf_base(s), sfb = sfa + 4u * MB * na_of(phs);
                        for (int h = 0; h < MB; ++h) {
                            // block h: its own accumulator columns, A rows and weight scales
                            const uint32_t dh = d + (uint32_t)(h * p.tile_rows);
                            const uint64_t adh = ad0 + (uint64_t)(h * a_blk);
                            const uint32_t sfah = sfa + 4u * (uint32_t)(h * na_of(phs));
                            if (ksteps == 8)
                                issue_stage_mmas<8, 4>(dh, adh, bd0, a_box, b_box, idesc_even,
                                                       idesc_odd, sfah, sfb, 0, !first);
                            else if (ksteps == 4)
                                issue_stage_mmas<4, 4>(dh, adh, bd0, a_box, b_box, idesc_even,
                                                       idesc_odd, sfah, sfb, 0, !first);
                            else
                                issue_stage_mmas<2, 2>(dh, adh, bd0, a_box, b_box, idesc_even,
                                                       idesc_odd, sfah, sfb, 0, !first);
                        }
                        tc_commit(&empty[s]);
                    }
                    __syncwarp();
                    pre = rd != 0;
                    s = sn;
                    ph = pn;
                    first = false;
                }
                if (!ok) break;
                // every MMA warp arrives once per item (a warp without stages in it too)
                if (lane == 0) tc_commit(&tfull[a]);
                __syncwarp();
                if (++a == p.acc_bufs) {
                    a = 0;
                    aph ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            // Wait for every MMA/copy this warp issued before TMEM is freed.
            tc_commit(&drain[w]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&drain[w]), 0)) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    atomicOr(status, kErrTimeoutDrain);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------------------------ scale layout
        bool copied = false;  // this warp issued scale-factor copies (drained below)
        int gw = 0;           // stages that used the two-atom staging buffers so far
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
#pragma unroll kPhaseUnroll
        for (int phs = 0; phs < 2; ++phs) {
            if (!ok) break;
            const StageGeom& q = p.g[phs];
            for (int m = 0, it = item_of(phs, 0); it >= 0 && ok; it = item_of(phs, ++m)) {
                const Item x = decode_item(q, p.ws.tiles, it, tcache);
                if (!moe_check(item_in_range(p, x, num_tiles), status)) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                for (int ks = x.ks0; ks < x.ks1; ++ks) {
                    if (!mbar_wait_warp(&sfull[s], ph, status, kErrTimeoutFull, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + (size_t)s * p.slot_bytes;
                    const int qmb = mb_of(phs), qna = na_of(phs);
                    if (kWide && p.wide_sf && (qna & 1) == 0) {
                        // Two-atom copies from staging buffer b = gw % 2: first wait
                        // until the copies that read it two stages ago have run.
                        const int b = gw & 1;
                        if (gw >= 2 && !mbar_wait_warp(&sbuf[b], (uint32_t)((gw >> 1) - 1) & 1u, status,
                                                       kErrTimeoutFull, abort_flag)) {
                            ok = false;
                            break;
                        }
                        uint8_t* wb = smem + p.off_sfw + (uint32_t)b * p.sfw_bytes;
                        const int pairs = qna / 2;
                        for (int h = 0; h < qmb; ++h)
                            wide_sf_rows(st + q.off_sa + h * 128 * q.sr_a, q.sr_a, qna, wb + h * pairs * 4096, lane);
                        wide_sf_rows(st + q.off_sb, 16, qna, wb + qmb * pairs * 4096, lane);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tc_fence_after();
                            const uint32_t sfa = tmem_base + p.sf_col0 + (uint32_t)s * p.sf_cols;
                            const uint32_t sfb = sfa + 4u * (uint32_t)(qmb * qna);
                            for (int i = 0; i < (qmb + 1) * pairs; ++i) {
                                // block i / pairs (qmb: the route tile), atom pair i % pairs
                                const int h = i / pairs, pp = i - h * pairs;
                                const uint32_t col = (h < qmb ? sfa + 4u * (uint32_t)(h * qna) : sfb) + 8u * (uint32_t)pp;
                                tmem_cp_128x256b(col, smem_desc(smem_u32(wb + i * 4096), 128, 256, 0));
                            }
                            tc_commit(&sfready[s]);
                            tc_commit(&sbuf[b]);
                            copied = true;
                        }
                        __syncwarp();
                        ++gw;
                        if (++s == NS) {
                            s = 0;
                            ph ^= 1u;
                        }
                        continue;
                    }
                    // block h's rows sit at h * 128 * sr_a; its natoms atoms replace them
                    // in place (128 * sr_a == natoms * 512)
                    for (int h = 0; h < qmb; ++h)
                        sf_to_atoms(st + q.off_sa + h * 128 * q.sr_a, q.sr_a, qna, st + q.off_sa + h * qna * 512,
                                    lane);
                    sf_to_atoms(st + q.off_sb, 16, qna, st + q.off_sb, lane);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (kSfByLayoutWarp) {
                            // the scale factors to TMEM as well; sfready completes once the
                            // copies have run (the slot's previous stage has finished: its
                            // MMAs freed the slot before this stage's copies were issued)
                            tc_fence_after();
                            const uint32_t sfa = tmem_base + p.sf_col0 + (uint32_t)s * p.sf_cols;
                            const uint32_t sfb = sfa + 4u * (uint32_t)(qmb * qna);
                            const uint64_t da = smem_desc(smem_u32(st + q.off_sa), 0, 128, 0);
                            const uint64_t db = smem_desc(smem_u32(st + q.off_sb), 0, 128, 0);
                            for (int c = 0; c < qmb * qna; ++c)
                                tmem_cp_sf(sfa + 4u * (uint32_t)c, da + (uint64_t)(32 * c));
                            for (int c = 0; c < qna; ++c)
                                tmem_cp_sf(sfb + 4u * (uint32_t)c, db + (uint64_t)(32 * c));
                            tc_commit(&sfready[s]);
                            copied = true;
                        } else {
                            mbar_arrive(&sfready[s]);
                        }
                    }
                    if (++s == NS) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
        if (lane == 0 && copied) {
            // every copy this warp issued has run before TMEM is freed
            tc_commit(&drain[2]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&drain[2]), 0)) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    atomicOr(status, kErrTimeoutDrain);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        // The groups of four warps take items in turn, so one item's global
        // traffic overlaps the next item's TMEM reads.  Each group covers the 128
        // TMEM lanes (warp % 4 = lane quadrant).
        const uint32_t q4 = warp & 3u;           // TMEM lane quadrant of this warp
        const int grp = (int)(warp - 4) >> 2;    // epilogue group
        const uint32_t bar_id = 1u + (uint32_t)grp;
        float* xg = xchg + grp * (kXchgBytes / 4);
        const int R = p.R;
        constexpr int MW = kMW;
        int local = 0;
        int a_next = 0;         // accumulator buffer of the CTA's item `local`
        uint32_t aph_next = 0;  // and its use parity
        int g0 = 0;             // index of the item's first stage (as the MMA warps count)
        bool ok = true;
        if (front) {
            front_quant(p, fpos, qfirst);
            // the slots' route ids and weights come from CTA 0 (ready word)
            int got = 1;
            if (warp == 4 && lane == 0)
                got = poll_word(p.ws.status + 15, kFrontReady, true, status, kErrTimeoutFront, abort_flag) ? 1 : 0;
            ok = named_bar_and(3, 256, got != 0);
        }
#pragma unroll kPhaseUnroll
        for (int phs = 0; phs < 2; ++phs) {
            if (!ok) break;
            const StageGeom& q = p.g[phs];
            const int per = q.kstages;  // stages per item
            const int MB = mb_of(phs);
            for (int m = 0, it = item_of(phs, 0); it >= 0; it = item_of(phs, ++m), ++local) {
                const int a = a_next;
                const uint32_t aph = aph_next;
                if (++a_next == p.acc_bufs) {
                    a_next = 0;
                    aph_next ^= 1u;
                }
                const int gbeg = g0;
                g0 += per;
                if (local % kEpi != grp) continue;
                const Item x = decode_item(q, p.ws.tiles, it, tcache);
                if (!moe_check(item_in_range(p, x, num_tiles), status)) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                // Route metadata, fetched before waiting for the accumulator.  Stage 1,
                // and stage 2 with two weight blocks per item (narrow tiles): the ids
                // (and weights) of the tile's first 16 slots (lane & 15; later chunks
                // are loaded a chunk ahead).  Stage 2 with one weight block: the ids and
                // weights of all the tile's slots, lane l holding rows l, l + 32, l + 64
                // and l + 96 (sentinel past the tile's rows): there a chunk of 16 stores
                // takes less time than one load from L2, and loading a chunk ahead left
                // every chunk waiting for its metadata (measured prefill T=4096: GEMM
                // kernel 485 -> 440 us).
                const int MBi = mb_of(phs);
                int rid_pre = 0;
                float w_pre = 0.0f;
                int rid4[4] = {R, R, R, R};
                float w4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if (phs == 0 || MBi > 1) {
                    const int slot0 = x.row0 + (int)(lane & 15);
                    rid_pre = ld_route(front, p.ws.sorted_ids + slot0);
                    if (phs == 1) w_pre = ld_route(front, p.ws.sorted_w + slot0);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int r = 32 * j + (int)lane;
                        if (r < x.nrows) {
                            rid4[j] = ld_route(front, p.ws.sorted_ids + x.row0 + r);
                            w4[j] = ld_route(front, p.ws.sorted_w + x.row0 + r);
                        }
                    }
                }
                if (!mbar_wait_warp(&tfull[a], aph, status, kErrTimeoutTmemFull, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tacc_item = tmem_base + ((q4 * 32u) << 16) + (uint32_t)a * p.acc_cols;
                uint32_t tacc = tacc_item;  // block 0; stage 2 moves it per block
                const int nchunks = x.nrows / 16;
                // MMA warp w wrote an accumulator for this item iff one of the item's
                // stages g has g % MW == w.
                const int nst = x.ks1 - x.ks0;
                const bool has1 = MW == 2 && (((gbeg & 1) == 1) || nst > 1);
                const bool has0 = MW == 1 || ((gbeg & 1) == 0) || nst > 1;
                // v = sum of the MMA warps' partial accumulators, warp 0's first
                auto load_acc = [&](int c, float (&v)[16]) {
                    // MMA warp 1's accumulator starts MB * tile_rows columns after warp 0's
                    const uint32_t w1off = (uint32_t)(MB * p.tile_rows);
                    if (has0 && has1) {
                        float t[16];
                        tmem_ld16(tacc + 16u * c, v);
                        tmem_ld16(tacc + w1off + 16u * c, t);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 16; ++k) v[k] = v[k] + t[k];
                    } else {
                        tmem_ld16(tacc + (has0 ? 0u : w1off) + 16u * c, v);
                        tmem_ld_wait();
                    }
                };
                auto release = [&]() {
                    tc_fence_before();
                    mbar_arrive(&tempty[a]);
                };
                bool released = false;
                if (phs == 0) {
                    const int n0 = x.f * 64;  // first feature of the tile
                    {
                        // Per chunk of 16 routes, in two halves of 8: the four warps put
                        // their accumulator rows (gate features 0-31, 32-63, up 0-31,
                        // 32-63) into the exchange buffer; then thread t takes route
                        // t / 16 of the half, feature block (t / 8) % 2 and its 4 features
                        // 4 (t % 8) .. +3, so the block's amax spans 8 lanes and every
                        // thread does the same independent work.  A half whose 8 slots
                        // are all padding is skipped (the same decision in every warp).
                        const int tq = (int)(q4 * 32u + lane);
                        const int ri = tq >> 4, bb = (tq >> 3) & 1, sub = tq & 7;
                        const int feat0 = n0 + 32 * bb;  // first feature of this thread's block
                        int rid_nx = rid_pre;  // the next chunk's route ids, loaded a chunk ahead
                        for (int c = 0; c < nchunks; ++c) {
                            const int rid_l = rid_nx;
                            if (c + 1 < nchunks)
                                rid_nx = ld_route(front, p.ws.sorted_ids + x.row0 + 16 * (c + 1) + (int)(lane & 15));
                            float v[16];
                            load_acc(c, v);
                            if (c + 1 == nchunks) {
                                release();
                                released = true;
                            }
                            const uint32_t valid = __ballot_sync(0xffffffffu, rid_l < R);
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                if (((valid >> (8 * hh)) & 0xffu) == 0u) continue;  // all padding
#pragma unroll
                                for (int i = 0; i < 8; ++i) xg[(q4 * 8 + i) * 32 + lane] = v[8 * hh + i];
                                named_bar_sync(bar_id, 128);
                                const float4 g4 = *reinterpret_cast<const float4*>(xg + (bb * 8 + ri) * 32 + sub * 4);
                                const float4 u4 =
                                    *reinterpret_cast<const float4*>(xg + ((2 + bb) * 8 + ri) * 32 + sub * 4);
                                const float gs[4] = {g4.x, g4.y, g4.z, g4.w};
                                const float us[4] = {u4.x, u4.y, u4.z, u4.w};
                                float hv[4];
                                uint32_t amax = 0;
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const float sg = gs[j] / (1.0f + expf(-gs[j]));
                                    // features past the logical d_inter (padding): zero
                                    hv[j] = feat0 < p.Il ? __bfloat162float(__float2bfloat16_rn(sg * us[j])) : 0.0f;
                                    amax = max(amax, __float_as_uint(hv[j]) & 0x7fffffffu);
                                }
                                amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                                amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                                amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
                                const uint32_t sbyte = mx_scale_byte(amax);
                                const float inv = mx_inv_scale(sbyte == 255u ? 0u : sbyte);
                                uint32_t half16 = 0;  // 4 codes, low nibble = lower feature
#pragma unroll
                                for (int j = 0; j < 4; ++j) half16 |= e2m1_code(hv[j], sbyte, inv) << (4 * j);
                                const uint32_t next16 = __shfl_down_sync(0xffffffffu, half16, 1);
                                const int rid = __shfl_sync(0xffffffffu, rid_l, 8 * hh + ri);
                                const int slot = x.row0 + 16 * c + 8 * hh + ri;
                                if (rid < R) {
                                    if ((sub & 1) == 0)
                                        *reinterpret_cast<uint32_t*>(p.ws.a2q + (size_t)slot * (p.I / 2) + feat0 / 2 +
                                                                     sub * 2) = half16 | (next16 << 16);
                                    if (sub == 0) p.ws.a2s[(size_t)slot * p.a2s_stride + feat0 / 32] = (uint8_t)sbyte;
                                }
                                named_bar_sync(bar_id, 128);  // the buffer is refilled next
                            }
                        }
                        // This feature tile of the route tile is written: count it for the
                        // stage-2 producers, whose TMA copies (async proxy) read it.
                        fence_proxy_async_global();
                        named_bar_sync(bar_id, 128);
                        if (q4 == 0 && lane == 0) {
                            __threadfence();
                            if (atomicAdd(p.ws.tile_done + x.tile, 1u) >= (uint32_t)q.n_ftiles)
                                atomicOr(status, kErrCounterState);
                        }
                    }
                } else if (MB > 1) {
                    // chunk qi = (block h, 16 routes c); the next chunk's route ids and
                    // weights (lanes & 15) are loaded while this chunk is stored
                    int rid_l = rid_pre;
                    float w_l = w_pre;
                    const int total = MB * nchunks;
                    for (int qi = 0; qi < total; ++qi) {
                        const int h = qi / nchunks, c = qi - h * nchunks;
                        tacc = tacc_item + (uint32_t)(h * p.tile_rows);
                        // output feature of this lane in block h
                        const int n = (x.f * MB + h) * 128 + 32 * (int)q4 + (int)lane;
                        int rid_n = 0;
                        float w_n = 0.0f;
                        if (qi + 1 < total) {
                            const int cn = c + 1 < nchunks ? c + 1 : 0;
                            const int sl = x.row0 + 16 * cn + (int)(lane & 15);
                            rid_n = ld_route(front, p.ws.sorted_ids + sl);
                            w_n = ld_route(front, p.ws.sorted_w + sl);
                        }
                        float v[16];
                        load_acc(c, v);
                        if (qi + 1 == total) {
                            release();
                            released = true;
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int rid = __shfl_sync(0xffffffffu, rid_l, i);
                            const float wv = __shfl_sync(0xffffffffu, w_l, i);
                            if (rid < R) p.ws.P[(size_t)rid * p.D + n] = wv * v[i];
                        }
                        rid_l = rid_n;
                        w_l = w_n;
                    }
                } else {
                    // one weight block: chunk c = rows 16c .. 16c + 15 of the tile, held
                    // by lanes 16 (c & 1) .. +15 in register c >> 1
                    // output feature of this lane
                    const int n = x.f * 128 + 32 * (int)q4 + (int)lane;
                    for (int c = 0; c < nchunks; ++c) {
                        const int j = c >> 1;
                        const int rid_l = j == 0 ? rid4[0] : j == 1 ? rid4[1] : j == 2 ? rid4[2] : rid4[3];
                        const float w_l = j == 0 ? w4[0] : j == 1 ? w4[1] : j == 2 ? w4[2] : w4[3];
                        const int lb = (c & 1) * 16;
                        float v[16];
                        load_acc(c, v);
                        if (c + 1 == nchunks) {
                            release();
                            released = true;
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int rid = __shfl_sync(0xffffffffu, rid_l, lb + i);
                            const float wv = __shfl_sync(0xffffffffu, w_l, lb + i);
                            if (rid < R) p.ws.P[(size_t)rid * p.D + n] = wv * v[i];
                        }
                    }
                }
                if (!released) release();
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tmem_base, p.tmem_cols);
    if (front && threadIdx.x == 0) front_exit(p, num_tiles);
}

cudaError_t launch_gemm(const CUtensorMap* maps, const GemmParams& p, int grid,
                        cudaStream_t stream) {
    // copy scheme and MMA warps: MMA-warp copies with two MMA warps, layout-warp
    // copies with one or (one chunk per copy) two
    if (p.mma_warps != 1 && p.mma_warps != 2) return cudaErrorInvalidValue;
    if (!p.sf_by_layout_warp && p.mma_warps != 2) return cudaErrorInvalidValue;
    if (p.wide_sf && (!p.sf_by_layout_warp || p.mma_warps != 1)) return cudaErrorInvalidValue;
    // instantiation: copy scheme, front end, the stage shapes of the common
    // configurations (decode-like, dense-like, prefill-like) and the epilogue
    // groups, else a generic one with two epilogue groups
    const int ks1 = p.g[0].kstage_elems / 64, ks2 = p.g[1].kstage_elems / 64, mb2 = p.g[1].mblocks;
    const bool f = p.fused_front != 0;
    const int mode = !p.sf_by_layout_warp ? 0 : p.wide_sf ? 2 : p.mma_warps == 2 ? 3 : 1;
    const bool three = p.epi_groups == 3 && !f;
    using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                              CUtensorMap, CUtensorMap, GemmParams);
    // spec = the index into the table below (per front-end variant)
    int spec;
    if (mode == 0)
        spec = (ks1 == 8 && ks2 == 4 && mb2 == 2) ? 0 : 1;
    else if (mode == 1)
        spec = (ks1 == 8 && ks2 == 8 && mb2 == 1)   ? 2
               : (ks1 == 8 && ks2 == 4 && mb2 == 1) ? (three ? 8 : 3)
               : (ks1 == 8 && ks2 == 4 && mb2 == 2) ? 5
                                                    : 4;
    else if (mode == 2)
        spec = (ks1 == 8 && ks2 == 4 && mb2 == 2) ? 6 : 7;
    else
        spec = (ks1 == 8 && ks2 == 4 && mb2 == 2) ? 9 : 10;
    // weights narrower than the run widths: the generic instantiation of the scheme
    // (only it compiles the per-K-box weight copies)
    if (p.kt_boxes) spec = mode == 0 ? 1 : mode == 1 ? 4 : mode == 2 ? 7 : 10;
    static const KernelFn kernels[2][11] = {
        {moe_gemm_kernel<0, false, 8, 4, 2, 2>, moe_gemm_kernel<0, false, 0, 0, 0, 2>,
         moe_gemm_kernel<1, false, 8, 8, 1, 2>, moe_gemm_kernel<1, false, 8, 4, 1, 2>,
         moe_gemm_kernel<1, false, 0, 0, 0, 2>, moe_gemm_kernel<1, false, 8, 4, 2, 2>,
         moe_gemm_kernel<2, false, 8, 4, 2, 2>, moe_gemm_kernel<2, false, 0, 0, 0, 2>,
         moe_gemm_kernel<1, false, 8, 4, 1, 3>,
         moe_gemm_kernel<3, false, 8, 4, 2, 2>, moe_gemm_kernel<3, false, 0, 0, 0, 2>},
        {moe_gemm_kernel<0, true, 8, 4, 2, 2>, moe_gemm_kernel<0, true, 0, 0, 0, 2>,
         moe_gemm_kernel<1, true, 8, 8, 1, 2>, moe_gemm_kernel<1, true, 8, 4, 1, 2>,
         moe_gemm_kernel<1, true, 0, 0, 0, 2>, moe_gemm_kernel<1, true, 8, 4, 2, 2>,
         moe_gemm_kernel<2, true, 8, 4, 2, 2>, moe_gemm_kernel<2, true, 0, 0, 0, 2>,
         moe_gemm_kernel<1, true, 8, 4, 1, 2>,
         moe_gemm_kernel<3, true, 8, 4, 2, 2>, moe_gemm_kernel<3, true, 0, 0, 0, 2>}};
    const int epi = (spec == 8 && !f) ? 3 : 2;  // the instantiation's epilogue groups
    // an epilogue group's accumulator-barrier parity is unambiguous only with at
    // least as many buffers as groups (gemm_geometry keeps it so)
    if (p.acc_bufs < epi) return cudaErrorInvalidValue;
    const KernelFn kernel = kernels[f ? 1 : 0][spec];
    // Raise the dynamic shared-memory limit once per device and instantiation.
    static bool limit_set[64][2][11];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!limit_set[dev][f ? 1 : 0][spec]) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmemLimit);
        if (err != cudaSuccess) return err;
        limit_set[dev][f ? 1 : 0][spec] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(128 + 128 * epi);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, maps[0], maps[1], maps[2], maps[3], maps[4],
                              maps[5], maps[6], maps[7], p);
}

}  // namespace moe
