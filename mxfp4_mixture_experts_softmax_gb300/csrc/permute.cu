// permute.cu -- stable counting sort of (token, slot) pairs by expert with
// tile-aligned buckets, in one CTA.
//
// Tokens are grouped by expert in fixed-height row tiles so that the grouped
// GEMMs see whole tiles of one expert (VibeSys Qwen3.5-397B on 4x MI300A,
// section "cheaper prefill and collectives": 32-row MoE tiles).  The pages
// report that parallelising the routing preparation gained nothing (section
// "what did not help"), so one CTA of 1024 threads does all of it:
//
//  1. warp w counts the experts of its contiguous slice of pairs into its own
//     shared-memory histogram row (32 rows x Et counters);
//  2. per expert, an exclusive scan over the 32 warp rows gives each warp's
//     starting rank inside the bucket; the bucket sizes rounded up to tile_m
//     are scanned over experts to give the offsets;
//  3. padding positions, the tile -> expert map and the tails are written;
//  4. each warp walks its slice in order, 32 pairs at a time; lanes naming
//     the same expert find each other with __match_any_sync and take
//     consecutive positions in lane order.
// Slices are contiguous and in warp order, so the result is the stable sort.
//
// route_permute_kernel runs the routing (route_device.cuh) of a small batch and
// this permutation in the same block, one launch instead of two; the ids it
// permutes were written by the block itself, so they are read with ordinary
// (not read-only cached) loads after a block barrier.
//
// Large batches (at least 8 pairs per expert and 8192 pairs) take a
// multi-block version of the same sort, four launches, so that the scattered
// stores of sorted_pairs and inv are spread over many SMs instead of one:
//  1. block b counts the experts of its contiguous slice of pairs into
//     scratch row b (scratch = inv_pairs, which holds T * Kt >= blocks * Et
//     ints and is rewritten in step 4), and fills its share of sorted_pairs
//     with -1 (padding and tail stay -1);
//  2. one block turns the rows into each (block, expert)'s first position:
//     bucket offset + the counts of earlier blocks; and writes the offsets
//     and the tile count;
//  3. block b scatters its slice from its row of positions exactly as the
//     single-block kernel does (warp sub-slices, lane order within a warp);
//  4. inv[sorted_pairs[p]] = p for the used positions; -1 for pairs whose id
//     is outside [0, Et); the tile -> expert map by binary search in the
//     offsets.
// The bulk stores of steps 1 and 4 are spread over the grid: written by the
// one block of step 2 they took ~30 us at 90k pairs.
// Slices are contiguous in pair order at every level, so the result is the
// same stable sort, bit for bit.
#include <stdlib.h>

#include <algorithm>

#include "moe_internal.h"
#include "route_device.cuh"

namespace moe {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

// ids written earlier by this kernel must not come through the read-only path
template <bool kOwnIds>
__device__ __forceinline__ int load_id(const int32_t* ids, int q) {
    return kOwnIds ? ids[q] : __ldg(ids + q);
}

// Exclusive scan of the bucket sizes padded to tile_m, over e = 0..Et (the
// entry Et counts 0, so off[Et] is the total); every thread of the block
// takes two entries (Et + 1 <= 2048).  cnt, off, wsum in shared memory.
__device__ __forceinline__ void padded_offsets(const int32_t* cnt, int Et, int tile_m, int32_t* off,
                                               int32_t* wsum) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i0 = 2 * tid, i1 = 2 * tid + 1;
    const int p0 = i0 < Et ? (cnt[i0] + tile_m - 1) / tile_m * tile_m : 0;
    const int p1 = i1 < Et ? (cnt[i1] + tile_m - 1) / tile_m * tile_m : 0;
    const int mine = p0 + p1;
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = wsum[lane];
        int wi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += n;
        }
        wsum[lane] = wi - v;  // exclusive prefix of warp totals
    }
    __syncthreads();
    const int excl = wsum[warp] + incl - mine;
    if (i0 <= Et) off[i0] = excl;
    if (i1 <= Et) off[i1] = excl + p0;
}

// Offsets out, tile count, bucket padding and the tail of sorted_pairs, the
// tile -> expert map and its tail (cnt and off complete in shared memory).
__device__ __forceinline__ void write_layout(const int32_t* cnt, const int32_t* off, int Et,
                                             int tile_m, int cap, int max_tiles,
                                             int32_t* __restrict__ sorted_pairs,
                                             int32_t* __restrict__ offsets_out,
                                             int32_t* __restrict__ tile_expert,
                                             int32_t* __restrict__ num_tiles) {
    const int tid = threadIdx.x;
    for (int e = tid; e <= Et; e += blockDim.x) offsets_out[e] = off[e];
    const int used = off[Et];
    const int nt = used / tile_m;
    if (tid == 0) *num_tiles = nt;
    for (int e = tid; e < Et; e += blockDim.x) {
        for (int p = off[e] + cnt[e]; p < off[e + 1]; ++p) sorted_pairs[p] = -1;
        for (int i = off[e] / tile_m; i < off[e + 1] / tile_m; ++i) tile_expert[i] = e;
    }
    for (int p = used + tid; p < cap; p += blockDim.x) sorted_pairs[p] = -1;
    for (int i = nt + tid; i < max_tiles; i += blockDim.x) tile_expert[i] = -1;
}

// Stable scatter of pairs [q_begin, q_end) (this warp's sub-slice) from the
// warp's write cursors my_hist[e]; with inv, also the inverse map.
template <bool kOwnIds>
__device__ __forceinline__ void scatter_warp(const int32_t* ids, int q_begin, int q_end, int Et,
                                             int32_t* my_hist, int32_t* __restrict__ sorted_pairs,
                                             int32_t* __restrict__ inv) {
    const int lane = threadIdx.x & 31;
    for (int base = q_begin; base < q_end; base += 32) {
        const int q = base + lane;
        int e = q < q_end ? load_id<kOwnIds>(ids, q) : -1;
        const bool valid = (unsigned)e < (unsigned)Et;
        if (inv && q < q_end && !valid) inv[q] = -1;
        if (!valid) e = -1 - lane;  // unique per lane: matches nobody
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
        int b = 0;
        if (valid) {
            b = my_hist[e];
            const int pos = b + __popc(peers & lanemask_lt());
            sorted_pairs[pos] = q;
            if (inv) inv[q] = pos;
        }
        __syncwarp();
        if (valid && (peers & lanemask_lt()) == 0) my_hist[e] = b + __popc(peers);
        __syncwarp();
    }
}

template <bool kOwnIds>
__device__ __forceinline__ void permute_block(const int32_t* ids, int P, int Et, int tile_m,
                                              int cap, int max_tiles,
                                              int32_t* __restrict__ sorted_pairs,
                                              int32_t* __restrict__ offsets_out,
                                              int32_t* __restrict__ inv,
                                              int32_t* __restrict__ tile_expert,
                                              int32_t* __restrict__ num_tiles) {
    extern __shared__ int32_t smem[];
    int32_t* hist = smem;                      // [kWarps][Et]: counts, then write cursors
    int32_t* cnt = hist + kWarps * Et;         // [Et]
    int32_t* off = cnt + Et;                   // [Et + 1]
    int32_t* wsum = off + Et + 1;              // [kWarps]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < kWarps * Et; i += kThreads) hist[i] = 0;
    __syncthreads();

    const int chunk = (P + kWarps - 1) / kWarps;
    const int q_begin = min(P, warp * chunk), q_end = min(P, q_begin + chunk);
    int32_t* my_hist = hist + warp * Et;
    for (int q = q_begin + lane; q < q_end; q += 32) {
        const int e = load_id<kOwnIds>(ids, q);
        if ((unsigned)e < (unsigned)Et) atomicAdd(&my_hist[e], 1);
    }
    __syncthreads();

    // per-expert exclusive scan over warps
    for (int e = tid; e < Et; e += kThreads) {
        int run = 0;
        for (int w = 0; w < kWarps; ++w) {
            const int c = hist[w * Et + e];
            hist[w * Et + e] = run;
            run += c;
        }
        cnt[e] = run;
    }
    __syncthreads();

    padded_offsets(cnt, Et, tile_m, off, wsum);
    __syncthreads();

    for (int i = tid; i < kWarps * Et; i += kThreads) hist[i] += off[i % Et];
    write_layout(cnt, off, Et, tile_m, cap, max_tiles, sorted_pairs, offsets_out, tile_expert,
                 num_tiles);
    __syncthreads();

    scatter_warp<kOwnIds>(ids, q_begin, q_end, Et, my_hist, sorted_pairs, inv);
}

// ------------------------------------------------- multi-block (large batches)

// 1. scratch[b][e] = pairs of block b's slice with expert e; sorted_pairs
//    filled with -1
__global__ void __launch_bounds__(kThreads) permute_count_kernel(const int32_t* __restrict__ ids,
                                                                 int P, int Et, int slice, int cap,
                                                                 int32_t* __restrict__ scratch,
                                                                 int32_t* __restrict__ sorted_pairs) {
    pdl_begin();
    extern __shared__ int32_t sh[];  // [Et]
    for (int p = blockIdx.x * kThreads + threadIdx.x; p < cap; p += gridDim.x * kThreads)
        sorted_pairs[p] = -1;
    for (int i = threadIdx.x; i < Et; i += kThreads) sh[i] = 0;
    __syncthreads();
    const int q0 = min(P, blockIdx.x * slice), q1 = min(P, q0 + slice);
    for (int q = q0 + threadIdx.x; q < q1; q += kThreads) {
        const int e = __ldg(ids + q);
        if ((unsigned)e < (unsigned)Et) atomicAdd(&sh[e], 1);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < Et; i += kThreads) scratch[(size_t)blockIdx.x * Et + i] = sh[i];
    pdl_end();
}

// 2. one block: scratch[b][e] = off[e] + pairs of expert e in blocks < b;
//    offsets and the tile count.  The work is split into units of one
//    expert's counts in 16 consecutive blocks (a chunk), spread over all the
//    block's threads (all 16 loads of a unit issued before any store that
//    depends on them: a store to the same array would otherwise order every
//    later load behind it).  csum holds each unit's sum, then its first
//    position within the expert.
__global__ void __launch_bounds__(kThreads, 1)
    permute_scan_kernel(int nb, int Et, int tile_m, int32_t* __restrict__ scratch,
                        int32_t* __restrict__ offsets_out, int32_t* __restrict__ num_tiles) {
    pdl_begin();
    extern __shared__ int32_t sh[];
    int32_t* cnt = sh;              // [Et]
    int32_t* off = cnt + Et;        // [Et + 1]
    int32_t* wsum = off + Et + 1;   // [kWarps]
    int32_t* csum = wsum + kWarps;  // [chunks][Et]
    constexpr int kChunk = 16;
    const int nch = (nb + kChunk - 1) / kChunk;
    const int units = nch * Et;  // unit u: expert u % Et, chunk u / Et
    for (int u = threadIdx.x; u < units; u += kThreads) {
        const int e = u % Et, b0 = (u / Et) * kChunk;
        int c[kChunk];
#pragma unroll
        for (int j = 0; j < kChunk; ++j) c[j] = b0 + j < nb ? scratch[(size_t)(b0 + j) * Et + e] : 0;
        int sum = 0;
#pragma unroll
        for (int j = 0; j < kChunk; ++j) sum += c[j];
        csum[u] = sum;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < Et; e += kThreads) {
        int run = 0;
        for (int k = 0; k < nch; ++k) {
            const int v = csum[k * Et + e];
            csum[k * Et + e] = run;
            run += v;
        }
        cnt[e] = run;
    }
    __syncthreads();
    padded_offsets(cnt, Et, tile_m, off, wsum);
    __syncthreads();
    for (int u = threadIdx.x; u < units; u += kThreads) {
        const int e = u % Et, b0 = (u / Et) * kChunk;
        int c[kChunk];
#pragma unroll
        for (int j = 0; j < kChunk; ++j) c[j] = b0 + j < nb ? scratch[(size_t)(b0 + j) * Et + e] : 0;
        int run = off[e] + csum[u];
#pragma unroll
        for (int j = 0; j < kChunk; ++j)
            if (b0 + j < nb) {
                scratch[(size_t)(b0 + j) * Et + e] = run;
                run += c[j];
            }
    }
    for (int e = threadIdx.x; e <= Et; e += kThreads) offsets_out[e] = off[e];
    if (threadIdx.x == 0) *num_tiles = off[Et] / tile_m;
    pdl_end();
}

// 3. block b scatters its slice from its row of first positions
__global__ void __launch_bounds__(kThreads, 1)
    permute_scatter_kernel(const int32_t* __restrict__ ids, int P, int Et, int slice,
                           const int32_t* __restrict__ scratch,
                           int32_t* __restrict__ sorted_pairs) {
    pdl_begin();
    extern __shared__ int32_t sh[];
    int32_t* hist = sh;  // [kWarps][Et]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < kWarps * Et; i += kThreads) hist[i] = 0;
    __syncthreads();
    const int q0 = min(P, blockIdx.x * slice), q1 = min(P, q0 + slice);
    const int chunk = (q1 - q0 + kWarps - 1) / kWarps;
    const int qb = min(q1, q0 + warp * chunk), qe = min(q1, qb + chunk);
    int32_t* my_hist = hist + warp * Et;
    for (int q = qb + lane; q < qe; q += 32) {
        const int e = __ldg(ids + q);
        if ((unsigned)e < (unsigned)Et) atomicAdd(&my_hist[e], 1);
    }
    __syncthreads();
    for (int e = tid; e < Et; e += kThreads) {
        int run = scratch[(size_t)blockIdx.x * Et + e];
        for (int w = 0; w < kWarps; ++w) {
            const int c = hist[w * Et + e];
            hist[w * Et + e] = run;
            run += c;
        }
    }
    __syncthreads();
    scatter_warp<false>(ids, qb, qe, Et, my_hist, sorted_pairs, nullptr);
    pdl_end();
}

// 4. the inverse map, -1 for pairs with an id outside [0, Et), and the tile
//    -> expert map (the expert whose bucket [off[e], off[e+1]) holds the
//    tile's first row; -1 past the used tiles)
__global__ void __launch_bounds__(256) permute_inverse_kernel(const int32_t* __restrict__ ids, int P,
                                                              int Et,
                                                              const int32_t* __restrict__ sorted_pairs,
                                                              const int32_t* __restrict__ offsets,
                                                              const int32_t* __restrict__ num_tiles,
                                                              int tile_m, int cap, int max_tiles,
                                                              int32_t* __restrict__ inv,
                                                              int32_t* __restrict__ tile_expert) {
    pdl_begin();
    const int nt = min(max(__ldg(num_tiles), 0), max_tiles);
    const int used = min(nt * tile_m, cap);
    const int n = max(max(P, used), max_tiles);
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        if (i < used) {
            const int q = __ldg(sorted_pairs + i);
            if ((unsigned)q < (unsigned)P) inv[q] = i;
        }
        if (i < P && (unsigned)__ldg(ids + i) >= (unsigned)Et) inv[i] = -1;
        if (i < max_tiles) {
            int e = -1;
            if (i < nt) {  // largest e with off[e] <= row (off is non-decreasing, off[0] = 0)
                const int row = i * tile_m;
                int lo = 0, hi = Et;  // invariant: off[lo] <= row < off[hi]
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (__ldg(offsets + mid) <= row) lo = mid;
                    else hi = mid;
                }
                e = lo;
            }
            tile_expert[i] = e;
        }
    }
    pdl_end();
}

__global__ void __launch_bounds__(kThreads, 1)
    permute_kernel(const int32_t* __restrict__ ids, int P, int Et, int tile_m, int cap,
                   int max_tiles, int32_t* __restrict__ sorted_pairs,
                   int32_t* __restrict__ offsets_out, int32_t* __restrict__ inv,
                   int32_t* __restrict__ tile_expert, int32_t* __restrict__ num_tiles) {
    pdl_begin();
    // one block on one SM: the next kernel may start right away (every kernel
    // of the layer waits on this one before it reads what it writes; one that
    // needs none of it overlaps it, see rows_to_f16_kernel)
    pdl_end();
    permute_block<false>(ids, P, Et, tile_m, cap, max_tiles, sorted_pairs, offsets_out, inv,
                         tile_expert, num_tiles);
}

template <int VPL>
__global__ void __launch_bounds__(kThreads, 1)
    route_permute_kernel(const float* __restrict__ logits, const float* __restrict__ shared_w,
                         int T, int E, int K, int with_shared, int renormalize, int tile_m, int cap,
                         int max_tiles, int32_t* topk_ids, float* __restrict__ topk_w,
                         int32_t* __restrict__ sorted_pairs, int32_t* __restrict__ offsets_out,
                         int32_t* __restrict__ inv, int32_t* __restrict__ tile_expert,
                         int32_t* __restrict__ num_tiles) {
    pdl_begin();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int Kt = K + (with_shared ? 1 : 0);
    for (int t = warp; t < T; t += kWarps)
        route_token<VPL>(logits + (size_t)t * E, E, K, with_shared, renormalize,
                         shared_w ? __ldg(shared_w + t) : 1.0f, topk_ids + (size_t)t * Kt,
                         topk_w + (size_t)t * Kt, lane);
    __syncthreads();  // the block's id writes are visible to the whole block
    permute_block<true>(topk_ids, T * Kt, E + (with_shared ? 1 : 0), tile_m, cap, max_tiles,
                        sorted_pairs, offsets_out, inv, tile_expert, num_tiles);
    pdl_end();
}

template <int VPL>
cudaError_t launch_fused(const float* logits, const float* sw, int T, int E, int K, int ws,
                         int rn, int tile_m, int cap, int max_tiles, int32_t* ids, float* w,
                         int32_t* sorted_pairs, int32_t* offsets, int32_t* inv,
                         int32_t* tile_expert, int32_t* num_tiles, cudaStream_t s) {
    const size_t smem = permute_smem_bytes(E + (ws ? 1 : 0));
    cudaError_t err = ensure_dynamic_smem((const void*)route_permute_kernel<VPL>, smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(route_permute_kernel<VPL>, dim3(1), dim3(kThreads), smem, s, logits, sw, T, E,
                      K, ws, rn, tile_m, cap, max_tiles, ids, w, sorted_pairs, offsets, inv,
                      tile_expert, num_tiles);
}

}  // namespace

size_t permute_smem_bytes(int Et) { return sizeof(int32_t) * ((size_t)kWarps * Et + 2 * Et + 1 + kWarps); }

// Blocks of the multi-block sort for P pairs over Et experts, or 0 for the
// single-block kernel.  MOE_PERMUTE_MULTI=0 / 1 forces either where both
// are possible (the multi-block scratch needs blocks * Et <= P).
int permute_blocks(int P, int Et) {
    const int nb = std::min(P / std::max(Et, 1), 160);
    const char* f = getenv("MOE_PERMUTE_MULTI");
    if (f && f[0] == '0') return 0;
    if (f && f[0] == '1') return nb >= 2 ? nb : 0;
    return (nb >= 8 && P >= 8192) ? nb : 0;
}

cudaError_t launch_permute(const int32_t* ids, int T, int Kt, int Et, int tile_m, int cap,
                           int max_tiles, int32_t* sorted_pairs, int32_t* offsets, int32_t* inv,
                           int32_t* tile_expert, int32_t* num_tiles, cudaStream_t s) {
    const int P = T * Kt;
    const int nb = permute_blocks(P, Et);
    if (nb == 0) {
        const size_t smem = permute_smem_bytes(Et);
        cudaError_t err = ensure_dynamic_smem((const void*)permute_kernel, smem);
        if (err != cudaSuccess) return err;
        return launch_pdl(permute_kernel, dim3(1), dim3(kThreads), smem, s, ids, P, Et, tile_m, cap,
                          max_tiles, sorted_pairs, offsets, inv, tile_expert, num_tiles);
    }
    const int slice = (P + nb - 1) / nb;
    int32_t* scratch = inv;  // nb * Et <= P ints, rewritten by the last step
    const size_t hist_smem = sizeof(int32_t) * (size_t)kWarps * Et;
    const size_t scan_smem =
        sizeof(int32_t) * (2 * (size_t)Et + 1 + kWarps + (size_t)((nb + 15) / 16) * Et);
    cudaError_t err = ensure_dynamic_smem((const void*)permute_scatter_kernel, hist_smem);
    if (err == cudaSuccess) err = ensure_dynamic_smem((const void*)permute_scan_kernel, scan_smem);
    if (err == cudaSuccess)
        err = launch_pdl(permute_count_kernel, dim3(nb), dim3(kThreads), sizeof(int32_t) * Et, s,
                         ids, P, Et, slice, cap, scratch, sorted_pairs);
    if (err == cudaSuccess)
        err = launch_pdl(permute_scan_kernel, dim3(1), dim3(kThreads), scan_smem, s, nb, Et, tile_m,
                         scratch, offsets, num_tiles);
    if (err == cudaSuccess)
        err = launch_pdl(permute_scatter_kernel, dim3(nb), dim3(kThreads), hist_smem, s, ids, P, Et,
                         slice, (const int32_t*)scratch, sorted_pairs);
    if (err == cudaSuccess)
        err = launch_pdl(permute_inverse_kernel, dim3(std::min((std::max(P, cap) + 255) / 256,
                                                               num_sms() * 8)),
                         dim3(256), 0, s, ids, P, Et, (const int32_t*)sorted_pairs,
                         (const int32_t*)offsets, (const int32_t*)num_tiles, tile_m, cap, max_tiles,
                         inv, tile_expert);
    return err;
}

}  // namespace moe

namespace moe {

cudaError_t launch_route_permute(const float* logits, const float* shared_w, int T, int E, int K,
                                 int with_shared, int renormalize, int tile_m, int cap,
                                 int max_tiles, int32_t* ids, float* w, int32_t* sorted_pairs,
                                 int32_t* offsets, int32_t* inv, int32_t* tile_expert,
                                 int32_t* num_tiles, cudaStream_t s) {
#define MOE_FUSED(V)                                                                           \
    return launch_fused<V>(logits, shared_w, T, E, K, with_shared, renormalize, tile_m, cap,     \
                           max_tiles, ids, w, sorted_pairs, offsets, inv, tile_expert, num_tiles, \
                           s)
    if (E <= 32) MOE_FUSED(1);
    if (E <= 64) MOE_FUSED(2);
    if (E <= 128) MOE_FUSED(4);
    if (E <= 256) MOE_FUSED(8);
    if (E <= 512) MOE_FUSED(16);
    MOE_FUSED(32);
#undef MOE_FUSED
}

}  // namespace moe
