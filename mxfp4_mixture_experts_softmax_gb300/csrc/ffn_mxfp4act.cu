// ffn_mxfp4act.cu -- the expert FFN with MXFP4-quantised activations: x and
// the SwiGLU output are quantised to MXFP4 and both GEMMs run as block-scaled
// MXFP4 x MXFP4 contractions on the 5th-generation tensor cores
// (tcgen05.mma kind::mxf4, E8M0 scales applied by the MMA itself).
//
// The pages fuse the activation with an MXFP4 quantisation that feeds an
// MXFP4 GEMM and measure the matmuls against the MXFP4 peak (OpenRelay,
// "Gemma 4 31B from B200 to MI355X", section "optimisation 4" and section
// "how far from the ceiling").  Quantisation follows the OCP Microscaling v1.0
// conversion: per 32 consecutive values, shared exponent e = floor(log2 amax)
// - 2 (clamped to >= -127; scale byte e + 127, byte 0 for an all-zero block),
// each value v / 2^e rounded to the nearest E2M1 value (ties to even,
// saturating at 6) by the hardware conversion cvt.rn.satfinite.e2m1x2.f32.
//
// GEMM work item = one tile of N = tile_m token rows of one expert x one
// block of 128 weight rows (64 gate + 64 up rows for gate_up; 128 rows of W2
// for down); weights are the MMA's M side, tokens its N side.  Persistent
// CTAs (one per SM), 320 threads:
//   * producer warp: 2D TMA loads (128-byte swizzle) of the weight codes (two
//     64-row boxes) and of the tile's activation codes (one N-row box), 256 k
//     per stage, one transaction barrier per pair of stages; with K % 512 ==
//     0 also the pair's 16 scale bytes of every weight row and token row;
//   * MMA warp: one thread issues the four K = 64 MMAs of each stage, waits
//     and commits once per pair of stages;
//   * 4 scale warps, one per tensor-memory lane quadrant: write the stage's
//     scale factors into tensor memory (tcgen05.st), read from the pair's
//     shared-memory slot (or, for other K, loaded from global memory).  The MMA reads the
//     weight row r's scale at lane r, column base + r / 32 (quadrant q reads
//     column q), and token column n's at lane 32 q + n % 32, column base +
//     n / 32 in every quadrant q; byte j of a 32-bit cell is k group j of a
//     128-k chunk, the MMA's scale id (0 or 2) picks the pair of groups;
//   * epilogue warps: down (one warp per lane quadrant and 32-column chunk)
//     stages the accumulator of the positions holding a pair as f16 rows by
//     sorted position, scaled by a power of two per (8 rows, 32 positions)
//     (store_y16_chunk); the combine gathers each token's positions from it
//     and applies the routing weight there; gate_up (4 warps) passes each
//     32-column slice of the accumulator through shared memory (transposed),
//     so each thread holds 16 consecutive i of one token: SwiGLU in fp32, then
//     MXFP4 quantisation of each 32-block of i (two threads per block), codes
//     and scale stored.
// Every wait is bounded (see mbar_wait); after a timeout each role stops, the
// MMA thread drains its own MMAs (bounded), and tensor memory is freed.
#include <algorithm>

#include "moe_internal.h"
#include "tcgen05.cuh"

namespace moe {

namespace {

constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kScaleWarp0 = 2;   // 2..5: warp % 4 covers every lane quadrant
constexpr int kEpiWarp0 = 6;     // 6..9 (gate_up), 6.. (down)
constexpr int kEpiThreads = 128;  // gate_up's epilogue warps, which meet at named barrier 1
// the down epilogue (staging y as f16, store-bound) has one warp per lane
// quadrant and 32-column chunk (two per quadrant at N = 256, where registers
// allow no more), warp h of a quadrant draining chunks h, h + 2, ...
// (skewed 8192-token MXFP4 step, down GEMM: 4 warps 422 us, 8: 366, 16: 349)
template <int MODE, int N>
constexpr int mx_epi_warps() { return MODE == 1 ? (N == 256 ? 8 : 4 * (N / 32)) : 4; }
template <int MODE, int N>
constexpr int mx_threads() { return (kEpiWarp0 + mx_epi_warps<MODE, N>()) * 32; }
constexpr int kBK = 256;                         // k per stage: one 128-byte row of packed codes
constexpr int kRowBytes = kBK / 2;
constexpr int kABytes = 128 * kRowBytes;         // 16 KB weight stage
constexpr int kABox = 64;                        // weight rows per TMA box
constexpr int kPrefetch = 8;                     // weight stages prefetched into L2 ahead

constexpr int kSmemLimit = 232448;               // dynamic shared memory per block

template <int MODE, int N>
struct MxLayout {
    static constexpr int kBBytes = N * kRowBytes;
    static constexpr int kStage = kABytes + kBBytes;  // multiple of 1024
    // scale bytes of one pair of stages (16 per row: 512 k), TMA-loaded
    static constexpr int kSfaBytes = 128 * 16;
    static constexpr int kSfPairBytes = kSfaBytes + N * 16;
    static constexpr int kStgRow = 132;             // fp32 staging row (one column), padded
    static constexpr int kStgBytes = MODE == 0 ? 32 * kStgRow * 4 : 0;  // gate_up epilogue only
    // the deepest even ring that fits (at most 10 stages)
    static constexpr int kFit = (kSmemLimit - 1024 - 256 - kStgBytes) / (kStage + kSfPairBytes / 2);
    static constexpr int kStages = (kFit > 10 ? 10 : kFit) & ~1;
    static_assert(kStages >= 4, "ring depth");
    static constexpr int kPairs = kStages / 2;
    static constexpr int kRing = kStages * kStage;
    static constexpr int kSf = kRing;               // scale slots, one per pair
    static constexpr int kStg = kSf + kPairs * kSfPairBytes;
    static constexpr int kBar = kStg + kStgBytes;
    static constexpr int kTotal = kBar + 256 + 1024;  // + barriers, alignment slack
    static_assert(kTotal <= kSmemLimit, "shared memory");
    static constexpr int kNJ = N / 32;              // 32-column groups of the tile
    // tensor memory (512 columns): accumulators, then per stage 32 columns of
    // scale factors, each 128-k chunk's block starting on a multiple of 8
    // columns: weights (4 columns used) at +0 and +8, tokens (kNJ <= 8
    // columns) at +16 and +24
    static constexpr int kSfCols = 32;
    static constexpr int kAccBufs = 2 * N + kStages * kSfCols <= 512 ? 2 : 1;
    static constexpr int kSfCol0 = kAccBufs * N;
    static_assert(kSfCol0 + kStages * kSfCols <= 512, "tensor memory");
};

// Instruction descriptor, kind::mxf4: E2M1 x E2M1 -> fp32, E8M0 scales, both
// operands K-major, M x N, scale id `sf` for both operands.
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N, int sf) {
    return ((uint32_t)sf << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(M >> 4) << 24) | ((uint32_t)sf << 29);
}

// D (tensor memory) += A * B, both from shared memory, scale factors of A
// and B in tensor memory (block size 32 along K).
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], "
        "[%5], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

template <int NC>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t* v);
template <>
__device__ __forceinline__ void tmem_st_cols<1>(uint32_t taddr, const uint32_t* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v[0]) : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_cols<2>(uint32_t taddr, const uint32_t* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1,%2};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1])
                 : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_cols<4>(uint32_t taddr, const uint32_t* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                 : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_cols<8>(uint32_t taddr, const uint32_t* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                     taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                 "r"(v[7])
                 : "memory");
}

// ------------------------------------------------------------ quantisation

// Two values -> one byte of E2M1 codes (lo in the low nibble), rounded to
// nearest even with saturation to +-6 by the hardware conversion.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// Scale byte of a block whose largest magnitude is amax (>= 0):
// floor(log2 amax) - 2 + 127 = biased exponent - 2, clamped at 0 (zero and
// subnormal amax, and blocks whose exponent would fall below -127).
__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
    return (uint32_t)max((int)((__float_as_uint(amax) >> 23) & 0xFFu) - 2, 0);
}

// 2^-(sbyte - 127) as fp32 (sbyte <= 252, so the exponent field 254 - sbyte
// stays finite).
__device__ __forceinline__ float mx_inv_scale(uint32_t sbyte) {
    return __uint_as_float((254u - sbyte) << 23);
}

// Eight values times f -> four bytes of codes (v[0] in the lowest nibble).
__device__ __forceinline__ uint32_t e2m1x8(const float* v, float f) {
    return e2m1x2(v[0] * f, v[1] * f) | (e2m1x2(v[2] * f, v[3] * f) << 8) |
           (e2m1x2(v[4] * f, v[5] * f) << 16) | (e2m1x2(v[6] * f, v[7] * f) << 24);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// One thread per 32-value block: 64 bytes of bf16 in, 16 bytes of codes and
// one scale byte out.  Blocks are numbered row-major, so block i of the
// whole matrix starts at element 32 i.
__global__ void __launch_bounds__(256) quantize_mxfp4_kernel(const uint4* __restrict__ x,
                                                             long long nblocks,
                                                             uint4* __restrict__ codes,
                                                             uint8_t* __restrict__ scales) {
    pdl_begin();
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nblocks;
         i += (long long)gridDim.x * blockDim.x) {
        float v[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 w = __ldg(x + 4 * i + c);
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[8 * c + 2 * j] = bf16_lo(u[j]);
                v[8 * c + 2 * j + 1] = bf16_hi(u[j]);
            }
        }
        float amax = 0.0f;
#pragma unroll
        for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(v[k]));
        const uint32_t sb = mx_scale_byte(amax);
        const float f = mx_inv_scale(sb);
        codes[i] = make_uint4(e2m1x8(v, f), e2m1x8(v + 8, f), e2m1x8(v + 16, f), e2m1x8(v + 24, f));
        scales[i] = (uint8_t)sb;
    }
    pdl_end();
}

// ------------------------------------------------------------------ GEMM

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

// silu(g) * u in fp32 with the fast exponential and division (a few ulp from
// the correctly rounded operations).
__device__ __forceinline__ float swiglu(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

template <int MODE, int N>
__global__ void __launch_bounds__(mx_threads<MODE, N>(), 1)
    mxf4_gemm_kernel(const GroupedGemm g, const __grid_constant__ CUtensorMap a_map,
                     const __grid_constant__ CUtensorMap b_map,
                     const __grid_constant__ CUtensorMap sfa_map,
                     const __grid_constant__ CUtensorMap sfb_map) {
    pdl_begin();
    using L = MxLayout<MODE, N>;
    constexpr int kStages = L::kStages, kPairs = L::kPairs, kNJ = L::kNJ;
    constexpr int kAccBufs = L::kAccBufs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float* stg = reinterpret_cast<float*>(smem + L::kStg);
    uint64_t* tma_full = reinterpret_cast<uint64_t*>(smem + L::kBar);  // per pair
    uint64_t* sf_full = tma_full + kPairs;        // scale factors written, per pair
    uint64_t* stage_free = sf_full + kPairs;      // MMAs done with a pair
    uint64_t* acc_full = stage_free + kPairs;     // [2]
    uint64_t* acc_free = acc_full + 2;            // [2]
    uint64_t* drain = acc_free + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    auto stage_a = [&](int s) { return smem + s * L::kStage; };
    auto stage_b = [&](int s) { return smem + s * L::kStage + kABytes; };
    auto sf_slot = [&](int pr) { return smem + L::kSf + pr * L::kSfPairBytes; };
    const bool sf_tma = g.sf_tma != 0;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = g.K, KG = K / 32;
    const int nk = ((K + kBK - 1) / kBK + 1) & ~1;  // stages per item, whole pairs
    const int row_blocks = MODE == 0 ? g.I / 64 : g.rows / 128;
    const int items = checked_tiles(g) * row_blocks;
    constexpr uint32_t kTmemCols = 512;

    if (tid == 0) {
        for (int p = 0; p < kPairs; ++p) {
            mbar_init(&tma_full[p], 1);
            mbar_init(&sf_full[p], 4);
            mbar_init(&stage_free[p], 1);
        }
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_free[b], mx_epi_warps<MODE, N>());
        }
        mbar_init(drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            uint32_t gs = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
                const int tile = item / row_blocks, block = item % row_blocks;
                const int e = checked_expert(g, tile, block == 0);
                if (e < 0) continue;  // skipped by every role
                const int ar0 = e * g.rows + (MODE == 0 ? block * 64 : block * 128);
                const int ar1 = MODE == 0 ? e * g.rows + g.I + block * 64 : ar0 + kABox;
                for (int st = 0; st < kPrefetch && st < nk; ++st) {
                    tma_prefetch_l2_2d(&a_map, st * kRowBytes, ar0);
                    tma_prefetch_l2_2d(&a_map, st * kRowBytes, ar1);
                }
                for (int st = 0; st < nk; ++st, ++gs) {
                    const int s = gs % kStages, pr = (gs >> 1) % kPairs;
                    if (st + kPrefetch < nk) {
                        tma_prefetch_l2_2d(&a_map, (st + kPrefetch) * kRowBytes, ar0);
                        tma_prefetch_l2_2d(&a_map, (st + kPrefetch) * kRowBytes, ar1);
                    }
                    if ((gs & 1) == 0) {  // both slots of a pair come free with one commit
                        if (gs >= kStages && !mbar_wait(&stage_free[pr], ((gs / kStages) - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&tma_full[pr],
                                              (uint32_t)(2 * L::kStage + (sf_tma ? L::kSfPairBytes : 0)));
                        if (sf_tma) {  // the pair's 16 scale groups of each row
                            const uint32_t sfd = smem_u32(sf_slot(pr));
                            const int kx = (st >> 1) * 16;
                            tma_load_2d(sfd, &sfa_map, kx, ar0, &tma_full[pr]);
                            tma_load_2d(sfd + kABox * 16, &sfa_map, kx, ar1, &tma_full[pr]);
                            tma_load_2d(sfd + L::kSfaBytes, &sfb_map, kx, tile * N, &tma_full[pr]);
                        }
                    }
                    const uint32_t a = smem_u32(stage_a(s));
                    tma_load_2d(a, &a_map, st * kRowBytes, ar0, &tma_full[pr]);
                    tma_load_2d(a + kABox * kRowBytes, &a_map, st * kRowBytes, ar1, &tma_full[pr]);
                    tma_load_2d(smem_u32(stage_b(s)), &b_map, st * kRowBytes, tile * N, &tma_full[pr]);
                }
            }
            // wait (bounded) until the last loads landed before the CTA can exit
            for (int d = 0; d < kStages && d < (int)gs; d += 2) {
                const uint32_t u = gs - 1 - d;
                if (!mbar_wait(&tma_full[(u >> 1) % kPairs], (u / kStages) & 1)) break;
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t idesc0 = idesc_mxf4(128, N, 0), idesc2 = idesc_mxf4(128, N, 2);
            uint32_t gs = 0, it = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
                if (checked_expert(g, item / row_blocks, false) < 0) continue;
                const uint32_t b = it % kAccBufs;
                if (it >= (uint32_t)kAccBufs && !mbar_wait(&acc_free[b], ((it / kAccBufs) - 1) & 1)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + b * N;
                for (int st = 0; st < nk; st += 2, gs += 2) {
                    const int pr = (gs >> 1) % kPairs;
                    const uint32_t par = (gs / kStages) & 1;
                    if (!mbar_wait(&tma_full[pr], par) || !mbar_wait(&sf_full[pr], par)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int s = (gs + h2) % kStages;
                        const uint64_t ad = sdesc_sw128(smem_u32(stage_a(s)));
                        const uint64_t bd = sdesc_sw128(smem_u32(stage_b(s)));
                        const uint32_t sf = tmem + (uint32_t)(L::kSfCol0 + s * L::kSfCols);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {  // K = 64 each: +32 bytes in the swizzle atom
                            const int c = kk >> 1;
                            mma_mxf4(d_tmem, ad + 2u * kk, bd + 2u * kk, (kk & 1) ? idesc2 : idesc0,
                                     sf + 8u * c, sf + 16u + 8u * c, (st | h2 | kk) != 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(&stage_free[pr]);
                }
                if (ok) mma_commit(&acc_full[b]);
                ++it;  // items processed (skipped ones use no accumulator)
            }
            mma_commit(drain);  // every MMA this thread issued has completed when this arrives
            mbar_wait(drain, 0);
        }
    } else if (warp >= kScaleWarp0 && warp < kEpiWarp0) {
        // ---------------------------------------------------- scale factors
        const int quad = warp & 3;
        const int rho = 32 * quad + lane;  // weight row of the stage = accumulator lane
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)L::kSfCol0;
        uint32_t gs = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
            const int tile = item / row_blocks, block = item % row_blocks;
            const int e = checked_expert(g, tile, false);
            if (e < 0) continue;
            const int wrow = MODE == 0 ? (rho < 64 ? block * 64 + rho : g.I + block * 64 + rho - 64)
                                       : block * 128 + rho;
            const uint8_t* sa = g.scales + ((size_t)e * g.rows + wrow) * (size_t)KG;
            const uint8_t* sb[kNJ];
#pragma unroll
            for (int j = 0; j < kNJ; ++j) {
                const int p = tile * N + 32 * j + lane;
                if (sf_tma) {
                    sb[j] = nullptr;
                } else if (MODE == 0) {
                    const int q = checked_pair(g, p);
                    sb[j] = q < 0 ? nullptr : g.act_scales + (size_t)(q / g.Kt) * KG;
                } else {
                    sb[j] = g.act_scales + (size_t)p * KG;
                }
            }
            for (int st = 0; st < nk; st += 2, gs += 2) {
                const int pr = (gs >> 1) % kPairs;
                // hc = 2 * (stage of the pair) + chunk: 4 scale bytes of a 128-k chunk
                uint32_t av[4], bv[4][kNJ];
                if (sf_tma) {
                    // the pair's slot is filled once the producer saw the MMAs
                    // that last read these tensor-memory columns complete
                    if (!mbar_wait_warp(&tma_full[pr], (gs / kStages) & 1)) {
                        ok = false;
                        break;
                    }
                    const uint4 a4 = lds128(sf_slot(pr) + rho * 16);
                    av[0] = a4.x, av[1] = a4.y, av[2] = a4.z, av[3] = a4.w;
#pragma unroll
                    for (int j = 0; j < kNJ; ++j) {
                        const uint4 b4 = lds128(sf_slot(pr) + L::kSfaBytes + (32 * j + lane) * 16);
                        bv[0][j] = b4.x, bv[1][j] = b4.y, bv[2][j] = b4.z, bv[3][j] = b4.w;
                    }
                } else {
                    // global loads first (they do not touch the ring)
#pragma unroll
                    for (int hc = 0; hc < 4; ++hc) {
                        const int grp = 8 * st + 4 * hc;
                        av[hc] = grp < KG ? __ldg(reinterpret_cast<const uint32_t*>(sa + grp)) : 0u;
#pragma unroll
                        for (int j = 0; j < kNJ; ++j)
                            bv[hc][j] = (sb[j] && grp < KG)
                                            ? __ldg(reinterpret_cast<const uint32_t*>(sb[j] + grp))
                                            : 0u;
                    }
                    if (gs >= kStages && !mbar_wait_warp(&stage_free[pr], ((gs / kStages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                }
                tc_fence_after();  // after the MMAs that last read these columns
#pragma unroll
                for (int hc = 0; hc < 4; ++hc) {
                    const int s = (gs + (hc >> 1)) % kStages, c = hc & 1;
                    const uint32_t col = lane_base + (uint32_t)(s * L::kSfCols);
                    tmem_st_cols<1>(col + 8u * c + (uint32_t)quad, &av[hc]);
                    tmem_st_cols<kNJ>(col + 16u + 8u * c, bv[hc]);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sf_full[pr]);
            }
        }
    } else {
        // -------------------------------------------------------- epilogue
        const int quad = warp & 3;                        // lanes 32 quad .. 32 quad + 31
        const int et = (warp - kEpiWarp0) * 32 + lane;    // 0..127
        uint32_t it = 0;
        // down: the tile's pair indices, loaded one item ahead (qn holds those
        // of `item` at the top of the loop); the positions that hold a pair
        // are a prefix of the tile (padding follows an expert's pairs), so
        // their count bounds the stores
        int qn[kNJ];
        auto load_pairs = [&](int item) {
            if (MODE == 1 && item < items) {
#pragma unroll
                for (int u = 0; u < kNJ; ++u) qn[u] = checked_pair(g, (item / row_blocks) * N + 32 * u + lane);
            }
        };
        load_pairs(blockIdx.x);
        for (int item = blockIdx.x; item < items; item += gridDim.x) {
            const int tile = item / row_blocks, block = item % row_blocks;
            const int e = checked_expert(g, tile, false);
            if (e < 0) {
                load_pairs(item + gridDim.x);
                continue;
            }
            const uint32_t b = it % kAccBufs;
            int nvalid = 0;
            if (MODE == 1) {
#pragma unroll
                for (int u = 0; u < kNJ; ++u) nvalid += __popc(__ballot_sync(0xFFFFFFFFu, qn[u] >= 0));
            }
            // one outcome for the warp, and in gate_up for all four epilogue
            // warps, which meet at named barrier 1 below: none may go on to
            // that barrier while another stopped
            bool acc_ok = mbar_wait_warp(&acc_full[b], (it / kAccBufs) & 1);
            if (MODE == 0) acc_ok = all_at_barrier(acc_ok, 1, kEpiThreads);
            if (!acc_ok) break;
            tc_fence_after();
            load_pairs(item + gridDim.x);
            // down: warp h of a quadrant drains chunks 32 h, 32 (h + kPerQuad), ...
            constexpr int kPerQuad = mx_epi_warps<MODE, N>() / 4;
            const int half = MODE == 1 ? (warp - kEpiWarp0) >> 2 : 0;
            constexpr int kCStep = 32 * kPerQuad;
            if (32 * half >= N) {  // no chunk for this warp (narrow tiles)
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_free[b]);
            }
#pragma unroll 1
            for (int c0 = 32 * half; c0 < N; c0 += kCStep) {
                uint32_t v[32];
                const uint32_t taddr = tmem + ((uint32_t)(32 * quad) << 16) + b * N + (uint32_t)c0;
                tmem_ld16_nowait(taddr, v);
                tmem_ld16_nowait(taddr + 16, v + 16);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (c0 + kCStep >= N) {  // this warp's part is drained: the next item may use it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acc_free[b]);
                }
                if (MODE == 1) {  // the raw accumulator of the positions holding a pair, staged as f16
                    const int nc = nvalid - c0;  // warp-uniform
                    store_y16_chunk(g, v, 1.0f, block, quad, lane, tile * N + c0, nc,
                                    block * 128 + 32 * quad + lane < g.rows);
                } else {
                    // transpose through shared memory: stg[column][accumulator row]
#pragma unroll
                    for (int i = 0; i < 32; ++i) stg[i * L::kStgRow + 32 * quad + lane] = __uint_as_float(v[i]);
                    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
                    // thread -> (column, 32-block of i, half): rows 0..63 are the
                    // gate rows of i = block * 64 + row, rows 64..127 the up rows
                    const int half = et & 1, col = (et >> 1) & 31, blk = et >> 6;
                    const float* gp = stg + col * L::kStgRow + 32 * blk + 16 * half;
                    float a[16];
                    float amax = 0.0f;
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const float4 gv = *reinterpret_cast<const float4*>(gp + 4 * k4);
                        const float4 uv = *reinterpret_cast<const float4*>(gp + 64 + 4 * k4);
                        a[4 * k4 + 0] = swiglu(gv.x, uv.x);
                        a[4 * k4 + 1] = swiglu(gv.y, uv.y);
                        a[4 * k4 + 2] = swiglu(gv.z, uv.z);
                        a[4 * k4 + 3] = swiglu(gv.w, uv.w);
                    }
#pragma unroll
                    for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(a[k]));
                    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
                    const uint32_t sbyte = mx_scale_byte(amax);
                    const float f = mx_inv_scale(sbyte);
                    const size_t p = (size_t)tile * N + c0 + col;
                    const int i0 = block * 64 + 32 * blk + 16 * half;
                    *reinterpret_cast<uint2*>(g.hq_codes + p * (size_t)(g.I / 2) + i0 / 2) =
                        make_uint2(e2m1x8(a, f), e2m1x8(a + 8, f));
                    if (half == 0) g.hq_scales[p * (size_t)(g.I / 32) + i0 / 32] = (uint8_t)sbyte;
                    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
                }
            }
            ++it;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
    pdl_end();
}

template <int MODE, int N>
cudaError_t launch_n(const GroupedGemm& g, cudaStream_t s) {
    const size_t smem = MxLayout<MODE, N>::kTotal;
    cudaError_t err = ensure_dynamic_smem((const void*)mxf4_gemm_kernel<MODE, N>, smem);
    if (err != cudaSuccess) return err;
    CUtensorMap a_map, b_map, sfa_map, sfb_map;
    err = encode_codes_map(&a_map, g.codes, g.K / 2, (uint64_t)g.num_experts * g.rows, kRowBytes, kABox);
    if (err != cudaSuccess) return err;
    err = encode_codes_map(&b_map, g.act, g.K / 2, (uint64_t)g.act_rows, kRowBytes, N);
    if (err != cudaSuccess) return err;
    if (g.sf_tma) {  // scale rows of K/32 bytes (a multiple of 16), 16-byte boxes
        err = encode_2d_map(&sfa_map, g.scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.K / 32,
                            (uint64_t)g.num_experts * g.rows, (uint64_t)(g.K / 32), 16, kABox,
                            CU_TENSOR_MAP_SWIZZLE_NONE);
        if (err != cudaSuccess) return err;
        err = encode_2d_map(&sfb_map, g.act_scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.K / 32,
                            (uint64_t)g.act_rows, (uint64_t)(g.K / 32), 16, N,
                            CU_TENSOR_MAP_SWIZZLE_NONE);
        if (err != cudaSuccess) return err;
    } else {  // not read
        sfa_map = a_map;
        sfb_map = b_map;
    }
    const int row_blocks = MODE == 0 ? g.I / 64 : g.rows / 128;
    const long long max_items = (long long)g.max_tiles * row_blocks;
    const int grid = (int)std::min<long long>(max_items, (long long)num_sms());
    return launch_pdl(mxf4_gemm_kernel<MODE, N>, dim3(grid), dim3(mx_threads<MODE, N>()), smem, s, g, a_map,
                      b_map, sfa_map, sfb_map);
}

template <int MODE>
cudaError_t launch_mode(const GroupedGemm& g, cudaStream_t s) {
    if (g.max_tiles == 0) return cudaSuccess;
    switch (g.tile_m) {
        case 32: return launch_n<MODE, 32>(g, s);
        case 64: return launch_n<MODE, 64>(g, s);
        case 128: return launch_n<MODE, 128>(g, s);
        case 256: return launch_n<MODE, 256>(g, s);
        default: return cudaErrorInvalidValue;
    }
}

// The token rows of the used tiles in tile order, MXFP4 encoded: codes
// (cb16 16-byte units per row) and, when sb16 > 0, scales (sb16 units per
// row); zeros for padding positions.  One warp per row, rows grid-strided.
__global__ void __launch_bounds__(256) gather_mx_rows_kernel(const uint4* __restrict__ xc,
                                                             const uint4* __restrict__ xs,
                                                             int cb16, int sb16,
                                                             const int32_t* __restrict__ sorted_pairs,
                                                             const int32_t* __restrict__ num_tiles,
                                                             int tile_m, int Kt, int cap,
                                                             int num_pairs, uint4* __restrict__ xgc,
                                                             uint4* __restrict__ xgs) {
    pdl_begin();
    const int rows = min(max(__ldg(num_tiles), 0) * tile_m, cap);
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int p = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); p < rows; p += warps) {
        int q = __ldg(sorted_pairs + p);
        if (q >= num_pairs) {
            if (lane == 0) flag_index_error();
            q = -1;
        }
        const size_t t = q < 0 ? 0 : (size_t)(q / Kt);
        for (int c = lane; c < cb16; c += 32)
            xgc[(size_t)p * cb16 + c] = q < 0 ? make_uint4(0, 0, 0, 0) : __ldg(xc + t * cb16 + c);
        for (int c = lane; c < sb16; c += 32)
            xgs[(size_t)p * sb16 + c] = q < 0 ? make_uint4(0, 0, 0, 0) : __ldg(xs + t * sb16 + c);
    }
    pdl_end();
}

// w_pos[p] = topk_w[q] (times rscale[p] when given) for the used positions p
// holding pair q, else 0.
__global__ void __launch_bounds__(256) position_weights_kernel(const int32_t* __restrict__ sorted_pairs,
                                                               const float* __restrict__ topk_w,
                                                               const float* __restrict__ rscale,
                                                               const int32_t* __restrict__ num_tiles,
                                                               int tile_m, int cap, int num_pairs,
                                                               float* __restrict__ w_pos) {
    pdl_begin();
    const int rows = min(max(__ldg(num_tiles), 0) * tile_m, cap);
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < rows; p += gridDim.x * blockDim.x) {
        const int q = __ldg(sorted_pairs + p);
        float w = (q >= 0 && q < num_pairs) ? __ldg(topk_w + q) : 0.0f;
        if (rscale) w = __fmul_rn(w, __ldg(rscale + p));
        w_pos[p] = w;
    }
    pdl_end();
}

}  // namespace

cudaError_t launch_position_weights(const int32_t* sorted_pairs, const float* topk_w,
                                    const float* rscale, const int32_t* num_tiles, int tile_m,
                                    int cap, int num_pairs, float* w_pos, cudaStream_t s) {
    if (cap <= 0) return cudaSuccess;
    const int blocks = std::min((cap + 255) / 256, num_sms() * 4);
    return launch_pdl(position_weights_kernel, dim3(blocks), dim3(256), 0, s, sorted_pairs, topk_w,
                      rscale, num_tiles, tile_m, cap, num_pairs, w_pos);
}

cudaError_t launch_gather_mx_rows(const uint8_t* xc, const uint8_t* xs, int H, bool with_scales,
                                  const int32_t* sorted_pairs, const int32_t* num_tiles, int tile_m,
                                  int Kt, int cap, int num_pairs, uint8_t* xgc, uint8_t* xgs,
                                  cudaStream_t s) {
    if (cap <= 0) return cudaSuccess;
    const int blocks = std::min((cap + 7) / 8, num_sms() * 8);
    return launch_pdl(gather_mx_rows_kernel, dim3(blocks), dim3(256), 0, s,
                      reinterpret_cast<const uint4*>(xc), reinterpret_cast<const uint4*>(xs), H / 32,
                      with_scales ? H / 512 : 0, sorted_pairs, num_tiles, tile_m, Kt, cap, num_pairs,
                      reinterpret_cast<uint4*>(xgc), reinterpret_cast<uint4*>(xgs));
}

cudaError_t launch_quantize_mxfp4(const uint16_t* x, int rows, int cols, uint8_t* codes,
                                  uint8_t* scales, cudaStream_t s) {
    const long long nblocks = (long long)rows * (cols / 32);
    if (nblocks <= 0) return cudaSuccess;
    const int blocks = (int)std::min<long long>((nblocks + 255) / 256, (long long)num_sms() * 8);
    return launch_pdl(quantize_mxfp4_kernel, dim3(blocks), dim3(256), 0, s,
                      reinterpret_cast<const uint4*>(x), nblocks, reinterpret_cast<uint4*>(codes),
                      scales);
}

bool mxfp4act_tile_supported(int tile_m) {
    return tile_m == 32 || tile_m == 64 || tile_m == 128 || tile_m == 256;
}
bool mxfp4act_shape_supported(int H, int I) { return H % 128 == 0 && I % 128 == 0; }
cudaError_t launch_mxfp4act_gate_up(const GroupedGemm& g, cudaStream_t s) { return launch_mode<0>(g, s); }
cudaError_t launch_mxfp4act_down(const GroupedGemm& g, cudaStream_t s) { return launch_mode<1>(g, s); }

cudaError_t read_device_error_mxfp4act(int* flag, int clear) {
    int wait = 0, index = 0;
    cudaError_t err = cudaMemcpyFromSymbol(&wait, g_device_error, sizeof(int));
    if (err == cudaSuccess) err = cudaMemcpyFromSymbol(&index, g_index_error, sizeof(int));
    if (err != cudaSuccess) return err;
    *flag = (wait ? 1 : 0) | (index ? 2 : 0);
    if (!clear) return cudaSuccess;
    const int zero = 0;
    err = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    return err == cudaSuccess ? cudaMemcpyToSymbol(g_index_error, &zero, sizeof(int)) : err;
}

}  // namespace moe
