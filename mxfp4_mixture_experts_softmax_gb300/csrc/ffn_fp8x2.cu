// ffn_fp8x2.cu -- the expert FFN with bf16 activations on the block-scaled
// tensor cores: the MXFP4 weights go into tcgen05.mma kind::mxf8f6f4 as they
// are stored (E2M1 codes, one E8M0 scale per 32 k), and each bf16 activation
// (x, and the SwiGLU output h) as the sum of two E4M3 terms with E8M0 scales of
// their own per 32 values.  Nothing is converted on the SMs inside the GEMM.
//
// The pages keep the activations in bf16 and dequantise the MXFP4 weights for
// the prefill GEMMs (padded and tuned prefill GEMM: VibeSys Qwen3.5-397B on 4x
// MI300A, section "baseline"; separate large-M launcher: vLLM MiniMax M3 on
// MI355X, section "local shape and tiling").  Here the block-scaled MMA applies
// the weight scales itself, and the two-term split carries a bf16 value
// exactly:
//   per 32 consecutive values v with largest magnitude amax (biased fp32
//   exponent b), the high term's scale is 2^(S_hi) with scale byte
//   s_hi = max(b - 7, 0) (S_hi = s_hi - 127), so that u = v / 2^S_hi < 2^8;
//   hi = E4M3(u) (nearest even); the low term's scale byte is
//   s_lo = max(s_hi - 5, 0) and lo = E4M3((u - hi) * 2^(s_hi - s_lo)).
//   u - hi is exact in fp32.  A bf16 u has 8 significant bits; for
//   |u| >= 2^-7 (every element within 2^14 of amax) hi keeps the top 4 bits
//   and the remainder, at most 4 significant bits on the grid 2^-9 once
//   shifted by 2^5, is an E4M3 value: hi * 2^S_hi + lo * 2^S_lo == v exactly.
//   Smaller elements are rounded to a multiple of 2^(S_hi - 14), an error
//   below amax * 2^-21.
// Each GEMM then computes D_hi + D_lo, with both terms as B columns of one MMA:
// a tile of N token rows is 2N B rows (N high-term rows, then N low-term
// rows), the accumulator has 2N columns, and the epilogue adds column c and
// column N + c in fp32.  Two E4M3 operand sets cost the MMA what one f16 set
// costs, and the weights cross shared memory once per k step.
//
// GEMM work item = one tile of N token rows of one expert x one block of 128
// weight rows (64 gate + 64 up rows for gate_up; 128 rows of W2 for down).
// Persistent CTAs (one per SM, or CTA pairs from 96-row tiles: see
// fp8x2_gemm_kernel); each CTA first tabulates its items' experts in shared
// memory.  Warp roles:
//   * producer warp: 2D TMA loads per 128-k stage: the block's codes, which
//     the TMA unpacks into the 16-byte-per-16-codes layout the MMA reads
//     (data type 16U4_ALIGN16B, 128-byte swizzle), and the tile's activation
//     rows (E4M3 bytes, 128-byte swizzle); once per group of 8 stages (4 when
//     the item's stages do not split into 8s) the group's scale bytes of every
//     weight row and activation row, one 32-byte (16-byte) box row each, into a
//     two-slot ring; an L2 prefetch cursor runs 16 stages ahead, across items;
//   * MMA warp: one thread issues the stage's four K = 32 MMAs (M = 128 or
//     256, N = 2 tile rows, scale id = k step) and commits them to the stage's
//     barrier, which frees the stage;
//   * 4 scale warps, one per tensor-memory lane quadrant: copy each stage's
//     scale bytes into tensor memory (tcgen05.st) as soon as the group has
//     landed and the columns are free, then wait for the stage's operands and
//     arrive on the MMA's barrier.  The MMA reads weight row r's scale at lane
//     r, column base + r / 32, and B column n's at lane 32 q + n % 32, column
//     base + 8 + n / 32 in every quadrant q; byte j of a 32-bit cell is k group
//     j of the stage;
//   * 8 epilogue warps in two groups of four, group h draining the 32-column
//     chunks h and h + 2 of D_hi + D_lo: each warp copies its chunks out of
//     tensor memory and releases the accumulator before computing.  gate_up
//     passes each chunk through its group's shared-memory buffer (transposed)
//     so each thread holds 16 consecutive i of one token: SwiGLU in fp32, h
//     rounded to bf16 (the oracle's rounding), then split into the two E4M3
//     terms of the down GEMM's B rows; down stages y as f16 rows by sorted
//     position (store_y16_chunk) for the combine, or writes y by pair times the
//     routing weight.
// Every wait is bounded (see mbar_wait); after a timeout each role stops, the
// MMA thread drains its own MMAs (bounded), and tensor memory is freed.
#include <cuda_fp16.h>

#include <algorithm>

#include "moe_internal.h"
#include "tcgen05.cuh"

namespace moe {

namespace {

constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kScaleWarp0 = 2;   // 2..5: warp % 4 covers every lane quadrant
constexpr int kEpiWarp0 = 6;
constexpr int kEpiThreads = 128;  // one epilogue group (4 warps); gate_up's meet at named barrier 1 + group
// two groups of four warps (one per lane quadrant); group h drains the
// 32-column chunks h and h + 2 of the accumulator
template <int MODE>
__host__ __device__ constexpr int x2_epi_warps() { return 8; }
template <int MODE>
__host__ __device__ constexpr int x2_threads() { return (kEpiWarp0 + x2_epi_warps<MODE>()) * 32; }
constexpr int kBK = 128;                 // k per stage: one 128-byte shared-memory row per operand row
constexpr int kRowBytes = 128;
constexpr int kABytes = 128 * kRowBytes;  // 16 KB weight stage (unpacked codes)
constexpr int kABox = 64;                 // weight rows per TMA box
constexpr int kSfGroupMax = 8;           // stages whose scale bytes one load brings
constexpr int kItemTab = 512;            // work items whose expert a CTA tabulates at its start
constexpr int kPrefetch = 16;             // weight stages prefetched into L2 ahead, across items
constexpr int kSmemLimit = 232448;

template <int MODE, int N, bool PAIR>
struct X2Layout {
    static constexpr int kBRows = 2 * N;               // high-term rows, then low-term rows
    static constexpr int kBRowsCta = PAIR ? N : kBRows;  // a pair's CTA loads one term's rows
    static constexpr int kBBytes = kBRowsCta * kRowBytes;
    // scale bytes of a group of up to 8 stages (4 per stage and row): the
    // weight rows, then all 2N B rows; two slots
    static constexpr int kSfRows = 128 + kBRows;
    static constexpr int kSfSlotBytes = kSfRows * 4 * kSfGroupMax;
    static constexpr int kStage = kABytes + kBBytes;
    static_assert(kStage % 1024 == 0 && kSfSlotBytes % 128 == 0, "alignment");
    static constexpr int kStgRow = 132;
    static constexpr int kStgBytes = MODE == 0 ? 2 * 32 * kStgRow * 4 : 0;  // one per epilogue group
    static constexpr int kFit =
        (kSmemLimit - 1024 - 512 - kStgBytes - 2 * kSfSlotBytes - kItemTab * 4) / kStage;
    static constexpr int kStages = kFit > 8 ? 8 : kFit;
    static_assert(kStages >= 3, "ring depth");
    static constexpr int kSf = kStages * kStage;
    static constexpr int kStg = kSf + 2 * kSfSlotBytes;
    static constexpr int kItems = kStg + kStgBytes;  // the CTA's item -> expert table
    static constexpr int kBar = kItems + kItemTab * 4;
    static constexpr int kTotal = kBar + 512 + 1024;  // + barriers, alignment slack
    static_assert(kTotal <= kSmemLimit, "shared memory");
    static constexpr int kBJ = kBRows / 32;             // B scale columns
    static constexpr int kBJst = kBJ <= 2 ? kBJ : (kBJ <= 4 ? 4 : 8);  // columns stored
    static_assert(kBJ <= 8, "B scale columns");
    // tensor memory (512 columns): accumulators of 2N columns, then 16
    // scale columns per stage (weights at +0, B columns at +8)
    static constexpr int kSfCols = 16;
    static constexpr int kAccCols = kBRows;
    static constexpr int kAccBufs = 2 * kAccCols + kStages * kSfCols <= 512 ? 2 : 1;
    static constexpr int kSfCol0 = kAccBufs * kAccCols;
    static_assert(kSfCol0 + kStages * kSfCols <= 512, "tensor memory");
};

// Instruction descriptor, kind::mxf8f6f4: A = E2M1 (the weights), B = E4M3
// (the activation terms), fp32 accumulator, E8M0 scales, both operands
// K-major, M x N, scale id `sf` (the k group of the stage) for both operands.
__host__ __device__ constexpr uint32_t idesc_x2(int M, int N, int sf) {
    return ((uint32_t)sf << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(M >> 4) << 24) | ((uint32_t)sf << 29);
}

// D (tensor memory) += A * B, both from shared memory, scale factors of A
// and B in tensor memory (one per 32 k).
__device__ __forceinline__ void mma_x2(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
        "[%5], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// The CTA-pair form (issued by the pair's even CTA): M = 256, A and the
// scale factors of A from each CTA's own shared and tensor memory, B's N
// columns from the two CTAs' halves.
__device__ __forceinline__ void mma_x2_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
        "[%5], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

template <int NC>
__device__ __forceinline__ void tmem_st_x(uint32_t taddr, const uint32_t* v);
template <>
__device__ __forceinline__ void tmem_st_x<1>(uint32_t taddr, const uint32_t* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v[0]) : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_x<2>(uint32_t taddr, const uint32_t* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1,%2};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1])
                 : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_x<4>(uint32_t taddr, const uint32_t* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                 : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_x<8>(uint32_t taddr, const uint32_t* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                     taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                 "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)));
    return v;
}

// ------------------------------------------------------- two-term split

// Two fp32 -> two E4M3 bytes (a in the low byte), nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

// Two E4M3 bytes (low byte first) -> their values (exact).
__device__ __forceinline__ float2 e4m3x2_value(uint32_t v) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)v));
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// The high term's scale byte of a block whose largest magnitude is amax.
__device__ __forceinline__ uint32_t x2_scale_hi(float amax) {
    return (uint32_t)max((int)((__float_as_uint(amax) >> 23) & 0xFFu) - 7, 0);
}
__device__ __forceinline__ uint32_t x2_scale_lo(uint32_t s_hi) { return s_hi >= 5u ? s_hi - 5u : 0u; }

// 16 values of one block -> 16 high-term and 16 low-term bytes (v[0] lowest).
__device__ __forceinline__ void x2_split16(const float* v, uint32_t s_hi, uint32_t s_lo, uint4& hi,
                                           uint4& lo) {
    const float f_hi = __uint_as_float((254u - s_hi) << 23);        // 2^-(s_hi - 127)
    const float f_lo = __uint_as_float((127u + s_hi - s_lo) << 23);  // 2^(s_hi - s_lo)
    uint32_t h[8], l[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float u0 = v[2 * k] * f_hi, u1 = v[2 * k + 1] * f_hi;
        h[k] = e4m3x2(u0, u1);
        const float2 hv = e4m3x2_value(h[k]);
        l[k] = e4m3x2((u0 - hv.x) * f_lo, (u1 - hv.y) * f_lo);
    }
    hi = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
    lo = make_uint4(l[0] | (l[1] << 16), l[2] | (l[3] << 16), l[4] | (l[5] << 16), l[6] | (l[7] << 16));
}

// Rows of bf16 values (cols a multiple of 32) -> the two E4M3 terms and
// their scale bytes.  One warp per row, lane j taking the 32-value blocks j,
// j + 32, ...  With sorted_pairs: row p of the used tiles takes token
// sorted_pairs[p] / Kt (zeros for padding) and lands in row
// (p / tile_n) * 2 tile_n + p % tile_n of q_hi / s_hi and the same row of
// q_lo / s_lo (the caller passes q_lo = q_hi + tile_n rows); without: row p
// in, row p out.
__global__ void __launch_bounds__(256) split_rows_kernel(
    const uint4* __restrict__ x, int cols, int nrows, const int32_t* __restrict__ sorted_pairs,
    const int32_t* __restrict__ num_tiles, int tile_n, int Kt, int cap, int num_pairs,
    uint8_t* __restrict__ q_hi, uint8_t* __restrict__ q_lo, uint8_t* __restrict__ s_hi,
    uint8_t* __restrict__ s_lo) {
    pdl_begin();
    // used tiles, at most the cap / tile_n the output rows hold
    const int rows = sorted_pairs ? min(max(__ldg(num_tiles), 0), cap / tile_n) * tile_n : nrows;
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    const int nb = cols / 32;
    for (int p = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); p < rows; p += warps) {
        long long t = p;
        if (sorted_pairs) {
            int q = __ldg(sorted_pairs + p);
            if (q >= num_pairs) {
                if (lane == 0) flag_index_error();
                q = -1;
            }
            t = q < 0 ? -1 : q / Kt;
        }
        const size_t orow = tile_n > 0 ? (size_t)(p / tile_n) * 2 * tile_n + p % tile_n : (size_t)p;
        for (int b = lane; b < nb; b += 32) {
            float v[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 w = t < 0 ? make_uint4(0, 0, 0, 0) : __ldg(x + (size_t)t * (cols / 8) + 4 * b + c);
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[8 * c + 2 * j] = __uint_as_float(u[j] << 16);
                    v[8 * c + 2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
                }
            }
            float amax = 0.0f;
#pragma unroll
            for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(v[k]));
            const uint32_t sh = x2_scale_hi(amax), sl = x2_scale_lo(sh);
            uint4 h0, l0, h1, l1;
            x2_split16(v, sh, sl, h0, l0);
            x2_split16(v + 16, sh, sl, h1, l1);
            uint4* dh = reinterpret_cast<uint4*>(q_hi + orow * (size_t)cols + 32 * b);
            uint4* dl = reinterpret_cast<uint4*>(q_lo + orow * (size_t)cols + 32 * b);
            dh[0] = h0;
            dh[1] = h1;
            dl[0] = l0;
            dl[1] = l1;
            s_hi[orow * nb + b] = (uint8_t)sh;
            s_lo[orow * nb + b] = (uint8_t)sl;
        }
    }
    pdl_end();
}

// ------------------------------------------------------------------ GEMM

// PAIR: launched as clusters of two CTAs; a work item is one tile x two
// adjacent weight blocks, block 2 grp + rank in CTA `rank`.  Each CTA loads
// its block's codes, one term's N B rows (the high terms in the even CTA, the
// low terms in the odd one, at the same shared-memory offset) and the scale
// bytes of its weight rows and of all 2N B columns, which its scale warps
// write into its own tensor memory; the even CTA's MMA thread issues M = 256
// MMAs for both and commits to the barriers of both CTAs.  The odd CTA's
// scale and epilogue warps arrive on the even CTA's barriers.  Each stage of
// B then crosses L2 -> shared memory once per 256 weight rows.
template <int MODE, int N, bool PAIR>
__global__ void __launch_bounds__(x2_threads<MODE>(), 1)
    fp8x2_gemm_kernel(const GroupedGemm g, const __grid_constant__ CUtensorMap a_map,
                      const __grid_constant__ CUtensorMap b_map,
                      const __grid_constant__ CUtensorMap sfa_map,
                      const __grid_constant__ CUtensorMap sfb_map) {
    pdl_begin();
    using L = X2Layout<MODE, N, PAIR>;
    constexpr int kStages = L::kStages, kAccBufs = L::kAccBufs, kAccCols = L::kAccCols;
    constexpr int kCtas = PAIR ? 2 : 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float* stg = reinterpret_cast<float*>(smem + L::kStg);
    uint64_t* tma_full = reinterpret_cast<uint64_t*>(smem + L::kBar);  // per stage, this CTA's loads
    uint64_t* sf_full = tma_full + kStages;       // scale factors in tensor memory (even CTA: both)
    uint64_t* stage_free = sf_full + kStages;     // the stage's MMAs completed
    uint64_t* sf_loaded = stage_free + kStages;   // [2] a scale group's bytes landed
    uint64_t* sf_done = sf_loaded + 2;            // [2] the scale warps read the group
    uint64_t* acc_full = sf_done + 2;             // [2]
    uint64_t* acc_free = acc_full + 2;            // [2] drained (even CTA: by both)
    uint64_t* drain = acc_free + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    auto stage_a = [&](int s) { return smem + s * L::kStage; };
    auto stage_b = [&](int s) { return smem + s * L::kStage + kABytes; };
    auto sf_slot = [&](int k) { return smem + L::kSf + k * L::kSfSlotBytes; };
    auto arrive0 = [&](uint64_t* bar) {  // on the barrier the even CTA waits on
        if (PAIR)
            mbar_arrive_remote(bar, 0);
        else
            mbar_arrive(bar);
    };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = PAIR ? (int)(blockIdx.x & 1u) : 0;
    const int cta0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;  // first item
    const int cstep = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;   // item stride
    const int nk = g.K / kBK;  // K % 512 == 0
    // stages per scale group: 8 (32-byte rows) when the item's stages split
    // into whole groups of 8, else 4 (16-byte rows); the launcher's scale
    // maps use the same width
    const int sfg = nk % 8 == 0 ? 8 : 4;
    const int row_blocks = MODE == 0 ? g.I / 64 : g.rows / 128;
    const int row_groups = PAIR ? row_blocks / 2 : row_blocks;  // even for pairs (K % 512 widths)
    const int items = checked_tiles(g) * row_groups;
    auto block_of = [&](int item) { return PAIR ? 2 * (item % row_groups) + rank : item % row_groups; };
    constexpr uint32_t kTmemCols = 512;

    // The expert of each of the CTA's first kItemTab work items (item cta0 +
    // k cstep at k), read once here by all threads together, so that no role
    // waits on a global load at the start of an item; later items read it
    // when they start.  -1: an expert out of range (flagged), skipped by
    // every role.
    int32_t* item_e = reinterpret_cast<int32_t*>(smem + L::kItems);
    for (int k = tid; k < kItemTab && cta0 + k * cstep < items; k += blockDim.x) {
        const int item = cta0 + k * cstep;
        item_e[k] = checked_expert(g, item / row_groups, block_of(item) == 0);
    }
    auto expert_of = [&](int item) {
        const int k = (item - cta0) / cstep;
        return k < kItemTab ? item_e[k] : checked_expert(g, item / row_groups, false);
    };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&tma_full[s], 1);
            mbar_init(&sf_full[s], 4 * kCtas);
            mbar_init(&stage_free[s], 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&sf_loaded[k], 1);
            mbar_init(&sf_done[k], 4);
        }
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_free[b], x2_epi_warps<MODE>() * kCtas);
        }
        mbar_init(drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) tmem_alloc<PAIR>(tmem_slot, kTmemCols);
    tc_fence_before();
    // a pair's barriers are initialised and its tensor memory allocated in
    // both CTAs before anything arrives there or an MMA writes it
    if (PAIR)
        cluster_sync_all();
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            // the weight rows of a work item: gate and up halves (gate_up) or
            // two 64-row halves (down); -1 for an item every role skips
            auto item_rows = [&](int item, int& r0, int& r1) {
                const int block = block_of(item);
                const int e = expert_of(item);
                r0 = e < 0 ? -1 : e * g.rows + (MODE == 0 ? block * 64 : block * 128);
                r1 = MODE == 0 ? e * g.rows + g.I + block * 64 : r0 + kABox;
            };
            // L2 prefetch cursor, kPrefetch stages ahead of the loads and
            // running on into the CTA's next items, so an item's first
            // stages are not fetched from memory only when it starts
            int pf_item = cta0, pf_st = 0, pf_r0 = -1, pf_r1 = -1;
            if (pf_item < items) item_rows(pf_item, pf_r0, pf_r1);
            auto prefetch_next = [&]() {
                while (pf_item < items && pf_r0 < 0) {  // skipped items
                    pf_item += cstep;
                    if (pf_item < items) item_rows(pf_item, pf_r0, pf_r1);
                }
                if (pf_item >= items) return;
                tma_prefetch_l2_2d(&a_map, pf_st * kBK, pf_r0);
                tma_prefetch_l2_2d(&a_map, pf_st * kBK, pf_r1);
                if (++pf_st == nk) {
                    pf_st = 0;
                    pf_item += cstep;
                    pf_r0 = -1;
                    if (pf_item < items) item_rows(pf_item, pf_r0, pf_r1);
                }
            };
            for (int i = 0; i < kPrefetch; ++i) prefetch_next();
            uint32_t gs = 0, gc = 0;  // stages and scale groups issued
            bool ok = true;
            for (int item = cta0; item < items && ok; item += cstep) {
                const int tile = item / row_groups, block = block_of(item);
                const int e = (item - cta0) / cstep < kItemTab ? expert_of(item)
                                                               : checked_expert(g, tile, block == 0);
                if (e < 0) continue;  // skipped by every role (of both CTAs)
                const int ar0 = e * g.rows + (MODE == 0 ? block * 64 : block * 128);
                const int ar1 = MODE == 0 ? e * g.rows + g.I + block * 64 : ar0 + kABox;
                const int br = tile * 2 * N;  // the tile's first B row (high terms)
                for (int st = 0; st < nk; ++st, ++gs) {
                    const int s = gs % kStages;
                    prefetch_next();
                    if (st % sfg == 0) {  // the scale bytes of stages st .. st + sfg - 1, one load per row
                        const int k = gc & 1;
                        if (gc >= 2 && !mbar_wait(&sf_done[k], ((gc >> 1) - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        const int w = 4 * sfg;  // bytes per row
                        mbar_arrive_expect_tx(&sf_loaded[k], (uint32_t)(L::kSfRows * w));
                        const uint32_t sfd = smem_u32(sf_slot(k));
                        tma_load_2d(sfd, &sfa_map, 4 * st, ar0, &sf_loaded[k]);
                        tma_load_2d(sfd + kABox * w, &sfa_map, 4 * st, ar1, &sf_loaded[k]);
                        tma_load_2d(sfd + 128 * w, &sfb_map, 4 * st, br, &sf_loaded[k]);
                        ++gc;
                    }
                    if (gs >= (uint32_t)kStages && !mbar_wait(&stage_free[s], ((gs / kStages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    // the unpacking loads write 8 bytes per 16 codes (the gaps
                    // between them are not written): the weight stage counts
                    // its packed size
                    mbar_arrive_expect_tx(&tma_full[s], (uint32_t)(kABytes / 2 + L::kBBytes));
                    const uint32_t a = smem_u32(stage_a(s));
                    tma_load_2d(a, &a_map, st * kBK, ar0, &tma_full[s]);
                    tma_load_2d(a + kABox * kRowBytes, &a_map, st * kBK, ar1, &tma_full[s]);
                    tma_load_2d(smem_u32(stage_b(s)), &b_map, st * kRowBytes, br + rank * N, &tma_full[s]);
                }
            }
            // wait (bounded) until the last loads landed before the CTA can exit
            for (int d = 0; d < kStages && d < (int)gs; ++d) {
                const uint32_t u = gs - 1 - d;
                if (!mbar_wait(&tma_full[u % kStages], (u / kStages) & 1)) break;
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA
        if (lane == 0 && rank == 0) {
            constexpr int kM = PAIR ? 256 : 128;
            constexpr uint32_t id0 = idesc_x2(kM, 2 * N, 0), id1 = idesc_x2(kM, 2 * N, 1);
            constexpr uint32_t id2 = idesc_x2(kM, 2 * N, 2), id3 = idesc_x2(kM, 2 * N, 3);
            uint32_t gs = 0, it = 0;
            bool ok = true;
            for (int item = cta0; item < items && ok; item += cstep) {
                if (expert_of(item) < 0) continue;
                const uint32_t b = it % kAccBufs;
                if (it >= (uint32_t)kAccBufs && !mbar_wait(&acc_free[b], ((it / kAccBufs) - 1) & 1)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + b * kAccCols;
                for (int st = 0; st < nk; ++st, ++gs) {
                    const int s = gs % kStages;
                    // the scale warps (of both CTAs) arrive once their stage's
                    // loads have landed and its scale factors are in tensor memory
                    if (!mbar_wait(&sf_full[s], (gs / kStages) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sdesc_sw128(smem_u32(stage_a(s)));
                    const uint64_t bd = sdesc_sw128(smem_u32(stage_b(s)));
                    const uint32_t sfa = tmem + (uint32_t)(L::kSfCol0 + s * L::kSfCols);
                    const uint32_t sfb = sfa + 8u;
                    // K = 32 each: +32 bytes in the swizzle atom, scale byte kk
                    if (PAIR) {
                        mma_x2_pair(d_tmem, ad, bd, id0, sfa, sfb, st != 0 ? 1u : 0u);
                        mma_x2_pair(d_tmem, ad + 2u, bd + 2u, id1, sfa, sfb, 1u);
                        mma_x2_pair(d_tmem, ad + 4u, bd + 4u, id2, sfa, sfb, 1u);
                        mma_x2_pair(d_tmem, ad + 6u, bd + 6u, id3, sfa, sfb, 1u);
                        mma_commit_pair(&stage_free[s]);
                    } else {
                        mma_x2(d_tmem, ad, bd, id0, sfa, sfb, st != 0 ? 1u : 0u);
                        mma_x2(d_tmem, ad + 2u, bd + 2u, id1, sfa, sfb, 1u);
                        mma_x2(d_tmem, ad + 4u, bd + 4u, id2, sfa, sfb, 1u);
                        mma_x2(d_tmem, ad + 6u, bd + 6u, id3, sfa, sfb, 1u);
                        mma_commit(&stage_free[s]);
                    }
                }
                if (ok) {
                    if (PAIR)
                        mma_commit_pair(&acc_full[b]);
                    else
                        mma_commit(&acc_full[b]);
                }
                ++it;  // items processed (skipped ones use no accumulator)
            }
            // every MMA this thread issued has completed when this arrives
            if (PAIR)
                mma_commit_pair(drain);
            else
                mma_commit(drain);
            mbar_wait(drain, 0);
        } else if (PAIR && lane == 0) {
            // the odd CTA: the pair's MMAs, and the commits arriving on this
            // CTA's barriers as they complete, are done before it exits
            mbar_wait(drain, 0);
        }
    } else if (warp >= kScaleWarp0 && warp < kEpiWarp0) {
        // ---------------------------------------------------- scale factors
        const int quad = warp & 3;
        const int rho = 32 * quad + lane;  // weight row of the stage = accumulator lane
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)L::kSfCol0;
        const int w = 4 * sfg;  // scale bytes per row in a group slot
        uint32_t gs = 0, gc = 0;
        bool ok = true;
        for (int item = cta0; item < items && ok; item += cstep) {
            if (expert_of(item) < 0) continue;
            for (int st = 0; st < nk; ++st, ++gs) {
                const int s = gs % kStages, k = gc & 1;
                // the stage's scale factors go into tensor memory as soon as
                // the group's bytes are here and the MMAs that last read those
                // columns have completed, ahead of the stage's operands
                if ((st % sfg == 0 && !mbar_wait_warp(&sf_loaded[k], (gc >> 1) & 1)) ||
                    (gs >= (uint32_t)kStages && !mbar_wait_warp(&stage_free[s], ((gs / kStages) - 1) & 1))) {
                    ok = false;
                    break;
                }
                const uint8_t* sf = sf_slot(k) + 4 * (st % sfg);
                uint32_t av[1], bv[L::kBJst];
                av[0] = lds32(sf + rho * w);
#pragma unroll
                for (int j = 0; j < L::kBJst; ++j)
                    bv[j] = j < L::kBJ ? lds32(sf + (128 + 32 * j + lane) * w) : 0u;
                tc_fence_after();
                const uint32_t col = lane_base + (uint32_t)(s * L::kSfCols);
                tmem_st_x<1>(col + (uint32_t)quad, av);
                tmem_st_x<L::kBJst>(col + 8u, bv);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                if (st % sfg == sfg - 1) {  // this warp's reads of the group are done
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sf_done[k]);
                    ++gc;
                }
                // then this CTA's operands of the stage
                if (!mbar_wait_warp(&tma_full[s], (gs / kStages) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive0(&sf_full[s]);
            }
        }
    } else {
        // -------------------------------------------------------- epilogue
        // Each warp copies its (at most two) chunks of D_hi + D_lo out of
        // tensor memory, releases the accumulator, and only then computes
        // and stores: the next item's MMAs wait for the copies alone.
        static_assert(N <= 128, "two chunks per epilogue warp");
        constexpr int kChunks = (N + 63) / 64;  // per warp
        const int quad = warp & 3;                              // lanes 32 quad .. 32 quad + 31
        const int grp = (warp - kEpiWarp0) >> 2;                // chunks 32 grp, 32 grp + 64
        const int et = ((warp - kEpiWarp0) & 3) * 32 + lane;    // gate_up: 0..127 within the group
        float* stg_g = stg + grp * 32 * L::kStgRow;
        uint32_t it = 0;
        for (int item = cta0; item < items; item += cstep) {
            const int tile = item / row_groups, block = block_of(item);
            if (expert_of(item) < 0) continue;
            const uint32_t b = it % kAccBufs;
            // down: the pair of this lane's position in each of the warp's chunks
            int q[kChunks];
#pragma unroll
            for (int j = 0; j < kChunks; ++j) q[j] = -1;
            if (MODE == 1) {
#pragma unroll
                for (int j = 0; j < kChunks; ++j)
                    if (32 * grp + 64 * j < N) q[j] = checked_pair(g, tile * N + 32 * grp + 64 * j + lane);
            }
            // one outcome for the warp, and in gate_up for the group's four
            // warps, which meet at a named barrier below: none may go on to
            // that barrier while another stopped
            bool acc_ok = mbar_wait_warp(&acc_full[b], (it / kAccBufs) & 1);
            if (MODE == 0) acc_ok = all_at_barrier(acc_ok, 1 + grp, kEpiThreads);
            if (!acc_ok) break;
            tc_fence_after();
            uint32_t v[kChunks][32];
#pragma unroll
            for (int j = 0; j < kChunks; ++j) {
                const int c0 = 32 * grp + 64 * j;
                if (c0 >= N) continue;
                const uint32_t taddr = tmem + ((uint32_t)(32 * quad) << 16) + b * kAccCols + (uint32_t)c0;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {  // D_hi + D_lo, 16 columns at a time
                    uint32_t dh[16], dl[16];
                    tmem_ld16_nowait(taddr + 16u * hf, dh);
                    tmem_ld16_nowait(taddr + (uint32_t)N + 16u * hf, dl);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        v[j][16 * hf + i] = __float_as_uint(__uint_as_float(dh[i]) + __uint_as_float(dl[i]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive0(&acc_free[b]);  // this warp's part is drained: the next item may use it
#pragma unroll
            for (int j = 0; j < kChunks; ++j) {
                const int c0 = 32 * grp + 64 * j;
                if (c0 >= N) continue;
                if (MODE == 1) {
                    const int nc = __popc(__ballot_sync(0xFFFFFFFFu, q[j] >= 0));  // pairs form a prefix
                    const int row = block * 128 + 32 * quad + lane;
                    if (g.y_blocked) {
                        store_y16_chunk(g, v[j], 1.0f, block, quad, lane, tile * N + c0, nc, row < g.rows);
                    } else {  // y by pair, times the routing weight
                        const float wq = q[j] >= 0 ? __ldg(g.topk_w + q[j]) : 0.0f;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int qi = __shfl_sync(0xFFFFFFFFu, q[j], i);
                            const float wi = __shfl_sync(0xFFFFFFFFu, wq, i);
                            if (qi >= 0 && row < g.rows)
                                g.y_out[(size_t)qi * g.rows + row] = __uint_as_float(v[j][i]) * wi;
                        }
                    }
                } else {
                    // transpose through shared memory: stg[column][accumulator row]
#pragma unroll
                    for (int i = 0; i < 32; ++i) stg_g[i * L::kStgRow + 32 * quad + lane] = __uint_as_float(v[j][i]);
                    asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(kEpiThreads) : "memory");
                    // thread -> (column, 32-block of i, half): rows 0..63 are the
                    // gate rows of i = block * 64 + row, rows 64..127 the up rows
                    const int hh = et & 1, col = (et >> 1) & 31, blk = et >> 6;
                    const float* gp = stg_g + col * L::kStgRow + 32 * blk + 16 * hh;
                    float a[16];
                    float amax = 0.0f;
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const float4 gv = *reinterpret_cast<const float4*>(gp + 4 * k4);
                        const float4 uv = *reinterpret_cast<const float4*>(gp + 64 + 4 * k4);
                        const float gg[4] = {gv.x, gv.y, gv.z, gv.w}, uu[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            // h = bf16(silu(g) * u), kept as its fp32 value
                            const float hv = __uint_as_float(
                                (uint32_t)f32_to_bf16_bits(silu_fast(gg[k]) * uu[k]) << 16);
                            a[4 * k4 + k] = hv;
                            amax = fmaxf(amax, fabsf(hv));
                        }
                    }
                    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
                    const uint32_t sh = x2_scale_hi(amax), sl = x2_scale_lo(sh);
                    uint4 hq, lq;
                    x2_split16(a, sh, sl, hq, lq);
                    const size_t hrow = (size_t)tile * 2 * N + c0 + col;  // high term; low term N rows on
                    const int i0 = block * 64 + 32 * blk + 16 * hh;
                    *reinterpret_cast<uint4*>(g.hq_codes + hrow * (size_t)g.I + i0) = hq;
                    *reinterpret_cast<uint4*>(g.hq_codes + (hrow + N) * (size_t)g.I + i0) = lq;
                    g.hq_scales[(hrow + (hh ? N : 0)) * (size_t)(g.I / 32) + i0 / 32] = (uint8_t)(hh ? sl : sh);
                    asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(kEpiThreads) : "memory");
                }
            }
            ++it;
        }
    }

    tc_fence_before();
    // neither CTA of a pair releases its tensor memory or shared memory while
    // the other may still arrive there or the pair's MMAs may still run
    if (PAIR)
        cluster_sync_all();
    else
        __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc<PAIR>(tmem, kTmemCols);
    }
    pdl_end();
}

template <int MODE, int N, bool PAIR>
cudaError_t launch_n(const GroupedGemm& g, cudaStream_t s) {
    using L = X2Layout<MODE, N, PAIR>;
    const size_t smem = L::kTotal;
    const void* fn = (const void*)fp8x2_gemm_kernel<MODE, N, PAIR>;
    cudaError_t err = ensure_dynamic_smem(fn, smem);
    if (err != cudaSuccess) return err;
    CUtensorMap a_map, b_map, sfa_map, sfb_map;
    const uint64_t wrows = (uint64_t)g.num_experts * g.rows;
    // codes [wrows][K/2] bytes, unpacked by the TMA to 16 bytes per 16 codes
    err = encode_2d_map(&a_map, g.codes, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, g.K, wrows,
                        (uint64_t)(g.K / 2), kBK, kABox, CU_TENSOR_MAP_SWIZZLE_128B);
    if (err != cudaSuccess) return err;
    err = encode_codes_map(&b_map, g.act, g.K, (uint64_t)g.act_rows, kRowBytes, L::kBRowsCta);
    if (err != cudaSuccess) return err;
    // scale rows of K/32 bytes, boxes of one scale group (the kernel's width)
    const int sfw = 4 * ((g.K / kBK) % 8 == 0 ? 8 : 4);
    err = encode_2d_map(&sfa_map, g.scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.K / 32, wrows,
                        (uint64_t)(g.K / 32), sfw, kABox, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (err != cudaSuccess) return err;
    err = encode_2d_map(&sfb_map, g.act_scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.K / 32,
                        (uint64_t)g.act_rows, (uint64_t)(g.K / 32), sfw, 2 * N, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (err != cudaSuccess) return err;
    const int row_blocks = MODE == 0 ? g.I / 64 : g.rows / 128;
    const long long max_items = (long long)g.max_tiles * (PAIR ? row_blocks / 2 : row_blocks);
    if constexpr (PAIR) {
        // one wave of pairs: as many as can be resident at once (a pair needs
        // two SMs of one GPC)
        int resident = 0;
        err = max_active_pairs(fn, x2_threads<MODE>(), smem, &resident);
        if (err != cudaSuccess) return err;
        const int pairs = (int)std::min<long long>(max_items, (long long)std::max(resident, 1));
        return launch_pdl_cluster(fp8x2_gemm_kernel<MODE, N, true>, dim3(2 * pairs), dim3(x2_threads<MODE>()),
                                  smem, s, 2u, g, a_map, b_map, sfa_map, sfb_map);
    } else {
        const int grid = (int)std::min<long long>(max_items, (long long)num_sms());
        return launch_pdl(fp8x2_gemm_kernel<MODE, N, false>, dim3(grid), dim3(x2_threads<MODE>()), smem, s,
                          g, a_map, b_map, sfa_map, sfb_map);
    }
}

template <int MODE>
cudaError_t launch_mode(const GroupedGemm& g, cudaStream_t s) {
    if (g.max_tiles == 0) return cudaSuccess;
    // CTA pairs from 96-row tiles up; 32- and 64-row tiles run one CTA per
    // weight block (1536-token prefill, 64-row tiles: gate_up 647 us single,
    // 797 us in pairs; skewed 8192-token prefill, 128-row tiles: 1386 us
    // single, 1226 us in pairs)
    switch (g.tile_m) {
        case 32: return launch_n<MODE, 32, false>(g, s);
        case 64: return launch_n<MODE, 64, false>(g, s);
        case 96: return launch_n<MODE, 96, true>(g, s);
        case 128: return launch_n<MODE, 128, true>(g, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool fp8x2_tile_supported(int tile_m) { return tile_m == 32 || tile_m == 64 || tile_m == 96 || tile_m == 128; }
bool fp8x2_shape_supported(int H, int I) { return H % 512 == 0 && I % 512 == 0; }
cudaError_t launch_fp8x2_gate_up(const GroupedGemm& g, cudaStream_t s) { return launch_mode<0>(g, s); }
cudaError_t launch_fp8x2_down(const GroupedGemm& g, cudaStream_t s) { return launch_mode<1>(g, s); }

cudaError_t launch_split_rows(const uint16_t* x, int cols, int rows, const int32_t* sorted_pairs,
                              const int32_t* num_tiles, int tile_n, int Kt, int cap, int num_pairs,
                              uint8_t* q_hi, uint8_t* q_lo, uint8_t* s_hi, uint8_t* s_lo,
                              cudaStream_t s) {
    const int n = sorted_pairs ? cap : rows;
    if (n <= 0) return cudaSuccess;
    const int blocks = std::min((n + 7) / 8, num_sms() * 8);
    return launch_pdl(split_rows_kernel, dim3(blocks), dim3(256), 0, s, reinterpret_cast<const uint4*>(x),
                      cols, rows, sorted_pairs, num_tiles, tile_n, Kt, cap, num_pairs, q_hi, q_lo, s_hi,
                      s_lo);
}

cudaError_t read_device_error_fp8x2(int* flag, int clear) {
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
