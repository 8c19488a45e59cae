// ffn_decode.cu -- small-M grouped MXFP4 GEMMs (decode path) and the combine.
//
// Decode steps move every touched expert's MXFP4 weights once and do little
// arithmetic per byte, so the kernels are built around the weight stream
// (fused MXFP4 MoE kernel with in-register dequantisation: VibeSys
// Qwen3.5-397B on 4x MI300A, sections "baseline" and "kernels and graph
// capture"; narrow N tiles for small M: vLLM MiniMax M3 on MI355X, section
// "local shape and tiling").
//
// A CTA owns one tile (tile_m token rows of one expert, from moe_permute) and
// a block of 256 weight rows (gate_up: 128 gate rows and the 128 matching up
// rows, so the SwiGLU epilogue has g and u in the same registers; down: 256
// rows).  One producer warp streams the block's packed codes into a 4-stage
// shared-memory ring with 2D TMA loads (two 128-row x 128-byte boxes per
// stage, hardware 128-byte swizzle, mbarrier transaction counts); 16
// consumer warps each own 16 rows:
//   * ldmatrix.x4 hands lane c of every row quad the c-th 32-bit word (8
//     codes) of a 32-wide scale group, so each pair of m16n8k16 MMAs sees one
//     scale group per row;
//   * the hardware E2M1 -> f16x2 conversion turns each code byte into two
//     f16 values (every E2M1 value is exact in f16): one conversion per two
//     values, against three integer ops for a bit-placed bf16 pair;
//   * the MMA takes both operands in one type, so the activation rows are
//     carried as f16 scaled by a power of two per row (rows_to_f16_kernel:
//     the row's largest magnitude lands in [2^14, 2^15), so every element at
//     least 2^-29 of it converts exactly and smaller ones are rounded with an
//     error below 2^-39 of it); the row factor is undone in the epilogue;
//   * a staging warp bulk-copies the tile's rows into a double-buffered chunk
//     ahead of the consumers; each group's two MMAs go into a fresh fp32
//     partial that is added to the accumulator times 2^(s-126), an exact
//     power-of-two FMA (the 2^-1 left over is folded into the row factor).
// With consecutive codes converted pairwise, the MMA's k slots of lane c are
// k = 8c .. 8c+7 of the group, so one 16-byte shared load per n-tile gives
// both MMAs' B fragments; a row pitch of 64 bytes past a multiple of 128
// keeps those loads conflict-free.
#include <algorithm>

#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kLoadWarp = kConsumerWarps;        // TMA of the weight codes
constexpr int kStageWarp = kConsumerWarps + 1;   // activation staging
constexpr int kThreads = kConsumers + 64;
constexpr int kRows = 256;                   // weight rows per CTA
constexpr int kStageK = 256;                 // k per pipeline stage
constexpr int kRowBytes = kStageK / 2;       // code bytes per row per stage (one TMA box row)
constexpr int kBoxRows = 128;                // rows per TMA box
constexpr int kStages = 4;
constexpr int kStageBytes = kRows * kRowBytes;
constexpr int kXBytes = 32 * 1024;           // one staged activation chunk (two buffers)
// the group factor is 2^(s-126); the row factor carries the remaining 2^-1
constexpr float kGroupFactorBias = 0.5f;

template <int NT>
struct DecodeSmem {
    static constexpr int TM = NT * 8;
    static constexpr int KC = kXBytes / (TM * 2);  // k per staged activation chunk
    static constexpr int kPitch = KC * 2 + 64;     // bytes per staged row: +4 bank groups per row
    static constexpr int kXBuf = TM * kPitch;      // one staged chunk
    static constexpr int kX = kStages * kStageBytes;
    static constexpr int kBars = kX + 2 * kXBuf;
    static constexpr int kTotal = kBars + (2 * kStages + 4) * 8 + 1024;  // + alignment slack
};

// Weight row (within the expert) held in CTA row rho, or -1 past the end.
template <int MODE>
__device__ __forceinline__ int cta_weight_row(int rho, int block, int I, int rows) {
    if (MODE == 0) {
        const int n = block * 128 + (rho & 127);
        return n < I ? (rho < 128 ? n : I + n) : -1;
    }
    const int m = block * kRows + rho;
    return m < rows ? m : -1;
}

// Eight codes (two per byte, the even k in the low nibble) -> four f16x2:
// out[i] = (code 2i, code 2i + 1), low half first.
__device__ __forceinline__ void codes_to_f16x2(uint32_t w, uint32_t out[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
        : "r"(w));
}

// Persistent kernel: CTA b processes work items b, b + gridDim.x, ... where
// item = tile * row_blocks + block.  Two helper warps run ahead of the 16
// consumer warps across items: one streams the weight codes (TMA ring), one
// copies the tiles' f16 activation rows into a double-buffered chunk.
// Consumers only wait on mbarriers.
template <int MODE, int NT>
__global__ void __launch_bounds__(kThreads, 1)
    decode_gemm_kernel(const GroupedGemm g, const __grid_constant__ CUtensorMap codes_map) {
    pdl_begin();
    using L = DecodeSmem<NT>;
    constexpr int TM = L::TM;
    constexpr int KC = L::KC;
    extern __shared__ uint8_t smem_raw[];
    // the 128-byte swizzle pattern repeats every 1024 bytes: align the ring
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* codes_s = smem;
    uint8_t* xs_s = smem + L::kX;  // [2][TM] rows of kPitch bytes
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBars);
    uint64_t* empty = full + kStages;
    uint64_t* xfull = empty + kStages;  // [2] staged chunk ready
    uint64_t* xempty = xfull + 2;       // [2] staged chunk consumed

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = g.K;
    const int nsteps = (K + kStageK - 1) / kStageK;
    const int nchunks = (K + KC - 1) / KC;
    const int row_blocks = MODE == 0 ? (g.I + 127) / 128 : (g.rows + kRows - 1) / kRows;
    const int items = checked_tiles(g) * row_blocks;

    // staged rows past K and padding rows are never copied: start them at zero
    for (int i = tid; i < 2 * L::kXBuf / 16; i += kThreads)
        reinterpret_cast<uint4*>(xs_s)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&xfull[b], 1);
            mbar_init(&xempty[b], kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kLoadWarp) {
        // ------------------------------------------------- weight codes (TMA)
        if (lane == 0) {
            uint32_t gs = 0;
            for (int item = blockIdx.x; item < items; item += gridDim.x) {
                const int tile = item / row_blocks, block = item % row_blocks;
                const int e = checked_expert(g, tile, block == 0);
                if (e < 0) continue;  // skipped by every role
                // rows of the two boxes in the map's row space (experts stacked);
                // rows past this expert's block are loaded too and never used
                const int row0 = e * g.rows + (MODE == 0 ? block * 128 : block * kRows);
                const int row1 = MODE == 0 ? e * g.rows + g.I + block * 128 : row0 + kBoxRows;
                for (int st = 0; st < nsteps; ++st, ++gs) {
                    const int s = gs % kStages;
                    if (gs >= kStages && !mbar_wait(&empty[s], ((gs / kStages) - 1) & 1)) return;
                    mbar_arrive_expect_tx(&full[s], (uint32_t)kStageBytes);
                    const uint32_t dst = smem_u32(codes_s + s * kStageBytes);
                    tma_load_2d(dst, &codes_map, st * kRowBytes, row0, &full[s]);
                    tma_load_2d(dst + kBoxRows * kRowBytes, &codes_map, st * kRowBytes, row1, &full[s]);
                }
            }
        }
        return;
    }

    if (warp == kStageWarp) {
        // ------------------------------------------- activation staging
        // the f16 activation rows (rows_to_f16_kernel) are plain contiguous
        // copies: one bulk copy per tile row per chunk
        uint32_t gc = 0;
        for (int item = blockIdx.x; item < items; item += gridDim.x) {
            const int tile = item / row_blocks;
            if (checked_expert(g, tile, false) < 0) continue;
            int arow[TM > 32 ? 2 : 1];
            uint32_t valid = 0;
#pragma unroll
            for (int h = 0; h < (TM > 32 ? 2 : 1); ++h) {
                const int j = lane + 32 * h;
                const int q = j < TM ? checked_pair(g, tile * TM + j) : -1;
                arow[h] = q < 0 ? -1 : (g.act_by_token ? q / g.Kt : tile * TM + j);
                valid += __popc(__ballot_sync(0xFFFFFFFFu, arow[h] >= 0));
            }
            for (int c = 0; c < nchunks; ++c, ++gc) {
                const int b = gc & 1;
                if (gc >= 2 && !mbar_wait_warp(&xempty[b], ((gc >> 1) - 1) & 1)) return;
                const int kc = c * KC;
                const uint32_t bytes = (uint32_t)min(KC, K - kc) * 2u;
                if (lane == 0) mbar_arrive_expect_tx(&xfull[b], valid * bytes);
                __syncwarp();
                const uint32_t dst = smem_u32(xs_s) + b * L::kXBuf;
#pragma unroll
                for (int h = 0; h < (TM > 32 ? 2 : 1); ++h) {
                    const int j = lane + 32 * h;
                    if (arow[h] >= 0)
                        bulk_copy_g2s(dst + j * L::kPitch, g.act + (size_t)arow[h] * K + kc, bytes,
                                      &xfull[b]);
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int r = lane >> 2, c = lane & 3;
    const bool scales_vec = (K % kStageK) == 0 && ((reinterpret_cast<uintptr_t>(g.scales) & 7) == 0);
    const size_t sbytes = (size_t)K / 32;
    // ldmatrix: matrix j = lane / 8 (0: rows r, group 2gp; 1: rows r + 8, group
    // 2gp; 2, 3: the same for group 2gp + 1).  The TMA swizzle stores 16-byte
    // chunk q of row rho at chunk q ^ (rho % 8), here q = 2gp + j/2.
    const int mj = lane >> 3, mi = lane & 7;
    const int lrho = MODE == 0 ? ((mj & 1) ? 128 : 0) + 8 * warp + mi : 16 * warp + (mj & 1) * 8 + mi;
    uint32_t lm_off[4];
#pragma unroll
    for (int gp = 0; gp < 4; ++gp)
        lm_off[gp] = smem_u32(codes_s) + lrho * kRowBytes + (((2 * gp + (mj >> 1)) ^ mi) << 4);
    // staged activations of row r: group gl of a stage at byte 64 * gl + 16 * c
    const uint32_t xb = smem_u32(xs_s) + (uint32_t)(r * L::kPitch + c * 16);

    uint32_t gs = 0, gc = 0;
    bool failed = false;
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const int tile = item / row_blocks, block = item % row_blocks;
        const int e = checked_expert(g, tile, false);
        if (e < 0) continue;
        int qj[NT][2];  // pair index of this lane's two columns per n-tile (-1 = padding)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int u = 0; u < 2; ++u) qj[n][u] = checked_pair(g, tile * TM + n * 8 + 2 * c + u);
        const int rho0 = MODE == 0 ? 8 * warp + r : 16 * warp + r;
        const int rho1 = MODE == 0 ? 128 + 8 * warp + r : 16 * warp + 8 + r;
        const int wr0 = cta_weight_row<MODE>(rho0, block, g.I, g.rows);
        const int wr1 = cta_weight_row<MODE>(rho1, block, g.I, g.rows);
        const uint8_t* sp0 = g.scales + ((size_t)e * g.rows + max(wr0, 0)) * sbytes;
        const uint8_t* sp1 = g.scales + ((size_t)e * g.rows + max(wr1, 0)) * sbytes;
        auto load_scales = [&](int st, uint2& s0, uint2& s1) {
            if (scales_vec) {
                s0 = wr0 >= 0 ? __ldg(reinterpret_cast<const uint2*>(sp0 + st * 8)) : make_uint2(0, 0);
                s1 = wr1 >= 0 ? __ldg(reinterpret_cast<const uint2*>(sp1 + st * 8)) : make_uint2(0, 0);
            } else {
                uint32_t a[2] = {0, 0}, bb[2] = {0, 0};
                for (int gl = 0; gl < 8; ++gl) {
                    const int gidx = st * 8 + gl;
                    if (gidx * 32 < K) {
                        if (wr0 >= 0) a[gl >> 2] |= (uint32_t)__ldg(sp0 + gidx) << (8 * (gl & 3));
                        if (wr1 >= 0) bb[gl >> 2] |= (uint32_t)__ldg(sp1 + gidx) << (8 * (gl & 3));
                    }
                }
                s0 = make_uint2(a[0], a[1]);
                s1 = make_uint2(bb[0], bb[1]);
            }
        };
        uint2 nsc0, nsc1;
        load_scales(0, nsc0, nsc1);
        float acc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;

        uint32_t xbuf = 0;
        for (int st = 0; st < nsteps; ++st, ++gs) {
            const int kst = st * kStageK;
            if (kst % KC == 0) {  // first stage of a staged chunk
                xbuf = (gc & 1) * L::kXBuf;
                if (!failed && !mbar_wait_warp(&xfull[gc & 1], (gc >> 1) & 1)) failed = true;
            }
            const int s = gs % kStages;
            const uint2 sc0 = nsc0, sc1 = nsc1;
            if (st + 1 < nsteps) load_scales(st + 1, nsc0, nsc1);
            if (!failed && !mbar_wait_warp(&full[s], (gs / kStages) & 1)) failed = true;
            if (!failed) {
                const uint32_t soff = s * kStageBytes;
                const uint32_t xoff = xbuf + (uint32_t)(kst % KC) * 2u;  // bytes into the staged rows
#pragma unroll
                for (int gp = 0; gp < 4; ++gp) {
                    uint32_t w[4];
                    ldmatrix_x4(lm_off[gp] + soff, w);
#pragma unroll
                    for (int gi = 0; gi < 2; ++gi) {
                        const int gl = 2 * gp + gi;
                        const uint32_t b0 = __byte_perm(gl < 4 ? sc0.x : sc0.y, 0, 0x4440 + (gl & 3));
                        const uint32_t b1 = __byte_perm(gl < 4 ? sc1.x : sc1.y, 0, 0x4440 + (gl & 3));
                        // 2^(s - 126) as fp32 bits: (s + 1) << 23, by multiply-add
                        const float f0 = __uint_as_float(b0 * g.exp_one + g.exp_bias);
                        const float f1 = __uint_as_float(b1 * g.exp_one + g.exp_bias);
                        uint32_t ta[4], tb[4];
                        codes_to_f16x2(w[gi ? 2 : 0], ta);
                        codes_to_f16x2(w[gi ? 3 : 1], tb);
                        const uint32_t xa = xb + xoff + 64u * gl;
#pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            uint4 bv;
                            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                         : "=r"(bv.x), "=r"(bv.y), "=r"(bv.z), "=r"(bv.w)
                                         : "r"(xa + (uint32_t)(n * 8 * L::kPitch)));
                            float t4[4];
                            mma_f16_16816_z(t4, ta[0], tb[0], ta[1], tb[1], bv.x, bv.y);
                            mma_f16_16816_acc(t4, ta[2], tb[2], ta[3], tb[3], bv.z, bv.w);
                            acc[n][0] = fmaf(t4[0], f0, acc[n][0]);
                            acc[n][1] = fmaf(t4[1], f0, acc[n][1]);
                            acc[n][2] = fmaf(t4[2], f1, acc[n][2]);
                            acc[n][3] = fmaf(t4[3], f1, acc[n][3]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if ((kst + kStageK) % KC == 0 || st + 1 == nsteps) {  // last stage of the chunk
                if (lane == 0) mbar_arrive(&xempty[gc & 1]);
                ++gc;
            }
        }

        if (!failed) {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int j = n * 8 + 2 * c + u;
                    const int q = qj[n][u];
                    if (q < 0) continue;
                    if (MODE == 0) {
                        const float rs = __ldg(g.act_rscale + q / g.Kt) * kGroupFactorBias;
                        if (wr0 >= 0)
                            g.h_out[(size_t)(tile * TM + j) * g.I + wr0] =
                                f32_to_bf16_bits(silu(acc[n][u] * rs) * (acc[n][2 + u] * rs));
                    } else {
                        const float wq = __ldg(g.topk_w + q);
                        const float rs = __ldg(g.act_rscale + tile * TM + j) * kGroupFactorBias;
                        float* y = g.y_out + (size_t)q * g.rows;
                        if (wr0 >= 0) y[wr0] = wq * (acc[n][u] * rs);
                        if (wr1 >= 0) y[wr1] = wq * (acc[n][2 + u] * rs);
                    }
                }
            }
        }
    }
    pdl_end();
}

template <int MODE, int NT>
cudaError_t launch_nt(const GroupedGemm& g, const CUtensorMap& map, cudaStream_t s) {
    const size_t smem = DecodeSmem<NT>::kTotal;
    cudaError_t err = ensure_dynamic_smem((const void*)decode_gemm_kernel<MODE, NT>, smem);
    if (err != cudaSuccess) return err;
    const int row_blocks = MODE == 0 ? (g.I + 127) / 128 : (g.rows + kRows - 1) / kRows;
    const long long max_items = (long long)g.max_tiles * row_blocks;
    const int grid = (int)std::min<long long>(max_items, (long long)num_sms());
    return launch_pdl(decode_gemm_kernel<MODE, NT>, dim3(grid), dim3(kThreads), smem, s, g, map);
}

template <int MODE>
cudaError_t launch_mode(const GroupedGemm& g, cudaStream_t s) {
    if (g.max_tiles == 0) return cudaSuccess;
    // the packed codes of all experts as one 2D uint8 tensor [Et * rows, K / 2]
    CUtensorMap map;
    cudaError_t err = encode_codes_map(&map, g.codes, g.K / 2, (uint64_t)g.num_experts * g.rows,
                                       kRowBytes, kBoxRows);
    if (err != cudaSuccess) return err;
    switch (g.tile_m) {
        case 8: return launch_nt<MODE, 1>(g, map, s);
        case 16: return launch_nt<MODE, 2>(g, map, s);
        case 32: return launch_nt<MODE, 4>(g, map, s);
        case 64: return launch_nt<MODE, 8>(g, map, s);
        default: return cudaErrorInvalidValue;
    }
}

// One warp per row: dst[row] = f16(src[row] * 2^sigma) and rscale[row] =
// 2^-sigma, with sigma = 14 - floor(log2(max |src[row]|)) clamped to
// [-113, 112] (0 for an all-zero row), so the row's largest magnitude lands
// in [2^14, 2^15).  bf16 has fewer significant bits than f16, so every
// element that stays in the f16 normal range converts exactly.  Rows are
// either all `rows` rows, or (sorted_pairs given) the positions of the used
// tiles that hold a pair.  src may equal dst: each lane reads its elements
// before it writes them.  independent: the rows are the caller's input (x),
// read and written by no kernel between the last one that waited on its
// predecessors and this one, so the work runs before the wait on the
// previous kernel and overlaps it (the permutation, which signals its
// dependents as soon as its own wait is over); every thread still waits
// before it exits, so this grid completes only after its predecessor has.
__global__ void __launch_bounds__(256) rows_to_f16_kernel(const uint16_t* src, uint16_t* dst,
                                                          int cols, int rows,
                                                          const int32_t* __restrict__ sorted_pairs,
                                                          const int32_t* __restrict__ num_tiles,
                                                          int tile_m, float* __restrict__ rscale,
                                                          int independent) {
    if (!independent) pdl_begin();
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    bool active = row < rows;
    if (active && sorted_pairs)
        active = row < __ldg(num_tiles) * tile_m && __ldg(sorted_pairs + row) >= 0;
    if (active) {
        const uint4* s4 = reinterpret_cast<const uint4*>(src + (size_t)row * cols);
        uint4* d4 = reinterpret_cast<uint4*>(dst + (size_t)row * cols);
        const int n16 = cols / 8;
        uint32_t mx = 0;  // max |bf16| bit pattern (orders like the magnitude)
        for (int i = lane; i < n16; i += 32) {
            const uint4 v = s4[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) mx = max(mx, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        const int sigma = row_f16_shift(mx);
        const float up = __uint_as_float((uint32_t)(127 + sigma) << 23);
        for (int i = lane; i < n16; i += 32) {
            const uint4 v = s4[i];
            d4[i] = make_uint4(bf16x2_to_f16x2_scaled(v.x, up), bf16x2_to_f16x2_scaled(v.y, up),
                               bf16x2_to_f16x2_scaled(v.z, up), bf16x2_to_f16x2_scaled(v.w, up));
        }
        if (lane == 0) rscale[row] = __uint_as_float((uint32_t)(127 - sigma) << 23);
    }
    if (independent) pdl_begin();
    pdl_end();
}

// out[t][m] = bf16(sum over j ascending of y[t*Kt + j][m], then + y2[t][m] when
// y2 is given: a shared expert run as a separate dense MLP comes last, where
// the fused shared slot K would be); four columns per thread.  Four slots'
// loads are issued before their adds (the sum keeps slot order): a thread
// then waits on about Kt / 4 load round trips instead of Kt.
__global__ void __launch_bounds__(256) combine_kernel(const float4* __restrict__ y,
                                                      const float4* __restrict__ y2, int T, int H4,
                                                      int Kt, uint2* __restrict__ out) {
    pdl_begin();
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)T * H4) return;
    const size_t t = i / H4, m = i % H4;
    const float4* yt = y + t * Kt * H4 + m;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < Kt; j0 += 4) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (j0 + u < Kt) v[u] = __ldg(yt + (size_t)(j0 + u) * H4);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (j0 + u >= Kt) break;
            a.x += v[u].x;
            a.y += v[u].y;
            a.z += v[u].z;
            a.w += v[u].w;
        }
    }
    if (y2) {
        const float4 v = __ldg(y2 + t * H4 + m);
        a.x += v.x;
        a.y += v.y;
        a.z += v.z;
        a.w += v.w;
    }
    uint2 o;
    o.x = (uint32_t)f32_to_bf16_bits(a.x) | ((uint32_t)f32_to_bf16_bits(a.y) << 16);
    o.y = (uint32_t)f32_to_bf16_bits(a.z) | ((uint32_t)f32_to_bf16_bits(a.w) << 16);
    out[i] = o;
    pdl_end();
}

}  // namespace

bool decode_tile_supported(int tile_m) {
    return tile_m == 8 || tile_m == 16 || tile_m == 32 || tile_m == 64;
}

cudaError_t launch_decode_gate_up(const GroupedGemm& g, cudaStream_t s) { return launch_mode<0>(g, s); }
cudaError_t launch_decode_down(const GroupedGemm& g, cudaStream_t s) { return launch_mode<1>(g, s); }

cudaError_t launch_rows_to_f16(const uint16_t* src, uint16_t* dst, int cols, int rows,
                               const int32_t* sorted_pairs, const int32_t* num_tiles, int tile_m,
                               float* rscale, cudaStream_t s, bool independent) {
    if (rows <= 0) return cudaSuccess;
    return launch_pdl(rows_to_f16_kernel, dim3((rows + 7) / 8), dim3(256), 0, s, src, dst, cols,
                      rows, sorted_pairs, num_tiles, tile_m, rscale, independent ? 1 : 0);
}

// Waits on a barrier that nothing arrives at: the bounded wait gives up after
// limit_ns, raises the device error flag and the kernel returns.
static __global__ void wait_selftest_kernel(unsigned long long limit_ns) {
    pdl_begin();
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_for(&bar, 0, limit_ns);
    pdl_end();
}

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t s) {
    return launch_pdl(wait_selftest_kernel, dim3(1), dim3(32), 0, s, limit_ns);
}

// Two warps whose waits end differently: warp 0 waits on a barrier nothing
// arrives at (gives up after limit_ns), warp 1 on one whose phase has already
// completed.  Each warp makes its outcome uniform, the two reduce it at named
// barrier 1, and only if both succeeded do they meet there again -- the
// pattern of the GEMM epilogues, whose warps meet at a named barrier after
// their accumulator wait.  outcome[w] = the outcome warp w acted on (0: both
// stop; warp 1 is not left waiting at the barrier for warp 0).
static __global__ void wait_split_selftest_kernel(unsigned long long limit_ns, int32_t* outcome) {
    pdl_begin();
    __shared__ uint64_t bar[2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive(&bar[1]);  // phase 0 of bar[1] completes
    }
    __syncthreads();
    bool ok = mbar_wait_for(&bar[warp], 0, warp == 0 ? limit_ns : kWaitLimitNs);
    ok = __all_sync(0xFFFFFFFFu, ok) != 0;
    ok = all_at_barrier(ok, 1, 64);
    if (ok) asm volatile("bar.sync 1, 64;" ::: "memory");
    if (lane == 0) outcome[warp] = ok ? 1 : 0;
    pdl_end();
}

cudaError_t launch_wait_split_selftest(unsigned long long limit_ns, int32_t* outcome,
                                       cudaStream_t s) {
    return launch_pdl(wait_split_selftest_kernel, dim3(1), dim3(64), 0, s, limit_ns, outcome);
}

cudaError_t read_device_error_decode(int* flag, int clear) {
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

cudaError_t launch_combine(const float* y, const float* y2, int T, int H, int Kt, uint16_t* out,
                           cudaStream_t s) {
    const size_t n = (size_t)T * (H / 4);
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    const unsigned blocks = (unsigned)((n + threads - 1) / threads);
    return launch_pdl(combine_kernel, dim3(blocks), dim3(threads), 0, s,
                      reinterpret_cast<const float4*>(y), reinterpret_cast<const float4*>(y2), T,
                      H / 4, Kt, reinterpret_cast<uint2*>(out));
}

// The trivial grouping of a single dense expert over all T tokens (Kt = 1):
// sorted_pairs[p] = p for p < T, -1 after; every used tile belongs to expert
// 0; weights fill `w` with 1 when no per-token weights are given.
static __global__ void __launch_bounds__(256) identity_perm_kernel(int T, int tile_m, int cap,
                                                            int max_tiles,
                                                            int32_t* __restrict__ sorted_pairs,
                                                            int32_t* __restrict__ tile_expert,
                                                            int32_t* __restrict__ num_tiles,
                                                            float* __restrict__ ones) {
    pdl_begin();
    const int nt = (T + tile_m - 1) / tile_m;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < cap; i += gridDim.x * blockDim.x) {
        sorted_pairs[i] = i < T ? i : -1;
        if (i < max_tiles) tile_expert[i] = i < nt ? 0 : -1;
        if (ones && i < T) ones[i] = 1.0f;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) *num_tiles = nt;
    pdl_end();
}

cudaError_t launch_identity_perm(int T, int tile_m, int cap, int max_tiles, int32_t* sorted_pairs,
                                 int32_t* tile_expert, int32_t* num_tiles, float* ones,
                                 cudaStream_t s) {
    const int blocks = std::max(1, std::min((cap + 255) / 256, num_sms() * 4));
    return launch_pdl(identity_perm_kernel, dim3(blocks), dim3(256), 0, s, T, tile_m, cap,
                      max_tiles, sorted_pairs, tile_expert, num_tiles, ones);
}

}  // namespace moe
