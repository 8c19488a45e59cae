// moe_internal.h -- launchers shared between the libmoe translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe_device.cuh"

namespace moe {

// Raises a kernel's dynamic shared memory limit once per device (idempotent;
// the attribute is per function, so it stays set for later calls).
cudaError_t ensure_dynamic_smem(const void* func, size_t bytes);

// 2D TMA descriptor of a packed uint8 matrix [rows, row_bytes] (row-major),
// box [box_rows, box_bytes], 128-byte swizzle, zero fill out of bounds.
cudaError_t encode_codes_map(CUtensorMap* map, const void* base, int row_bytes, uint64_t rows,
                             int box_bytes, int box_rows);

// General 2D TMA descriptor: `inner` elements per row, `rows` rows,
// `row_stride` bytes between rows, box [box_rows, box_inner] elements.
cudaError_t encode_2d_map(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int inner,
                          uint64_t rows, uint64_t row_stride, int box_inner, int box_rows,
                          CUtensorMapSwizzle swizzle);

cudaError_t launch_route(const float* logits, const float* shared_w, int T, int E, int K,
                         int with_shared, int renormalize, int32_t* ids, float* w, cudaStream_t s);
// Routing and permutation in one single-block launch (small batches).
cudaError_t launch_route_permute(const float* logits, const float* shared_w, int T, int E, int K,
                                 int with_shared, int renormalize, int tile_m, int cap,
                                 int max_tiles, int32_t* ids, float* w, int32_t* sorted_pairs,
                                 int32_t* offsets, int32_t* inv, int32_t* tile_expert,
                                 int32_t* num_tiles, cudaStream_t s);

size_t permute_smem_bytes(int Et);
cudaError_t launch_permute(const int32_t* ids, int T, int Kt, int Et, int tile_m, int cap,
                           int max_tiles, int32_t* sorted_pairs, int32_t* offsets, int32_t* inv,
                           int32_t* tile_expert, int32_t* num_tiles, cudaStream_t s);

// Arguments of one grouped MXFP4 GEMM (swap-AB: weight rows are the MMA's M
// side, the tile's token rows its N side).
struct GroupedGemm {
    const uint8_t* codes;        // [Et][rows][K/2]
    const uint8_t* scales;       // [Et][rows][K/32]
    int rows;                    // weight rows per expert (2I for gate_up, H for down)
    int K;                       // reduction length (H for gate_up, I for down)
    const uint16_t* act;         // B rows: x [T][H] (gate_up) or h [cap][I] (down); bf16,
                                 // or f16 scaled per row (decode path)
    const float* act_rscale;     // decode path: factor undoing each act row's scaling
    int act_by_token;            // 1: B row = token q / Kt of the pair; 0: B row = sorted position
    const int32_t* sorted_pairs;
    const int32_t* tile_expert;
    const int32_t* num_tiles;
    int Kt;
    int num_experts;             // Et (experts stacked in codes / scales)
    int act_rows;                // rows of `act` (T for x, cap for h)
    int tile_m;
    int max_tiles;
    int num_pairs;               // T * Kt: valid pair indices are [0, num_pairs)
    int I;                       // SwiGLU: gate rows [0, I), up rows [I, 2I)
    uint16_t* h_out;             // SwiGLU output h [cap][I] (bf16)
    float* y_out;                // weighted output [T*Kt][H] (fp32)
    const float* topk_w;
    // MXFP4-activation GEMMs: B rows are packed E2M1 codes ([act_rows][K/2],
    // passed in `act`) with E8M0 scales act_scales ([T][K/32] by token for
    // gate_up, [cap][K/32] by sorted position for down); gate_up writes h as
    // codes hq_codes [cap][I/2] and scales hq_scales [cap][I/32]
    const uint8_t* act_scales;
    uint8_t* hq_codes;
    uint8_t* hq_scales;
    // 1: B scales are tile-ordered rows ([cap][K/32], K % 512 == 0) that the
    // producer loads by TMA with the codes; 0: scale warps load them (by
    // token for gate_up, by position for down)
    int sf_tma;
    int y_blocked;               // down: y by sorted position instead of [pair][rows], without
                                 // the column factor, staged as the f16 rows below
    // y16_out [act_rows][y_rows_pad] holds f16(y * 2^shift),
    // y_shift [ceil(act_rows/32)][y_rows_pad/8] the shift of each (8 output
    // rows, 32 positions) group, y_rows_pad = rows rounded up to 128
    uint16_t* y16_out = nullptr;
    int8_t* y_shift = nullptr;
    int y_rows_pad = 0;
    // decode group factor 2^(s-126) as fp32 bits s * exp_one + exp_bias,
    // taken as runtime values so the multiply-add stays one instruction
    uint32_t exp_one = 1u << 23, exp_bias = 1u << 23;
};

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel in the stream is still running; every kernel of
// the library begins with pdl_begin(), which waits for that kernel to finish.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// launch_pdl for a kernel launched as clusters of `cluster_x` CTAs along x
// (gridDim.x a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t s, unsigned cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Clusters of two CTAs of `func` (block threads, dynamic shared memory
// bytes) that can be resident at once on the current device (cached per
// device and function).
cudaError_t max_active_pairs(const void* func, int threads, size_t smem, int* pairs);

// Streaming multiprocessors of the current device (cached per device).
int num_sms();

bool decode_tile_supported(int tile_m);
bool prefill_tile_supported(int tile_m);
bool prefill_shape_supported(int H, int I);

cudaError_t launch_decode_gate_up(const GroupedGemm& g, cudaStream_t s);
// dst[row] = f16(src[row] * 2^sigma_row), rscale[row] = 2^-sigma_row (the
// decode GEMMs' B rows); every row, or with sorted_pairs the used positions
// that hold a pair.  src may equal dst.  independent: src is the layer's
// input, touched by no kernel since the last one that waited on all before
// it, so the conversion may overlap its predecessor (see rows_to_f16_kernel).
cudaError_t launch_rows_to_f16(const uint16_t* src, uint16_t* dst, int cols, int rows,
                               const int32_t* sorted_pairs, const int32_t* num_tiles, int tile_m,
                               float* rscale, cudaStream_t s, bool independent = false);
cudaError_t launch_decode_down(const GroupedGemm& g, cudaStream_t s);
cudaError_t launch_prefill_gate_up(const GroupedGemm& g, cudaStream_t s);
// xg[p] = f16(x[t] * 2^sigma_t), t = sorted_pairs[p] / Kt, for the rows of
// the used tiles (0 for pads), rscale[t] = 2^-sigma_t (the conversion of
// launch_rows_to_f16, applied while gathering x (bf16) into tile order)
cudaError_t launch_gather_rows_f16(const uint16_t* x, int H, const int32_t* sorted_pairs,
                                   const int32_t* num_tiles, int tile_m, int Kt, int cap,
                                   int num_pairs, uint16_t* xg, float* rscale, cudaStream_t s);
cudaError_t launch_prefill_down(const GroupedGemm& g, cudaStream_t s);
cudaError_t read_device_error_prefill(int* flag, int clear);
// one block waiting on a barrier that never completes, for limit_ns
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t s);
// two warps, one wait giving up and one completing; outcome[2] (device) gets
// the outcome each warp acted on
cudaError_t launch_wait_split_selftest(unsigned long long limit_ns, int32_t* outcome,
                                       cudaStream_t s);
cudaError_t read_device_error_decode(int* flag, int clear);
// out = bf16(sum of the Kt slot rows of y, then + y2's row when y2 is not null)
cudaError_t launch_combine(const float* y, const float* y2, int T, int H, int Kt, uint16_t* out,
                           cudaStream_t s);
// Items of a grouped GEMM launch: the device's tile count, clamped to the
// tiles the buffers hold (a larger count is flagged as an index error).
__device__ __forceinline__ int checked_tiles(const GroupedGemm& g) {
    const int nt = __ldg(g.num_tiles);
    if (nt < 0 || nt > g.max_tiles) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag_index_error();
        return nt < 0 ? 0 : g.max_tiles;
    }
    return nt;
}

// The expert of a tile, or -1 (flagged) when it is outside [0, num_experts).
__device__ __forceinline__ int checked_expert(const GroupedGemm& g, int tile, bool flag) {
    const int e = __ldg(g.tile_expert + tile);
    if ((unsigned)e >= (unsigned)g.num_experts) {
        if (flag) flag_index_error();
        return -1;
    }
    return e;
}

// A sorted position's pair index, or -1 for padding and (flagged) out of range.
__device__ __forceinline__ int checked_pair(const GroupedGemm& g, int pos) {
    const int q = __ldg(g.sorted_pairs + pos);
    if (q >= g.num_pairs) {
        flag_index_error();
        return -1;
    }
    return q;
}

// One 32-column chunk of a down item's y (the prefill and MXFP4-activation
// down GEMMs), staged as f16 rows by sorted position (y16_out [act_rows][y_rows_pad]) scaled by a power of two per
// (8 output rows, 32 positions): lane `lane` of quadrant
// `quad` holds output row 32 quad + lane of the block, v[i] the accumulator of
// column col0 + i (col0 = the chunk's first sorted position, a multiple of 32), fr
// the row factor.  The largest |y| over the chunk's nc columns that hold a
// pair and the 8 rows of the lane's group (three exchanges) sets the shift
// that moves it into [2^14, 2^15); each element is stored as f16(y * 2^shift)
// (relative error at most 2^-11 for every element within 2^28 of that
// largest) and the group's shift as one byte at
// y_shift[col0 / 32][(block * 128 + row) / 8].  row_ok = the output row
// exists.  All 32 lanes call it.
__device__ __forceinline__ void store_y16_chunk(const GroupedGemm& g, const uint32_t v[32], float fr,
                                                int block, int quad, int lane, int col0, int nc,
                                                bool row_ok) {
    float y[32];
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        y[i] = __uint_as_float(v[i]) * fr;
        if (i < nc) mx = fmaxf(mx, fabsf(y[i]));
    }
    if (!row_ok) mx = 0.0f;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    if (!row_ok) return;
    const int sh = f32_f16_shift(__float_as_uint(mx));
    const float up = __uint_as_float((uint32_t)(127 + sh) << 23);
    const int row = block * 128 + 32 * quad + lane;
    uint16_t* yb = g.y16_out + (size_t)col0 * g.y_rows_pad + row;
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const __half2 h = __floats2half2_rn(y[i] * up, y[i + 1] * up);
        if (i < nc) yb[(size_t)i * g.y_rows_pad] = __half_as_ushort(__low2half(h));
        if (i + 1 < nc) yb[(size_t)(i + 1) * g.y_rows_pad] = __half_as_ushort(__high2half(h));
    }
    if ((lane & 7) == 0) g.y_shift[(size_t)(col0 / 32) * (g.y_rows_pad / 8) + row / 8] = (int8_t)sh;
}

// MXFP4 activations: codes [rows][cols/2] and scales [rows][cols/32] of bf16
// rows (cols a multiple of 32), OCP MX rounding (see ffn_mxfp4act.cu).
cudaError_t launch_quantize_mxfp4(const uint16_t* x, int rows, int cols, uint8_t* codes,
                                  uint8_t* scales, cudaStream_t s);
bool mxfp4act_tile_supported(int tile_m);
bool mxfp4act_shape_supported(int H, int I);
// MXFP4 token rows into tile order: codes [T][H/2] -> [cap][H/2] and, when
// with_scales (H % 512 == 0), scales [T][H/32] -> [cap][H/32]; zeros for pads
cudaError_t launch_gather_mx_rows(const uint8_t* xc, const uint8_t* xs, int H, bool with_scales,
                                  const int32_t* sorted_pairs, const int32_t* num_tiles, int tile_m,
                                  int Kt, int cap, int num_pairs, uint8_t* xgc, uint8_t* xgs,
                                  cudaStream_t s);
// w_pos[p] = topk_w[sorted_pairs[p]] (times rscale[p] when given) for the
// used positions, 0 for padding
cudaError_t launch_position_weights(const int32_t* sorted_pairs, const float* topk_w,
                                    const float* rscale, const int32_t* num_tiles, int tile_m,
                                    int cap, int num_pairs, float* w_pos, cudaStream_t s);
// out[t, m] = bf16(sum over the Kt slots j ascending of f[p] * y[p][m]), p =
// inv[t * Kt + j], for y staged by the down epilogues (store_y16_chunk) as f16
// rows by position with a power-of-two shift per (8 output rows, 32
// positions): y = y16 * 2^-shift (exact); f null: factor 1
cudaError_t launch_combine_blocked_f16(const uint16_t* y16, const int8_t* shift, const int32_t* inv,
                                       const float* f, int T, int H, int Kt, int cap, uint16_t* out,
                                       cudaStream_t s);
// block-scaled MXFP4 x MXFP4 grouped GEMMs (tcgen05 kind::mxf4)
cudaError_t launch_mxfp4act_gate_up(const GroupedGemm& g, cudaStream_t s);
cudaError_t launch_mxfp4act_down(const GroupedGemm& g, cudaStream_t s);
cudaError_t read_device_error_mxfp4act(int* flag, int clear);

// bf16 activations as two E4M3 terms on the block-scaled tensor cores
// (tcgen05 kind::mxf8f6f4, ffn_fp8x2.cu).  B rows of a tile of N positions:
// N high-term rows, then N low-term rows (act [max_tiles * 2N][K] bytes, E8M0
// scales act_scales [max_tiles * 2N][K/32]); gate_up writes h in the same form
// (hq_codes [max_tiles * 2N][I], hq_scales [max_tiles * 2N][I/32]).
bool fp8x2_tile_supported(int tile_m);
bool fp8x2_shape_supported(int H, int I);
cudaError_t launch_fp8x2_gate_up(const GroupedGemm& g, cudaStream_t s);
cudaError_t launch_fp8x2_down(const GroupedGemm& g, cudaStream_t s);
// The two terms of bf16 rows [rows][cols]: with sorted_pairs, the token rows
// of the used positions p (zeros for padding) land in row
// (p / tile_n) * 2 tile_n + p % tile_n of q_hi / s_hi and q_lo / s_lo (the
// caller passes them tile_n rows apart); without, row p lands in row p.
cudaError_t launch_split_rows(const uint16_t* x, int cols, int rows, const int32_t* sorted_pairs,
                              const int32_t* num_tiles, int tile_n, int Kt, int cap, int num_pairs,
                              uint8_t* q_hi, uint8_t* q_lo, uint8_t* s_hi, uint8_t* s_lo,
                              cudaStream_t s);
cudaError_t read_device_error_fp8x2(int* flag, int clear);

// grouping of one dense expert over T tokens (Kt = 1); ones[T] = 1 if given
cudaError_t launch_identity_perm(int T, int tile_m, int cap, int max_tiles, int32_t* sorted_pairs,
                                 int32_t* tile_expert, int32_t* num_tiles, float* ones,
                                 cudaStream_t s);

}  // namespace moe
