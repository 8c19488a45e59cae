// ffn_decode.cu -- small-M grouped MXFP4 GEMMs (decode path) and the combine.
//
// Decode steps move every touched expert's MXFP4 weights once and do little
// arithmetic per byte, so the kernels are built around the weight stream:
// each warp streams 16 weight rows with 16-byte loads straight into
// registers, dequantises them there (fused MXFP4 MoE kernel with in-register
// dequantisation: VibeSys Qwen3.5-397B on 4x MI300A, sections "baseline" and
// "kernels and graph capture") and feeds legacy warp MMAs in a swap-AB
// arrangement: the weight rows are the MMA's 16-row M side, the tile's tokens
// its 8-column N side (narrow N tiles for small M: vLLM MiniMax M3 on MI355X,
// section "local shape and tiling").
//
// A CTA owns one tile (tile_m rows of one expert, from moe_permute) and a
// block of weight rows (gate_up: 64 gate rows + the 64 matching up rows, so
// the SwiGLU epilogue has g and u in the same registers; down: 128 rows).
// The tile's activation rows are staged once per 512-wide K chunk into shared
// memory in the pair-interleaved, XOR-swizzled layout the B fragments read
// conflict-free.
//
// K mapping inside one 256-wide K step: lane (r, c) = (lane/4, lane%4) loads
// bytes [32c, 32c+32) of the step's 128 code bytes of its two rows, i.e.
// k = 64c .. 64c+63 (two scale groups).  Word i of those bytes (codes
// k = 64c+8i .. +7) feeds two MMAs: codes (0,4),(1,5) and (2,6),(3,7).  The
// MMA's k slots are therefore a permutation of k; the activations in shared
// memory use the same permutation, so every product pairs the right x[k].
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kThreads = 256;
constexpr int kKC = 512;              // K per staged activation chunk
constexpr int kChunks16 = kKC / 8;    // 16-byte chunks per staged row

template <int MODE, int NT>
__global__ void __launch_bounds__(kThreads, 2) decode_gemm_kernel(const GroupedGemm g) {
    constexpr int TM = NT * 8;
    extern __shared__ uint4 smem_u4[];
    uint4* xs = smem_u4;                                      // [TM][kChunks16]
    int32_t* qrow = reinterpret_cast<int32_t*>(xs + TM * kChunks16);  // [TM]

    const int tile = blockIdx.x;
    if (tile >= __ldg(g.num_tiles)) return;
    const int e = __ldg(g.tile_expert + tile);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, c = lane & 3;

    for (int j = threadIdx.x; j < TM; j += kThreads) qrow[j] = __ldg(g.sorted_pairs + tile * TM + j);

    int row0, row1;
    bool warp_valid;
    if (MODE == 0) {
        const int n0 = blockIdx.y * 64 + warp * 8;
        warp_valid = n0 < g.I;
        row0 = n0 + r;
        row1 = g.I + n0 + r;
    } else {
        const int m0 = blockIdx.y * 128 + warp * 16;
        warp_valid = m0 < g.rows;
        row0 = m0 + r;
        row1 = m0 + r + 8;
    }
    if (!warp_valid) row0 = row1 = 0;  // keep addresses in range; no loads are issued
    const int K = g.K;
    const size_t cbytes = (size_t)K / 2, sbytes = (size_t)K / 32;
    const uint8_t* cp0 = g.codes + ((size_t)e * g.rows + row0) * cbytes;
    const uint8_t* cp1 = g.codes + ((size_t)e * g.rows + row1) * cbytes;
    const uint8_t* sp0 = g.scales + ((size_t)e * g.rows + row0) * sbytes;
    const uint8_t* sp1 = g.scales + ((size_t)e * g.rows + row1) * sbytes;

    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;

    const int nsteps = (K + 255) / 256;
    // code registers: [row][half] 16 bytes each, plus their scale bytes
    uint4 nxt[2][2];
    uint32_t nsc[2][2];
    auto load_step = [&](int st) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int kb = st * 256 + 64 * c + 32 * h;
            const bool ok = warp_valid && kb < K;
            nxt[0][h] = ok ? ldg_stream_v4(cp0 + kb / 2) : make_uint4(0, 0, 0, 0);
            nxt[1][h] = ok ? ldg_stream_v4(cp1 + kb / 2) : make_uint4(0, 0, 0, 0);
            nsc[0][h] = ok ? (uint32_t)__ldg(sp0 + kb / 32) : 127u;
            nsc[1][h] = ok ? (uint32_t)__ldg(sp1 + kb / 32) : 127u;
        }
    };
    load_step(0);

    for (int st = 0; st < nsteps; ++st) {
        if ((st * 256) % kKC == 0) {
            __syncthreads();
            const int kc = st * 256;
            for (int idx = threadIdx.x; idx < TM * kChunks16; idx += kThreads) {
                const int j = idx / kChunks16, L = idx % kChunks16;
                const int k = kc + L * 8;
                const int q = qrow[j];
                uint4 v = make_uint4(0, 0, 0, 0);
                if (k < K && q >= 0) {
                    const size_t arow = g.act_by_token ? (size_t)(q / g.Kt) : (size_t)(tile * TM + j);
                    v = pair_interleave8(__ldg(reinterpret_cast<const uint4*>(g.act + arow * K + k)));
                }
                const int phys = L ^ (((L >> 3) & 3) | ((j & 1) << 2));
                xs[j * kChunks16 + phys] = v;
            }
            __syncthreads();
        }
        uint4 cur[2][2];
        uint32_t csc[2][2];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                cur[a][h] = nxt[a][h];
                csc[a][h] = nsc[a][h];
            }
        if (st + 1 < nsteps) load_step(st + 1);
        if (!warp_valid) continue;

        const int lbase = ((st * 256) % kKC) / 8 + 8 * c;  // step-local chunk of word 0
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t m0lo = e8m0_mult_lo(csc[0][h]), m1lo = e8m0_mult_lo(csc[1][h]);
            const bool big = __any_sync(0xFFFFFFFFu, (csc[0][h] > 128u) | (csc[1][h] > 128u));
            const uint32_t w0[4] = {cur[0][h].x, cur[0][h].y, cur[0][h].z, cur[0][h].w};
            const uint32_t w1[4] = {cur[1][h].x, cur[1][h].y, cur[1][h].z, cur[1][h].w};
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
                uint32_t d0[4], d1[4];
                mxfp4_word_to_bf16x2(w0[i4], m0lo, d0);
                mxfp4_word_to_bf16x2(w1[i4], m1lo, d1);
                if (big) {
                    bf16x2_scale(d0, e8m0_mult_hi(csc[0][h]));
                    bf16x2_scale(d1, e8m0_mult_hi(csc[1][h]));
                }
                const int i = 4 * h + i4;
                const int L = lbase + i;
                const int phys = L ^ (c | ((r & 1) << 2));
                const uint32_t aA[4] = {d0[0], d1[0], d0[1], d1[1]};
                const uint32_t aB[4] = {d0[2], d1[2], d0[3], d1[3]};
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const uint4 b = xs[(n * 8 + r) * kChunks16 + phys];
                    mma_bf16_16816(acc[n], aA, b.x, b.y);
                    mma_bf16_16816(acc[n], aB, b.z, b.w);
                }
            }
        }
    }

    if (!warp_valid) return;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int j = n * 8 + 2 * c + u;
            const int q = qrow[j];
            if (q < 0) continue;
            const int p = tile * TM + j;
            if (MODE == 0) {
                const float gv = acc[n][u], uv = acc[n][2 + u];
                g.h_out[(size_t)p * g.I + row0] = f32_to_bf16_bits(silu(gv) * uv);
            } else {
                const float wq = __ldg(g.topk_w + q);
                float* y = g.y_out + (size_t)q * g.rows;
                y[row0] = wq * acc[n][u];
                y[row1] = wq * acc[n][2 + u];
            }
        }
    }
}

template <int MODE, int NT>
cudaError_t launch_nt(const GroupedGemm& g, cudaStream_t s) {
    const size_t smem = (size_t)NT * 8 * kChunks16 * sizeof(uint4) + NT * 8 * sizeof(int32_t);
    cudaError_t err = ensure_dynamic_smem((const void*)decode_gemm_kernel<MODE, NT>, smem);
    if (err != cudaSuccess) return err;
    const int row_blocks = MODE == 0 ? (g.I + 63) / 64 : (g.rows + 127) / 128;
    dim3 grid(g.max_tiles, row_blocks);
    decode_gemm_kernel<MODE, NT><<<grid, kThreads, smem, s>>>(g);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_mode(const GroupedGemm& g, cudaStream_t s) {
    if (g.max_tiles == 0) return cudaSuccess;
    switch (g.tile_m) {
        case 8: return launch_nt<MODE, 1>(g, s);
        case 16: return launch_nt<MODE, 2>(g, s);
        case 32: return launch_nt<MODE, 4>(g, s);
        case 64: return launch_nt<MODE, 8>(g, s);
        default: return cudaErrorInvalidValue;
    }
}

// out[t][m] = bf16(sum over j ascending of y[t*Kt + j][m]); four columns per thread.
__global__ void __launch_bounds__(256) combine_kernel(const float4* __restrict__ y, int T, int H4,
                                                      int Kt, uint2* __restrict__ out) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)T * H4) return;
    const size_t t = i / H4, m = i % H4;
    const float4* yt = y + t * Kt * H4 + m;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < Kt; ++j) {
        const float4 v = __ldg(yt + (size_t)j * H4);
        a.x += v.x;
        a.y += v.y;
        a.z += v.z;
        a.w += v.w;
    }
    uint2 o;
    o.x = (uint32_t)f32_to_bf16_bits(a.x) | ((uint32_t)f32_to_bf16_bits(a.y) << 16);
    o.y = (uint32_t)f32_to_bf16_bits(a.z) | ((uint32_t)f32_to_bf16_bits(a.w) << 16);
    out[i] = o;
}

}  // namespace

bool decode_tile_supported(int tile_m) {
    return tile_m == 8 || tile_m == 16 || tile_m == 32 || tile_m == 64;
}

cudaError_t launch_decode_gate_up(const GroupedGemm& g, cudaStream_t s) { return launch_mode<0>(g, s); }
cudaError_t launch_decode_down(const GroupedGemm& g, cudaStream_t s) { return launch_mode<1>(g, s); }

cudaError_t launch_combine(const float* y, int T, int H, int Kt, uint16_t* out, cudaStream_t s) {
    const size_t n = (size_t)T * (H / 4);
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    const unsigned blocks = (unsigned)((n + threads - 1) / threads);
    combine_kernel<<<blocks, threads, 0, s>>>(reinterpret_cast<const float4*>(y), T, H / 4, Kt,
                                              reinterpret_cast<uint2*>(out));
    return cudaGetLastError();
}

}  // namespace moe
