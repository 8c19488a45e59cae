// ffn_prefill.cu -- large-M grouped MXFP4 GEMMs on the 5th-generation tensor
// cores (tcgen05 MMA, accumulators in tensor memory).
//
// Prefill chunks put tens to thousands of rows on each expert, so the GEMMs
// become dense contractions (separate large-M launcher regime: vLLM MiniMax M3
// on MI355X, section "local shape and tiling"; padded and tuned prefill GEMM:
// VibeSys Qwen3.5-397B on 4x MI300A, section "baseline").
//
// One CTA computes a 128-row block of one expert's weight matrix against one
// tile of tile_m token rows (swap-AB: weights are the MMA's M = 128 side, the
// tile's tokens its N = tile_m side), accumulating D[128, N] in fp32 in tensor
// memory over the whole reduction:
//   * per 64-wide K stage every thread dequantises one weight row (64 E2M1
//     codes, exact to bf16) into the stage's A buffer and the tile's token rows
//     are copied into the B buffer with cp.async (zero-filled for padding);
//     both buffers use the 128-byte swizzled K-major layout the MMA reads;
//   * one thread issues the four K = 16 MMAs of the stage and commits them to
//     the stage's mbarrier, which frees the buffers for reuse kStages later;
//   * the epilogue reads the accumulator from tensor memory (each warp its 32
//     lanes) and applies SwiGLU (gate_up, gate and up rows interleaved so the
//     partner value is one lane away) or the routing weight (down).
// Every wait is bounded by the global timer; on timeout the kernel raises the
// library's device error flag, drains its own MMAs (bounded), frees its tensor
// memory and returns.
#include "moe_internal.h"

namespace moe {

__device__ int g_device_error = 0;

namespace {

constexpr int kThreads = 128;
constexpr int kBK = 64;                       // K elements per stage (one 128-B row)
constexpr int kStages = 4;
constexpr int kABytes = 128 * kBK * 2;        // 16 KB per A stage
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzled layout: 8-row groups of 128-byte rows, 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);          // start address
    d |= (uint64_t)1u << 16;                          // leading byte offset (unused here)
    d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;    // stride byte offset: next 8 rows
    d |= (uint64_t)1u << 46;                          // descriptor version
    d |= (uint64_t)2u << 61;                          // 128-byte swizzle
    return d;
}

// Instruction descriptor: bf16 x bf16 -> fp32, both operands K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t r[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

template <int N>
struct PrefillSmem {
    static constexpr int kBBytes = N * kBK * 2;
    static constexpr int kBars = 1024 * 0 + kStages * (kABytes + kBBytes);  // offset of barriers
    static constexpr int kTotal = kBars + 256 + N * 4 + 1024;              // + alignment slack
};

template <int MODE, int N>
__global__ void __launch_bounds__(kThreads, 1) prefill_gemm_kernel(const GroupedGemm g) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * kABytes;
    constexpr int kBBytes = PrefillSmem<N>::kBBytes;
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + PrefillSmem<N>::kBars);
    uint64_t* done = empty + kStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    int32_t* qrow = reinterpret_cast<int32_t*>(tmem_slot + 4);

    const int tile = blockIdx.x;
    if (tile >= __ldg(g.num_tiles)) return;  // uniform, before any barrier or tensor memory
    const int e = __ldg(g.tile_expert + tile);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = g.K;

    for (int j = tid; j < N; j += kThreads) qrow[j] = __ldg(g.sorted_pairs + tile * N + j);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&empty[s], 1);
        mbar_init(done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"((uint32_t)N)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // this thread's weight row of the 128-row block
    int arow;
    bool rvalid;
    if (MODE == 0) {
        const int n = blockIdx.y * 64 + (tid >> 1);
        rvalid = n < g.I;
        arow = (tid & 1) ? g.I + n : n;
    } else {
        arow = blockIdx.y * 128 + tid;
        rvalid = arow < g.rows;
    }
    if (!rvalid) arow = 0;
    const uint8_t* cp = g.codes + ((size_t)e * g.rows + arow) * (size_t)(K / 2);
    const uint8_t* sp = g.scales + ((size_t)e * g.rows + arow) * (size_t)(K / 32);

    const int nk = (K + kBK - 1) / kBK;
    uint4 nc[2];
    uint32_t ns[2];
    auto load_chunk = [&](int kc) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int kb = kc * kBK + 32 * h;
            const bool ok = rvalid && kb < K;
            nc[h] = ok ? __ldg(reinterpret_cast<const uint4*>(cp + kb / 2)) : make_uint4(0, 0, 0, 0);
            ns[h] = ok ? (uint32_t)__ldg(sp + kb / 32) : 127u;
        }
    };
    load_chunk(0);

    constexpr uint32_t idesc = idesc_bf16(128, N);
    bool failed = false;
    for (int kc = 0; kc < nk; ++kc) {
        const int s = kc % kStages;
        if (kc >= kStages && !mbar_wait(&empty[s], (uint32_t)((kc / kStages - 1) & 1))) failed = true;
        if (__syncthreads_or(failed)) {
            failed = true;
            break;
        }
        // B: the tile's token rows, 8 x 16 bytes per row, swizzled
        uint8_t* b_st = sB + s * kBBytes;
        for (int i = tid; i < N * 8; i += kThreads) {
            const int j = i >> 3, ch = i & 7;
            const int k = kc * kBK + ch * 8;
            const int q = qrow[j];
            const uint16_t* src = g.act;
            uint32_t bytes = 0;
            if (q >= 0 && k < K) {
                const size_t brow = g.act_by_token ? (size_t)(q / g.Kt) : (size_t)(tile * N + j);
                src = g.act + brow * K + k;
                bytes = 16;
            }
            cp_async_16(smem_u32(b_st + j * 128 + ((ch ^ (j & 7)) << 4)), src, bytes);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        // A: dequantise this thread's row (64 codes) into natural k order
        const uint4 cc[2] = {nc[0], nc[1]};
        const uint32_t cs[2] = {ns[0], ns[1]};
        if (kc + 1 < nk) load_chunk(kc + 1);
        uint8_t* a_row = sA + s * kABytes + tid * 128;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t mlo = e8m0_mult_lo(cs[h]);
            const bool big = cs[h] > 128u;
            const uint32_t w4[4] = {cc[h].x, cc[h].y, cc[h].z, cc[h].w};
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
                uint32_t d[4];
                mxfp4_word_to_bf16x2(w4[i4], mlo, d);
                if (big) bf16x2_scale(d, e8m0_mult_hi(cs[h]));
                uint4 v;
                v.x = __byte_perm(d[0], d[1], 0x5410);  // (k0, k1)
                v.y = __byte_perm(d[2], d[3], 0x5410);  // (k2, k3)
                v.z = __byte_perm(d[0], d[1], 0x7632);  // (k4, k5)
                v.w = __byte_perm(d[2], d[3], 0x7632);  // (k6, k7)
                const int ch = 4 * h + i4;
                *reinterpret_cast<uint4*>(a_row + ((ch ^ (tid & 7)) << 4)) = v;
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint64_t ad = sdesc_sw128(smem_u32(sA + s * kABytes));
            const uint64_t bd = sdesc_sw128(smem_u32(b_st));
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)  // +32 bytes per K = 16 step inside the atom
                mma_bf16_ss(tmem, ad + 2u * k, bd + 2u * k, idesc, (kc | k) != 0 ? 1u : 0u);
            mma_commit(&empty[s]);
        }
    }
    if (tid == 0) mma_commit(done);  // tracks every MMA this thread issued
    const bool drained = mbar_wait(done, 0);
    tc_fence_after();
    if (!failed && drained) {
#pragma unroll 1
        for (int c0 = 0; c0 < N; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, v);
            const int r = 32 * warp + lane;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int j = c0 + i;
                const float acc = __uint_as_float(v[i]);
                if (MODE == 0) {
                    const float partner = __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
                    const int n = blockIdx.y * 64 + (r >> 1);
                    const int q = qrow[j];
                    if (!(lane & 1) && n < g.I && q >= 0)
                        g.h_out[(size_t)(tile * N + j) * g.I + n] = f32_to_bf16_bits(silu(acc) * partner);
                } else {
                    const int m = blockIdx.y * 128 + r;
                    const int q = qrow[j];
                    if (m < g.rows && q >= 0) g.y_out[(size_t)q * g.rows + m] = __ldg(g.topk_w + q) * acc;
                }
            }
        }
    }
    if ((failed || !drained) && tid == 0) atomicExch(&g_device_error, 1);
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"((uint32_t)N)
                     : "memory");
}

template <int MODE, int N>
cudaError_t launch_n(const GroupedGemm& g, cudaStream_t s) {
    const size_t smem = PrefillSmem<N>::kTotal;
    cudaError_t err = ensure_dynamic_smem((const void*)prefill_gemm_kernel<MODE, N>, smem);
    if (err != cudaSuccess) return err;
    const int row_blocks = MODE == 0 ? (g.I + 63) / 64 : (g.rows + 127) / 128;
    dim3 grid(g.max_tiles, row_blocks);
    prefill_gemm_kernel<MODE, N><<<grid, kThreads, smem, s>>>(g);
    return cudaGetLastError();
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

}  // namespace

bool prefill_tile_supported(int tile_m) {
    return tile_m == 32 || tile_m == 64 || tile_m == 128 || tile_m == 256;
}
bool prefill_shape_supported(int H, int I) { return H % 32 == 0 && I % 32 == 0; }
cudaError_t launch_prefill_gate_up(const GroupedGemm& g, cudaStream_t s) { return launch_mode<0>(g, s); }
cudaError_t launch_prefill_down(const GroupedGemm& g, cudaStream_t s) { return launch_mode<1>(g, s); }

cudaError_t read_device_error(int* flag, int clear) {
    cudaError_t err = cudaMemcpyFromSymbol(flag, g_device_error, sizeof(int));
    if (err != cudaSuccess || !clear) return err;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

}  // namespace moe
