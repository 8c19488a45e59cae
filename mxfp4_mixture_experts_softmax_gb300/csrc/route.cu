// route.cu -- softmax top-K routing, one warp per token.
//
// Softmax-scored top-K selection at E=512, K=10 as one fused kernel
// (InferenceX MI355X Qwen3.5 blog, optimisations section, PR #21421), with
// the shared expert appended as slot K (same blog, PR #20736).
//
// Each lane holds E/32 logits in registers (lane l owns experts l, l+32, ...,
// so every load is a coalesced 128-byte row segment).  The softmax max and
// denominator are warp reductions.  The K winners come from K rounds of a
// warp arg-max on a 64-bit key (order-preserving logit bits, then the
// complemented expert index), so equal logits resolve to the lower index and
// the selection is exact.  Lane k keeps the k-th winner and writes it.
#include "moe_internal.h"

namespace moe {

namespace {

// Monotone map of a float to uint32 (larger float -> larger key); -0 is
// folded onto +0 first so that the two zeros tie.
__device__ __forceinline__ uint32_t order_key(float v) {
    if (v == 0.0f) v = 0.0f;
    uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

template <int VPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E,
                                                    int K, int with_shared, int renormalize,
                                                    int32_t* __restrict__ topk_ids,
                                                    float* __restrict__ topk_w) {
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* l = logits + (size_t)t * E;

    float v[VPL];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldg(l + e) : -INFINITY;
        m = fmaxf(m, v[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));

    float z = 0.0f;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
        if (lane + 32 * i < E) z += expf(v[i] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);

    uint32_t taken = 0;
    int my_id = 0;
    float my_logit = 0.0f;
    for (int k = 0; k < K; ++k) {
        unsigned long long best = 0ull;  // below every valid key
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u)) {
                unsigned long long key =
                    ((unsigned long long)order_key(v[i]) << 32) | (0xFFFFFFFFu - (uint32_t)e);
                best = key > best ? key : best;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
            best = other > best ? other : best;
        }
        const int e = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
        if ((e & 31) == lane) taken |= 1u << (e >> 5);
        if (lane == k) {
            my_id = e;
            my_logit = key_to_float((uint32_t)(best >> 32));
        }
    }

    const float p = lane < K ? expf(my_logit - m) / z : 0.0f;
    float s = p;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);

    const int Kt = K + (with_shared ? 1 : 0);
    if (lane < K) {
        topk_ids[(size_t)t * Kt + lane] = my_id;
        topk_w[(size_t)t * Kt + lane] = renormalize ? p / s : p;
    }
    if (with_shared && lane == 0) {
        topk_ids[(size_t)t * Kt + K] = E;
        topk_w[(size_t)t * Kt + K] = 1.0f;
    }
}

template <int VPL>
cudaError_t launch(const float* logits, int T, int E, int K, int ws, int rn, int32_t* ids,
                   float* w, cudaStream_t s) {
    const int warps = 8;
    dim3 grid((T + warps - 1) / warps);
    return launch_pdl(route_kernel<VPL>, dim3(grid), dim3(warps * 32), 0, s, logits, T, E, K, ws, rn,
                      ids, w);
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int K, int with_shared,
                         int renormalize, int32_t* ids, float* w, cudaStream_t s) {
    if (E <= 32) return launch<1>(logits, T, E, K, with_shared, renormalize, ids, w, s);
    if (E <= 64) return launch<2>(logits, T, E, K, with_shared, renormalize, ids, w, s);
    if (E <= 128) return launch<4>(logits, T, E, K, with_shared, renormalize, ids, w, s);
    if (E <= 256) return launch<8>(logits, T, E, K, with_shared, renormalize, ids, w, s);
    if (E <= 512) return launch<16>(logits, T, E, K, with_shared, renormalize, ids, w, s);
    return launch<32>(logits, T, E, K, with_shared, renormalize, ids, w, s);
}

}  // namespace moe
