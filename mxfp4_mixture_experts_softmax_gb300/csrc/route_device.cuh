// route_device.cuh -- softmax top-K routing of one token by one warp, shared by
// the routing kernel and the fused routing + permutation kernel.
//
// Softmax-scored top-K selection as one fused step (InferenceX MI355X Qwen3.5
// blog, optimisations section, PR #21421), with the shared expert appended as
// slot K (same blog, PR #20736).  Lane l holds logits l, l+32, ... in
// registers (coalesced 128-byte loads); the softmax max and denominator are
// warp reductions; the K winners come from K rounds of a warp arg-max on the
// order-preserving logit bits, ties going to the lower expert index, so the
// selection is exact.  Lane k keeps the k-th winner and writes it.
#pragma once

#include "moe_device.cuh"

namespace moe {

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

// Routes logits row l (E values) into ids / w (Kt entries each); called by all
// 32 lanes of a warp.  shared_weight is the shared slot's weight.
template <int VPL>
__device__ __forceinline__ void route_token(const float* __restrict__ l, int E, int K,
                                            int with_shared, int renormalize, float shared_weight,
                                            int32_t* ids, float* w, int lane) {
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

    int my_id = 0;
    float my_logit = 0.0f;
    if constexpr (VPL <= 16) {
        // 32-bit order keys built once; a taken key is set to 0 (below every
        // valid key).  Each round: the warp's largest key (one max reduction),
        // then the lowest expert index holding it (one min reduction) -- the
        // same winner as an arg-max on (key, lower index first).
        uint32_t key[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) key[i] = lane + 32 * i < E ? order_key(v[i]) : 0u;
        for (int k = 0; k < K; ++k) {
            uint32_t lm = 0u;
#pragma unroll
            for (int i = 0; i < VPL; ++i) lm = max(lm, key[i]);
            const uint32_t best = __reduce_max_sync(0xFFFFFFFFu, lm);
            uint32_t le = 0xFFFFFFFFu;  // this lane's lowest expert holding `best`
#pragma unroll
            for (int i = VPL - 1; i >= 0; --i)
                if (best != 0u && key[i] == best) le = (uint32_t)(lane + 32 * i);
            const int e = (int)__reduce_min_sync(0xFFFFFFFFu, le);  // -1 if none is left
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if (lane + 32 * i == e) key[i] = 0u;
            if (lane == k) {
                my_id = e;
                my_logit = key_to_float(best);
            }
        }
    } else {
        // many values per lane: keys rebuilt each round (fewer live registers)
        uint32_t taken = 0;
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
    }

    const float p = lane < K ? expf(my_logit - m) / z : 0.0f;
    float s = p;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);

    if (lane < K) {
        ids[lane] = my_id;
        w[lane] = renormalize ? p / s : p;
    }
    if (with_shared && lane == 0) {
        ids[K] = E;
        w[K] = shared_weight;
    }
}

}  // namespace moe
