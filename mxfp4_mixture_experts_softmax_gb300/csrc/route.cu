// route.cu -- softmax top-K routing, one warp per token (route_device.cuh).
#include "moe_internal.h"
#include "route_device.cuh"

namespace moe {

namespace {

template <int VPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits,
                                                    const float* __restrict__ shared_w, int T,
                                                    int E, int K, int with_shared, int renormalize,
                                                    int32_t* __restrict__ topk_ids,
                                                    float* __restrict__ topk_w) {
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const int Kt = K + (with_shared ? 1 : 0);
    route_token<VPL>(logits + (size_t)t * E, E, K, with_shared, renormalize,
                     shared_w ? __ldg(shared_w + t) : 1.0f, topk_ids + (size_t)t * Kt,
                     topk_w + (size_t)t * Kt, lane);
    pdl_end();
}

template <int VPL>
cudaError_t launch(const float* logits, const float* sw, int T, int E, int K, int ws, int rn,
                   int32_t* ids, float* w, cudaStream_t s) {
    const int warps = 8;
    dim3 grid((T + warps - 1) / warps);
    return launch_pdl(route_kernel<VPL>, dim3(grid), dim3(warps * 32), 0, s, logits, sw, T, E, K,
                      ws, rn, ids, w);
}

}  // namespace

cudaError_t launch_route(const float* logits, const float* shared_w, int T, int E, int K,
                         int with_shared, int renormalize, int32_t* ids, float* w, cudaStream_t s) {
    const int ws = with_shared, rn = renormalize;
    if (E <= 32) return launch<1>(logits, shared_w, T, E, K, ws, rn, ids, w, s);
    if (E <= 64) return launch<2>(logits, shared_w, T, E, K, ws, rn, ids, w, s);
    if (E <= 128) return launch<4>(logits, shared_w, T, E, K, ws, rn, ids, w, s);
    if (E <= 256) return launch<8>(logits, shared_w, T, E, K, ws, rn, ids, w, s);
    if (E <= 512) return launch<16>(logits, shared_w, T, E, K, ws, rn, ids, w, s);
    return launch<32>(logits, shared_w, T, E, K, ws, rn, ids, w, s);
}

}  // namespace moe
