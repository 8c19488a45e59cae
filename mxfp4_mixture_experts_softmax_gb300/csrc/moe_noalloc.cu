// moe_noalloc.cu -- moe_ffn for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the layer:
// code running under a CUDA stream capture that must not allocate, runtimes
// that hand out only fixed, pre-registered device memory, or plugins that do
// not own an allocator.  For them moe_ffn_noalloc runs the same three FFN
// kernels as moe_ffn with its workspace (the bf16 SwiGLU intermediate and the
// fp32 per-pair outputs) in the fixed device array below instead of a
// caller-provided buffer.  Inputs and outputs are still the caller's.
#include <mutex>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace {

// The scratch lives in every GPU that loads the library, from module load
// until the process exits.
__device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The host-side
// name g_noalloc_scratch is only a stand-in for the symbol; the address a
// kernel may use is looked up once per device (the first call on a device
// does this set-up) and cached.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" moe_status_t moe_ffn_noalloc(const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                                        const uint8_t* w2, const uint8_t* s2, const float* topk_w,
                                        const int32_t* sorted_pairs,
                                        const int32_t* expert_offsets, const int32_t* inv_pairs,
                                        const int32_t* tile_expert, const int32_t* num_tiles, int T,
                                        int H, int I, int Et, int Kt, int tile_m, uint16_t* out,
                                        cudaStream_t stream) {
    const size_t need = moe_ffn_workspace_size(T, H, I, Et, Kt, tile_m);
    if (need == 0 && T != 0) return MOE_ERR_INVALID_ARG;
    if (need > (size_t)MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return moe_ffn(x, w13, s13, w2, s2, topk_w, sorted_pairs, expert_offsets,
                               inv_pairs, tile_expert, num_tiles, T, H, I, Et, Kt, tile_m, out,
                               nullptr, 0, stream);
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    // Nothing in the scratch has to start at zero: every workspace element
    // the kernels read is written earlier in the same call.
    return moe_ffn(x, w13, s13, w2, s2, topk_w, sorted_pairs, expert_offsets, inv_pairs,
                   tile_expert, num_tiles, T, H, I, Et, Kt, tile_m, out, scratch,
                   (size_t)MOE_NOALLOC_SCRATCH_BYTES, stream);
}
