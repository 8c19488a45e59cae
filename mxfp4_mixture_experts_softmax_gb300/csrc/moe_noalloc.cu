// moe_noalloc.cu -- moe_ffn for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the layer:
// code running under a CUDA stream capture that must not allocate, runtimes
// that hand out only fixed, pre-registered device memory, or plugins that do
// not own an allocator.  For them moe_ffn_noalloc runs the same FFN kernels
// as moe_ffn with the whole moe_ffn workspace (moe_ffn_workspace_size bytes)
// in the fixed device array below instead of a caller-provided buffer.
// Inputs and outputs are still the caller's.
#include <mutex>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace {

// The scratch lives in every GPU that loads the library, from module load
// until the process exits.
__device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}

// A __device__ array has one address per CUDA context (the module is loaded
// into each context), so the cache is keyed by the current context's ID,
// which the driver never reuses within a process: a context destroyed and
// created again (cudaDeviceReset) or a caller's own non-primary context gets
// its own lookup.
struct ScratchEntry {
    unsigned long long ctx_id;
    void* addr;
};
constexpr int kMaxContexts = 64;
std::mutex g_scratch_mu;
ScratchEntry g_scratch_cache[kMaxContexts] = {};
int g_scratch_next = 0;

cudaError_t current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (!get_current || !get_id) return cudaErrorNotSupported;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorContextIsDestroyed;
    if (!ctx) {
        // no context bound to this thread yet: the runtime binds the current
        // device's primary context on its first call that needs one
        void* p = nullptr;
        cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorContextIsDestroyed;
    }
    return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorContextIsDestroyed;
}

// Device address of the scratch array in the current context.  The host-side
// name g_noalloc_scratch is only a stand-in for the symbol; the address a
// kernel may use is looked up by the first call in each context (with that
// context current) and cached.
cudaError_t scratch_address(void** out) {
    unsigned long long id = 0;
    cudaError_t err = current_context_id(&id);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    for (const ScratchEntry& e : g_scratch_cache)
        if (e.addr && e.ctx_id == id) {
            *out = e.addr;
            return cudaSuccess;
        }
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_cache[g_scratch_next] = ScratchEntry{id, p};
    g_scratch_next = (g_scratch_next + 1) % kMaxContexts;
    *out = p;
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
