// moe_api.cu -- the extern "C" entry points of libmoe: argument checks on the
// host, workspace layout, path choice and kernel launches.  Everything runs
// on the caller's stream; nothing here allocates or synchronises.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <initializer_list>
#include <mutex>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace moe {


cudaError_t ensure_dynamic_smem(const void* func, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    struct Entry {
        const void* func;
        int device;
        size_t bytes;
    };
    static std::mutex mu;
    static Entry seen[256];
    static int n_seen = 0;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_seen; ++i)
        if (seen[i].func == func && seen[i].device == dev && seen[i].bytes >= bytes) return cudaSuccess;
    err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (err != cudaSuccess) return err;
    if (n_seen < 256) seen[n_seen++] = Entry{func, dev, bytes};
    return cudaSuccess;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library).
static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

cudaError_t encode_2d_map(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int inner,
                          uint64_t rows, uint64_t row_stride, int box_inner, int box_rows,
                          CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)(rows > 0 ? rows : 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)row_stride};
    const cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_codes_map(CUtensorMap* map, const void* base, int row_bytes, uint64_t rows,
                             int box_bytes, int box_rows) {
    return encode_2d_map(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, row_bytes, rows,
                         (uint64_t)row_bytes, box_bytes, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

int num_sms() {
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

cudaError_t max_active_pairs(const void* func, int threads, size_t smem, int* pairs) {
    struct Entry {
        const void* func;
        int device;
        size_t smem;
        int pairs;
    };
    static std::mutex mu;
    static Entry seen[64];
    static int n_seen = 0;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_seen; ++i)
        if (seen[i].func == func && seen[i].device == dev && seen[i].smem == smem) {
            *pairs = seen[i].pairs;
            return cudaSuccess;
        }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 1024);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    err = cudaOccupancyMaxActiveClusters(&n, func, &cfg);
    if (err != cudaSuccess) return err;
    *pairs = n;
    if (n_seen < 64) seen[n_seen++] = Entry{func, dev, smem, n};
    return cudaSuccess;
}

static bool trace_enabled() {
    static int v = -1;
    if (v < 0) {
        const char* s = getenv("MOE_TRACE");
        v = (s && s[0] && s[0] != '0') ? 1 : 0;
    }
    return v == 1;
}

static moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Profiling hook (moe_set_gemm_events): events recorded on the caller's stream
// right before and right after the GEMM kernel launch of each FFN call.
static std::mutex g_gemm_ev_mu;
static cudaEvent_t g_gemm_ev_before = nullptr, g_gemm_ev_after = nullptr;

template <typename F>
static cudaError_t launch_gemm_timed(F launch, cudaStream_t stream) {
    cudaEvent_t before, after;
    {
        std::lock_guard<std::mutex> lock(g_gemm_ev_mu);
        before = g_gemm_ev_before;
        after = g_gemm_ev_after;
    }
    cudaError_t err = before ? cudaEventRecord(before, stream) : cudaSuccess;
    if (err != cudaSuccess) return err;
    err = launch();
    if (err == cudaSuccess && after) err = cudaEventRecord(after, stream);
    return err;
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

static size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static int64_t capacity64(int T, int Kt, int Et, int tile_m) {
    if (T < 0 || Kt < 1 || Et < 1 || tile_m < 1) return -1;
    return (int64_t)T * Kt + (int64_t)Et * (tile_m - 1);
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status_t status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: null, negative or misaligned argument";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE: size outside the supported limits";
        case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL: workspace smaller than moe_ffn_workspace_size()";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA launch failed (see cudaGetLastError)";
        case MOE_ERR_INTERNAL: return "MOE_ERR_INTERNAL: internal error";
    }
    return "MOE_ERR_UNKNOWN: unknown status code";
}

int moe_version(void) { return 100; }

moe_status_t moe_device_error(int* flag, int clear) {
    if (!flag) return MOE_ERR_INVALID_ARG;
    int a = 0, b = 0;
    int c = 0, d = 0;
    cudaError_t err = read_device_error_prefill(&a, clear);
    if (err == cudaSuccess) err = read_device_error_decode(&b, clear);
    if (err == cudaSuccess) err = read_device_error_mxfp4act(&c, clear);
    if (err == cudaSuccess) err = read_device_error_fp8x2(&d, clear);
    *flag = a | b | c | d;
    return cuda_status(err);
}

moe_status_t moe_set_gemm_events(cudaEvent_t before, cudaEvent_t after) {
    if ((before == nullptr) != (after == nullptr)) return MOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_gemm_ev_mu);
    g_gemm_ev_before = before;
    g_gemm_ev_after = after;
    return MOE_OK;
}

moe_status_t moe_selftest_wait_timeout(int limit_us, cudaStream_t stream) {
    if (limit_us < 1 || limit_us > 1000000) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_wait_selftest((unsigned long long)limit_us * 1000ull, stream));
}

moe_status_t moe_selftest_wait_split(int limit_us, int32_t* outcome, cudaStream_t stream) {
    if (limit_us < 1 || limit_us > 1000000 || !outcome || !aligned(outcome, 4))
        return MOE_ERR_INVALID_ARG;
    return cuda_status(
        launch_wait_split_selftest((unsigned long long)limit_us * 1000ull, outcome, stream));
}

static moe_status_t check_route(const float* logits, const float* shared_w, int T, int E, int K,
                                int with_shared, const int32_t* topk_ids, const float* topk_w) {
    if (T < 0 || E < 1 || K < 1) return MOE_ERR_INVALID_ARG;
    if (E > 1024 || K > 32 || K > E) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4)) return MOE_ERR_INVALID_ARG;
    if (shared_w && (!with_shared || !aligned(shared_w, 4))) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status_t moe_route_ex(const float* logits, const float* shared_w, int T, int E, int K,
                          int with_shared, int renormalize, int32_t* topk_ids, float* topk_w,
                          cudaStream_t stream) {
    const moe_status_t st = check_route(logits, shared_w, T, E, K, with_shared, topk_ids, topk_w);
    if (st != MOE_OK || T == 0) return st;
    return cuda_status(launch_route(logits, shared_w, T, E, K, with_shared ? 1 : 0,
                                    renormalize ? 1 : 0, topk_ids, topk_w, stream));
}

moe_status_t moe_route(const float* logits, int T, int E, int K, int with_shared, int renormalize,
                       int32_t* topk_ids, float* topk_w, cudaStream_t stream) {
    return moe_route_ex(logits, nullptr, T, E, K, with_shared, renormalize, topk_ids, topk_w,
                        stream);
}

size_t moe_permute_capacity(int T, int Kt, int Et, int tile_m) {
    const int64_t cap = capacity64(T, Kt, Et, tile_m);
    return cap < 0 ? 0 : (size_t)cap;
}

size_t moe_permute_max_tiles(int T, int Kt, int Et, int tile_m) {
    const int64_t cap = capacity64(T, Kt, Et, tile_m);
    return cap < 0 ? 0 : (size_t)(cap / tile_m);
}

static moe_status_t check_permute(const int32_t* topk_ids, int T, int Kt, int Et, int tile_m,
                                  const int32_t* sorted_pairs, const int32_t* expert_offsets,
                                  const int32_t* inv_pairs, const int32_t* tile_expert,
                                  const int32_t* num_tiles, int64_t* cap_out) {
    const int64_t cap = capacity64(T, Kt, Et, tile_m);
    if (cap < 0) return MOE_ERR_INVALID_ARG;
    if (Kt > 33 || Et > 1025 || tile_m > 256 || cap >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!expert_offsets || !num_tiles) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_ids || !inv_pairs)) return MOE_ERR_INVALID_ARG;
    if (cap > 0 && !sorted_pairs) return MOE_ERR_INVALID_ARG;
    if (cap / tile_m > 0 && !tile_expert) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {topk_ids, sorted_pairs, expert_offsets, inv_pairs, tile_expert, num_tiles};
    for (const void* p : ptrs)
        if (p && !aligned(p, 4)) return MOE_ERR_INVALID_ARG;
    *cap_out = cap;
    return MOE_OK;
}

moe_status_t moe_permute(const int32_t* topk_ids, int T, int Kt, int Et, int tile_m,
                         int32_t* sorted_pairs, int32_t* expert_offsets, int32_t* inv_pairs,
                         int32_t* tile_expert, int32_t* num_tiles, cudaStream_t stream) {
    int64_t cap = 0;
    const moe_status_t st = check_permute(topk_ids, T, Kt, Et, tile_m, sorted_pairs,
                                          expert_offsets, inv_pairs, tile_expert, num_tiles, &cap);
    if (st != MOE_OK) return st;
    return cuda_status(launch_permute(topk_ids, T, Kt, Et, tile_m, (int)cap, (int)(cap / tile_m),
                                      sorted_pairs, expert_offsets, inv_pairs, tile_expert,
                                      num_tiles, stream));
}

moe_status_t moe_route_permute(const float* logits, const float* shared_w, int T, int E, int K,
                               int with_shared, int renormalize, int tile_m, int32_t* topk_ids,
                               float* topk_w, int32_t* sorted_pairs, int32_t* expert_offsets,
                               int32_t* inv_pairs, int32_t* tile_expert, int32_t* num_tiles,
                               cudaStream_t stream) {
    moe_status_t st = check_route(logits, shared_w, T, E, K, with_shared, topk_ids, topk_w);
    if (st != MOE_OK) return st;
    const int Kt = K + (with_shared ? 1 : 0), Et = E + (with_shared ? 1 : 0);
    int64_t cap = 0;
    st = check_permute(topk_ids, T, Kt, Et, tile_m, sorted_pairs, expert_offsets, inv_pairs,
                       tile_expert, num_tiles, &cap);
    if (st != MOE_OK) return st;
    if (T == 0 || T > MOE_ROUTE_PERMUTE_FUSED_MAX_T) {
        // larger batches: the routing is spread over many blocks
        st = moe_route_ex(logits, shared_w, T, E, K, with_shared, renormalize, topk_ids, topk_w,
                          stream);
        if (st != MOE_OK) return st;
        return moe_permute(topk_ids, T, Kt, Et, tile_m, sorted_pairs, expert_offsets, inv_pairs,
                           tile_expert, num_tiles, stream);
    }
    return cuda_status(launch_route_permute(logits, shared_w, T, E, K, with_shared ? 1 : 0,
                                            renormalize ? 1 : 0, tile_m, (int)cap,
                                            (int)(cap / tile_m), topk_ids, topk_w, sorted_pairs,
                                            expert_offsets, inv_pairs, tile_expert, num_tiles,
                                            stream));
}

// Tile heights of the paths that gather B rows into tile order and stage y
// by sorted position (prefill, and the two-term path's 96).
static bool staged_tile(int tile_m) { return prefill_tile_supported(tile_m) || fp8x2_tile_supported(tile_m); }

static size_t y_offset(int64_t cap, int I) { return round_up((size_t)cap * I * sizeof(uint16_t), 256); }

// y: fp32 [T*Kt, H] by pair, or, for prefill tile heights, also room for the
// f16 rows by position moe_ffn_down_combine writes ([cap][H rounded up to 128]).
static size_t y_bytes(int64_t cap, int T, int H, int Kt, int tile_m) {
    size_t n = (size_t)T * Kt * H * sizeof(float);
    if (staged_tile(tile_m))
        n = std::max(n, (size_t)((H + 127) / 128) * 128 * (size_t)cap * sizeof(uint16_t));
    return round_up(n, 256);
}

// After y: x as scaled f16 rows [T, H] (both paths), the prefill path's
// tile-ordered copy of them [cap, H] (prefill tile heights only), the fp32
// row factors of x [T] and of h [cap], and the routing weight of each sorted
// position [cap].
static size_t x16_offset(int64_t cap, int T, int H, int I, int Kt, int tile_m) {
    return y_offset(cap, I) + y_bytes(cap, T, H, Kt, tile_m);
}

static size_t xg_offset(int64_t cap, int T, int H, int I, int Kt, int tile_m) {
    return x16_offset(cap, T, H, I, Kt, tile_m) + round_up((size_t)T * H * sizeof(uint16_t), 256);
}

static size_t rs_offset(int64_t cap, int T, int H, int I, int Kt, int tile_m) {
    const size_t xg = staged_tile(tile_m) ? round_up((size_t)cap * H * sizeof(uint16_t), 256) : 0;
    return xg_offset(cap, T, H, I, Kt, tile_m) + xg;
}

static size_t wpos_offset(int64_t cap, int T, int H, int I, int Kt, int tile_m) {
    return rs_offset(cap, T, H, I, Kt, tile_m) + round_up((size_t)(T + cap) * sizeof(float), 256);
}

// After the position weights: the shifts of y staged as f16 by the prefill
// down GEMMs, one byte per (8 output rows, 32 positions) [ceil(cap/32)][H
// rounded up to 128, / 8].
static size_t yshift_offset(int64_t cap, int T, int H, int I, int Kt, int tile_m) {
    return wpos_offset(cap, T, H, I, Kt, tile_m) + round_up((size_t)cap * sizeof(float), 256);
}

// After the shifts: the scale bytes of h's two E4M3 terms on the
// MOE_PATH_PREFILL_FP8X2 path [2 cap][I/32] (its tile heights only).
static size_t x2s_offset(int64_t cap, int T, int H, int I, int Kt, int tile_m) {
    const size_t shifts =
        staged_tile(tile_m) ? (size_t)((cap + 31) / 32) * (size_t)((H + 127) / 128 * 16) : 0;
    return yshift_offset(cap, T, H, I, Kt, tile_m) + round_up(shifts, 256);
}

size_t moe_ffn_workspace_size(int T, int H, int I, int Et, int Kt, int tile_m) {
    const int64_t cap = capacity64(T, Kt, Et, tile_m);
    if (cap < 0 || H <= 0 || I <= 0) return 0;
    const size_t x2s = fp8x2_tile_supported(tile_m) ? (size_t)cap * 2 * (size_t)(I / 32) : 0;
    return x2s_offset(cap, T, H, I, Kt, tile_m) + round_up(x2s, 256);
}

moe_path_t moe_ffn_auto_path(int T, int Kt, int Et, int tile_m) {
    // mean rows per expert; the decode path wins while most experts see only
    // a few rows, so the weight stream, not the MMA, bounds the time
    // (the large-M regime's tile heights: the f16 prefill path's and the two-term path's 96)
    const double rows_per_expert = Et > 0 ? (double)T * Kt / Et : 0.0;
    if (rows_per_expert >= 16.0 && staged_tile(tile_m)) return MOE_PATH_PREFILL;
    if (decode_tile_supported(tile_m)) return MOE_PATH_DECODE;
    return staged_tile(tile_m) ? MOE_PATH_PREFILL : MOE_PATH_DECODE;
}

// Shape/path checks shared by the FFN calls.  Resolves AUTO (and the
// MOE_FORCE_PATH environment override) to a concrete path.
static moe_status_t check_ffn_shape(int T, int H, int I, int Et, int Kt, int tile_m,
                                    moe_path_t* path) {
    const int64_t cap = capacity64(T, Kt, Et, tile_m);
    if (cap < 0 || H <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
    if (H % 32 || I % 32 || H > 65536 || I > 65536 || Kt > 33 || Et > 1025 || tile_m > 256 ||
        cap >= ((int64_t)1 << 31))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    moe_path_t p = *path;
    if (p != MOE_PATH_AUTO && p != MOE_PATH_DECODE && p != MOE_PATH_PREFILL &&
        p != MOE_PATH_PREFILL_FP8X2)
        return MOE_ERR_INVALID_ARG;
    if (p == MOE_PATH_AUTO) {
        const char* f = getenv("MOE_FORCE_PATH");
        if (f && !strcmp(f, "decode")) p = MOE_PATH_DECODE;
        else if (f && !strcmp(f, "prefill")) p = MOE_PATH_PREFILL;
        else if (f && !strcmp(f, "prefill_fp8x2")) p = MOE_PATH_PREFILL_FP8X2;
        else {
            p = moe_ffn_auto_path(T, Kt, Et, tile_m);
            // the large-M regime: the block-scaled two-term path where it applies
            if (p == MOE_PATH_PREFILL && fp8x2_tile_supported(tile_m) && fp8x2_shape_supported(H, I))
                p = MOE_PATH_PREFILL_FP8X2;
        }
    }
    if (p == MOE_PATH_DECODE && !decode_tile_supported(tile_m)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (p == MOE_PATH_PREFILL && (!prefill_tile_supported(tile_m) || !prefill_shape_supported(H, I)))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (p == MOE_PATH_PREFILL_FP8X2 && (!fp8x2_tile_supported(tile_m) || !fp8x2_shape_supported(H, I)))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    *path = p;
    return MOE_OK;
}

moe_path_t moe_ffn_auto_path_shape(int T, int H, int I, int Et, int Kt, int tile_m) {
    moe_path_t p = MOE_PATH_AUTO;
    return check_ffn_shape(T, H, I, Et, Kt, tile_m, &p) == MOE_OK ? p : MOE_PATH_AUTO;
}

static bool ptrs_ok(std::initializer_list<const void*> ptrs, size_t align) {
    for (const void* p : ptrs)
        if (!p || !aligned(p, align)) return false;
    return true;
}

static GroupedGemm base_gemm(const int32_t* sorted_pairs, const int32_t* tile_expert,
                             const int32_t* num_tiles, int T, int I, int Et, int Kt, int tile_m,
                             int max_tiles) {
    GroupedGemm g{};
    g.num_pairs = T * Kt;
    g.num_experts = Et;
    g.sorted_pairs = sorted_pairs;
    g.tile_expert = tile_expert;
    g.num_tiles = num_tiles;
    g.Kt = Kt;
    g.tile_m = tile_m;
    g.max_tiles = max_tiles;
    g.I = I;
    return g;
}

static void trace(const char* step, int T, int H, int I, int Et, int Kt, int tile_m, moe_path_t p) {
    if (trace_enabled())
        fprintf(stderr, "[libmoe] %s T=%d H=%d I=%d Et=%d Kt=%d tile_m=%d path=%s\n", step, T, H, I,
                Et, Kt, tile_m,
                p == MOE_PATH_DECODE ? "decode" : (p == MOE_PATH_PREFILL_FP8X2 ? "prefill_fp8x2" : "prefill"));
}

size_t moe_ffn_y_offset(int T, int I, int Et, int Kt, int tile_m) {
    const int64_t cap = capacity64(T, Kt, Et, tile_m);
    if (cap < 0 || I <= 0) return 0;
    return y_offset(cap, I);
}

moe_status_t moe_ffn_gate_up(const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                             const int32_t* sorted_pairs, const int32_t* tile_expert,
                             const int32_t* num_tiles, int T, int H, int I, int Et, int Kt,
                             int tile_m, void* workspace, size_t ws_bytes, moe_path_t path,
                             cudaStream_t stream) {
    moe_status_t st = check_ffn_shape(T, H, I, Et, Kt, tile_m, &path);
    if (st != MOE_OK || T == 0) return st;
    if (!ptrs_ok({x, w13, workspace}, 16) || !ptrs_ok({s13, sorted_pairs, tile_expert, num_tiles}, 4))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_ffn_workspace_size(T, H, I, Et, Kt, tile_m)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    const int64_t cap = capacity64(T, Kt, Et, tile_m);
    const int max_tiles = (int)(cap / tile_m);
    trace("moe_ffn_gate_up", T, H, I, Et, Kt, tile_m, path);
    GroupedGemm g = base_gemm(sorted_pairs, tile_expert, num_tiles, T, I, Et, Kt, tile_m, max_tiles);
    g.codes = w13;
    g.scales = s13;
    g.rows = 2 * I;
    g.K = H;
    g.h_out = reinterpret_cast<uint16_t*>(workspace);
    if (path == MOE_PATH_PREFILL_FP8X2) {
        if (!aligned(w13, 32)) return MOE_ERR_INVALID_ARG;  // unpacking TMA loads
        // x as two E4M3 terms in tile order, 2 tile_m rows per tile (in the
        // area of the tile-ordered copy), their scale bytes in the y area
        // (free until the down GEMM); h comes out in the same form (the h
        // area, and its scale bytes after the shifts)
        char* ws = reinterpret_cast<char*>(workspace);
        uint8_t* xq = reinterpret_cast<uint8_t*>(ws + xg_offset(cap, T, H, I, Kt, tile_m));
        uint8_t* xs = reinterpret_cast<uint8_t*>(ws + y_offset(cap, I));
        cudaError_t err = launch_split_rows(x, H, 0, sorted_pairs, num_tiles, tile_m, Kt, (int)cap,
                                            T * Kt, xq, xq + (size_t)tile_m * H, xs,
                                            xs + (size_t)tile_m * (H / 32), stream);
        if (err != cudaSuccess) return MOE_ERR_CUDA;
        g.act = reinterpret_cast<const uint16_t*>(xq);
        g.act_rows = max_tiles * 2 * tile_m;
        g.act_scales = xs;
        g.hq_codes = reinterpret_cast<uint8_t*>(ws);
        g.hq_scales = reinterpret_cast<uint8_t*>(ws + x2s_offset(cap, T, H, I, Kt, tile_m));
        return cuda_status(launch_gemm_timed([&] { return launch_fp8x2_gate_up(g, stream); }, stream));
    }
    // both GEMMs take f16 B rows scaled per row by a power of two: x here,
    // and h (in place) once the GEMM has written it
    char* ws = reinterpret_cast<char*>(workspace);
    uint16_t* x16 = reinterpret_cast<uint16_t*>(ws + x16_offset(cap, T, H, I, Kt, tile_m));
    float* rs_x = reinterpret_cast<float*>(ws + rs_offset(cap, T, H, I, Kt, tile_m));
    g.act_rscale = rs_x;  // indexed by token
    cudaError_t err;
    if (path == MOE_PATH_DECODE) {
        err = launch_rows_to_f16(x, x16, H, T, nullptr, nullptr, tile_m, rs_x, stream,
                                 /*independent=*/true);
        if (err != cudaSuccess) return MOE_ERR_CUDA;
        g.act = x16;
        g.act_rows = T;
        g.act_by_token = 1;
        err = launch_gemm_timed([&] { return launch_decode_gate_up(g, stream); }, stream);
    } else {
        // the prefill GEMM reads its token rows as one box per stage: gather
        // them into tile order, converted to scaled f16 on the way
        uint16_t* xg = reinterpret_cast<uint16_t*>(ws + xg_offset(cap, T, H, I, Kt, tile_m));
        err = launch_gather_rows_f16(x, H, sorted_pairs, num_tiles, tile_m, Kt, (int)cap, T * Kt, xg,
                                     rs_x, stream);
        if (err != cudaSuccess) return MOE_ERR_CUDA;
        g.act = xg;
        g.act_rows = (int)cap;
        g.act_by_token = 0;
        err = launch_gemm_timed([&] { return launch_prefill_gate_up(g, stream); }, stream);
    }
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    err = launch_rows_to_f16(g.h_out, g.h_out, I, (int)cap, sorted_pairs, num_tiles, tile_m,
                             rs_x + T, stream);
    return cuda_status(err);
}

moe_status_t moe_ffn_down(const uint8_t* w2, const uint8_t* s2, const float* topk_w,
                          const int32_t* sorted_pairs, const int32_t* tile_expert,
                          const int32_t* num_tiles, int T, int H, int I, int Et, int Kt,
                          int tile_m, void* workspace, size_t ws_bytes, moe_path_t path,
                          cudaStream_t stream) {
    moe_status_t st = check_ffn_shape(T, H, I, Et, Kt, tile_m, &path);
    if (st != MOE_OK || T == 0) return st;
    if (!ptrs_ok({w2, workspace}, 16) || !ptrs_ok({s2, topk_w, sorted_pairs, tile_expert, num_tiles}, 4))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_ffn_workspace_size(T, H, I, Et, Kt, tile_m)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    const int64_t cap = capacity64(T, Kt, Et, tile_m);
    const int max_tiles = (int)(cap / tile_m);
    trace("moe_ffn_down", T, H, I, Et, Kt, tile_m, path);
    GroupedGemm g = base_gemm(sorted_pairs, tile_expert, num_tiles, T, I, Et, Kt, tile_m, max_tiles);
    g.codes = w2;
    g.scales = s2;
    g.rows = H;
    g.K = I;
    g.act = reinterpret_cast<const uint16_t*>(workspace);
    g.act_rscale = reinterpret_cast<const float*>(reinterpret_cast<const char*>(workspace) +
                                                  rs_offset(cap, T, H, I, Kt, tile_m)) + T;
    g.act_rows = (int)cap;
    g.act_by_token = 0;
    g.y_out = reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) + y_offset(cap, I));
    g.topk_w = topk_w;
    if (path == MOE_PATH_PREFILL_FP8X2) {  // h as two E4M3 terms, y by pair
        if (!aligned(w2, 32)) return MOE_ERR_INVALID_ARG;
        g.act_rows = max_tiles * 2 * tile_m;
        g.act_scales = reinterpret_cast<const uint8_t*>(workspace) + x2s_offset(cap, T, H, I, Kt, tile_m);
        g.act_rscale = nullptr;
        return cuda_status(launch_gemm_timed([&] { return launch_fp8x2_down(g, stream); }, stream));
    }
    cudaError_t err = launch_gemm_timed(
        [&] { return path == MOE_PATH_DECODE ? launch_decode_down(g, stream) : launch_prefill_down(g, stream); },
        stream);
    return cuda_status(err);
}

moe_status_t moe_ffn_down_combine(const uint8_t* w2, const uint8_t* s2, const float* topk_w,
                                  const int32_t* sorted_pairs, const int32_t* inv_pairs,
                                  const int32_t* tile_expert, const int32_t* num_tiles, int T, int H,
                                  int I, int Et, int Kt, int tile_m, uint16_t* out, void* workspace,
                                  size_t ws_bytes, moe_path_t path, cudaStream_t stream) {
    moe_status_t st = check_ffn_shape(T, H, I, Et, Kt, tile_m, &path);
    if (st != MOE_OK || T == 0) return st;
    if (!ptrs_ok({w2, out, workspace}, 16) ||
        !ptrs_ok({s2, topk_w, sorted_pairs, inv_pairs, tile_expert, num_tiles}, 4))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_ffn_workspace_size(T, H, I, Et, Kt, tile_m)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    char* ws = reinterpret_cast<char*>(workspace);
    float* y = reinterpret_cast<float*>(ws + moe_ffn_y_offset(T, I, Et, Kt, tile_m));
    if (path == MOE_PATH_DECODE) {  // y by pair, then the slot-ordered combine
        st = moe_ffn_down(w2, s2, topk_w, sorted_pairs, tile_expert, num_tiles, T, H, I, Et, Kt,
                          tile_m, workspace, ws_bytes, path, stream);
        return st != MOE_OK ? st : moe_combine(y, T, H, Kt, out, stream);
    }
    // prefill: y by sorted position, staged as f16 with a power-of-two shift
    // per (8 output rows, 32 positions), without the column factor; the
    // factor per position (routing weight x h row factor) is applied by the
    // combine, which gathers each token's positions in slot order
    const int64_t cap = capacity64(T, Kt, Et, tile_m);
    const bool x2 = path == MOE_PATH_PREFILL_FP8X2;
    if (x2 && !aligned(w2, 32)) return MOE_ERR_INVALID_ARG;  // unpacking TMA loads
    float* w_pos = reinterpret_cast<float*>(ws + wpos_offset(cap, T, H, I, Kt, tile_m));
    const float* h_rscale = reinterpret_cast<const float*>(ws + rs_offset(cap, T, H, I, Kt, tile_m)) + T;
    trace("moe_ffn_down_combine", T, H, I, Et, Kt, tile_m, path);
    // the two-term path's h needs no row factor
    cudaError_t err = launch_position_weights(sorted_pairs, topk_w, x2 ? nullptr : h_rscale, num_tiles,
                                              tile_m, (int)cap, T * Kt, w_pos, stream);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    GroupedGemm g = base_gemm(sorted_pairs, tile_expert, num_tiles, T, I, Et, Kt, tile_m,
                              (int)(cap / tile_m));
    g.codes = w2;
    g.scales = s2;
    g.rows = H;
    g.K = I;
    g.act = reinterpret_cast<const uint16_t*>(workspace);
    g.act_rscale = h_rscale;
    g.act_rows = (int)cap;
    g.act_by_token = 0;
    g.y_out = y;
    g.y_blocked = 1;
    g.y16_out = reinterpret_cast<uint16_t*>(y);
    g.y_shift = reinterpret_cast<int8_t*>(ws + yshift_offset(cap, T, H, I, Kt, tile_m));
    g.y_rows_pad = (H + 127) / 128 * 128;
    g.topk_w = topk_w;
    if (x2) {
        g.act_rows = (int)(cap / tile_m) * 2 * tile_m;
        g.act_scales = reinterpret_cast<const uint8_t*>(ws + x2s_offset(cap, T, H, I, Kt, tile_m));
        g.act_rscale = nullptr;
    }
    err = launch_gemm_timed(
        [&] { return x2 ? launch_fp8x2_down(g, stream) : launch_prefill_down(g, stream); }, stream);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_status(launch_combine_blocked_f16(g.y16_out, g.y_shift, inv_pairs, w_pos, T, H, Kt,
                                                  (int)cap, out, stream));
}

moe_status_t moe_combine_ex(const float* y, const float* y_extra, int T, int H, int Kt,
                            uint16_t* out, cudaStream_t stream) {
    if (T < 0 || H <= 0 || Kt < 1) return MOE_ERR_INVALID_ARG;
    if (H % 4 || Kt > 33) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    if (!ptrs_ok({y, out}, 16) || (y_extra && !aligned(y_extra, 16))) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_combine(y, y_extra, T, H, Kt, out, stream));
}

moe_status_t moe_combine(const float* y, int T, int H, int Kt, uint16_t* out, cudaStream_t stream) {
    return moe_combine_ex(y, nullptr, T, H, Kt, out, stream);
}

// ---------------------------------------------- shared expert of another width
// Workspace: the routed layer's moe_ffn workspace, then the dense expert's
// grouping (sorted_pairs [cap_s], tile_expert [cap_s / tile_m], num_tiles,
// unit weights [T]), then the dense expert's own moe_ffn workspace.
struct DenseSharedLayout {
    size_t routed, perm, ones, tiles, count, dense, total;
    int64_t cap_s;
};

static bool dense_shared_layout(int T, int H, int I, int Et, int Kt, int Is, int tile_m,
                                DenseSharedLayout* L) {
    const size_t r = moe_ffn_workspace_size(T, H, I, Et, Kt, tile_m);
    const size_t d = moe_ffn_workspace_size(T, H, Is, 1, 1, tile_m);
    const int64_t cap_s = capacity64(T, 1, 1, tile_m);
    if ((r == 0 && T != 0) || (d == 0 && T != 0) || cap_s < 0) return false;
    L->cap_s = cap_s;
    L->routed = 0;
    L->perm = round_up(r, 256);
    L->tiles = L->perm + round_up((size_t)cap_s * 4, 256);
    L->count = L->tiles + round_up((size_t)(cap_s / tile_m + 1) * 4, 256);
    L->ones = L->count + 256;
    L->dense = L->ones + round_up((size_t)T * 4 + 4, 256);
    L->total = L->dense + d;
    return true;
}

size_t moe_ffn_dense_shared_workspace_size(int T, int H, int I, int Et, int Kt, int Is, int tile_m) {
    DenseSharedLayout L;
    return dense_shared_layout(T, H, I, Et, Kt, Is, tile_m, &L) ? L.total : 0;
}

moe_status_t moe_ffn_dense_shared(const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                                  const uint8_t* w2, const uint8_t* s2, const float* topk_w,
                                  const int32_t* sorted_pairs, const int32_t* expert_offsets,
                                  const int32_t* inv_pairs, const int32_t* tile_expert,
                                  const int32_t* num_tiles, int T, int H, int I, int Et, int Kt,
                                  int tile_m, const uint8_t* w13s, const uint8_t* s13s,
                                  const uint8_t* w2s, const uint8_t* s2s, int Is,
                                  const float* shared_w, uint16_t* out, void* workspace,
                                  size_t ws_bytes, cudaStream_t stream) {
    moe_path_t p_routed = MOE_PATH_AUTO, p_dense = MOE_PATH_AUTO;
    moe_status_t st = check_ffn_shape(T, H, I, Et, Kt, tile_m, &p_routed);
    if (st != MOE_OK) return st;
    st = check_ffn_shape(T, H, Is, 1, 1, tile_m, &p_dense);
    if (st != MOE_OK || T == 0) return st;
    if (!ptrs_ok({x, w13, w2, w13s, w2s, out, workspace}, 16) ||
        !ptrs_ok({s13, s2, s13s, s2s, topk_w, sorted_pairs, expert_offsets, inv_pairs, tile_expert,
                  num_tiles}, 4) ||
        (shared_w && !aligned(shared_w, 4)))
        return MOE_ERR_INVALID_ARG;
    DenseSharedLayout L;
    if (!dense_shared_layout(T, H, I, Et, Kt, Is, tile_m, &L)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    char* ws = reinterpret_cast<char*>(workspace);
    const size_t r_bytes = moe_ffn_workspace_size(T, H, I, Et, Kt, tile_m);
    const size_t d_bytes = moe_ffn_workspace_size(T, H, Is, 1, 1, tile_m);
    // the routed experts
    st = moe_ffn_gate_up(x, w13, s13, sorted_pairs, tile_expert, num_tiles, T, H, I, Et, Kt, tile_m,
                         ws, r_bytes, p_routed, stream);
    if (st != MOE_OK) return st;
    st = moe_ffn_down(w2, s2, topk_w, sorted_pairs, tile_expert, num_tiles, T, H, I, Et, Kt, tile_m,
                      ws, r_bytes, p_routed, stream);
    if (st != MOE_OK) return st;
    // the shared expert over every token, weight shared_w[t] (1 when null)
    int32_t* sp_s = reinterpret_cast<int32_t*>(ws + L.perm);
    int32_t* te_s = reinterpret_cast<int32_t*>(ws + L.tiles);
    int32_t* nt_s = reinterpret_cast<int32_t*>(ws + L.count);
    float* ones = reinterpret_cast<float*>(ws + L.ones);
    char* dws = ws + L.dense;
    if (launch_identity_perm(T, tile_m, (int)L.cap_s, (int)(L.cap_s / tile_m), sp_s, te_s, nt_s,
                             shared_w ? nullptr : ones, stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    st = moe_ffn_gate_up(x, w13s, s13s, sp_s, te_s, nt_s, T, H, Is, 1, 1, tile_m, dws, d_bytes,
                         p_dense, stream);
    if (st != MOE_OK) return st;
    st = moe_ffn_down(w2s, s2s, shared_w ? shared_w : ones, sp_s, te_s, nt_s, T, H, Is, 1, 1, tile_m,
                      dws, d_bytes, p_dense, stream);
    if (st != MOE_OK) return st;
    // routed slots in order, then the shared expert
    const float* y = reinterpret_cast<const float*>(ws + moe_ffn_y_offset(T, I, Et, Kt, tile_m));
    const float* ys = reinterpret_cast<const float*>(dws + moe_ffn_y_offset(T, Is, 1, 1, tile_m));
    return moe_combine_ex(y, ys, T, H, Kt, out, stream);
}

moe_status_t moe_ffn_path(const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                          const uint8_t* w2, const uint8_t* s2, const float* topk_w,
                          const int32_t* sorted_pairs, const int32_t* expert_offsets,
                          const int32_t* inv_pairs, const int32_t* tile_expert,
                          const int32_t* num_tiles, int T, int H, int I, int Et, int Kt,
                          int tile_m, uint16_t* out, void* workspace, size_t ws_bytes,
                          moe_path_t path, cudaStream_t stream) {
    moe_status_t st = check_ffn_shape(T, H, I, Et, Kt, tile_m, &path);
    if (st != MOE_OK || T == 0) return st;
    if (!ptrs_ok({x, w13, w2, out, workspace}, 16) ||
        !ptrs_ok({s13, s2, topk_w, sorted_pairs, expert_offsets, inv_pairs, tile_expert, num_tiles}, 4))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_ffn_workspace_size(T, H, I, Et, Kt, tile_m)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    st = moe_ffn_gate_up(x, w13, s13, sorted_pairs, tile_expert, num_tiles, T, H, I, Et, Kt, tile_m,
                         workspace, ws_bytes, path, stream);
    if (st != MOE_OK) return st;
    return moe_ffn_down_combine(w2, s2, topk_w, sorted_pairs, inv_pairs, tile_expert, num_tiles, T, H,
                                I, Et, Kt, tile_m, out, workspace, ws_bytes, path, stream);
}

moe_status_t moe_ffn(const uint16_t* x, const uint8_t* w13, const uint8_t* s13, const uint8_t* w2,
                     const uint8_t* s2, const float* topk_w, const int32_t* sorted_pairs,
                     const int32_t* expert_offsets, const int32_t* inv_pairs,
                     const int32_t* tile_expert, const int32_t* num_tiles, int T, int H, int I,
                     int Et, int Kt, int tile_m, uint16_t* out, void* workspace, size_t ws_bytes,
                     cudaStream_t stream) {
    return moe_ffn_path(x, w13, s13, w2, s2, topk_w, sorted_pairs, expert_offsets, inv_pairs,
                        tile_expert, num_tiles, T, H, I, Et, Kt, tile_m, out, workspace, ws_bytes,
                        MOE_PATH_AUTO, stream);
}

// ------------------------------------------------ MXFP4-quantised activations
// Workspace: x codes [T, H/2], x scales [T, H/32], x codes and scales
// gathered into tile order [cap, H/2] and [cap, H/32], h codes [cap, I/2], h
// scales [cap, I/32], routing weight per position fp32 [cap], y staged as f16
// rows by position [cap, Hpad] and its shift bytes [ceil(cap/32), Hpad/8]
// (Hpad = H rounded up to 128); each region starts on a 256-byte boundary.
struct MxLayoutWs {
    size_t xc, xs, xg, xgs, hc, hs, wpos, y, ysh, total;
};

static bool mx_layout(int T, int H, int I, int Et, int Kt, int tile_m, MxLayoutWs* L) {
    const int64_t cap = capacity64(T, Kt, Et, tile_m);
    if (cap < 0 || T < 0 || H <= 0 || I <= 0 || Kt <= 0) return false;
    L->xc = 0;
    L->xs = L->xc + round_up((size_t)T * (H / 2), 256);
    L->xg = L->xs + round_up((size_t)T * (H / 32), 256);
    L->xgs = L->xg + round_up((size_t)cap * (H / 2), 256);
    L->hc = L->xgs + round_up((size_t)cap * (H / 32), 256);
    L->hs = L->hc + round_up((size_t)cap * (I / 2), 256);
    L->wpos = L->hs + round_up((size_t)cap * (I / 32), 256);
    L->y = L->wpos + round_up((size_t)cap * sizeof(float), 256);
    const size_t hpad = (size_t)(H + 127) / 128 * 128;
    L->ysh = L->y + round_up((size_t)cap * hpad * sizeof(uint16_t), 256);
    L->total = L->ysh + round_up((size_t)((cap + 31) / 32) * (hpad / 8), 256);
    return true;
}

size_t moe_ffn_mxfp4act_workspace_size(int T, int H, int I, int Et, int Kt, int tile_m) {
    MxLayoutWs L;
    return mx_layout(T, H, I, Et, Kt, tile_m, &L) ? L.total : 0;
}

moe_status_t moe_ffn_mxfp4act_h_offsets(int T, int H, int I, int Et, int Kt, int tile_m,
                                        size_t* codes_offset, size_t* scales_offset) {
    MxLayoutWs L;
    if (!codes_offset || !scales_offset || !mx_layout(T, H, I, Et, Kt, tile_m, &L))
        return MOE_ERR_INVALID_ARG;
    *codes_offset = L.hc;
    *scales_offset = L.hs;
    return MOE_OK;
}

static moe_status_t check_mx_shape(int T, int H, int I, int Et, int Kt, int tile_m) {
    moe_path_t p = MOE_PATH_PREFILL;  // the general limits; the tile heights are checked below
    const int64_t cap = capacity64(T, Kt, Et, tile_m);
    if (cap < 0 || H <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
    if (!mxfp4act_tile_supported(tile_m) || !mxfp4act_shape_supported(H, I))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    return check_ffn_shape(T, H, I, Et, Kt, tile_m, &p);
}

moe_status_t moe_split_e4m3x2(const uint16_t* x, int rows, int cols, uint8_t* q_hi, uint8_t* q_lo,
                              uint8_t* s_hi, uint8_t* s_lo, cudaStream_t stream) {
    if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (cols % 32 || (int64_t)rows * cols >= ((int64_t)1 << 40) || rows >= (1 << 30))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!ptrs_ok({x, q_hi, q_lo}, 16) || !s_hi || !s_lo) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_split_rows(x, cols, rows, nullptr, nullptr, 0, 1, 0, 0, q_hi, q_lo, s_hi,
                                         s_lo, stream));
}

moe_status_t moe_quantize_mxfp4(const uint16_t* x, int rows, int cols, uint8_t* codes,
                                uint8_t* scales, cudaStream_t stream) {
    if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (cols % 32 || (int64_t)rows * cols >= ((int64_t)1 << 40)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!ptrs_ok({x, codes}, 16) || !scales) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_quantize_mxfp4(x, rows, cols, codes, scales, stream));
}

moe_status_t moe_ffn_mxfp4act_gate_up(const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                                      const int32_t* sorted_pairs, const int32_t* tile_expert,
                                      const int32_t* num_tiles, int T, int H, int I, int Et,
                                      int Kt, int tile_m, void* workspace, size_t ws_bytes,
                                      cudaStream_t stream) {
    moe_status_t st = check_mx_shape(T, H, I, Et, Kt, tile_m);
    if (st != MOE_OK || T == 0) return st;
    if (!ptrs_ok({x, w13, workspace}, 16) || !ptrs_ok({s13, sorted_pairs, tile_expert, num_tiles}, 4))
        return MOE_ERR_INVALID_ARG;
    MxLayoutWs L;
    mx_layout(T, H, I, Et, Kt, tile_m, &L);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    const int64_t cap = capacity64(T, Kt, Et, tile_m);
    char* ws = reinterpret_cast<char*>(workspace);
    cudaError_t err = launch_quantize_mxfp4(x, T, H, reinterpret_cast<uint8_t*>(ws + L.xc),
                                            reinterpret_cast<uint8_t*>(ws + L.xs), stream);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    // the GEMM reads each tile's token rows as one box per stage: gather the
    // code rows (H/2 bytes each) into tile order, and the scale rows (H/32
    // bytes) too when they are whole 16-byte units (then the GEMM loads them
    // by TMA; otherwise its scale warps read them by token)
    const bool sf_tma = H % 512 == 0;
    err = launch_gather_mx_rows(reinterpret_cast<const uint8_t*>(ws + L.xc),
                                reinterpret_cast<const uint8_t*>(ws + L.xs), H, sf_tma, sorted_pairs,
                                num_tiles, tile_m, Kt, (int)cap, T * Kt,
                                reinterpret_cast<uint8_t*>(ws + L.xg),
                                reinterpret_cast<uint8_t*>(ws + L.xgs), stream);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    GroupedGemm g = base_gemm(sorted_pairs, tile_expert, num_tiles, T, I, Et, Kt, tile_m,
                              (int)(cap / tile_m));
    g.codes = w13;
    g.scales = s13;
    g.rows = 2 * I;
    g.K = H;
    g.act = reinterpret_cast<const uint16_t*>(ws + L.xg);
    g.act_rows = (int)cap;
    g.act_scales = reinterpret_cast<const uint8_t*>(ws + (sf_tma ? L.xgs : L.xs));
    g.sf_tma = sf_tma ? 1 : 0;
    g.hq_codes = reinterpret_cast<uint8_t*>(ws + L.hc);
    g.hq_scales = reinterpret_cast<uint8_t*>(ws + L.hs);
    trace("moe_ffn_mxfp4act_gate_up", T, H, I, Et, Kt, tile_m, MOE_PATH_PREFILL);
    return cuda_status(launch_gemm_timed([&] { return launch_mxfp4act_gate_up(g, stream); }, stream));
}

moe_status_t moe_ffn_mxfp4act_down(const uint8_t* w2, const uint8_t* s2, const float* topk_w,
                                   const int32_t* sorted_pairs, const int32_t* inv_pairs,
                                   const int32_t* tile_expert, const int32_t* num_tiles, int T,
                                   int H, int I, int Et, int Kt, int tile_m, uint16_t* out,
                                   void* workspace, size_t ws_bytes, cudaStream_t stream) {
    moe_status_t st = check_mx_shape(T, H, I, Et, Kt, tile_m);
    if (st != MOE_OK || T == 0) return st;
    if (!ptrs_ok({w2, out, workspace}, 16) ||
        !ptrs_ok({s2, topk_w, sorted_pairs, inv_pairs, tile_expert, num_tiles}, 4))
        return MOE_ERR_INVALID_ARG;
    MxLayoutWs L;
    mx_layout(T, H, I, Et, Kt, tile_m, &L);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    const int64_t cap = capacity64(T, Kt, Et, tile_m);
    char* ws = reinterpret_cast<char*>(workspace);
    GroupedGemm g = base_gemm(sorted_pairs, tile_expert, num_tiles, T, I, Et, Kt, tile_m,
                              (int)(cap / tile_m));
    g.codes = w2;
    g.scales = s2;
    g.rows = H;
    g.K = I;
    g.act = reinterpret_cast<const uint16_t*>(ws + L.hc);
    g.act_rows = (int)cap;
    g.act_scales = reinterpret_cast<const uint8_t*>(ws + L.hs);
    g.sf_tma = I % 512 == 0 ? 1 : 0;
    g.y_blocked = 1;
    g.y16_out = reinterpret_cast<uint16_t*>(ws + L.y);
    g.y_shift = reinterpret_cast<int8_t*>(ws + L.ysh);
    g.y_rows_pad = (H + 127) / 128 * 128;
    g.topk_w = topk_w;
    float* w_pos = reinterpret_cast<float*>(ws + L.wpos);
    trace("moe_ffn_mxfp4act_down", T, H, I, Et, Kt, tile_m, MOE_PATH_PREFILL);
    cudaError_t err = launch_position_weights(sorted_pairs, topk_w, nullptr, num_tiles, tile_m,
                                              (int)cap, T * Kt, w_pos, stream);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    err = launch_gemm_timed([&] { return launch_mxfp4act_down(g, stream); }, stream);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_status(launch_combine_blocked_f16(g.y16_out, g.y_shift, inv_pairs, w_pos, T, H, Kt,
                                                  (int)cap, out, stream));
}

moe_status_t moe_ffn_mxfp4act(const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                              const uint8_t* w2, const uint8_t* s2, const float* topk_w,
                              const int32_t* sorted_pairs, const int32_t* expert_offsets,
                              const int32_t* inv_pairs, const int32_t* tile_expert,
                              const int32_t* num_tiles, int T, int H, int I, int Et, int Kt,
                              int tile_m, uint16_t* out, void* workspace, size_t ws_bytes,
                              cudaStream_t stream) {
    moe_status_t st = check_mx_shape(T, H, I, Et, Kt, tile_m);
    if (st != MOE_OK || T == 0) return st;
    if (!ptrs_ok({expert_offsets, inv_pairs}, 4)) return MOE_ERR_INVALID_ARG;
    st = moe_ffn_mxfp4act_gate_up(x, w13, s13, sorted_pairs, tile_expert, num_tiles, T, H, I, Et,
                                  Kt, tile_m, workspace, ws_bytes, stream);
    if (st != MOE_OK) return st;
    return moe_ffn_mxfp4act_down(w2, s2, topk_w, sorted_pairs, inv_pairs, tile_expert, num_tiles, T,
                                 H, I, Et, Kt, tile_m, out, workspace, ws_bytes, stream);
}

}  // extern "C"
