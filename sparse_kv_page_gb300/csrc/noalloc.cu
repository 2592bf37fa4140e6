// noalloc.cu - a decode step for callers that cannot allocate device memory.
//
// Serving engines commonly reserve almost all of HBM for their own paged KV
// pool at start-up and hand plugins no allocator, and cudaMalloc itself may
// synchronise the device, which a latency-critical decode loop cannot afford.
// Such callers cannot provide the workspace that locks_decode_step needs. This
// file gives them one entry point whose scratch (the score table and the
// selection) lives in a fixed, file-scope device array instead. It runs the
// same two kernels as locks_decode_step by calling it with that array as the
// workspace; no existing code path changes.
#include <cudaTypedefs.h>

#include <mutex>

#include "locks_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(36) << 20;   // 36 MiB per GPU, held until exit
constexpr int kMaxContexts = 64;

// Device storage; in host code this name is only a stand-in for the symbol,
// its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// The array's address differs per CUDA context (each context loads the module
// anew), so the looked-up addresses are cached per (device, current context).
struct Entry {
    int dev;
    CUcontext ctx;
    void* ptr;
};
std::mutex g_mu;
Entry g_cache[kMaxContexts];
int g_n = 0;

// The driver's cuCtxGetCurrent, looked up once through the runtime.
PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
    static const PFN_cuCtxGetCurrent_v4000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return static_cast<PFN_cuCtxGetCurrent_v4000>(nullptr);
        }
        return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    }();
    return fn;
}

// Device address of the scratch array in the current device's current context
// (looked up with that device current on the first call in each context).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return LOCKS_ERR_CUDA;
    }
    const auto get = ctx_get_current();
    if (!get) return LOCKS_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS) return LOCKS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (ctx != nullptr) {
        for (int i = 0; i < g_n; ++i)
            if (g_cache[i].dev == dev && g_cache[i].ctx == ctx) {
                *out = g_cache[i].ptr;
                return LOCKS_OK;
            }
    }
    // First call in this context (or no context current yet: the lookup makes the
    // runtime's primary context of `dev` current, and it is cached under that one).
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return LOCKS_ERR_CUDA;
    }
    if (ctx == nullptr && (get(&ctx) != CUDA_SUCCESS || ctx == nullptr)) return LOCKS_ERR_CUDA;
    if (g_n < kMaxContexts) g_cache[g_n++] = {dev, ctx, p};
    *out = p;
    return LOCKS_OK;
}

}  // namespace

extern "C" LOCKS_API int locks_decode_step_noalloc(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                                                   const uint16_t* v_cache, locks_summaries_t summaries,
                                                   const int32_t* page_table, const int32_t* seq_pages,
                                                   int32_t budget_tokens, uint16_t* out, float* lse, void* stream) {
    size_t need = 0;
    int v = locks_workspace_size(dims, budget_tokens, &need);
    if (v != LOCKS_OK) return v;
    if (need > kNoAllocScratchBytes) return LOCKS_ERR_WORKSPACE_TOO_SMALL;
    void* scratch = nullptr;
    if ((v = scratch_address(&scratch)) != LOCKS_OK) return v;
    // Every part of the scratch is written before it is read within one call
    // (scores, then the selection); the status word is cleared so each call
    // starts from LOCKS_OK.
    if (cudaMemsetAsync(scratch, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return LOCKS_ERR_CUDA;
    }
    return locks_decode_step(dims, q, k_cache, v_cache, summaries, page_table, seq_pages, budget_tokens, out, lse,
                             nullptr, nullptr, nullptr, scratch, kNoAllocScratchBytes, stream);
}
