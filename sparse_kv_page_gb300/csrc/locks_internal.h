// locks_internal.h - launchers shared between the kernel files and the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "locks_common.cuh"

namespace locks {

// Raises a kernel's dynamic shared-memory limit (and allows 16-CTA clusters
// when asked) once per device instead of on every launch.
template <auto Kern>
cudaError_t ensure_kernel_attrs(int smem_bytes, bool nonportable_cluster = false) {
    static std::atomic<int> done[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire) >= smem_bytes + 1) return cudaSuccess;
    e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    if (nonportable_cluster) {
        e = cudaFuncSetAttribute(Kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    int prev = done[dev].load();
    while (prev < smem_bytes + 1 && !done[dev].compare_exchange_weak(prev, smem_bytes + 1)) {
    }
    return cudaSuccess;
}

// The scorer's persistent grid: one CTA per SM, at most kMaxScorerCtas (which bounds the
// size of its LSE partials). CTA c scores items [c * per, (c + 1) * per) of the
// batch * nchunks items, per = ceil(items / grid); an item is kStageUnits / Hkv
// consecutive logical pages of one sequence (all kv heads).
constexpr int kMaxScorerCtas = 256;
constexpr int kStageUnits = 64;
inline int score_grid(int total_items, int num_sms) {
    const int g = num_sms < kMaxScorerCtas ? num_sms : kMaxScorerCtas;
    return total_items < g ? total_items : g;
}
// LSE partial slots per (sequence, query head) in each scorer CTA: one per consumer warp
// that scores that head (two groups of 8 warps take alternate stages for GQA groups of up
// to 8 heads; for larger groups each group takes 8 of the heads; a group's 8 warps split
// a stage's pages over 8 / Hkv blocks).
__host__ __device__ constexpr int slot_warps(int hkv, int g) { return (g > 8 ? 1 : 2) * (8 / hkv); }

struct ScoreArgs {
    const float* q;
    const int8_t* mu;
    const uint8_t* basis;
    const int8_t* coef;
    const uint16_t* scales;
    const int32_t* page_table;
    const int32_t* seq_pages;
    float* scores;
    float* lse_partials;      // nullable: (max, sum exp) pairs [B][Hq][grid * slot_warps]: per
                              // (sequence, query head, scorer CTA, consumer warp), over the
                              // units that warp scored (-inf, 0 when none)
    int batch, hq, hkv, max_pages, num_phys;
    DeviceStatus st;
};
cudaError_t launch_score(const ScoreArgs& a, int num_sms, cudaStream_t stream);

struct SelectAttendArgs {
    // selection
    const float* scores;
    const float* lse_partials;   // nullable: the scorer's partials (ScoreArgs::lse_partials)
    int score_grid;           // the grid of the scorer launch that wrote them
    const int32_t* seq_pages;
    int32_t* selected;        // [B][Hkv][k_cap]
    int32_t* n_selected;      // [B][Hkv]
    float* sel_keys;          // nullable
    int budget_pages;         // budget_tokens / 16
    int k_cap;
    // attention
    const float* q;
    const uint16_t* k_cache;
    const uint16_t* v_cache;
    const int32_t* page_table;
    const int32_t* tail_tokens;   // nullable: tokens of each sequence's unfilled page (fused mode)
    uint16_t* out;
    float* lse;               // nullable
    // split attention (attention-only launches): `splits` clusters per (sequence, kv
    // head); per (b, q head) a zeroed arrival count and kMaxSplits (m, l, o[128]) partials
    int splits;
    int32_t* attn_cnt;        // nullable: no split
    float* attn_part;
    int batch, hq, hkv, max_pages, num_phys;
    DeviceStatus st;
    // K and V caches as 2D tensors [num_phys * hkv * 16 rows][128] bf16 for tiled TMA:
    // 64 x 16 boxes with 128-byte swizzle (filled by the launcher; unused by the selection)
    CUtensorMap tm_k, tm_v;
};
enum class SAMode { kSelect, kAttend, kSelectAttend };
constexpr int kMaxSplits = 4;
constexpr int kSplitPartFloats = 2 + 128;   // m, l, o[128] per (b, q head, split)
cudaError_t launch_select_attend(const SelectAttendArgs& a, SAMode mode, int cluster, cudaStream_t stream);
// Clusters of `cluster` CTAs (8, 12 or 16; 12 runs one CTA per SM) of the select/attend
// kernel that can be resident at once on the current device (0 if it cannot launch), and
// how many of its CTAs share an SM (1 or 2, from shared memory).
int select_attend_active_clusters(int max_pages, SAMode mode, int group, int cluster);
int select_attend_ctas_per_sm(int max_pages, SAMode mode, int cluster);
size_t select_attend_smem_bytes(int max_pages, int cluster, SAMode mode);

struct BuildArgs {
    const uint16_t* k_cache;
    const int32_t* phys_page_ids;
    int n_pages;
    int hkv;
    int num_phys;
    int8_t* mu;
    uint8_t* basis;
    int8_t* coef;
    uint16_t* scales;
    DeviceStatus st;
};
cudaError_t launch_build(const BuildArgs& a, int num_sms, cudaStream_t stream);

// Selector ablations (off the decode path). One argument block for the five kernels;
// each uses the fields its comment names.
struct AblationArgs {
    const float* q;           // [B][Hq][128]: queries (exact, variant, projection) or projected queries
    const uint16_t* k_cache;  // [num_phys][hkv][16][128] bf16
    const int32_t* page_table;
    const int32_t* seq_pages;
    float* scores;            // [B][Hq][max_pages] (exact, variant)
    int batch, hq, hkv, max_pages, num_phys;
    int rank;                 // variant: 1..15; shared basis / projection: 0..128
    int bits_mu, bits_v, bits_c;   // variant: 0 (unquantised) or 2..8
    float* moment;            // [B][Hkv][128][128] fp32 second moments (shared basis)
    float* basis;             // [B][Hkv][rank][128] (written by the shared basis, read by the projection)
    float* eigvals;           // nullable [B][Hkv][128] (shared basis)
    float* q_proj;            // [B][Hq][128] (projection output)
    DeviceStatus st;
};
cudaError_t launch_exact_scores(const AblationArgs& a, cudaStream_t stream);
cudaError_t launch_variant_scores(const AblationArgs& a, cudaStream_t stream);
cudaError_t launch_shared_basis(const AblationArgs& a, cudaStream_t stream);
cudaError_t launch_project_queries(const AblationArgs& a, cudaStream_t stream);

// Bounded-wait self test: one CTA waits on an mbarrier phase that never
// completes and must give up after the limit, recording LOCKS_ERR_TIMEOUT.
cudaError_t launch_wait_selftest(DeviceStatus st, cudaStream_t stream);

}  // namespace locks
