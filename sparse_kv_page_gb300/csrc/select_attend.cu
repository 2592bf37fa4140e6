// select_attend.cu - group-shared top-k page selection and sparse attention.
//
// One thread-block cluster of CL CTAs per (sequence b, kv head). The CTAs of
// a cluster split the sequence's pages (selection) and then the selected
// pages (attention) and combine their partial results through distributed
// shared memory, so selection and attention need no global scratch and no
// second launch. Attention-only launches over long selections may also split
// a (sequence, kv head) over several clusters, merged through the workspace
// by the last cluster to finish.
//
// Selection (gist.science summary of the LOCKS paper, 2.3 "group-shared
// selection"; LOCKS post, "Code": keep budget // 16 pages, sorted ascending):
//   L_h   = log sum_j exp(s_hj)                      (per query head)
//   key_j = log((1/g) sum_{h in group} exp(s_hj - L_h))
//   top-k by a radix select on the order-preserving uint32 image of key_j:
//   a first 8-bit pass over the range the keys' sum fixes, built with the
//   keys; its histograms summed across the cluster through DSMEM; then the
//   candidates (keys in and above the chosen bin) gathered into every CTA and
//   the bin ranked directly (an exact MSB-first radix out of line when that
//   fails). Equal keys are ranked by lower page id; the kept pages are written
//   in ascending page order.
// Attention (LOCKS post, "Code": scaled dot-product attention over the pages
// kept): each CTA takes a contiguous share of the selected pages; each warp
// streams its pages (K and V rows as four tiled TMA boxes of 16 tokens x 64
// dims, 128-byte swizzle; one or two ring slots per warp) and runs QK^T and PV
// on the tensor cores (mma.sync bf16 through ldmatrix, query split hi/lo,
// online softmax in fp32). Warp partials (m, l, o) are merged per CTA, then
// across the cluster (pulled through DSMEM, or, on 12-CTA clusters, pushed
// into the owning CTA).
//
// When the scoring kernel's LSE partials (one (max, sum exp) pair per scorer warp
// and query head) are given, the per-head normaliser L_h is reduced from them
// instead of from the full score table.
// 8- and 16-CTA instances keep to 128 registers per thread so that two CTAs
// share an SM; 12-CTA instances run one CTA per SM.
#include <cudaTypedefs.h>
#include <algorithm>
#include <climits>
#include <cstring>

#include "locks_internal.h"

namespace locks {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
// A page slot holds the page's K then V rows of one kv head as four TMA boxes of
// 16 rows x 64 dims (128-byte rows, 128-byte swizzle: 16-byte chunk c of row r
// sits at chunk c ^ (r & 7)), each 2 KiB and 1 KiB-aligned.
constexpr int kBoxBytes = kPage * 64 * 2;             // 2048 B
constexpr int kPageSlotBytes = 4 * kBoxBytes;         // 8192 B
constexpr int kPartStride = 2 + kD;                   // m, l, o[128]
static_assert(kPartStride == kSplitPartFloats, "split partials use the attention partial layout");
// the ring also holds the warps' attention partials after the page loop
constexpr int kWarpPartBytes = kWarps * LOCKS_MAX_GROUP * kPartStride * 4;
constexpr int kRingBytes = ((kWarps * kPageSlotBytes > kWarpPartBytes ? kWarps * kPageSlotBytes : kWarpPartBytes) +
                            1023) / 1024 * 1024;
constexpr int kMaxG = LOCKS_MAX_GROUP;
constexpr int kQRow = 136;                            // bf16 per staged query row (128 + 8 pad)
constexpr int kRankCap = 256;                         // radix early exit: largest bin ranked directly
constexpr int kCandCap = 768;                         // fast selection: candidates gathered per segment
constexpr int kCandListBytes = kCandCap * 12;         // a list of (key, logical page, physical page)
constexpr int kStageBytes = 64 * 1024;                // staged score rows (four heads) of a CTA's pages
static_assert(kStageBytes <= kRingBytes, "the staged scores share the attention ring's space");
// The 12-CTA cluster runs one CTA per SM: its launch asks for more shared memory than two
// CTAs can share. Eight such clusters are co-resident on this GPU (96 SMs), where eight
// 16-CTA clusters are packed two CTAs to an SM on 64 SMs. Its CTAs may stage up to
// 128 KiB of score rows (four heads of 8192 pages).
constexpr int kSpreadCluster = 12;
constexpr int kSpreadStageBytes = 128 * 1024;
constexpr int kSpreadSmemBytes = 120 * 1024;
__host__ __device__ constexpr int stage_cap(int cl) { return cl == kSpreadCluster ? kSpreadStageBytes : kStageBytes; }
__host__ __device__ constexpr int round_kib(int bytes) { return (bytes + 1023) / 1024 * 1024; }
// Attention ring: one page slot per warp, two for the 12-CTA cluster (a warp's next page
// is in flight while it attends the current one).
__host__ __device__ constexpr int slots_per_warp(int cl) { return cl == kSpreadCluster ? 2 : 1; }
__host__ __device__ constexpr int ring_bytes(int cl) {
    return round_kib(slots_per_warp(cl) * kWarps * kPageSlotBytes > kWarpPartBytes
                         ? slots_per_warp(cl) * kWarps * kPageSlotBytes
                         : kWarpPartBytes);
}
// Shared memory after SmallShared: region A (the keys, which overlay the staged score rows
// of four heads, then the attention ring), then (selection) the published and the gathered
// candidate lists.
// 12-CTA clusters merge the attention by pushing each CTA's per-head partial into the
// owning CTA's inbox (after every other region): slot (head / CL, source CTA), each
// [m, l, 2 pad, o[128]] floats; a CTA owns at most two of up to 16 heads.
constexpr int kInStride = 4 + kD;
constexpr int kInboxBytes = 2 * kSpreadCluster * kInStride * 4;
__host__ __device__ constexpr int region_a_bytes(int chunk, int cl) {
    return (4 * chunk * 4 <= stage_cap(cl) && round_kib(4 * chunk * 4) > ring_bytes(cl)) ? round_kib(4 * chunk * 4)
           : round_kib(chunk * 4) > ring_bytes(cl)                                        ? round_kib(chunk * 4)
                                                                                           : ring_bytes(cl);
}
// byte offset of the inbox from the region after SmallShared
__host__ __device__ constexpr int inbox_offset(int chunk, int cl, bool attend_only) {
    return attend_only ? ring_bytes(cl) : region_a_bytes(chunk, cl) + 2 * kCandListBytes;
}

struct SmallShared {
    uint16_t qs[2][16 * kQRow];           // query rows (group heads), bf16 high / low parts
    uint32_t hist[2][256];
    float part_m[kMaxG], part_l[kMaxG];   // this CTA's per-head LSE partial
    float Lh[kMaxG];
    float red_m[kWarps][kMaxG], red_l[kWarps][kMaxG];
    uint32_t tot[3][256];                 // radix pass: bin counts of all CTAs, lower-ranked CTAs, this CTA
    int wcnt[kWarps][2];
    int digit, above, above_low, above_own, eq_low, eq_own, inbin;
    // radix early exit: the chosen bin's keys (this CTA's, then all CTAs')
    int bin_cnt[16], nbin, rank_take, rank_eq, cnt4[4];
    int wtot[3][kWarps];                  // strided scans: flagged elements per (slot, warp)
    uint32_t rank_T;
    uint32_t bin_keys[256], rank_keys[256];
    uint8_t rank_src[256];
    uint64_t bar[2 * kWarps];             // attention ring slots (two per warp at most)
    uint64_t sbar;                        // staged score rows (selection)
    int pub_n;                            // fast selection: this CTA's published candidates
    int cnt_r[16];                        // ... and every CTA's count
    float cpart[kMaxG * kPartStride];     // this CTA's attention partial per head
    int split_last;                       // split attention: this cluster merges the splits of a head
};

// Two CTAs share an SM up to 4096 pages per CTA (the 1M-token context over 16 CTAs).
static_assert(sizeof(SmallShared) + 1024 + kRingBytes + 2 * kCandListBytes <= 113 * 1024,
              "shared memory of two select/attend CTAs per SM");

// Byte offset of (token row, dim) in a page slot's K (or V) half: box = dim / 64,
// 16-byte chunk (dim % 64) / 8 swizzled with the row.
__device__ __forceinline__ int swz_offset(int token, int dim) {
    return (dim >> 6) * kBoxBytes + token * 128 + ((((dim & 63) >> 3) ^ (token & 7)) << 4);
}

__device__ __forceinline__ void lse_combine(float& m, float& l, float m2, float l2) {
    const float M = fmaxf(m, m2);
    if (M == -INFINITY) return;
    l = l * fast_exp2((m - M) * kLog2e) + l2 * fast_exp2((m2 - M) * kLog2e);
    m = M;
}

// Stores into another CTA's shared memory (cluster-window addresses from dsmem_addr).
__device__ __forceinline__ void st_dsmem_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_dsmem_f32x2(uint32_t addr, float a, float b) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ void st_dsmem_f32x4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// ------------------------------------------------------------- selection
// Stores the group's query rows (scaled by log2(e)/sqrt(d)) in shared memory as bf16
// high and low parts; the attention's MMA A fragments are read back with ldmatrix.
__device__ __forceinline__ void store_query(const float (&qv)[16 * kD / kThreads], int g, SmallShared& sh) {
#pragma unroll
    for (int u = 0; u < 16 * kD / kThreads; ++u) {
        const int idx = threadIdx.x + u * kThreads, row = idx / kD, col = idx % kD;
        const float x = row < g ? qv[u] * (kInvSqrtD * kLog2e) : 0.f;
        const __nv_bfloat16 h = __float2bfloat16_rn(x);
        const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(h));
        sh.qs[0][row * kQRow + col] = __bfloat16_as_ushort(h);
        sh.qs[1][row * kQRow + col] = __bfloat16_as_ushort(lo);
    }
}
__device__ __forceinline__ void load_query(const SelectAttendArgs& a, int b, int kvh, int g,
                                           float (&qv)[16 * kD / kThreads]) {
#pragma unroll
    for (int u = 0; u < 16 * kD / kThreads; ++u) {
        const int idx = threadIdx.x + u * kThreads, row = idx / kD, col = idx % kD;
        qv[u] = row < g ? a.q[(static_cast<int64_t>(b) * a.hq + kvh * g + row) * kD + col] : 0.f;
    }
}

// Score reads: a thread takes kSL slabs of 4 consecutive pages per round (slab i of the
// round at page jr starts at jr + 4 (tid + i kThreads)) and kHB query heads at a time.
// A NaN score carries no mass (read as -inf), as do pages at or past j1 and heads >= g.
constexpr int kSL = 4;
constexpr int kRoundPages = kSL * 4 * kThreads;   // 4096
constexpr int kHB = 4;
struct ScoreRound {
    float4 v[kSL][kHB];
};

__device__ __forceinline__ float no_nan(float x) { return x == x ? x : -INFINITY; }

// From global memory (128-bit loads when rows are 16-byte aligned), heads [h0, h0 + kHB).
__device__ __forceinline__ void load_round(const float* srow, int64_t stride, int g, int h0, int jr, int j1,
                                           bool vec, ScoreRound& x) {
#pragma unroll
    for (int i = 0; i < kSL; ++i) {
        const int j = jr + 4 * (static_cast<int>(threadIdx.x) + i * kThreads);
#pragma unroll
        for (int hh = 0; hh < kHB; ++hh) {
            float4 v = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (h0 + hh < g && j < j1) {
                const float* p = srow + static_cast<int64_t>(h0 + hh) * stride + j;
                if (vec) {
                    v = __ldcg(reinterpret_cast<const float4*>(p));
                } else {
                    v.x = __ldcg(p);
                    if (j + 1 < j1) v.y = __ldcg(p + 1);
                    if (j + 2 < j1) v.z = __ldcg(p + 2);
                    if (j + 3 < j1) v.w = __ldcg(p + 3);
                }
            }
            x.v[i][hh] = v;
        }
    }
}
// From the staged rows in shared memory (row hh of the batch at stg + hh * chunk; off is
// the round's first page relative to the CTA's first page).
__device__ __forceinline__ void load_round_smem(const float* stg, int chunk, int nh, int off, int nloc,
                                                ScoreRound& x) {
#pragma unroll
    for (int i = 0; i < kSL; ++i) {
        const int jj = off + 4 * (static_cast<int>(threadIdx.x) + i * kThreads);
#pragma unroll
        for (int hh = 0; hh < kHB; ++hh) {
            float4 v = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (hh < nh && jj < nloc) v = *reinterpret_cast<const float4*>(stg + hh * chunk + jj);
            x.v[i][hh] = v;
        }
    }
}
__device__ __forceinline__ float round_val(const ScoreRound& x, int i, int hh, int e, int j, int j1) {
    const float4 v = x.v[i][hh];
    const float s = e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w));
    return j + e < j1 ? no_nan(s) : -INFINITY;
}

// The first radix digit of the selection (fast path). Keys are log mass shares that sum
// to 1 over the sequence (each head's shares sum to 1 and a key is the group mean), so at
// most K - 1 keys exceed -ln K, and the K-th largest lies above -ln P (P pages; the mean
// share is 1/P) unless K is a large fraction of P. The
// first pass counts the keys' order-preserving uint32 images u in 256 bins of 2^s images
// spanning [lo, hi], hi = -ln K + 1/4, lo = -ln P; keys below / above the span fall in
// bins 0 / 255 (bin 0 -- about half of the keys -- is counted by difference, without
// atomics). If the K-th key lands in bin 0 or 255 the selection
// restarts as a plain MSB-first radix over the whole key (exact either way).
struct RadixRange {
    uint32_t base;   // u of the first image of bin 0
    uint64_t top;    // one past the last image of bin 255 (<= 2^32)
    uint32_t last;   // top - 1
    int s;           // log2 of the bin width
};
__device__ __forceinline__ RadixRange fast_range(int K, int P) {
    const float hi = -logf(static_cast<float>(K)) + 0.25f;
    const float lo = -logf(static_cast<float>(P));
    const uint32_t uhi = orderable_key(hi), ulo = orderable_key(lo);   // hi > lo since K < P
    const uint64_t span = static_cast<uint64_t>(uhi) - ulo + 1;
    RadixRange r;
    r.s = 0;
    while ((256ull << r.s) < span) ++r.s;
    r.top = static_cast<uint64_t>(uhi) + 1;
    if (r.top > (256ull << r.s)) {
        r.base = static_cast<uint32_t>(r.top - (256ull << r.s));
    } else {
        r.base = 0u;
        r.top = 256ull << r.s;
    }
    r.last = static_cast<uint32_t>(r.top - 1);
    return r;
}
__device__ __forceinline__ uint32_t fast_digit(uint32_t u, const RadixRange& r) {
    return u < r.base ? 0u : min((u - r.base) >> r.s, 255u);   // above the range: bin 255
}
// The float key of an order-preserving image (orderable_key's inverse; image 0 gives NaN).
__device__ __forceinline__ float key_of_image(uint32_t u) {
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// Per-head normaliser L_h of sequence b into sh.Lh[0..g) (the same in every CTA).
// From the scorer's LSE partials (its launch of grid a.score_grid wrote one (max, sum exp)
// per scorer CTA and consumer warp that scored the head): warp w reduces heads w, w + 8
// over the partials of the scorer CTAs whose item range covers sequence b; no exchange.
// Without partials: each CTA reduces its own pages' scores (staged rows or global
// loads) and the CTAs exchange their (max, sum) through DSMEM.
// The normaliser from this CTA's own scores and a cluster exchange (launches without the
// scorer's partials): out of line, so that the partials path's code is contiguous.
template <int CL, int GM>
__device__ __noinline__ void normaliser_scores(const SelectAttendArgs& a, int b, int kvh, int g, int j0, int j1,
                                             bool staged, const float* stg, int chunk, SmallShared& sh) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // from this CTA's scores, then a cluster exchange
    const int64_t stride = a.max_pages;
    const float* srow = a.scores + (static_cast<int64_t>(b) * a.hq + kvh * g) * stride;
    const bool vec = (a.max_pages & 3) == 0 && (reinterpret_cast<uintptr_t>(a.scores) & 15) == 0;
    constexpr int kBatches = (GM + kHB - 1) / kHB;
    float m[GM], l[GM];
#pragma unroll
    for (int hh = 0; hh < GM; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.f;
    }
#pragma unroll 1
    for (int jr = j0; jr < j1; jr += kRoundPages) {
#pragma unroll
        for (int bt = 0; bt < kBatches; ++bt) {
            ScoreRound x;
            if (staged && bt == 0)
                load_round_smem(stg, chunk, min(g, kHB), jr - j0, j1 - j0, x);
            else
                load_round(srow, stride, g, bt * kHB, jr, j1, vec, x);
#pragma unroll
            for (int hh = 0; hh < kHB; ++hh) {
                const int h = bt * kHB + hh;
                if (h >= g || h >= GM) continue;
                float bm = -INFINITY;
#pragma unroll
                for (int i = 0; i < kSL; ++i) {
                    const int j = jr + 4 * (tid + i * kThreads);
#pragma unroll
                    for (int e = 0; e < 4; ++e) bm = fmaxf(bm, round_val(x, i, hh, e, j, j1));
                }
                if (bm == -INFINITY) continue;
                float z = 0.f;
#pragma unroll
                for (int i = 0; i < kSL; ++i) {
                    const int j = jr + 4 * (tid + i * kThreads);
#pragma unroll
                    for (int e = 0; e < 4; ++e) z += fast_exp2((round_val(x, i, hh, e, j, j1) - bm) * kLog2e);
                }
                lse_combine(m[h], l[h], bm, z);
            }
        }
    }
    // warp reduction: max first, then the sums rescaled to it
#pragma unroll
    for (int hh = 0; hh < GM; ++hh) {
        if (hh < g) {
            float M = m[hh];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            float z = (m[hh] == -INFINITY) ? 0.f : l[hh] * fast_exp2((m[hh] - M) * kLog2e);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
            if (lane == 0) {
                sh.red_m[warp][hh] = M;
                sh.red_l[warp][hh] = z;
            }
        }
    }
    __syncthreads();
    if (tid < g) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sh.red_m[w][tid]);
        float z = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w)
                if (sh.red_m[w][tid] != -INFINITY) z += sh.red_l[w][tid] * fast_exp2((sh.red_m[w][tid] - M) * kLog2e);
        }
        sh.part_m[tid] = M;
        sh.part_l[tid] = z;
    }
    cluster_sync_all();
    if (tid < g) {
        float pm[CL], pl[CL];   // all remote loads in flight before any use
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) {
            pm[r] = ld_dsmem_f32(dsmem_addr(&sh.part_m[tid], r));
            pl[r] = ld_dsmem_f32(dsmem_addr(&sh.part_l[tid], r));
        }
        float M = -INFINITY;
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) M = fmaxf(M, pm[r]);
        float z = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (uint32_t r = 0; r < CL; ++r)
                if (pm[r] != -INFINITY) z += pl[r] * fast_exp2((pm[r] - M) * kLog2e);
        }
        sh.Lh[tid] = (z > 0.f) ? M + logf(z) : -INFINITY;
    }
    __syncthreads();
}

template <int CL, int GM>
__device__ void normaliser(const SelectAttendArgs& a, int b, int kvh, int g, int j0, int j1, bool staged,
                           const float* stg, int chunk, SmallShared& sh) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (a.lse_partials) {
        const int np = kStageUnits / a.hkv;
        const int nchunks = (a.max_pages + np - 1) / np;
        const int grid = max(1, a.score_grid);
        const int per = max(1, (a.batch * nchunks + grid - 1) / grid);   // no items: c_hi < c_lo, n = 0
        const int W = slot_warps(a.hkv, g);
        const int c_lo = (b * nchunks) / per;
        const int c_hi = min(grid - 1, ((b + 1) * nchunks - 1) / per);
        const int n = (c_hi - c_lo + 1) * W;
#pragma unroll 1
        for (int hh = warp; hh < g; hh += kWarps) {
            const float2* row = reinterpret_cast<const float2*>(a.lse_partials) +
                                (static_cast<int64_t>(b) * a.hq + kvh * g + hh) * grid * W + c_lo * W;
            float m = -INFINITY, l = 0.f;
            // two (max, sum) pairs per 16-byte load (a slot row starts on an even pair: W is even)
#pragma unroll 1
            for (int i0 = 0; i0 < n; i0 += 2 * 32 * 8) {
                float4 v[8];   // all in flight before any use
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + 2 * (lane + 32 * u);
                    v[u] = i < n ? __ldcg(reinterpret_cast<const float4*>(row + i))
                                 : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
                }
                // an empty or corrupt pair (sum not > 0, or a NaN) contributes nothing
                float mm[16];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    mm[2 * u] = (v[u].y > 0.f && v[u].x == v[u].x) ? v[u].x : -INFINITY;
                    mm[2 * u + 1] = (v[u].w > 0.f && v[u].z == v[u].z) ? v[u].z : -INFINITY;
                }
                float M = m;
#pragma unroll
                for (int k = 0; k < 16; ++k) M = fmaxf(M, mm[k]);
                if (M != -INFINITY) {
                    float z = m == -INFINITY ? 0.f : l * fast_exp2((m - M) * kLog2e);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        z += mm[2 * u] == -INFINITY ? 0.f : v[u].y * fast_exp2((mm[2 * u] - M) * kLog2e);
                        z += mm[2 * u + 1] == -INFINITY ? 0.f : v[u].w * fast_exp2((mm[2 * u + 1] - M) * kLog2e);
                    }
                    m = M;
                    l = z;
                }
            }
            float M = m;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            float z = (m == -INFINITY) ? 0.f : l * fast_exp2((m - M) * kLog2e);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
            if (lane == 0) sh.Lh[hh] = (z > 0.f) ? M + logf(z) : -INFINITY;
        }
        __syncthreads();
        return;
    }
    normaliser_scores<CL, GM>(a, b, kvh, g, j0, j1, staged, stg, chunk, sh);
}

// Bulk copy of rows [h0, h0 + nh) of this CTA's score columns [j0, j0 + nloc) to the
// staging buffer (row hh at stg + hh * chunk), completing on sh.sbar. One thread.
__device__ __forceinline__ void stage_rows(const float* srow, int64_t stride, int h0, int nh, int j0, int nloc,
                                           int chunk, float* stg, SmallShared& sh) {
    const uint32_t bytes = static_cast<uint32_t>((nloc + 3) & ~3) * 4u;   // within the row: max_pages % 4 == 0
    mbar_arrive_expect_tx(&sh.sbar, bytes * static_cast<uint32_t>(nh));
    for (int hh = 0; hh < nh; ++hh) bulk_g2s(stg + hh * chunk, srow + (h0 + hh) * stride + j0, bytes, &sh.sbar);
}

// Loads the scores of heads [h0, h0 + kHB) of the 4-page slab at page j (relative jj to
// the CTA's first page) from the staged rows (row hh at stg + hh * chunk) or from global
// memory; heads >= g read as -inf. Values of pages at or past j1 are not meaningful.
__device__ __forceinline__ void load_slab(const float* stg, int chunk, const float* srow, int64_t stride, int g,
                                          int h0, int j, int jj, int j1, bool staged, bool vec, float4 (&v)[kHB]) {
#pragma unroll
    for (int hh = 0; hh < kHB; ++hh) {
        float4 x = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (h0 + hh < g) {
            if (staged) {
                x = *reinterpret_cast<const float4*>(stg + hh * chunk + jj);
            } else {
                const float* p = srow + static_cast<int64_t>(h0 + hh) * stride + j;
                if (vec) {
                    x = __ldcg(reinterpret_cast<const float4*>(p));
                } else {
                    x.x = __ldcg(p);
                    if (j + 1 < j1) x.y = __ldcg(p + 1);
                    if (j + 2 < j1) x.z = __ldcg(p + 2);
                    if (j + 3 < j1) x.w = __ldcg(p + 3);
                }
            }
        }
        v[hh] = x;
    }
}
__device__ __forceinline__ float comp(const float4& v, int e) {
    return e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w));
}

// Warp w's share [w0, w1) of a CTA's n keys: contiguous, a multiple of 4 long.
__device__ __forceinline__ void warp_span(int n, int w, int& w0, int& w1) {
    const int per = ((n + kWarps - 1) / kWarps + 3) & ~3;
    w0 = min(n, w * per);
    w1 = min(n, w0 + per);
}

// Pages whose unshifted sum underflowed in the staged key loop (every share below 2^-100,
// or none): the key again with the largest term factored out, from the scores in global
// memory (staged row 0 now holds the keys); the histogram is corrected. Out of line: rare.
__device__ __noinline__ void keys_underflow_fixup(const float* srow, int64_t stride, int g, int j0, int w0, int w1,
                                                  uint32_t* keys, float4 Lp4, float log_g, bool hist0,
                                                  const RadixRange fr, uint32_t* whist) {
    const float Lp[kHB] = {Lp4.x, Lp4.y, Lp4.z, Lp4.w};
#pragma unroll 1
    for (int jj = w0 + 4 * (threadIdx.x & 31); jj < w1; jj += 128) {
#pragma unroll 1
        for (int e = 0; e < 4 && jj + e < w1; ++e) {
            float x[kHB], m = -INFINITY;
#pragma unroll
            for (int hh = 0; hh < kHB; ++hh) {
                x[hh] = hh < g ? fmaf(no_nan(__ldcg(srow + hh * stride + j0 + jj + e)), kLog2e, -Lp[hh]) : -INFINITY;
                m = fmaxf(m, x[hh]);
            }
            float z = 0.f, zz = 0.f;
#pragma unroll
            for (int hh = 0; hh < kHB; ++hh) {
                z += fast_exp2(x[hh]);
                zz += fast_exp2(x[hh] - m);
            }
            const uint32_t old_u = keys[jj + e];
            if (old_u == 0u || z >= 7.9e-31f) continue;   // NaN key, or no underflow
            const float key2 = m == -INFINITY ? -INFINITY : m + fast_log2(zz);
            const uint32_t u = orderable_key(key2 * kLn2 - log_g);
            if (hist0) {
                const uint32_t d0 = fast_digit(old_u, fr), d1 = fast_digit(u, fr);
                if (d0 != 0u) atomicSub(&whist[(threadIdx.x >> 5) * 256 + d0], 1u);
                if (d1 != 0u) atomicAdd(&whist[(threadIdx.x >> 5) * 256 + d1], 1u);
            }
            keys[jj + e] = u;
        }
    }
}
// The optional key output (tests), once every thread's keys are final. Out of line.
__device__ __noinline__ void keys_out(float* kout, const uint32_t* keys, int nloc) {
    __syncthreads();
#pragma unroll 1
    for (int i = threadIdx.x; i < nloc; i += kThreads) kout[i] = key_of_image(keys[i]);
}

// group_keys for scores read with loads (rows not staged) or groups of more than four
// heads (staged four rows at a time). Returns whether a staging wait timed out. Called
// inline for large groups (their normal path) and out of line otherwise (rare), so that
// the staged path's code is contiguous.
template <int GM>
__device__ __forceinline__ bool group_keys_loads(const SelectAttendArgs& a, int b, int kvh, int j0, int j1, int chunk, uint32_t* keys,
                           SmallShared& sh, bool staged, const RadixRange fr, bool hist0, uint32_t* whist) {
    bool failed = false;
    const int tid = threadIdx.x;
    const int g = a.hq / a.hkv;
    const int nloc = j1 - j0;
    const int64_t stride = a.max_pages;
    const float* srow = a.scores + (static_cast<int64_t>(b) * a.hq + kvh * g) * stride;
    const bool vec = (a.max_pages & 3) == 0 && (reinterpret_cast<uintptr_t>(a.scores) & 15) == 0;
    const float* stg = reinterpret_cast<const float*>(keys);
    const float log_g = logf(static_cast<float>(g));
    float Lp[GM];
#pragma unroll
    for (int hh = 0; hh < GM; ++hh) Lp[hh] = hh < g ? sh.Lh[hh] * kLog2e : 0.f;
    float* kout = a.sel_keys ? a.sel_keys + (static_cast<int64_t>(b) * a.hkv + kvh) * a.max_pages : nullptr;
    // key of one page from its log2-domain total (m, z): the largest term 2^m, the sum
    // z of 2^(x - m); counts it and writes the optional key output
    auto finish = [&](int j, float key2) -> uint32_t {
        const float key = key2 * kLn2 - log_g;
        const uint32_t u = orderable_key(key);
        if (j < j1) {
            const uint32_t d = fast_digit(u, fr);
            if (hist0 && d != 0u) atomicAdd(&whist[(threadIdx.x >> 5) * 256 + d], 1u);   // this warp's counts
            if (kout) kout[j] = key;
        }
        return u;
    };
    if constexpr (GM <= kHB) {
        // a rolled loop over this thread's slabs (instruction fetch is part of this code's
        // latency: it runs about once per launch), the slab's four pages in parallel
#pragma unroll 1
        for (int jr = j0; jr < j1; jr += kRoundPages) {
#pragma unroll 1
            for (int i = 0; i < kSL; ++i) {
                const int j = jr + 4 * (tid + i * kThreads);   // consecutive threads, consecutive slabs
                if (j >= j1) break;
                float4 v[kHB];
                load_slab(stg, chunk, srow, stride, g, 0, j, j - j0, j1, staged, vec, v);
                uint32_t k4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float x[kHB], z = 0.f;
#pragma unroll
                    for (int hh = 0; hh < kHB; ++hh) {
                        x[hh] = hh < g ? fmaf(comp(v[hh], e), kLog2e, -Lp[hh]) : -INFINITY;
                        z += fast_exp2(x[hh]);
                    }
                    float key2 = fast_log2(z);
                    if (!(z >= 7.9e-31f) && z == z) {   // underflow (2^-100): factor out the largest term
                        float m = x[0];
#pragma unroll
                        for (int hh = 1; hh < kHB; ++hh) m = fmaxf(m, x[hh]);
                        float zz = 0.f;
#pragma unroll
                        for (int hh = 0; hh < kHB; ++hh) zz += fast_exp2(x[hh] - m);
                        key2 = m == -INFINITY ? -INFINITY : m + fast_log2(zz);
                    }
                    k4[e] = finish(j + e, key2);
                }
                // keys[] has room for whole slabs (chunk is a multiple of 8)
                *reinterpret_cast<uint4*>(keys + (j - j0)) = make_uint4(k4[0], k4[1], k4[2], k4[3]);
            }
        }
    } else {
        constexpr int kBatches = (GM + kHB - 1) / kHB;
        const int nbt = (g + kHB - 1) / kHB;
#pragma unroll 1
        for (int jr = j0; jr < j1; jr += kRoundPages) {
            float pm[kSL * 4], pz[kSL * 4];   // per page of this thread: largest term and sum (log2)
#pragma unroll
            for (int p = 0; p < kSL * 4; ++p) {
                pm[p] = -INFINITY;
                pz[p] = 0.f;
            }
#pragma unroll 1
            for (int bt = 0; bt < nbt && bt < kBatches; ++bt) {
                if (staged && bt > 0) {
                    // the next four rows into the staging buffer once every thread has read it
                    __syncthreads();
                    if (tid == 0) {
                        fence_proxy_async_smem();
                        stage_rows(srow, stride, bt * kHB, min(g - bt * kHB, kHB), j0, nloc, chunk,
                                   reinterpret_cast<float*>(keys), sh);
                    }
                }
                if (staged && !mbar_wait_bounded(&sh.sbar, static_cast<uint32_t>(bt & 1), a.st.wait_limit_ns))
                    failed = true;
                float Lb[kHB];
#pragma unroll
                for (int hh = 0; hh < kHB; ++hh) {
                    float L = 0.f;
#pragma unroll
                    for (int h = 0; h < GM; ++h) L = (h == bt * kHB + hh) ? Lp[h] : L;
                    Lb[hh] = L;
                }
#pragma unroll
                for (int i = 0; i < kSL; ++i) {
                    const int j = jr + 4 * (tid + i * kThreads);
                    if (j >= j1) continue;
                    float4 v[kHB];
                    load_slab(stg, chunk, srow, stride, g, bt * kHB, j, j - j0, j1, staged, vec, v);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int p = 4 * i + e;
                        float x[kHB], mr = -INFINITY;
#pragma unroll
                        for (int hh = 0; hh < kHB; ++hh) {
                            x[hh] = bt * kHB + hh < g ? fmaf(comp(v[hh], e), kLog2e, -Lb[hh]) : -INFINITY;
                            mr = fmaxf(mr, x[hh]);
                        }
                        if (mr == -INFINITY) continue;
                        float zr = 0.f;
#pragma unroll
                        for (int hh = 0; hh < kHB; ++hh) zr += fast_exp2(x[hh] - mr);
                        const float M = fmaxf(pm[p], mr);
                        pz[p] = pz[p] * fast_exp2(pm[p] - M) + zr * fast_exp2(mr - M);
                        pm[p] = M;
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < kSL; ++i) {
                const int j = jr + 4 * (tid + i * kThreads);
                if (j >= j1) continue;
                uint32_t k4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int p = 4 * i + e;
                    k4[e] = finish(j + e, pm[p] == -INFINITY ? -INFINITY : pm[p] + fast_log2(pz[p]));
                }
                *reinterpret_cast<uint4*>(keys + (j - j0)) = make_uint4(k4[0], k4[1], k4[2], k4[3]);
            }
        }
    }
    return failed;
}
template <int GM>
__device__ __noinline__ bool group_keys_loads_ool(const SelectAttendArgs& a, int b, int kvh, int j0, int j1, int chunk,
                                                  uint32_t* keys, SmallShared& sh, bool staged, const RadixRange fr,
                                                  bool hist0, uint32_t* whist) {
    return group_keys_loads<GM>(a, b, kvh, j0, j1, chunk, keys, sh, staged, fr, hist0, whist);
}

// The group keys of this CTA's pages [j0, j1) into keys[] (order-preserving uint32 images)
// and, when hist0, the fast first radix pass's histogram of them into sh.hist[0] (zeroed
// by the caller), from sh.Lh. In the log2 domain x_h = s_h log2 e - L_h log2 e <= 0 and
// key = log2(sum_h 2^x_h) ln 2 - ln g; each term is at most 1, so the sum needs no shift
// unless it underflows (every share below 2^-100), when the page is redone with its
// largest term factored out. A NaN score makes its page's key NaN (ranked last).
// Staged scores (see select_pages) are read from shared memory, a batch of four heads at
// a time (groups of more than four heads re-stage the next batch after each); keys[]
// overlays the first staged row, each thread reading a slab's scores before writing its
// keys. Otherwise the scores are read from global memory.
template <int GM>
__device__ void group_keys(const SelectAttendArgs& a, int b, int kvh, int j0, int j1, int chunk, uint32_t* keys,
                           SmallShared& sh, bool staged, const RadixRange& fr, bool hist0, uint32_t* whist,
                           bool& failed) {
    const int tid = threadIdx.x;
    const int g = a.hq / a.hkv;
    const int nloc = j1 - j0;
    const int64_t stride = a.max_pages;
    const float* srow = a.scores + (static_cast<int64_t>(b) * a.hq + kvh * g) * stride;
    const float* stg = reinterpret_cast<const float*>(keys);
    const float log_g = logf(static_cast<float>(g));
    float Lp[GM];
#pragma unroll
    for (int hh = 0; hh < GM; ++hh) Lp[hh] = hh < g ? sh.Lh[hh] * kLog2e : 0.f;
    float* kout = a.sel_keys ? a.sel_keys + (static_cast<int64_t>(b) * a.hkv + kvh) * a.max_pages : nullptr;
    if (GM <= kHB && staged) {
        // staged rows: warp w takes the pages of warp_span, lane l the slabs of 4 pages at
        // 4 l, 4 l + 128, ... of them (so warp w's histogram counts exactly that range);
        // shared memory by window address, the histogram by shared reductions; the rare
        // underflow and the optional key output are handled after the loop
        const uint32_t s_base = smem_u32(stg);
        const uint32_t wh = smem_u32(whist) + static_cast<uint32_t>(threadIdx.x >> 5) * 1024u;
        int w0, w1;
        warp_span(nloc, threadIdx.x >> 5, w0, w1);
        bool uf = false;
#pragma unroll 1
        for (int jj = w0 + 4 * (tid & 31); jj < w1; jj += 128) {
            float4 v[kHB];
#pragma unroll
            for (int hh = 0; hh < kHB; ++hh) {
                // rows past the group are not staged: read (inside the region) and ignored
                v[hh] = lds_f4(s_base + static_cast<uint32_t>(hh * chunk + jj) * 4u);
                if (hh >= g) v[hh] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
            uint32_t k4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float z = 0.f;
#pragma unroll
                for (int hh = 0; hh < kHB; ++hh) z += fast_exp2(fmaf(comp(v[hh], e), kLog2e, -Lp[hh]));
                uf |= !(z >= 7.9e-31f) && z == z;   // every share below 2^-100 (or none): redone below
                const uint32_t u = orderable_key(fast_log2(z) * kLn2 - log_g);
                const uint32_t d = fast_digit(u, fr);
                red_shared_add_if(hist0 && d != 0u && jj + e < w1, wh + d * 4u, 1u);
                k4[e] = u;
            }
            sts_u4(s_base + static_cast<uint32_t>(jj) * 4u, make_uint4(k4[0], k4[1], k4[2], k4[3]));
        }
        if (__syncthreads_or(uf))
            keys_underflow_fixup(srow, stride, g, j0, w0, w1, keys,
                                 make_float4(Lp[0], GM > 1 ? Lp[1 % GM] : 0.f, GM > 2 ? Lp[2 % GM] : 0.f,
                                             GM > 3 ? Lp[3 % GM] : 0.f),
                                 log_g, hist0, fr, whist);
        if (kout) keys_out(kout + j0, keys, nloc);
    } else if constexpr (GM > kHB) {   // the normal path of large groups: inline
        failed |= group_keys_loads<GM>(a, b, kvh, j0, j1, chunk, keys, sh, staged, fr, hist0, whist);
    } else {                           // unstaged rows: rare, out of line
        failed |= group_keys_loads_ool<GM>(a, b, kvh, j0, j1, chunk, keys, sh, staged, fr, hist0, whist);
    }
    __syncthreads();
    if (hist0) {
        // the warps' counts summed per bin; bin 0 (keys below the fast range) by difference
        uint32_t c = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) c += whist[w * 256 + tid];
        sh.hist[0][tid] = c;
        __syncthreads();
        if (tid < 32) {
            uint32_t t = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) t += sh.hist[0][8 * tid + k];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
            if (tid == 0) sh.hist[0][0] = static_cast<uint32_t>(nloc) - t;
        }
    }
}

// Ordered compaction: visits the keys kept by (T, take_eq) -- every key > T and the
// first take_eq keys == T in index order -- and calls emit(i, pos) with each kept
// index and its rank among the kept ones. Each warp walks one contiguous range,
// four groups of 32 keys per step (conflict-free; ranks from ballots).
template <typename F>
__device__ int ordered_keep(const uint32_t* keys, int n, uint32_t T, int take_eq, SmallShared& sh, F emit) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per_w = (((n + kWarps - 1) / kWarps) + 127) & ~127;
    const int w0 = min(n, warp * per_w), w1 = min(n, w0 + per_w);
    const unsigned lt = lanemask_lt();
    int ngt = 0, neq = 0;
    for (int i0 = w0; i0 < w1; i0 += 128) {
        uint32_t key[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + 32 * u + lane;
            key[u] = i < w1 ? keys[i] : 0u;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const bool valid = i0 + 32 * u + lane < w1;
            ngt += __popc(__ballot_sync(0xffffffffu, valid && key[u] > T));
            neq += __popc(__ballot_sync(0xffffffffu, valid && key[u] == T));
        }
    }
    if (lane == 0) {
        sh.wcnt[warp][0] = ngt;
        sh.wcnt[warp][1] = neq;
    }
    __syncthreads();
    int gt_pre = 0, eq_pre = 0, gt_all = 0, eq_all = 0;
    for (int w = 0; w < kWarps; ++w) {
        if (w < warp) {
            gt_pre += sh.wcnt[w][0];
            eq_pre += sh.wcnt[w][1];
        }
        gt_all += sh.wcnt[w][0];
        eq_all += sh.wcnt[w][1];
    }
    int pos = gt_pre + min(eq_pre, take_eq), eq_seen = eq_pre;
    for (int i0 = w0; i0 < w1; i0 += 128) {
        uint32_t key[4];
        unsigned eqb[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + 32 * u + lane;
            key[u] = i < w1 ? keys[i] : 0u;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) eqb[u] = __ballot_sync(0xffffffffu, i0 + 32 * u + lane < w1 && key[u] == T);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + 32 * u + lane;
            const bool eq = (eqb[u] >> lane) & 1u;
            const bool keep = i < w1 && (key[u] > T || (eq && eq_seen + __popc(eqb[u] & lt) < take_eq));
            const unsigned kb = __ballot_sync(0xffffffffu, keep);
            if (keep) emit(i, pos + __popc(kb & lt));
            pos += __popc(kb);
            eq_seen += __popc(eqb[u]);
        }
    }
    return gt_all + min(eq_all, take_eq);
}

// Exclusive ranks, in element order, of the flagged elements among three per thread held
// strided (thread t holds elements t, t + kThreads, t + 2 kThreads). Uses sh.wtot; one
// barrier.
__device__ __forceinline__ void scan_strided(const bool (&f)[3], int (&pos)[3], SmallShared& sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned bal[3];
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        bal[u] = __ballot_sync(0xffffffffu, f[u]);
        if (lane == 0) sh.wtot[u][warp] = __popc(bal[u]);
    }
    __syncthreads();
    const unsigned lt = lanemask_lt();
    int before = 0;
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        int in_u = 0, low = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const int c = sh.wtot[u][w];
            in_u += c;
            low += w < warp ? c : 0;
        }
        pos[u] = before + low + __popc(bal[u] & lt);
        before += in_u;
    }
}

// Candidate lists of the fast selection (after the CTA's keys region in shared memory,
// at the same offsets in every CTA): this CTA's published candidates (key, logical page,
// physical page), and all CTAs' candidates gathered in ascending page order (later the
// kept pages, compacted).
struct CandList {
    uint32_t* key;
    int32_t* logical;
    int32_t* phys;
};
__device__ __forceinline__ CandList cand_list(uint8_t* base) {
    CandList c;
    c.key = reinterpret_cast<uint32_t*>(base);
    c.logical = reinterpret_cast<int32_t*>(base + kCandCap * 4);
    c.phys = reinterpret_cast<int32_t*>(base + kCandCap * 8);
    return c;
}

// The gather when some CTA published more than its fixed share of slots: element e of the
// ascending list comes from the CTA whose offset range holds it (the counts read first),
// written to `to` (this CTA's gathered-list arrays) at index e. Returns the list length.
// Out of line: rare.
template <int CL>
__device__ __noinline__ int gather_by_offsets(const CandList pub, const CandList to, SmallShared& sh) {
    int off[CL + 1];
    off[0] = 0;
#pragma unroll
    for (int r = 0; r < CL; ++r)
        off[r + 1] = off[r] + static_cast<int>(ld_dsmem_u32(dsmem_addr(&sh.pub_n, static_cast<uint32_t>(r))));
    const int N = min(off[CL], kCandCap);
#pragma unroll 1
    for (int e = threadIdx.x; e < N; e += kThreads) {
        int r = 0, first = 0;
#pragma unroll
        for (int q = 1; q < CL; ++q) {
            r = e >= off[q] ? q : r;
            first = e >= off[q] ? off[q] : first;
        }
        const int k = e - first;
        to.key[e] = ld_dsmem_u32(dsmem_addr(&pub.key[k], static_cast<uint32_t>(r)));
        to.logical[e] = static_cast<int>(ld_dsmem_u32(dsmem_addr(&pub.logical[k], static_cast<uint32_t>(r))));
        to.phys[e] = static_cast<int>(ld_dsmem_u32(dsmem_addr(&pub.phys[k], static_cast<uint32_t>(r))));
    }
    return N;
}

// The candidates' publication when the keys were not computed by warp ranges (scores read
// with loads, or groups of more than four heads): an ordered compaction of the keys >= lo_u,
// then each candidate's physical page (the staged page-table entry, or global memory) and an
// L2 prefetch of its K/V when it is kept for sure (key >= hi_u). Returns the count. Inline
// for large groups (their normal path), out of line otherwise.
__device__ __forceinline__ int publish_ordered(const SelectAttendArgs& a, int b, int kvh, int j0, int nloc,
                                            const uint32_t* keys, uint32_t lo_u, uint64_t hi_u, const int32_t* ptab,
                                            bool ptab_staged, bool paged, const CandList pub, SmallShared& sh) {
    const int npub = ordered_keep(keys, nloc, lo_u - 1u, 0, sh, [&](int i, int pos) {
        if (pos < kCandCap) {   // always: the count was checked; the guard bounds a logic error
            pub.key[pos] = keys[i];
            pub.logical[pos] = j0 + i;
        }
    });
    __syncthreads();
    const int64_t kv_row = static_cast<int64_t>(kPage) * kD * 2;   // bytes per (page, kv head)
#pragma unroll 1
    for (int t = threadIdx.x; t < min(npub, kCandCap); t += kThreads) {
        int phys = 0;
        if (paged) {
            const int i = pub.logical[t] - j0;
            phys = ptab_staged ? ptab[i] : a.page_table[static_cast<int64_t>(b) * a.max_pages + j0 + i];
            if (phys < 0 || phys >= a.num_phys) {
                report_error(a.st, LOCKS_ERR_BAD_INDEX);
                phys = 0;
            }
            if (static_cast<uint64_t>(pub.key[t]) >= hi_u) {
                const int64_t unit = static_cast<int64_t>(phys) * a.hkv + kvh;
                prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(a.k_cache) + unit * kv_row, kv_row);
                prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(a.v_cache) + unit * kv_row, kv_row);
            }
        }
        pub.phys[t] = phys;
    }
    return npub;
}
__device__ __noinline__ int publish_ordered_ool(const SelectAttendArgs& a, int b, int kvh, int j0, int nloc,
                                                const uint32_t* keys, uint32_t lo_u, uint64_t hi_u, const int32_t* ptab,
                                                bool ptab_staged, bool paged, const CandList pub, SmallShared& sh) {
    return publish_ordered(a, b, kvh, j0, nloc, keys, lo_u, hi_u, ptab, ptab_staged, paged, pub, sh);
}

// One radix pass's cluster step: sums the CTAs' histograms `hist` (256 bins) through
// DSMEM (hv[r] = CTA r's count of this thread's bin) and finds the bin where the count of
// keys at or above it first reaches `remaining`, scanning from the top bin down. Leaves in
// sh: digit, above / above_low / above_own (keys in higher bins: all CTAs, lower-ranked
// CTAs, this CTA), eq_low / eq_own / inbin (keys in the bin: lower-ranked, own, all).
template <int CL>
__device__ __forceinline__ void pick_digit(const uint32_t* hist, int remaining, uint32_t rank, SmallShared& sh,
                                           uint32_t (&hv)[CL], const uint32_t* pushed = nullptr) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (pushed) {   // every CTA's histogram already pushed here: [rank][bin]
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) hv[r] = pushed[r * 256 + tid];
    } else {
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) hv[r] = ld_dsmem_u32(dsmem_addr(&hist[tid], r));   // all in flight
    }
    uint32_t all = 0u, low = 0u;
#pragma unroll
    for (uint32_t r = 0; r < CL; ++r) {
        all += hv[r];
        low += r < rank ? hv[r] : 0u;
    }
    sh.tot[0][tid] = all;
    sh.tot[1][tid] = low;
    sh.tot[2][tid] = hist[tid];
    __syncthreads();
    if (warp == 0) {
        // lane l holds bins 8l .. 8l + 7 of (all CTAs, lower-ranked CTAs, this CTA)
        int c[3][8], t[3], suf[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const uint4 h0 = *reinterpret_cast<const uint4*>(&sh.tot[k][8 * lane]);
            const uint4 h1 = *reinterpret_cast<const uint4*>(&sh.tot[k][8 * lane + 4]);
            c[k][0] = h0.x; c[k][1] = h0.y; c[k][2] = h0.z; c[k][3] = h0.w;
            c[k][4] = h1.x; c[k][5] = h1.y; c[k][6] = h1.z; c[k][7] = h1.w;
            t[k] = ((c[k][0] + c[k][1]) + (c[k][2] + c[k][3])) + ((c[k][4] + c[k][5]) + (c[k][6] + c[k][7]));
            suf[k] = t[k];
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const int y = __shfl_down_sync(0xffffffffu, suf[k], o);
                if (lane + o < 32) suf[k] += y;
            }
        }
        int ab[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) ab[k] = suf[k] - t[k];   // keys in the bins of higher lanes
#pragma unroll
        for (int i = 7; i >= 0; --i) {
            if (ab[0] < remaining && ab[0] + c[0][i] >= remaining) {
                sh.digit = 8 * lane + i;
                sh.above = ab[0];
                sh.above_low = ab[1];
                sh.above_own = ab[2];
                sh.eq_low = c[1][i];
                sh.eq_own = c[2][i];
                sh.inbin = c[0][i];
            }
#pragma unroll
            for (int k = 0; k < 3; ++k) ab[k] += c[k][i];
        }
    }
    __syncthreads();
}

// The general radix select (kept out of line: the fast candidate path runs otherwise),
// entered after the first pass over the fast range (its result in sh and sh.bin_cnt).
// restart: the K-th key lay outside the fast range, so the select starts over as an
// MSB-first radix over the whole key. Each later pass histograms the next 8 bits of the
// key's offset from the range's base among the keys matching the digits so far; once the
// chosen bin holds at most kRankCap keys across the cluster, every CTA publishes its keys
// of that bin, gathers all of them through DSMEM and ranks them directly. The kept keys
// are then written by an ordered compaction: the pass counts place each CTA's kept keys
// in the ascending output without a further exchange.
template <int CL>
__device__ __noinline__ int select_general(const SelectAttendArgs& a, int b, int kvh, uint32_t rank, int j0, int nloc,
                                           int K, const uint32_t* keys, SmallShared& sh, RadixRange fr,
                                           bool restart) {
    const int tid = threadIdx.x, lane = tid & 31;
    int32_t* out = a.selected + (static_cast<int64_t>(b) * a.hkv + kvh) * a.k_cap;
    uint32_t base = restart ? 0u : fr.base, pv = 0u;
    int shift = restart ? 24 : fr.s, prev = 32;
    int remaining = K;
    int gt_low = 0, gt_own = 0, eq_low = 0, eq_own = 0;
    uint32_t T = 0u;
    bool have = !restart;   // sh holds the result of the pass over (base, shift, prev)
#pragma unroll 1
    for (int pass = 1;; ++pass) {
        uint32_t hv[CL];
        if (!have) {
            uint32_t* hist = sh.hist[pass & 1];   // alternating: other CTAs read the previous one
            hist[tid] = 0u;
            __syncthreads();
            if (prev >= 32) {
                // whole-key first digit (the top byte takes few values): one shared atomic per
                // distinct bin per warp step
#pragma unroll 1
                for (int i0 = 0; i0 < nloc; i0 += kThreads) {
                    const int i = i0 + tid;
                    const uint32_t bin = i < nloc ? (keys[i] - base) >> shift : 0xffffffffu;
                    const unsigned peers = __match_any_sync(0xffffffffu, bin);
                    if (i < nloc && lane == __ffs(peers) - 1)
                        atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
                }
            } else {
                const uint32_t hp = pv >> prev, mask = (1u << (prev - shift)) - 1u;
#pragma unroll 1
                for (int i = tid; i < nloc; i += kThreads) {
                    const uint32_t v = keys[i] - base;
                    if ((v >> prev) == hp) atomicAdd(&hist[(v >> shift) & mask], 1u);
                }
            }
            __syncthreads();
            cluster_sync_all();
            pick_digit<CL>(hist, remaining, rank, sh, hv);
            if (tid == sh.digit) {
#pragma unroll
                for (uint32_t r = 0; r < CL; ++r) sh.bin_cnt[r] = static_cast<int>(hv[r]);
            }
        }
        have = false;
        const uint32_t digit = static_cast<uint32_t>(sh.digit);
        pv |= digit << shift;
        remaining -= sh.above;
        gt_low += sh.above_low;
        gt_own += sh.above_own;
        eq_low = sh.eq_low;
        eq_own = sh.eq_own;
        const int inbin = sh.inbin;
        if (shift > 0 && inbin <= kRankCap) {
            // The K-th largest key is one of the inbin keys of the chosen bin: every CTA
            // publishes its keys of that bin, every CTA gathers all of them through DSMEM and
            // ranks them directly instead of running the remaining passes.
            if (tid == 0) sh.nbin = 0;
            __syncthreads();
            const uint32_t want = pv >> shift;   // every bit of v at or above this pass's digit
#pragma unroll 1
            for (int i0 = 0; i0 < nloc; i0 += kThreads) {
                const int i = i0 + tid;
                const uint32_t key = i < nloc ? keys[i] : 0u;
                const bool m = i < nloc && ((key - base) >> shift) == want;
                const unsigned bal = __ballot_sync(0xffffffffu, m);
                int bpos = 0;
                if (lane == 0 && bal) bpos = atomicAdd(&sh.nbin, __popc(bal));
                bpos = __shfl_sync(0xffffffffu, bpos, 0);
                if (m) sh.bin_keys[bpos + __popc(bal & lanemask_lt())] = key;
            }
            cluster_sync_all();   // every CTA's bin keys are complete and visible
            if (tid < inbin) {
                int r = 0, first = 0;
#pragma unroll
                for (int q = 0; q < CL - 1; ++q) {
                    if (r == q && tid >= first + sh.bin_cnt[q]) {   // past rank q's keys: move on
                        first += sh.bin_cnt[q];
                        r = q + 1;
                    }
                }
                sh.rank_keys[tid] = ld_dsmem_u32(dsmem_addr(&sh.bin_keys[tid - first], static_cast<uint32_t>(r)));
                sh.rank_src[tid] = static_cast<uint8_t>(r);
            }
            if (tid < 4) sh.cnt4[tid] = 0;
            __syncthreads();
            if (tid < inbin) {
                const uint32_t key = sh.rank_keys[tid];
                int gt = 0, ge = 0;
#pragma unroll 1
                for (int q = 0; q < inbin; ++q) {
                    const uint32_t v = sh.rank_keys[q];
                    gt += v > key;
                    ge += v >= key;
                }
                if (gt < remaining && ge >= remaining) {   // key is the remaining-th largest of the bin
                    sh.rank_T = key;
                    sh.rank_take = remaining - gt;
                }
            }
            __syncthreads();
            T = sh.rank_T;
            if (tid < inbin) {
                const uint32_t key = sh.rank_keys[tid];
                const int r = sh.rank_src[tid];
                if ((key >= T) && r <= static_cast<int>(rank))
                    atomicAdd(&sh.cnt4[(key > T ? 0 : 2) + (r == static_cast<int>(rank) ? 1 : 0)], 1);
            }
            __syncthreads();
            gt_low += sh.cnt4[0];
            gt_own += sh.cnt4[1];
            eq_low = sh.cnt4[2];
            eq_own = sh.cnt4[3];
            remaining = sh.rank_take;
            break;
        }
        if (shift == 0) {   // every bit fixed: T is the K-th largest key (ties by page id)
            T = base + pv;
            break;
        }
        prev = shift;
        shift = max(0, shift - 8);
    }
    // T is the K-th largest key; the first `remaining` keys equal to it are kept. This CTA
    // keeps its keys > T and its first take_cta keys == T, written from position pos0 on
    // (the kept keys of lower-ranked CTAs come first).
    const int take_cta = max(0, min(remaining - eq_low, eq_own));
    const int pos0 = gt_low + min(eq_low, remaining);
    ordered_keep(keys, nloc, T, take_cta, sh, [&](int i, int pos) {
        if (pos0 + pos < K) out[pos0 + pos] = j0 + i;   // always < K; the guard only bounds a logic error
    });
    return K;
}

// Writes selected[b][kvh][0..K) and n_selected[b][kvh]; returns K. When the fast
// candidate path ran, *listed is set and the kept pages (logical, physical) are in the
// gathered candidate list, ascending, so the attention needs no further exchange.
// Cluster-wide radix select: each CTA histograms its own keys and every CTA sums the
// CTAs' histograms through DSMEM and picks the digit. The first pass takes the fast
// range (its histogram is built with the keys). If the chosen bin is inside that range
// and the keys in it and above it are few (<= kCandCap, the bin's <= kRankCap), every
// CTA publishes those candidate keys (in page order, with their physical pages; the sure
// ones above the bin also get an L2 prefetch of their K/V), gathers all CTAs' lists
// through DSMEM after one cluster barrier, ranks the bin's keys directly and keeps the
// K largest (equal keys by lower page id). Otherwise later passes take the next 8 bits of
// the key's offset from the range's base, ending, when the chosen bin holds at most
// kRankCap keys, in a direct ranking of that bin, and the kept keys are written by an
// ordered compaction (the pass counts place each CTA's kept keys in the output).
template <int CL, int GM>
__device__ int select_pages(const SelectAttendArgs& a, int b, int kvh, uint32_t rank, int chunk, uint8_t* big,
                            SmallShared& sh, bool stage_q, bool* listed, bool* preissued) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t* keys = reinterpret_cast<uint32_t*>(big);
    const CandList pub = cand_list(big + region_a_bytes(chunk, CL));
    const CandList cand = cand_list(big + region_a_bytes(chunk, CL) + kCandListBytes);
    *listed = false;
    *preissued = false;
    const int g = a.hq / a.hkv;
    // This CTA's nominal page range [jn0, jn0 + nn). Inputs go out before the wait for the
    // scorer (an L2 prefetch of the range's page-table entries, the query rows, the
    // sequence length), the range's score rows (bulk copies into the staging buffer)
    // right after it.
    const int jn0 = min(a.max_pages, static_cast<int>(rank) * chunk);
    const int nn = min(chunk, a.max_pages - jn0);
    const int64_t stride = a.max_pages;
    const float* srow = a.scores + (static_cast<int64_t>(b) * a.hq + kvh * g) * stride;
    const bool vec = (a.max_pages & 3) == 0 && (reinterpret_cast<uintptr_t>(a.scores) & 15) == 0;
    // groups of more than four heads read their scores with loads (staging them four rows at
    // a time would serialise the copies)
    const bool staged = GM <= kHB && vec && nn > 0 && kHB * chunk * 4 <= stage_cap(CL);
    if (tid == 32 && nn > 0 && a.page_table && vec && (reinterpret_cast<uintptr_t>(a.page_table) & 15) == 0)
        prefetch_l2_bulk(a.page_table + static_cast<int64_t>(b) * a.max_pages + jn0,
                         static_cast<uint32_t>((nn + 3) & ~3) * 4u);
    float qv[16 * kD / kThreads];
    if (stage_q) load_query(a, b, kvh, g, qv);
    const int seq_len = a.seq_pages[b];
    // the scores and partials come from the previous kernel (the scorer)
    grid_dependency_wait();
    allow_dependent_launch();   // the next kernel waits for this grid's completion itself
    if (tid == 0 && staged) stage_rows(srow, stride, 0, min(g, kHB), jn0, nn, chunk, reinterpret_cast<float*>(keys), sh);
    bool failed = false;
    if (staged && !a.lse_partials && !mbar_wait_bounded(&sh.sbar, 0, a.st.wait_limit_ns)) failed = true;

    const int P = max(0, min(seq_len, a.max_pages));
    const int j0 = min(P, jn0);
    const int j1 = min(P, j0 + chunk);
    const int nloc = j1 - j0;
    normaliser<CL, GM>(a, b, kvh, g, j0, j1, staged, reinterpret_cast<float*>(keys), chunk, sh);
    if (stage_q) store_query(qv, g, sh);   // read after the barriers below
    int K = min(a.budget_pages, min(P, a.k_cap));
    K = max(K, 0);
    const bool select = K > 0 && K < P;
    const RadixRange fr = fast_range(select ? K : 1, select ? P : 2);
    if (staged && a.lse_partials && !mbar_wait_bounded(&sh.sbar, 0, a.st.wait_limit_ns)) failed = true;
    // per-warp histograms of the keys in the (still unused) candidate-list space, zeroed by
    // the kernel's prologue
    uint32_t* whist = reinterpret_cast<uint32_t*>(pub.key);
    group_keys<GM>(a, b, kvh, j0, j1, chunk, keys, sh, staged, fr, select, whist, failed);
    // the page-table entries of this CTA's pages into the staged score rows that are free now
    // (rows 1..3; row 0 holds the keys), for the candidates' physical pages
    int32_t* ptab = reinterpret_cast<int32_t*>(keys) + chunk;
    const bool paged = a.page_table && a.k_cache && a.v_cache;
    const bool ptab_staged = vec && paged && nloc > 0 && select && 2 * chunk * 4 <= region_a_bytes(chunk, CL) &&
                             (reinterpret_cast<uintptr_t>(a.page_table) & 15) == 0;
    const uint32_t ptab_phase = staged ? 1u : 0u;   // the staging barrier's phases: scores, then this
    if (ptab_staged && tid == 0) {
        fence_proxy_async_smem();   // the rows' generic reads (the keys pass) before the async refill
        const uint32_t bytes = static_cast<uint32_t>((nloc + 3) & ~3) * 4u;
        mbar_arrive_expect_tx(&sh.sbar, bytes);
        bulk_g2s(ptab, a.page_table + static_cast<int64_t>(b) * a.max_pages + j0, bytes, &sh.sbar);
    }
    if (failed) report_error(a.st, LOCKS_ERR_TIMEOUT);

    int32_t* out = a.selected + (static_cast<int64_t>(b) * a.hkv + kvh) * a.k_cap;
    if (rank == 0 && tid == 0) a.n_selected[b * a.hkv + kvh] = K;
    if (K == 0) return 0;
    if (K == P) {
        for (int j = j0 + tid; j < j1; j += kThreads) out[j] = j;
        return K;
    }

    // pass 0 over the fast range (its histogram was built with the keys). 12-CTA clusters
    // push each bin to every CTA before the barrier (a table in the merge inbox, which is
    // unused until the attention), so the digit is picked from local memory.
    uint32_t* pushed = nullptr;
    if constexpr (CL == kSpreadCluster) {
        pushed = reinterpret_cast<uint32_t*>(big + inbox_offset(chunk, CL, false));
        static_assert(CL * 256 * 4 <= kInboxBytes, "the histogram table fits the inbox");
        const uint32_t mine = sh.hist[0][tid];   // written by this thread (bin 0: thread 0)
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) st_dsmem_u32(dsmem_addr(&pushed[rank * 256 + tid], r), mine);
    }
    cluster_sync_all();
    uint32_t hv[CL];
    pick_digit<CL>(sh.hist[0], K, rank, sh, hv, pushed);
    const uint32_t digit = static_cast<uint32_t>(sh.digit);
    if (tid == static_cast<int>(digit)) {
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) sh.bin_cnt[r] = static_cast<int>(hv[r]);
    }
    const int remaining = K - sh.above, inbin = sh.inbin;
    if (digit == 0u || digit == 255u || inbin > kRankCap || K - remaining + inbin > kCandCap) {
        // the staged page-table copy lands before that space is reused
        if (ptab_staged && !mbar_wait_bounded(&sh.sbar, ptab_phase & 1u, a.st.wait_limit_ns))
            report_error(a.st, LOCKS_ERR_TIMEOUT);
        __syncthreads();
        return select_general<CL>(a, b, kvh, rank, j0, nloc, K, keys, sh, fr, digit == 0u || digit == 255u);
    }

    // ---- fast candidate path
    const uint32_t lo_u = fr.base + (digit << fr.s);   // first key image of the chosen bin
    const uint64_t hi_u = static_cast<uint64_t>(fr.base) + (static_cast<uint64_t>(digit + 1) << fr.s);
    const int64_t kv_row = static_cast<int64_t>(kPage) * kD * 2;   // bytes per (page, kv head)
    // publish this CTA's candidates (keys >= lo_u) in page order by an ordered compaction,
    // then their physical pages (from the staged page-table entries) and an L2 prefetch of
    // the K/V of those above the bin, which are kept for sure (selection-only launches carry
    // no table or caches)
    bool pt_failed = ptab_staged && !mbar_wait_bounded(&sh.sbar, ptab_phase & 1u, a.st.wait_limit_ns);
    if (pt_failed) report_error(a.st, LOCKS_ERR_TIMEOUT);
    int npub = 0;
    if (GM <= kHB && staged) {
        // warp w computed the keys of warp_span w, so its candidates are counted by its
        // histogram's bins >= digit; the counts place every warp's candidates, which one
        // ordered pass over its keys then writes
        int cnt = 0;
        for (int d = static_cast<int>(digit) + lane; d < 256; d += 32) cnt += static_cast<int>(whist[warp * 256 + d]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        if (lane == 0) sh.wcnt[warp][0] = cnt;
        __syncthreads();   // counts visible, and the histograms (under the list) read by every warp
        int pos = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            pos += w < warp ? sh.wcnt[w][0] : 0;
            npub += sh.wcnt[w][0];
        }
        int w0, w1;
        warp_span(nloc, warp, w0, w1);
        const bool pt_direct = paged && ptab_staged;
        const uint32_t kaddr = smem_u32(keys), paddr = pt_direct ? smem_u32(ptab) : kaddr;
        const uint32_t pkey = smem_u32(pub.key), plog = smem_u32(pub.logical), pphys = smem_u32(pub.phys);
        const int32_t* grow = a.page_table ? a.page_table + static_cast<int64_t>(b) * a.max_pages + j0 : nullptr;
        const unsigned lt = lanemask_lt();
        const int first = pos;
        bool bad = false;
        // straight-line code (predicated loads and stores): a branch into code not yet
        // fetched would wait on instruction memory
#pragma unroll 1
        for (int i0 = w0; i0 < w1; i0 += 128) {
            uint32_t key[4], pt[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = min(i0 + 32 * u + lane, w1 - 1);
                key[u] = lds_u32(kaddr + static_cast<uint32_t>(i) * 4u);
                pt[u] = lds_u32(paddr + static_cast<uint32_t>(i) * 4u);   // used when staged
                key[u] = i0 + 32 * u + lane < w1 ? key[u] : 0u;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + 32 * u + lane;
                const unsigned bal = __ballot_sync(0xffffffffu, key[u] >= lo_u);   // lo_u > 0: never past w1
                const int at = pos + __popc(bal & lt);
                // always below kCandCap (the count was checked); the test bounds a logic error
                const bool c = key[u] >= lo_u && at < kCandCap;
                // the physical page from the staged table (from global memory after the loop
                // otherwise: a conditional global load here slows the whole loop)
                int phys = pt_direct ? static_cast<int>(pt[u]) : 0;
                const bool out_of_range = phys < 0 || phys >= a.num_phys;
                bad |= c && out_of_range;
                phys = out_of_range ? 0 : phys;
                const uint32_t slot = static_cast<uint32_t>(min(at, kCandCap - 1)) * 4u;
                sts_u32_if(c, pkey + slot, key[u]);
                sts_u32_if(c, plog + slot, static_cast<uint32_t>(j0 + i));
                sts_u32_if(c, pphys + slot, static_cast<uint32_t>(phys));
                pos += __popc(bal);
            }
        }
        __syncwarp();
        if (paged && !ptab_staged) {
#pragma unroll 1
            for (int t = first + lane; t < min(pos, kCandCap); t += 32) {
                int phys = __ldg(grow + (pub.logical[t] - j0));
                const bool out_of_range = phys < 0 || phys >= a.num_phys;
                bad |= out_of_range;
                pub.phys[t] = out_of_range ? 0 : phys;
            }
            __syncwarp();
        }
        if (bad) report_error(a.st, LOCKS_ERR_BAD_INDEX);
        // an L2 prefetch of the K/V of this warp's candidates above the bin (kept for sure),
        // issued by one lane (a bulk prefetch takes one address per instruction)
        if (paged && lane == 0) {
#pragma unroll 1
            for (int t = first; t < min(pos, kCandCap); ++t) {
                if (static_cast<uint64_t>(pub.key[t]) < hi_u) continue;
                const int64_t unit = static_cast<int64_t>(pub.phys[t]) * a.hkv + kvh;
                prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(a.k_cache) + unit * kv_row, kv_row);
                prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(a.v_cache) + unit * kv_row, kv_row);
            }
        }
    } else {
        if constexpr (GM > kHB)   // the normal path of large groups: inline
            npub = publish_ordered(a, b, kvh, j0, nloc, keys, lo_u, hi_u, ptab, ptab_staged, paged, pub, sh);
        else
            npub = publish_ordered_ool(a, b, kvh, j0, nloc, keys, lo_u, hi_u, ptab, ptab_staged, paged, pub, sh);
    }
    if (tid == 0) {
        sh.pub_n = npub;
        sh.nbin = 0;
    }
    cluster_sync_all();   // every CTA's list is complete and visible
    // gather, one round of remote loads: element e = r kSlot + k is CTA r's k-th candidate,
    // read with CTA r's count, so ascending e is ascending page order; thread t holds
    // e = t, t + kThreads, t + 2 kThreads. A CTA with more than kSlot candidates (rare)
    // makes every CTA gather again by offsets.
    constexpr int kSlot = kCandCap / CL;
    static_assert(kSlot * CL == 3 * kThreads, "three gathered elements per thread");
    uint32_t ck[3];
    int cl[3], cp[3];
    bool cv[3], over = false;
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        const int e = tid + u * kThreads, r = e / kSlot, k = e - r * kSlot;
        const int cnt = static_cast<int>(ld_dsmem_u32(dsmem_addr(&sh.pub_n, static_cast<uint32_t>(r))));
        ck[u] = ld_dsmem_u32(dsmem_addr(&pub.key[k], static_cast<uint32_t>(r)));
        cl[u] = static_cast<int>(ld_dsmem_u32(dsmem_addr(&pub.logical[k], static_cast<uint32_t>(r))));
        cp[u] = static_cast<int>(ld_dsmem_u32(dsmem_addr(&pub.phys[k], static_cast<uint32_t>(r))));
        cv[u] = k < cnt;
        over |= k == 0 && cnt > kSlot;
    }
    // the bin's keys, unordered, for the ranking
    auto bin_keys = [&]() {
        // one shared atomic per warp for its three rounds
        bool m[3];
        unsigned bal[3];
#pragma unroll
        for (int u = 0; u < 3; ++u) {
            m[u] = cv[u] && static_cast<uint64_t>(ck[u]) < hi_u;
            bal[u] = __ballot_sync(0xffffffffu, m[u]);
        }
        const int n0 = __popc(bal[0]), n1 = __popc(bal[1]), n2 = __popc(bal[2]);
        int base = 0;
        if (lane == 0 && n0 + n1 + n2 > 0) base = atomicAdd(&sh.nbin, n0 + n1 + n2);
        base = __shfl_sync(0xffffffffu, base, 0);
        const unsigned lt = lanemask_lt();
#pragma unroll
        for (int u = 0; u < 3; ++u) {
            const int at = base + (u > 0 ? n0 : 0) + (u > 1 ? n1 : 0) + __popc(bal[u] & lt);
            if (m[u] && at < kRankCap) sh.rank_keys[at] = ck[u];   // always: the bin count was checked
        }
    };
    bin_keys();
    if (__syncthreads_or(over)) {
        const int N = gather_by_offsets<CL>(pub, cand, sh);
        __syncthreads();
#pragma unroll
        for (int u = 0; u < 3; ++u) {
            const int e = tid + u * kThreads;
            cv[u] = e < N;
            ck[u] = cv[u] ? cand.key[e] : 0u;
            cl[u] = cv[u] ? cand.logical[e] : 0;
            cp[u] = cv[u] ? cand.phys[e] : 0;
        }
        if (tid == 0) sh.nbin = 0;
        __syncthreads();
        bin_keys();
        __syncthreads();
    }
    // rank every bin key against all of them: G threads per key (consecutive lanes), each
    // over a strided share, as many as the block holds (G a power of two <= 8)
    const int nb = min(sh.nbin, kRankCap);
    const int G = nb <= kThreads / 8 ? 8 : (nb <= kThreads / 4 ? 4 : (nb <= kThreads / 2 ? 2 : 1));
    {
        const int kidx = tid / G, part = tid % G;
        const uint32_t key = kidx < nb ? sh.rank_keys[kidx] : 0u;
        int gt = 0, ge = 0;
        if (kidx < nb) {
#pragma unroll 4
            for (int q = part; q < nb; q += G) {
                const uint32_t v = sh.rank_keys[q];
                gt += v > key;
                ge += v >= key;
            }
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {   // sum over the key's G lanes (aligned groups)
            const int gt2 = __shfl_xor_sync(0xffffffffu, gt, o), ge2 = __shfl_xor_sync(0xffffffffu, ge, o);
            if (o < G) {
                gt += gt2;
                ge += ge2;
            }
        }
        if (kidx < nb && part == 0 && gt < remaining && ge >= remaining) {   // the remaining-th largest
            sh.rank_T = key;
            sh.rank_take = remaining - gt;
            sh.rank_eq = ge - gt;
        }
    }
    __syncthreads();
    const uint32_t T = sh.rank_T;
    const int take = sh.rank_take;
    // kept: every key > T, and the first `take` keys == T in page order (all of them when
    // T is not tied beyond `take`)
    bool kp[3];
    int pos[3];
    if (take == sh.rank_eq) {
#pragma unroll
        for (int u = 0; u < 3; ++u) kp[u] = cv[u] && ck[u] >= T;
    } else {
        bool eqf[3];
#pragma unroll
        for (int u = 0; u < 3; ++u) eqf[u] = cv[u] && ck[u] == T;
        scan_strided(eqf, pos, sh);
        __syncthreads();   // the scan's totals read by every thread
#pragma unroll
        for (int u = 0; u < 3; ++u) kp[u] = cv[u] && (ck[u] > T || (eqf[u] && pos[u] < take));
    }
    scan_strided(kp, pos, sh);
    // the kept list (ascending) into the gathered-list arrays; this CTA writes its share of
    // selected[]
    const int share = (K + CL - 1) / CL;
    const int s0 = static_cast<int>(rank) * share, s1 = min(K, s0 + share);
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        if (kp[u] && pos[u] < kCandCap) {
            cand.logical[pos[u]] = cl[u];
            cand.phys[pos[u]] = cp[u];
            if (pos[u] >= s0 && pos[u] < s1) out[pos[u]] = cl[u];
        }
    }
    // the first pages of every warp's attention share go out now: their K/V tiles into the
    // ring (free: the keys and page-table rows it overlays are no longer read; the cluster
    // barrier ordered every thread's reads before this fence), so the attention starts on
    // tiles in flight. Launches with tail pages divide the attention differently: not those.
    if (stage_q && paged && !a.tail_tokens) {
        constexpr int kSlots = slots_per_warp(CL);
        fence_proxy_async_smem();
#pragma unroll
        for (int u = 0; u < 3; ++u) {
            const int q = pos[u] - s0;
            if (kp[u] && pos[u] >= s0 && pos[u] < s1 && q < kSlots * kWarps) {
                const int sl = q / kWarps * kWarps + q % kWarps;   // slot k = q / kWarps of warp q % kWarps
                uint8_t* slot = big + sl * kPageSlotBytes;
                uint64_t* bar = &sh.bar[sl];
                const int y = static_cast<int>((static_cast<int64_t>(cp[u]) * a.hkv + kvh) * kPage);
                mbar_arrive_expect_tx(bar, kPageSlotBytes);
                tma_load_2d(slot, &a.tm_k, 0, y, bar);
                tma_load_2d(slot + kBoxBytes, &a.tm_k, 64, y, bar);
                tma_load_2d(slot + 2 * kBoxBytes, &a.tm_v, 0, y, bar);
                tma_load_2d(slot + 3 * kBoxBytes, &a.tm_v, 64, y, bar);
            }
        }
        *preissued = true;
    }
    *listed = true;
    __syncthreads();
    return K;
}
// ------------------------------------------------------------- attention
// Pages come from `sel` (global, logical ids, looked up through the page table), or, when
// list_log is given, from lists in shared memory of (logical, physical) pages.
template <int CL, int GM, bool SPLIT>
__device__ void attend_pages(const SelectAttendArgs& a, int b, int kvh, uint32_t rank, int n_sel,
                             const int32_t* sel, bool sel_coherent, bool q_staged, uint8_t* ring, SmallShared& sh,
                             float* inbox, const int32_t* list_log = nullptr, const int32_t* list_phys = nullptr,
                             bool preissued = false) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gid = lane >> 2, t = lane & 3;
    const int g = a.hq / a.hkv;
    bool failed = false, bad = false;
    // the sequence's tokens without a summary yet (fused mode): `tail` tokens on logical
    // pages tail_page, tail_page + 1, ... after the selected ones, attended whole
    int tail = 0, tail_page = 0;
    if (a.tail_tokens) {
        tail = a.tail_tokens[b];
        tail_page = a.seq_pages[b];
        const int npg = (tail + kPage - 1) / kPage;
        if (tail < 0 || tail > kPage * LOCKS_MAX_TAIL_PAGES ||
            (tail > 0 && (tail_page < 0 || tail_page + npg > a.max_pages))) {
            bad = true;
            tail = 0;
        }
    }
    const int n_all = n_sel + (tail + kPage - 1) / kPage;
    // split attention (attention-only launches): cluster z of S takes a contiguous
    // share of the pages, then each CTA a share of that
    const int S = static_cast<int>(gridDim.z), z = static_cast<int>(blockIdx.z);
    const int zper = (n_all + S - 1) / S;
    const int z0 = min(n_all, z * zper), z1 = min(n_all, z0 + zper);
    const int per = (z1 - z0 + CL - 1) / CL;
    const int p0 = min(z1, z0 + static_cast<int>(rank) * per);
    const int p1 = min(z1, p0 + per);

    if (!q_staged) {
        float qv[16 * kD / kThreads];
        load_query(a, b, kvh, g, qv);
        store_query(qv, g, sh);
        __syncthreads();
    }
    const int qrow = (lane & 7) + ((lane >> 3) & 1) * 8, qcol = (lane >> 4) * 8;
    float o[16][4];
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;   // rows gid, gid + 8

    // warp w attends pages p0 + w, p0 + w + kWarps, ...; page k of the warp goes to slot
    // k mod kSlots, refilled with page k + kSlots once page k is attended
    constexpr int kSlots = slots_per_warp(CL);
    auto issue = [&](int p, int sl) {
        int logical, phys;
        if (list_log && p < n_sel) {   // the fused launch's kept list (shared memory)
            logical = list_log[p];
            phys = list_phys[p];
        } else {
            logical = p < n_sel ? (sel_coherent ? __ldcg(sel + p) : sel[p]) : tail_page + (p - n_sel);
            if (logical < 0 || logical >= a.max_pages) {
                bad = true;
                logical = 0;
            }
            phys = a.page_table[static_cast<int64_t>(b) * a.max_pages + logical];
        }
        if (phys < 0 || phys >= a.num_phys) {
            bad = true;
            phys = 0;
        }
        const int y = static_cast<int>((static_cast<int64_t>(phys) * a.hkv + kvh) * kPage);   // the tile's first row
        uint8_t* slot = ring + (sl * kWarps + warp) * kPageSlotBytes;
        uint64_t* bar = &sh.bar[sl * kWarps + warp];
        fence_proxy_async_smem();   // earlier generic reads of the slot before the async refill
        __syncwarp();
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, kPageSlotBytes);
            tma_load_2d(slot, &a.tm_k, 0, y, bar);
            tma_load_2d(slot + kBoxBytes, &a.tm_k, 64, y, bar);
            tma_load_2d(slot + 2 * kBoxBytes, &a.tm_v, 0, y, bar);
            tma_load_2d(slot + 3 * kBoxBytes, &a.tm_v, 64, y, bar);
        }
    };
    if (!preissued) {   // (the fused launch's selection issues a warp's first pages itself)
#pragma unroll
        for (int k = 0; k < kSlots; ++k)
            if (p0 + warp + k * kWarps < p1) issue(p0 + warp + k * kWarps, k);
    }
    uint32_t phases = 0u;   // bit sl: the parity slot sl waits for next
    int sl = 0;
    for (int p = p0 + warp; p < p1; p += kWarps) {
        // tokens of the page that are attended
        const int valid = p < n_sel ? kPage : min(kPage, tail - (p - n_sel) * kPage);
        const uint8_t* slot = ring + (sl * kWarps + warp) * kPageSlotBytes;
        if (!mbar_wait_bounded(&sh.bar[sl * kWarps + warp], (phases >> sl) & 1u, a.st.wait_limit_ns)) failed = true;
        phases ^= 1u << sl;
        const uint8_t* kslot = slot;
        const uint8_t* vslot = slot + 2 * kBoxBytes;

        // S = Q K^T: two n-tiles of 8 tokens
        float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            uint32_t kb[4], qh[4], ql[4];
            const int mat = lane >> 3;
            const int token = (mat >> 1) * 8 + (lane & 7);
            const int dim = 16 * s + (mat & 1) * 8;
            ldmatrix_x4(kb, kslot + swz_offset(token, dim));
            ldmatrix_x4(qh, &sh.qs[0][qrow * kQRow + 16 * s + qcol]);
            ldmatrix_x4(ql, &sh.qs[1][qrow * kQRow + 16 * s + qcol]);
            mma_bf16_16816(sacc[0], qh, kb[0], kb[1]);
            mma_bf16_16816(sacc[0], ql, kb[0], kb[1]);
            mma_bf16_16816(sacc[1], qh, kb[2], kb[3]);
            mma_bf16_16816(sacc[1], ql, kb[2], kb[3]);
        }
        if (valid < kPage) {
            // the unfilled page: tokens >= valid take no part (logits -inf; their V rows,
            // which need not hold finite values, are zeroed before P V)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int tok = nt * 8 + 2 * t;
                if (tok >= valid) sacc[nt][0] = sacc[nt][2] = -INFINITY;
                if (tok + 1 >= valid) sacc[nt][1] = sacc[nt][3] = -INFINITY;
            }
            for (int idx = lane; idx < (kPage - valid) * 16; idx += 32) {
                const int r = valid + (idx >> 4), box = (idx >> 3) & 1, c = idx & 7;
                *reinterpret_cast<uint4*>(const_cast<uint8_t*>(vslot) + box * kBoxBytes + r * 128 + c * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }
        // online softmax (log2 domain); rows gid (c0, c1) and gid + 8 (c2, c3)
        float mx_a = fmaxf(fmaxf(sacc[0][0], sacc[0][1]), fmaxf(sacc[1][0], sacc[1][1]));
        float mx_b = fmaxf(fmaxf(sacc[0][2], sacc[0][3]), fmaxf(sacc[1][2], sacc[1][3]));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        const float corr_a = (m_a == -INFINITY) ? 0.f : fast_exp2(m_a - mn_a);
        const float corr_b = (m_b == -INFINITY) ? 0.f : fast_exp2(m_b - mn_b);
        m_a = mn_a;
        m_b = mn_b;
        float pr[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            pr[nt][0] = fast_exp2(sacc[nt][0] - mn_a);
            pr[nt][1] = fast_exp2(sacc[nt][1] - mn_a);
            pr[nt][2] = fast_exp2(sacc[nt][2] - mn_b);
            pr[nt][3] = fast_exp2(sacc[nt][3] - mn_b);
        }
        l_a = l_a * corr_a + pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1];
        l_b = l_b * corr_b + pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3];
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
            o[nd][0] *= corr_a;
            o[nd][1] *= corr_a;
            o[nd][2] *= corr_b;
            o[nd][3] *= corr_b;
        }
        const uint32_t pa[4] = {pack_bf16x2(pr[0][0], pr[0][1]), pack_bf16x2(pr[0][2], pr[0][3]),
                                pack_bf16x2(pr[1][0], pr[1][1]), pack_bf16x2(pr[1][2], pr[1][3])};
        // O += P V: 16 n-tiles of 8 dims, two per ldmatrix.x4.trans
#pragma unroll
        for (int nd = 0; nd < 16; nd += 2) {
            uint32_t vb[4];
            const int mat = lane >> 3;
            const int token = (mat & 1) * 8 + (lane & 7);
            const int dim = 8 * (nd + (mat >> 1));
            ldmatrix_x4_trans(vb, vslot + swz_offset(token, dim));
            mma_bf16_16816(o[nd], pa, vb[0], vb[1]);
            mma_bf16_16816(o[nd + 1], pa, vb[2], vb[3]);
        }
        __syncwarp();   // all lanes done reading the slot before it is refilled
        if (p + kSlots * kWarps < p1) issue(p + kSlots * kWarps, sl);
        sl = kSlots == 1 ? 0 : sl ^ 1;
    }
    if (failed) report_error(a.st, LOCKS_ERR_TIMEOUT);
    if (bad) report_error(a.st, LOCKS_ERR_BAD_INDEX);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);

    // warp partials into the (now idle) ring: [warp][head][m, l, o[128]]
    __syncthreads();
    float* wpart = reinterpret_cast<float*>(ring);
    {
        float* ra = wpart + (warp * kMaxG + gid) * kPartStride;
        float* rb = wpart + (warp * kMaxG + gid + 8) * kPartStride;
        // rows of heads >= g hold nothing and are never read
        if (gid < g) {
            if (t == 0) {
                ra[0] = m_a;
                ra[1] = l_a;
            }
#pragma unroll
            for (int nd = 0; nd < 16; ++nd) {
                const int d = 8 * nd + 2 * t;
                ra[2 + d] = o[nd][0];
                ra[2 + d + 1] = o[nd][1];
            }
        }
        if (gid + 8 < g) {
            if (t == 0) {
                rb[0] = m_b;
                rb[1] = l_b;
            }
#pragma unroll
            for (int nd = 0; nd < 16; ++nd) {
                const int d = 8 * nd + 2 * t;
                rb[2 + d] = o[nd][2];
                rb[2 + d + 1] = o[nd][3];
            }
        }
    }
    __syncthreads();
    // CTA merge over warps: thread -> (head, 4 consecutive dims)
    for (int idx = tid; idx < g * (kD / 4); idx += kThreads) {
        const int hh = idx / (kD / 4), d4 = (idx % (kD / 4)) * 4;
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wpart[(w * kMaxG + hh) * kPartStride]);
        float L = 0.f, acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
        if (M != -INFINITY) {
            for (int w = 0; w < kWarps; ++w) {
                const float* r = wpart + (w * kMaxG + hh) * kPartStride;
                if (r[0] == -INFINITY) continue;
                const float f = fast_exp2(r[0] - M);
                L += r[1] * f;
                acc0 += r[2 + d4] * f;
                acc1 += r[3 + d4] * f;
                acc2 += r[4 + d4] * f;
                acc3 += r[5 + d4] * f;
            }
        }
        if constexpr (CL == kSpreadCluster) {
            // into the owner's inbox: slot (hh / CL, this CTA)
            const uint32_t ra = dsmem_addr(inbox + ((hh / CL) * CL + static_cast<int>(rank)) * kInStride,
                                           static_cast<uint32_t>(hh % CL));
            if (d4 == 0) st_dsmem_f32x2(ra, M, L);
            st_dsmem_f32x4(ra + static_cast<uint32_t>(4 + d4) * 4u, acc0, acc1, acc2, acc3);
        } else {
            float* c = sh.cpart + hh * kPartStride;
            if (d4 == 0) {
                c[0] = M;
                c[1] = L;
            }
            c[2 + d4] = acc0;
            c[3 + d4] = acc1;
            c[4 + d4] = acc2;
            c[5 + d4] = acc3;
        }
    }
    cluster_sync_all();   // every CTA's partials delivered (pushed) or readable (pulled)
    // cluster merge: CTA r finalises heads r, r + CL, ...
    for (int hh = static_cast<int>(rank); hh < g; hh += CL) {
        const int64_t qh_idx = static_cast<int64_t>(b) * a.hq + kvh * g + hh;
        float M = -INFINITY, L = 0.f, acc = 0.f;
        if (tid < kD) {
            float mr[CL], lr[CL], orr[CL];   // all loads in flight before any use
            if constexpr (CL == kSpreadCluster) {
                const float* in = inbox + (hh / CL) * CL * kInStride;
#pragma unroll
                for (int r = 0; r < CL; ++r) {
                    mr[r] = in[r * kInStride];
                    lr[r] = in[r * kInStride + 1];
                    orr[r] = in[r * kInStride + 4 + tid];
                }
            } else {
                const float* c = sh.cpart + hh * kPartStride;
#pragma unroll
                for (uint32_t r = 0; r < CL; ++r) {
                    mr[r] = ld_dsmem_f32(dsmem_addr(c, r));
                    lr[r] = ld_dsmem_f32(dsmem_addr(c + 1, r));
                    orr[r] = ld_dsmem_f32(dsmem_addr(c + 2 + tid, r));
                }
            }
#pragma unroll
            for (uint32_t r = 0; r < CL; ++r) M = fmaxf(M, mr[r]);
            if (M != -INFINITY) {
#pragma unroll
                for (uint32_t r = 0; r < CL; ++r) {
                    if (mr[r] == -INFINITY) continue;
                    const float f = fast_exp2(mr[r] - M);
                    L += lr[r] * f;
                    acc += orr[r] * f;
                }
            }
        }
        if (SPLIT && S > 1) {
            // this cluster's (m, l, o) of the head into the workspace; the last of the S
            // clusters to arrive (an atomic count, no waiting) merges them
            float* gp = a.attn_part + (qh_idx * kMaxSplits + z) * kPartStride;
            if (tid < kD) {
                gp[2 + tid] = acc;
                if (tid == 0) {
                    gp[0] = M;
                    gp[1] = L;
                }
            }
            __threadfence();
            __syncthreads();
            if (tid == 0) sh.split_last = atomicAdd(&a.attn_cnt[qh_idx], 1) == S - 1;
            __syncthreads();
            if (!sh.split_last) continue;
            __threadfence();
            if (tid < kD) {
                const float* hp = a.attn_part + qh_idx * kMaxSplits * kPartStride;
                M = -INFINITY;
                for (int zz = 0; zz < S; ++zz) M = fmaxf(M, __ldcg(hp + zz * kPartStride));
                L = 0.f;
                acc = 0.f;
                if (M != -INFINITY) {
                    for (int zz = 0; zz < S; ++zz) {
                        const float mz = __ldcg(hp + zz * kPartStride);
                        if (mz == -INFINITY) continue;
                        const float f = fast_exp2(mz - M);
                        L += __ldcg(hp + zz * kPartStride + 1) * f;
                        acc += __ldcg(hp + zz * kPartStride + 2 + tid) * f;
                    }
                }
            }
        }
        if (tid < kD) {
            const float val = (L > 0.f) ? acc / L : 0.f;
            a.out[qh_idx * kD + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
            if (a.lse && tid == 0) a.lse[qh_idx] = (L > 0.f) ? (M + fast_log2(L)) * kLn2 : -INFINITY;
        }
    }
    // pulled partials stay readable until every CTA is done; pushed ones are local
    if constexpr (CL != kSpreadCluster) cluster_sync_all();
}

template <int CL, SAMode MODE, int GM>
__global__ void __launch_bounds__(kThreads, CL == kSpreadCluster ? 1 : 2) select_attend_kernel(const __grid_constant__ SelectAttendArgs a,
                                                                       int chunk) {
    extern __shared__ __align__(1024) uint8_t smem[];
    SmallShared& sh = *reinterpret_cast<SmallShared*>(smem);
    // the region after SmallShared, 1 KiB-aligned in the shared window (128-byte swizzle)
    const uint32_t small_end = smem_u32(smem) + static_cast<uint32_t>(sizeof(SmallShared));
    uint8_t* big = smem + (((small_end + 1023u) & ~1023u) - smem_u32(smem));
    const uint32_t rank = cluster_ctarank();
    const int seg = blockIdx.y;
    const int b = seg / a.hkv, kvh = seg % a.hkv;
    if (threadIdx.x < 2 * kWarps) mbar_init(&sh.bar[threadIdx.x], 1);
    if (threadIdx.x == 2 * kWarps) mbar_init(&sh.sbar, 1);
    if constexpr (MODE != SAMode::kAttend) {
        // the selection's per-warp key histograms (in the candidate-list space)
        uint32_t* whist = reinterpret_cast<uint32_t*>(big + region_a_bytes(chunk, CL));
        static_assert(kWarps * 256 * 4 <= kCandListBytes, "per-warp histograms fit a candidate list");
#pragma unroll 1
        for (int i = threadIdx.x; i < kWarps * 256; i += kThreads) whist[i] = 0u;
    }
    fence_barrier_init();
    // Launched with programmatic stream serialization: the set-up above overlaps the end
    // of the previous kernel (the scorer). The selection waits for it inside select_pages,
    // after loading inputs that kernel does not write (the query, sequence lengths and a
    // prefetch of the page table): every kernel of this library lets its dependents
    // launch only after its own wait, so the kernels before it are complete.
    if constexpr (MODE == SAMode::kAttend) {
        grid_dependency_wait();
        allow_dependent_launch();   // the next kernel waits for this grid's completion itself
    }
    __syncthreads();

    if constexpr (MODE == SAMode::kSelect) {
        bool listed = false, preissued = false;
        select_pages<CL, GM>(a, b, kvh, rank, chunk, big, sh, false, &listed, &preissued);
        cluster_sync_all();   // this CTA's shared data stays readable until every CTA is done with it
    } else if constexpr (MODE == SAMode::kAttend) {
        const int n = max(0, min(a.n_selected[b * a.hkv + kvh], a.k_cap));
        attend_pages<CL, GM, true>(a, b, kvh, rank, n, a.selected + (static_cast<int64_t>(b) * a.hkv + kvh) * a.k_cap,
                                   false, false, big, sh, reinterpret_cast<float*>(big + inbox_offset(chunk, CL, true)));
    } else {
        bool listed = false, preissued = false;
        const int n = select_pages<CL, GM>(a, b, kvh, rank, chunk, big, sh, true, &listed, &preissued);
        if (!listed) {
            // the selection went to global memory; make it visible to the cluster's CTAs
            asm volatile("fence.acq_rel.cluster;" ::: "memory");
            cluster_sync_all();
        }
        // fast selection: every CTA holds the kept pages, ascending, in its gathered list
        const CandList kept = cand_list(big + region_a_bytes(chunk, CL) + kCandListBytes);
        attend_pages<CL, GM, false>(a, b, kvh, rank, n, a.selected + (static_cast<int64_t>(b) * a.hkv + kvh) * a.k_cap,
                                    true, true, big, sh, reinterpret_cast<float*>(big + inbox_offset(chunk, CL, false)),
                                    listed ? kept.logical : nullptr, listed ? kept.phys : nullptr, preissued);
    }
}

int chunk_of(int max_pages, int cluster) {
    int c = (max_pages + cluster - 1) / cluster;
    return (c + 7) & ~7;   // whole 8-page blocks: 4-page slabs and 16-byte score loads stay aligned
}

// The driver's tiled tensor-map encoder, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        }
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// A K or V cache [num_phys][hkv][16][128] bf16 as a 2D tensor of num_phys * hkv * 16
// rows of 128 elements, read in 64 x 16 boxes with 128-byte swizzle.
cudaError_t encode_cache_map(CUtensorMap* map, const uint16_t* base, int64_t rows) {
    const auto fn = encode_tiled();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kPage)};
    const cuuint32_t elem_strides[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), dims, strides, box,
                          elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int CL, SAMode MODE, int GM>
cudaError_t launch_t(const SelectAttendArgs& args, cudaStream_t stream) {
    SelectAttendArgs a = args;
    std::memset(&a.tm_k, 0, sizeof(a.tm_k));
    std::memset(&a.tm_v, 0, sizeof(a.tm_v));
    if (MODE != SAMode::kSelect) {
        const int64_t rows = static_cast<int64_t>(a.num_phys) * a.hkv * kPage;   // TMA row coordinates are int32
        if (rows > INT_MAX) return cudaErrorInvalidValue;
        cudaError_t e = encode_cache_map(&a.tm_k, a.k_cache, rows);
        if (e == cudaSuccess) e = encode_cache_map(&a.tm_v, a.v_cache, rows);
        if (e != cudaSuccess) return e;
    }
    const int chunk = chunk_of(a.max_pages, CL);
    const size_t smem = select_attend_smem_bytes(a.max_pages, CL, MODE);
    auto kern = select_attend_kernel<CL, MODE, GM>;
    cudaError_t e = ensure_kernel_attrs<select_attend_kernel<CL, MODE, GM>>(static_cast<int>(smem), CL > 8);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    const int splits = (MODE == SAMode::kAttend && a.attn_part && a.attn_cnt) ? max(1, min(a.splits, kMaxSplits)) : 1;
    cfg.gridDim = dim3(CL, a.batch * a.hkv, splits);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, a, chunk);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int CL, int GM>
cudaError_t launch_cl(const SelectAttendArgs& a, SAMode mode, cudaStream_t stream) {
    switch (mode) {
        case SAMode::kSelect: return launch_t<CL, SAMode::kSelect, GM>(a, stream);
        case SAMode::kAttend: return launch_t<CL, SAMode::kAttend, GM>(a, stream);
        default: return launch_t<CL, SAMode::kSelectAttend, GM>(a, stream);
    }
}

template <int CL, SAMode MODE, int GM>
int active_clusters_t(size_t smem) {
    auto kern = select_attend_kernel<CL, MODE, GM>;
    if (ensure_kernel_attrs<select_attend_kernel<CL, MODE, GM>>(static_cast<int>(smem), CL > 8) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <int CL, int GM>
int active_clusters_cl(size_t smem, SAMode mode) {
    switch (mode) {
        case SAMode::kSelect: return active_clusters_t<CL, SAMode::kSelect, GM>(smem);
        case SAMode::kAttend: return active_clusters_t<CL, SAMode::kAttend, GM>(smem);
        default: return active_clusters_t<CL, SAMode::kSelectAttend, GM>(smem);
    }
}

}  // namespace

size_t select_attend_smem_bytes(int max_pages, int cluster, SAMode mode) {
    const size_t small = sizeof(SmallShared) + 1024;   // + alignment of the region after it
    const size_t need =
        mode == SAMode::kAttend
            ? small + static_cast<size_t>(ring_bytes(cluster))
            : small + static_cast<size_t>(region_a_bytes(chunk_of(max_pages, cluster), cluster)) + 2 * kCandListBytes;
    return cluster == kSpreadCluster ? std::max<size_t>(need + kInboxBytes, kSpreadSmemBytes) : need;
}

int group_bound(int g) { return g <= 4 ? 4 : 16; }

namespace {
template <int GM>
int active_clusters_g(size_t smem, SAMode mode, int cluster) {
    if (cluster == kSpreadCluster) return active_clusters_cl<kSpreadCluster, GM>(smem, mode);
    return cluster == 16 ? active_clusters_cl<16, GM>(smem, mode) : active_clusters_cl<8, GM>(smem, mode);
}
template <int GM>
cudaError_t launch_g(const SelectAttendArgs& a, SAMode mode, int cluster, cudaStream_t stream) {
    if (cluster == kSpreadCluster) return launch_cl<kSpreadCluster, GM>(a, mode, stream);
    return cluster == 16 ? launch_cl<16, GM>(a, mode, stream) : launch_cl<8, GM>(a, mode, stream);
}
}  // namespace

int select_attend_active_clusters(int max_pages, SAMode mode, int g, int cluster) {
    const size_t smem = select_attend_smem_bytes(max_pages, cluster, mode);
    return group_bound(g) == 4 ? active_clusters_g<4>(smem, mode, cluster) : active_clusters_g<16>(smem, mode, cluster);
}

int select_attend_ctas_per_sm(int max_pages, SAMode mode, int cluster) {
    int dev = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    const size_t per_cta = select_attend_smem_bytes(max_pages, cluster, mode) + 1024;   // + the per-CTA reserve
    return std::max(1, std::min(2, static_cast<int>(static_cast<size_t>(per_sm) / per_cta)));
}

cudaError_t launch_select_attend(const SelectAttendArgs& a, SAMode mode, int cluster, cudaStream_t stream) {
    if (a.batch * a.hkv == 0) return cudaSuccess;
    const int g = a.hq / a.hkv;
    return group_bound(g) == 4 ? launch_g<4>(a, mode, cluster, stream) : launch_g<16>(a, mode, cluster, stream);
}

}  // namespace locks
