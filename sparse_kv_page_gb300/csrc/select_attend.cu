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
//   top-k by an MSB-first radix select (4 passes of 8 bits) on the
//   order-preserving uint32 image of key_j; histograms are summed across the
//   cluster through DSMEM. Equal keys are ranked by lower page id; the output
//   is written in ascending page order by an ordered compaction.
// Attention (LOCKS post, "Code": scaled dot-product attention over the pages
// kept): each CTA takes a contiguous share of the selected pages; each warp
// streams one page at a time (its K and V rows as four tiled TMA boxes of 16
// tokens x 64 dims, 128-byte swizzle) and runs QK^T and PV on the tensor cores
// (mma.sync bf16 through ldmatrix, query split hi/lo, online softmax in fp32).
// Warp partials (m, l, o) are merged per CTA, then across the cluster.
//
// When the scoring kernel's per-8-page LSE partials are given, the per-head
// normaliser L_h is reduced from them instead of from the full score table.
// At most 128 registers per thread so that two CTAs share an SM.
#include <cudaTypedefs.h>
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
    int bin_cnt[16], nbin, rank_take, cnt4[4];
    uint32_t rank_T;
    uint32_t bin_keys[256], rank_keys[256];
    uint8_t rank_src[256];
    uint64_t bar[kWarps];
    float cpart[kMaxG * kPartStride];     // this CTA's attention partial per head
    int split_last;                       // split attention: this cluster merges the splits of a head
};

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

// ------------------------------------------------------------- selection
// Per-head normaliser L_h over the sequence (cluster-wide) and the group keys of
// this CTA's pages [j0, j1) into keys[] (order-preserving uint32 images).
// Scores are read in batches of kB pages per thread, each batch's loads issued
// one batch ahead (the first one before the normaliser's reduction, so its
// latency overlaps the cluster exchange). Loops stay rolled: this code runs
// about once per launch, and its instruction fetch is what it waits on.
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

// stage_q: also stage the query rows for the attention that follows (their loads
// overlap the normaliser's).
template <int CL, int GM>
__device__ void group_keys(const SelectAttendArgs& a, int b, int kvh, int j0, int j1, uint32_t* keys,
                           SmallShared& sh, bool stage_q) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = a.hq / a.hkv;
    const int nloc = j1 - j0;
    const float* srow = a.scores + (static_cast<int64_t>(b) * a.hq + kvh * g) * a.max_pages;
    constexpr int kB = GM <= 4 ? 4 : 1;   // pages per thread per batch
    constexpr int kStep = kB * kThreads;
    auto load_batch = [&](float (&x)[kB][GM], int jb) {
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const int j = jb + u * kThreads;
#pragma unroll
            for (int hh = 0; hh < GM; ++hh)
                x[u][hh] = (hh < g && j < j1) ? srow[static_cast<int64_t>(hh) * a.max_pages + j] : -INFINITY;
        }
    };
    // the first two batches of scores are in flight during the normaliser below, and
    // two stay in flight in the key loop
    float v[kB][GM], v2[kB][GM];
    load_batch(v, j0 + tid);
    load_batch(v2, j0 + tid + kStep);
    float qv[16 * kD / kThreads];
    if (stage_q) load_query(a, b, kvh, g, qv);

    // 1. per-head log-sum-exp over the sequence's pages: (m, l) per thread and head
    float m[GM], l[GM];
#pragma unroll
    for (int hh = 0; hh < GM; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.f;
    }
    if (a.lse_partials) {
        // from the scoring kernel's (max, sum) partials of 8-page blocks
        const int nblk = (a.max_pages + 7) / 8;
        const int blk0 = j0 / 8, blk1 = nloc > 0 ? (j1 + 7) / 8 : blk0;   // an empty range owns no block
        const float2* prow = reinterpret_cast<const float2*>(a.lse_partials) +
                             (static_cast<int64_t>(b) * a.hq + kvh * g) * nblk;
#pragma unroll 1
        for (int ib = blk0 + tid; ib < blk1; ib += kThreads) {
            float2 pv[GM];
#pragma unroll
            for (int hh = 0; hh < GM; ++hh)
                pv[hh] = hh < g ? prow[static_cast<int64_t>(hh) * nblk + ib] : make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int hh = 0; hh < GM; ++hh)
                if (hh < g) lse_combine(m[hh], l[hh], pv[hh].x, pv[hh].y);
        }
    } else {
        // from the scores themselves (reloading them later if they span several batches)
#pragma unroll 1
        for (int jb = j0 + tid; jb < j1; jb += kStep) {
            float x[kB][GM];
            if (jb == j0 + tid) {
#pragma unroll
                for (int u = 0; u < kB; ++u)
#pragma unroll
                    for (int hh = 0; hh < GM; ++hh) x[u][hh] = v[u][hh];
            } else if (jb == j0 + tid + kStep) {
#pragma unroll
                for (int u = 0; u < kB; ++u)
#pragma unroll
                    for (int hh = 0; hh < GM; ++hh) x[u][hh] = v2[u][hh];
            } else {
                load_batch(x, jb);
            }
#pragma unroll
            for (int hh = 0; hh < GM; ++hh) {
                if (hh < g) {
                    float bm = x[0][hh];
#pragma unroll
                    for (int u = 1; u < kB; ++u) bm = fmaxf(bm, x[u][hh]);
                    if (bm != -INFINITY) {
                        float z = 0.f;
#pragma unroll
                        for (int u = 0; u < kB; ++u) z += fast_exp2((x[u][hh] - bm) * kLog2e);
                        lse_combine(m[hh], l[hh], bm, z);
                    }
                }
            }
        }
    }
    if (stage_q) store_query(qv, g, sh);   // read after the barriers below
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

    // 2. group-mean mass-share keys
    // (log2 domain: x = (s - L_h) log2 e; key = (max + log2 sum exp2(x - max)) ln 2 - ln g)
    const float log_g = logf(static_cast<float>(g));
    float Lr[GM];
#pragma unroll
    for (int hh = 0; hh < GM; ++hh) Lr[hh] = hh < g ? sh.Lh[hh] : 0.f;
#pragma unroll 1
    for (int jb = j0 + tid; jb < j1; jb += kStep) {
        float w[kB][GM];
        const bool more = jb + 2 * kStep < j1;
        if (more) load_batch(w, jb + 2 * kStep);   // two batches in flight while this one is used
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const int j = jb + u * kThreads;
            if (j < j1) {
                float mx = -INFINITY;
                float x[GM];
#pragma unroll
                for (int hh = 0; hh < GM; ++hh) {
                    x[hh] = 0.f;
                    if (hh < g) {
                        x[hh] = (v[u][hh] - Lr[hh]) * kLog2e;
                        mx = fmaxf(mx, x[hh]);
                    }
                }
                float key;
                if (mx == -INFINITY) {
                    key = -INFINITY;
                } else {
                    float z = 0.f;
#pragma unroll
                    for (int hh = 0; hh < GM; ++hh)
                        if (hh < g) z += fast_exp2(x[hh] - mx);
                    key = (mx + fast_log2(z)) * kLn2 - log_g;
                }
                keys[j - j0] = orderable_key(key);
                if (a.sel_keys) a.sel_keys[(static_cast<int64_t>(b) * a.hkv + kvh) * a.max_pages + j] = key;
            }
        }
#pragma unroll
        for (int u = 0; u < kB; ++u)
#pragma unroll
            for (int hh = 0; hh < GM; ++hh) {
                v[u][hh] = v2[u][hh];
                if (more) v2[u][hh] = w[u][hh];
            }
    }
    __syncthreads();
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

// Writes selected[b][kvh][0..K) and n_selected[b][kvh]; returns K.
// One MSB-first radix select over the cluster (4 passes of 8 bits): each CTA
// histograms its own keys, every CTA sums the CTAs' histograms through DSMEM and
// picks the digit. The same pass also yields, per CTA, how many keys lie above
// the chosen bin in lower-ranked CTAs and in this one (and, in the last pass,
// how many equal T), which places this CTA's kept keys in the ascending output
// without a further exchange.
template <int CL, int GM>
__device__ int select_pages(const SelectAttendArgs& a, int b, int kvh, uint32_t rank, int chunk, uint32_t* keys,
                            SmallShared& sh, bool stage_q) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = max(0, min(a.seq_pages[b], a.max_pages));
    const int j0 = min(P, static_cast<int>(rank) * chunk);
    const int j1 = min(P, j0 + chunk);
    const int nloc = j1 - j0;

    group_keys<CL, GM>(a, b, kvh, j0, j1, keys, sh, stage_q);

    int K = min(a.budget_pages, min(P, a.k_cap));
    K = max(K, 0);
    int32_t* out = a.selected + (static_cast<int64_t>(b) * a.hkv + kvh) * a.k_cap;
    if (rank == 0 && tid == 0) a.n_selected[b * a.hkv + kvh] = K;
    if (K == 0) return 0;
    if (K == P) {
        for (int j = j0 + tid; j < j1; j += kThreads) out[j] = j;
        return K;
    }

    uint32_t prefix = 0;
    int remaining = K;
    int gt_low = 0, gt_own = 0, eq_low = 0, eq_own = 0;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        uint32_t* hist = sh.hist[pass & 1];   // alternating: other CTAs read the previous one
        hist[tid] = 0u;
        __syncthreads();
        if (pass == 0) {
            // the top byte takes few values: one shared atomic per distinct bin per warp step
            for (int i0 = 0; i0 < nloc; i0 += kThreads) {
                const int i = i0 + tid;
                const uint32_t bin = i < nloc ? keys[i] >> 24 : 0xffffffffu;
                const unsigned peers = __match_any_sync(0xffffffffu, bin);
                if (i < nloc && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
            }
        } else {
            const uint32_t hp = prefix >> (shift + 8);
#pragma unroll 4
            for (int i = tid; i < nloc; i += kThreads) {
                const uint32_t key = keys[i];
                if ((key >> (shift + 8)) == hp) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            }
        }
        __syncthreads();
        cluster_sync_all();
        uint32_t hv[CL];   // all remote loads in flight before any use
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) hv[r] = ld_dsmem_u32(dsmem_addr(&hist[tid], r));
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
            // lane l holds bins 8l .. 8l + 7 of (all CTAs, lower-ranked CTAs, this CTA);
            // the digit is the bin where the count of keys at or above it first
            // reaches `remaining`, scanning from the top bin down
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
        prefix |= static_cast<uint32_t>(sh.digit) << shift;
        remaining -= sh.above;
        gt_low += sh.above_low;
        gt_own += sh.above_own;
        eq_low = sh.eq_low;
        eq_own = sh.eq_own;
        const int inbin = sh.inbin;
        if (pass < 3 && inbin <= kRankCap) {
            // The K-th largest key is one of the inbin keys of the chosen bin: every CTA
            // publishes its keys of that bin, every CTA gathers all of them through DSMEM and
            // ranks them directly instead of running the remaining passes.
            if (tid == sh.digit) {
#pragma unroll
                for (uint32_t r = 0; r < CL; ++r) sh.bin_cnt[r] = static_cast<int>(hv[r]);
            }
            if (tid == 0) sh.nbin = 0;
            __syncthreads();
            const uint32_t want = prefix >> shift;   // every bit at or above this pass's digit
            for (int i0 = 0; i0 < nloc; i0 += kThreads) {
                const int i = i0 + tid;
                const uint32_t key = i < nloc ? keys[i] : 0u;
                const bool m = i < nloc && (key >> shift) == want;
                const unsigned bal = __ballot_sync(0xffffffffu, m);
                int base = 0;
                if (lane == 0 && bal) base = atomicAdd(&sh.nbin, __popc(bal));
                base = __shfl_sync(0xffffffffu, base, 0);
                if (m) sh.bin_keys[base + __popc(bal & lanemask_lt())] = key;
            }
            cluster_sync_all();   // every CTA's bin keys are complete and visible
            if (tid < inbin) {
                int r = 0, base = 0;
#pragma unroll
                for (int q = 0; q < CL - 1; ++q) {
                    if (r == q && tid >= base + sh.bin_cnt[q]) {   // past rank q's keys: move on
                        base += sh.bin_cnt[q];
                        r = q + 1;
                    }
                }
                sh.rank_keys[tid] = ld_dsmem_u32(dsmem_addr(&sh.bin_keys[tid - base], static_cast<uint32_t>(r)));
                sh.rank_src[tid] = static_cast<uint8_t>(r);
            }
            if (tid < 4) sh.cnt4[tid] = 0;
            __syncthreads();
            if (tid < inbin) {
                const uint32_t key = sh.rank_keys[tid];
                int gt = 0, ge = 0;
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
            const uint32_t T = sh.rank_T;
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
            prefix = T;
            remaining = sh.rank_take;
            break;
        }
    }
    // T = prefix is the K-th largest key; the first `remaining` keys equal to it are
    // kept. This CTA keeps its keys > T and its first take_cta keys == T, written from
    // position pos0 on (the kept keys of lower-ranked CTAs come first).
    const int take_cta = max(0, min(remaining - eq_low, eq_own));
    const int pos0 = gt_low + min(eq_low, remaining);
    ordered_keep(keys, nloc, prefix, take_cta, sh, [&](int i, int pos) {
        if (pos0 + pos < K) out[pos0 + pos] = j0 + i;   // always < K; the guard only bounds a logic error
    });
    return K;
}
// ------------------------------------------------------------- attention
template <int CL, int GM>
__device__ void attend_pages(const SelectAttendArgs& a, int b, int kvh, uint32_t rank, int n_sel,
                             const int32_t* sel, bool sel_coherent, bool q_staged, uint8_t* ring, SmallShared& sh) {
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

    uint8_t* slot = ring + warp * kPageSlotBytes;
    uint64_t* bar = &sh.bar[warp];
    uint32_t phase = 0;
    for (int p = p0 + warp; p < p1; p += kWarps) {
        // tokens of the page that are attended
        const int valid = p < n_sel ? kPage : min(kPage, tail - (p - n_sel) * kPage);
        int logical = p < n_sel ? (sel_coherent ? __ldcg(sel + p) : sel[p]) : tail_page + (p - n_sel);
        if (logical < 0 || logical >= a.max_pages) {
            bad = true;
            logical = 0;
        }
        int64_t phys = a.page_table[static_cast<int64_t>(b) * a.max_pages + logical];
        if (phys < 0 || phys >= a.num_phys) {
            bad = true;
            phys = 0;
        }
        const int y = static_cast<int>((phys * a.hkv + kvh) * kPage);   // first row of the page's tile
        fence_proxy_async_smem();   // earlier generic reads of the slot before the async refill
        __syncwarp();
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, kPageSlotBytes);
            tma_load_2d(slot, &a.tm_k, 0, y, bar);
            tma_load_2d(slot + kBoxBytes, &a.tm_k, 64, y, bar);
            tma_load_2d(slot + 2 * kBoxBytes, &a.tm_v, 0, y, bar);
            tma_load_2d(slot + 3 * kBoxBytes, &a.tm_v, 64, y, bar);
        }
        if (!mbar_wait_bounded(bar, phase, a.st.wait_limit_ns)) failed = true;
        phase ^= 1u;
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
        if (t == 0) {
            ra[0] = m_a;
            ra[1] = l_a;
            rb[0] = m_b;
            rb[1] = l_b;
        }
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
            const int d = 8 * nd + 2 * t;
            ra[2 + d] = o[nd][0];
            ra[2 + d + 1] = o[nd][1];
            rb[2 + d] = o[nd][2];
            rb[2 + d + 1] = o[nd][3];
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
    cluster_sync_all();
    // cluster merge: CTA r finalises heads r, r + CL, ...
    for (int hh = static_cast<int>(rank); hh < g; hh += CL) {
        const int64_t qh_idx = static_cast<int64_t>(b) * a.hq + kvh * g + hh;
        float M = -INFINITY, L = 0.f, acc = 0.f;
        if (tid < kD) {
            const float* c = sh.cpart + hh * kPartStride;
            float mr[CL], lr[CL], orr[CL];   // all remote loads in flight before any use
#pragma unroll
            for (uint32_t r = 0; r < CL; ++r) {
                mr[r] = ld_dsmem_f32(dsmem_addr(c, r));
                lr[r] = ld_dsmem_f32(dsmem_addr(c + 1, r));
                orr[r] = ld_dsmem_f32(dsmem_addr(c + 2 + tid, r));
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
        if (S > 1) {
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
    cluster_sync_all();   // partials stay readable until every CTA is done
}

template <int CL, SAMode MODE, int GM>
__global__ void __launch_bounds__(kThreads, 2) select_attend_kernel(const __grid_constant__ SelectAttendArgs a,
                                                                       int chunk) {
    extern __shared__ __align__(1024) uint8_t smem[];
    SmallShared& sh = *reinterpret_cast<SmallShared*>(smem);
    // the region after SmallShared, 1 KiB-aligned in the shared window (128-byte swizzle)
    const uint32_t small_end = smem_u32(smem) + static_cast<uint32_t>(sizeof(SmallShared));
    uint8_t* big = smem + (((small_end + 1023u) & ~1023u) - smem_u32(smem));
    const uint32_t rank = cluster_ctarank();
    const int seg = blockIdx.y;
    const int b = seg / a.hkv, kvh = seg % a.hkv;
    // a dependent kernel (the next layer's scorer) may be scheduled once every CTA
    // of this grid has started; it waits for this grid's completion itself
    allow_dependent_launch();
    if (threadIdx.x < kWarps) mbar_init(&sh.bar[threadIdx.x], 1);
    fence_barrier_init();
    // launched with programmatic stream serialization: the set-up above overlaps
    // the end of the previous kernel (the scorer); every global access follows
    grid_dependency_wait();
    __syncthreads();

    if constexpr (MODE == SAMode::kSelect) {
        select_pages<CL, GM>(a, b, kvh, rank, chunk, reinterpret_cast<uint32_t*>(big), sh, false);
        cluster_sync_all();   // this CTA's shared data stays readable until every CTA is done with it
    } else if constexpr (MODE == SAMode::kAttend) {
        const int n = max(0, min(a.n_selected[b * a.hkv + kvh], a.k_cap));
        attend_pages<CL, GM>(a, b, kvh, rank, n, a.selected + (static_cast<int64_t>(b) * a.hkv + kvh) * a.k_cap, false,
                             false, big, sh);
    } else {
        const int n = select_pages<CL, GM>(a, b, kvh, rank, chunk, reinterpret_cast<uint32_t*>(big), sh, true);
        // the selection went to global memory; make it visible to the cluster's CTAs
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
        cluster_sync_all();
        attend_pages<CL, GM>(a, b, kvh, rank, n, a.selected + (static_cast<int64_t>(b) * a.hkv + kvh) * a.k_cap, true,
                             true, big, sh);
    }
}

int chunk_of(int max_pages, int cluster) {
    int c = (max_pages + cluster - 1) / cluster;
    return (c + 7) & ~7;   // whole 8-page blocks (the LSE partials' granularity)
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
    const size_t keys = (mode == SAMode::kAttend) ? 0 : static_cast<size_t>(chunk_of(max_pages, cluster)) * 4;
    const size_t ring = (mode == SAMode::kSelect) ? 0 : static_cast<size_t>(kRingBytes);
    return small + (keys > ring ? keys : ring);
}

int group_bound(int g) { return g <= 4 ? 4 : 16; }

int select_attend_active_clusters(int max_pages, SAMode mode, int g, int cluster) {
    const size_t smem = select_attend_smem_bytes(max_pages, cluster, mode);
    if (group_bound(g) == 4)
        return cluster == 16 ? active_clusters_cl<16, 4>(smem, mode) : active_clusters_cl<8, 4>(smem, mode);
    return cluster == 16 ? active_clusters_cl<16, 16>(smem, mode) : active_clusters_cl<8, 16>(smem, mode);
}

cudaError_t launch_select_attend(const SelectAttendArgs& a, SAMode mode, int cluster, cudaStream_t stream) {
    if (a.batch * a.hkv == 0) return cudaSuccess;
    const int g = a.hq / a.hkv;
    if (group_bound(g) == 4) return cluster == 16 ? launch_cl<16, 4>(a, mode, stream) : launch_cl<8, 4>(a, mode, stream);
    return cluster == 16 ? launch_cl<16, 16>(a, mode, stream) : launch_cl<8, 16>(a, mode, stream);
}

}  // namespace locks
