// select_attend.cu - group-shared top-k page selection and sparse attention.
//
// One thread-block cluster of CL CTAs per (sequence b, kv head). The CTAs of
// a cluster split the sequence's pages (selection) and then the selected
// pages (attention) and combine their partial results through distributed
// shared memory, so no global scratch and no second launch is needed.
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
// streams one page at a time (16 K rows + 16 V rows, 256-byte bulk copies
// into padded shared rows) and runs QK^T and PV on the tensor cores
// (mma.sync bf16, query split hi/lo, online softmax in fp32). Warp partials
// (m, l, o) are merged per CTA, then across the cluster.
//
// When the scoring kernel's per-8-page LSE partials are given, the per-head
// normaliser L_h is reduced from them instead of from the full score table.
// At most 128 registers per thread so that two CTAs share an SM.
#include "locks_internal.h"

namespace locks {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowBytes = 272;                        // 256 B row + 16 B pad (conflict-free ldmatrix)
constexpr int kPageSlotBytes = 2 * kPage * kRowBytes; // K rows then V rows: 8704 B
constexpr int kRingBytes = kWarps * kPageSlotBytes;   // 69,632 B
constexpr int kPartStride = 2 + kD;                   // m, l, o[128]
constexpr int kMaxG = LOCKS_MAX_GROUP;
constexpr int kQRow = 136;                            // bf16 per staged query row (128 + 8 pad)

struct SmallShared {
    uint16_t qs[2][16 * kQRow];           // query rows (group heads), bf16 high / low parts
    uint32_t hist[2][256];
    float part_m[kMaxG], part_l[kMaxG];   // this CTA's per-head LSE partial
    float Lh[kMaxG];
    float red_m[kWarps][kMaxG], red_l[kWarps][kMaxG];
    int scan[kWarps + 1];
    int cnt[2];                           // this CTA's (greater, equal) counts
    int digit, above;
    uint64_t bar[kWarps];
    float cpart[kMaxG * kPartStride];     // this CTA's attention partial per head
};

__device__ __forceinline__ void lse_combine(float& m, float& l, float m2, float l2) {
    const float M = fmaxf(m, m2);
    if (M == -INFINITY) return;
    l = l * fast_exp2((m - M) * kLog2e) + l2 * fast_exp2((m2 - M) * kLog2e);
    m = M;
}

// Block-wide exclusive scan of one int per thread; returns (exclusive, total).
__device__ __forceinline__ int block_exclusive_scan(int v, int* scan, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scan[warp] = x;
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int w = 0; w < kWarps; ++w) {
            const int c = scan[w];
            scan[w] = acc;
            acc += c;
        }
        scan[kWarps] = acc;
    }
    __syncthreads();
    const int excl = scan[warp] + x - v;
    total = scan[kWarps];
    __syncthreads();
    return excl;
}

// ------------------------------------------------------------- selection
// Writes selected[b][kvh][0..k) and n_selected[b][kvh]; returns k.
template <int CL, int GM>
__device__ int select_pages(const SelectAttendArgs& a, int b, int kvh, uint32_t rank, int chunk,
                            uint32_t* keys, SmallShared& sh) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = a.hq / a.hkv;
    const int P = max(0, min(a.seq_pages[b], a.max_pages));
    const int j0 = min(P, static_cast<int>(rank) * chunk);
    const int j1 = min(P, j0 + chunk);
    const int nloc = j1 - j0;
    const float* srow = a.scores + (static_cast<int64_t>(b) * a.hq + kvh * g) * a.max_pages;

    // 1. per-head log-sum-exp over the sequence's pages
    float m[GM], l[GM];
#pragma unroll
    for (int hh = 0; hh < GM; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.f;
    }
    constexpr int kBatch = GM <= 4 ? 4 : 1;   // pages per thread whose loads are all issued before use
    if (a.lse_partials) {
        // from the scoring kernel's (max, sum) partials of 8-page blocks
        const int nblk = (a.max_pages + 7) / 8;
        const int blk0 = j0 / 8, blk1 = nloc > 0 ? (j1 + 7) / 8 : blk0;   // an empty range owns no block
        const float2* prow = reinterpret_cast<const float2*>(a.lse_partials) +
                             (static_cast<int64_t>(b) * a.hq + kvh * g) * nblk;
        for (int ib = blk0 + tid; ib < blk1; ib += kBatch * kThreads) {
            float2 v[kBatch][GM];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int blk = ib + u * kThreads;
#pragma unroll
                for (int hh = 0; hh < GM; ++hh)
                    v[u][hh] = (hh < g && blk < blk1) ? prow[static_cast<int64_t>(hh) * nblk + blk]
                                                      : make_float2(-INFINITY, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
#pragma unroll
                for (int hh = 0; hh < GM; ++hh)
                    if (hh < g) lse_combine(m[hh], l[hh], v[u][hh].x, v[u][hh].y);
        }
    } else {
        for (int jb = j0 + tid; jb < j1; jb += kBatch * kThreads) {
            float v[kBatch][GM];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int j = jb + u * kThreads;
#pragma unroll
                for (int hh = 0; hh < GM; ++hh)
                    v[u][hh] = (hh < g && j < j1) ? srow[static_cast<int64_t>(hh) * a.max_pages + j] : -INFINITY;
            }
#pragma unroll
            for (int hh = 0; hh < GM; ++hh) {
                if (hh < g) {
                    float bm = v[0][hh];
#pragma unroll
                    for (int u = 1; u < kBatch; ++u) bm = fmaxf(bm, v[u][hh]);
                    if (bm != -INFINITY) {
                        float z = 0.f;
#pragma unroll
                        for (int u = 0; u < kBatch; ++u) z += fast_exp2((v[u][hh] - bm) * kLog2e);
                        lse_combine(m[hh], l[hh], bm, z);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int hh = 0; hh < GM; ++hh) {
        if (hh < g) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float m2 = __shfl_xor_sync(0xffffffffu, m[hh], o);
                const float l2 = __shfl_xor_sync(0xffffffffu, l[hh], o);
                lse_combine(m[hh], l[hh], m2, l2);
            }
            if (lane == 0) {
                sh.red_m[warp][hh] = m[hh];
                sh.red_l[warp][hh] = l[hh];
            }
        }
    }
    __syncthreads();
    if (tid < g) {
        float mm = -INFINITY, ll = 0.f;
        for (int w = 0; w < kWarps; ++w) lse_combine(mm, ll, sh.red_m[w][tid], sh.red_l[w][tid]);
        sh.part_m[tid] = mm;
        sh.part_l[tid] = ll;
    }
    cluster_sync_all();
    if (tid < g) {
        float pm[CL], pl[CL];   // all remote loads in flight before any use
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) {
            pm[r] = ld_dsmem_f32(dsmem_addr(&sh.part_m[tid], r));
            pl[r] = ld_dsmem_f32(dsmem_addr(&sh.part_l[tid], r));
        }
        float mm = -INFINITY, ll = 0.f;
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) lse_combine(mm, ll, pm[r], pl[r]);
        sh.Lh[tid] = (ll > 0.f) ? mm + logf(ll) : -INFINITY;
    }
    __syncthreads();

    // 2. group-mean mass-share keys
    // (log2 domain: x = (s - L_h) log2 e; key = (max + log2 sum exp2(x - max)) ln 2 - ln g)
    const float log_g = logf(static_cast<float>(g));
    float Lr[GM];
#pragma unroll
    for (int hh = 0; hh < GM; ++hh) Lr[hh] = hh < g ? sh.Lh[hh] : 0.f;
    for (int jb = j0 + tid; jb < j1; jb += kBatch * kThreads) {
        float v[kBatch][GM];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int j = jb + u * kThreads;
#pragma unroll
            for (int hh = 0; hh < GM; ++hh)
                v[u][hh] = (hh < g && j < j1) ? srow[static_cast<int64_t>(hh) * a.max_pages + j] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int j = jb + u * kThreads;
            if (j >= j1) break;
            float mx = -INFINITY;
#pragma unroll
            for (int hh = 0; hh < GM; ++hh) {
                if (hh < g) {
                    v[u][hh] = (v[u][hh] - Lr[hh]) * kLog2e;
                    mx = fmaxf(mx, v[u][hh]);
                }
            }
            float key;
            if (mx == -INFINITY) {
                key = -INFINITY;
            } else {
                float z = 0.f;
#pragma unroll
                for (int hh = 0; hh < GM; ++hh)
                    if (hh < g) z += fast_exp2(v[u][hh] - mx);
                key = (mx + fast_log2(z)) * kLn2 - log_g;
            }
            keys[j - j0] = orderable_key(key);
            if (a.sel_keys) a.sel_keys[(static_cast<int64_t>(b) * a.hkv + kvh) * a.max_pages + j] = key;
        }
    }
    __syncthreads();

    int K = min(a.budget_pages, min(P, a.k_cap));
    K = max(K, 0);
    int32_t* out = a.selected + (static_cast<int64_t>(b) * a.hkv + kvh) * a.k_cap;
    if (rank == 0 && tid == 0) a.n_selected[b * a.hkv + kvh] = K;
    if (K == 0) {
        cluster_sync_all();
        return 0;
    }
    if (K == P) {
        for (int j = j0 + tid; j < j1; j += kThreads) out[j] = j;
        cluster_sync_all();
        return K;
    }

    // 3. radix select of the K-th largest key
    uint32_t prefix = 0;
    int remaining = K;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        uint32_t* hist = sh.hist[pass & 1];
        hist[tid] = 0;
        __syncthreads();
        // warp-aggregated: one shared atomic per distinct bin per warp step
        for (int i0 = 0; i0 < nloc; i0 += kThreads) {
            const int i = i0 + tid;
            bool take = false;
            uint32_t bin = 0xffffffffu;
            if (i < nloc) {
                const uint32_t key = keys[i];
                take = pass == 0 || (key >> (shift + 8)) == (prefix >> (shift + 8));
                if (take) bin = (key >> shift) & 255u;
            }
            const unsigned peers = __match_any_sync(0xffffffffu, bin);
            if (take && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
        }
        __syncthreads();
        cluster_sync_all();
        uint32_t hv[CL];
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) hv[r] = ld_dsmem_u32(dsmem_addr(&hist[tid], r));
        int total_d = 0;
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) total_d += static_cast<int>(hv[r]);
        // suffix count S[d] = sum_{d' >= d} total[d'] = grand - exclusive prefix(d)
        int grand;
        const int excl = block_exclusive_scan(total_d, sh.scan, grand);
        const int S = grand - excl;
        if (S >= remaining && S - total_d < remaining) {
            sh.digit = tid;
            sh.above = S - total_d;
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(sh.digit) << shift;
        remaining -= sh.above;
        __syncthreads();
    }
    const uint32_t T = prefix;   // the K-th largest key; `remaining` keys equal to T are kept

    // 4. ordered compaction: keys > T, then the first `remaining` keys == T
    const int per_t = (nloc + kThreads - 1) / kThreads;
    const int i0 = min(nloc, tid * per_t), i1 = min(nloc, i0 + per_t);
    int ngt = 0, neq = 0;
    for (int i = i0; i < i1; ++i) {
        ngt += keys[i] > T;
        neq += keys[i] == T;
    }
    int cta_gt, cta_eq;
    block_exclusive_scan(ngt, sh.scan, cta_gt);
    const int eq_pre = block_exclusive_scan(neq, sh.scan, cta_eq);
    if (tid == 0) {
        sh.cnt[0] = cta_gt;
        sh.cnt[1] = cta_eq;
    }
    cluster_sync_all();
    int base_gt = 0, base_eq = 0;
    {
        uint32_t cg[CL], ce[CL];
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) {
            cg[r] = r < rank ? ld_dsmem_u32(dsmem_addr(&sh.cnt[0], r)) : 0u;
            ce[r] = r < rank ? ld_dsmem_u32(dsmem_addr(&sh.cnt[1], r)) : 0u;
        }
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) {
            base_gt += static_cast<int>(cg[r]);
            base_eq += static_cast<int>(ce[r]);
        }
    }
    const int take_cta = max(0, min(remaining - base_eq, cta_eq));
    const int pos0 = base_gt + min(base_eq, remaining);
    const int take_thr = max(0, min(take_cta - eq_pre, neq));
    int dummy;
    const int sel_pre = block_exclusive_scan(ngt + take_thr, sh.scan, dummy);
    int pos = pos0 + sel_pre, eq_seen = eq_pre;
    for (int i = i0; i < i1; ++i) {
        const uint32_t key = keys[i];
        const bool keep = key > T || (key == T && eq_seen < take_cta);
        eq_seen += key == T;
        if (keep) {
            if (pos < K) out[pos] = j0 + i;   // pos < K always; the guard only bounds a logic error
            ++pos;
        }
    }
    cluster_sync_all();   // keep this CTA's counters alive for the others
    return K;
}

// ------------------------------------------------------------- attention
template <int CL, int GM>
__device__ void attend_pages(const SelectAttendArgs& a, int b, int kvh, uint32_t rank, int n_sel,
                             const int32_t* sel, bool sel_coherent, uint8_t* ring, SmallShared& sh) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gid = lane >> 2, t = lane & 3;
    const int g = a.hq / a.hkv;
    const int per = (n_sel + CL - 1) / CL;
    const int p0 = min(n_sel, static_cast<int>(rank) * per);
    const int p1 = min(n_sel, p0 + per);

    // query rows of the group (scaled by log2(e)/sqrt(d)) staged in shared memory as bf16
    // high and low parts; the MMA A fragments are read back with ldmatrix
    {
        const float c = kInvSqrtD * kLog2e;
        for (int idx = tid; idx < 16 * kD; idx += kThreads) {
            const int row = idx / kD, col = idx % kD;
            const float x = row < g ? a.q[(static_cast<int64_t>(b) * a.hq + kvh * g + row) * kD + col] * c : 0.f;
            const __nv_bfloat16 h = __float2bfloat16_rn(x);
            const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(h));
            sh.qs[0][row * kQRow + col] = __bfloat16_as_ushort(h);
            sh.qs[1][row * kQRow + col] = __bfloat16_as_ushort(lo);
        }
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
    bool failed = false, bad = false;
    const int64_t head_stride = static_cast<int64_t>(kPage) * kD;   // elements per (page, kv head)
    for (int p = p0 + warp; p < p1; p += kWarps) {
        int logical = sel_coherent ? __ldcg(sel + p) : sel[p];
        if (logical < 0 || logical >= a.max_pages) {
            bad = true;
            logical = 0;
        }
        int64_t phys = a.page_table[static_cast<int64_t>(b) * a.max_pages + logical];
        if (phys < 0 || phys >= a.num_phys) {
            bad = true;
            phys = 0;
        }
        const int64_t off = (phys * a.hkv + kvh) * head_stride;
        fence_proxy_async_smem();   // earlier generic reads of the slot before the async refill
        if (lane == 0) mbar_arrive_expect_tx(bar, 2 * kPage * kD * 2);
        __syncwarp();
        {
            const int row = lane & 15;
            const uint16_t* src = (lane < 16 ? a.k_cache : a.v_cache) + off + row * kD;
            bulk_g2s(slot + (lane < 16 ? 0 : kPage * kRowBytes) + row * kRowBytes, src, kD * 2, bar);
        }
        if (!mbar_wait_bounded(bar, phase, a.st.wait_limit_ns)) failed = true;
        phase ^= 1u;
        const uint8_t* kslot = slot;
        const uint8_t* vslot = slot + kPage * kRowBytes;

        // S = Q K^T: two n-tiles of 8 tokens
        float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            uint32_t kb[4], qh[4], ql[4];
            const int mat = lane >> 3;
            const int token = (mat >> 1) * 8 + (lane & 7);
            const int dim = 16 * s + (mat & 1) * 8;
            ldmatrix_x4(kb, kslot + token * kRowBytes + dim * 2);
            ldmatrix_x4(qh, &sh.qs[0][qrow * kQRow + 16 * s + qcol]);
            ldmatrix_x4(ql, &sh.qs[1][qrow * kQRow + 16 * s + qcol]);
            mma_bf16_16816(sacc[0], qh, kb[0], kb[1]);
            mma_bf16_16816(sacc[0], ql, kb[0], kb[1]);
            mma_bf16_16816(sacc[1], qh, kb[2], kb[3]);
            mma_bf16_16816(sacc[1], ql, kb[2], kb[3]);
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
            ldmatrix_x4_trans(vb, vslot + token * kRowBytes + dim * 2);
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
        if (tid < kD) {
            const float* c = sh.cpart + hh * kPartStride;
            float mr[CL], lr[CL], orr[CL];   // all remote loads in flight before any use
#pragma unroll
            for (uint32_t r = 0; r < CL; ++r) {
                mr[r] = ld_dsmem_f32(dsmem_addr(c, r));
                lr[r] = ld_dsmem_f32(dsmem_addr(c + 1, r));
                orr[r] = ld_dsmem_f32(dsmem_addr(c + 2 + tid, r));
            }
            float M = -INFINITY;
#pragma unroll
            for (uint32_t r = 0; r < CL; ++r) M = fmaxf(M, mr[r]);
            float L = 0.f, acc = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (uint32_t r = 0; r < CL; ++r) {
                    if (mr[r] == -INFINITY) continue;
                    const float f = fast_exp2(mr[r] - M);
                    L += lr[r] * f;
                    acc += orr[r] * f;
                }
            }
            const int64_t qh_idx = static_cast<int64_t>(b) * a.hq + kvh * g + hh;
            const float val = (L > 0.f) ? acc / L : 0.f;
            a.out[qh_idx * kD + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
            if (a.lse && tid == 0) a.lse[qh_idx] = (L > 0.f) ? (M + fast_log2(L)) * kLn2 : -INFINITY;
        }
    }
    cluster_sync_all();   // partials stay readable until every CTA is done
}

template <int CL, SAMode MODE, int GM>
__global__ void __launch_bounds__(kThreads, 2) select_attend_kernel(SelectAttendArgs a, int chunk) {
    extern __shared__ __align__(128) uint8_t smem[];
    SmallShared& sh = *reinterpret_cast<SmallShared*>(smem);
    uint8_t* big = smem + ((sizeof(SmallShared) + 127) / 128) * 128;
    const uint32_t rank = cluster_ctarank();
    const int seg = blockIdx.y;
    const int b = seg / a.hkv, kvh = seg % a.hkv;
    if (threadIdx.x < kWarps) mbar_init(&sh.bar[threadIdx.x], 1);
    fence_barrier_init();
    __syncthreads();

    if constexpr (MODE == SAMode::kSelect) {
        select_pages<CL, GM>(a, b, kvh, rank, chunk, reinterpret_cast<uint32_t*>(big), sh);
    } else if constexpr (MODE == SAMode::kAttend) {
        const int n = max(0, min(a.n_selected[b * a.hkv + kvh], a.k_cap));
        attend_pages<CL, GM>(a, b, kvh, rank, n, a.selected + (static_cast<int64_t>(b) * a.hkv + kvh) * a.k_cap, false,
                         big, sh);
    } else {
        const int n = select_pages<CL, GM>(a, b, kvh, rank, chunk, reinterpret_cast<uint32_t*>(big), sh);
        // the selection went to global memory; make it visible to the cluster's CTAs
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
        cluster_sync_all();
        attend_pages<CL, GM>(a, b, kvh, rank, n, a.selected + (static_cast<int64_t>(b) * a.hkv + kvh) * a.k_cap, true,
                         big, sh);
    }
}

int chunk_of(int max_pages, int cluster) {
    int c = (max_pages + cluster - 1) / cluster;
    return (c + 7) & ~7;   // whole 8-page blocks (the LSE partials' granularity)
}

template <int CL, SAMode MODE, int GM>
cudaError_t launch_t(const SelectAttendArgs& a, cudaStream_t stream) {
    const int chunk = chunk_of(a.max_pages, CL);
    const size_t smem = select_attend_smem_bytes(a.max_pages, CL, MODE);
    auto kern = select_attend_kernel<CL, MODE, GM>;
    cudaError_t e = ensure_kernel_attrs<select_attend_kernel<CL, MODE, GM>>(static_cast<int>(smem), CL > 8);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL, a.batch * a.hkv, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
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
    const size_t small = ((sizeof(SmallShared) + 127) / 128) * 128;
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
