// score.cu - LOCKS page scoring from the resident summaries alone.
//
// Computes, for every (sequence b, query head h, logical page j), the score of
// the LOCKS post ("How LOCKS works") and of the gist.science summary, 2.2:
//     s = log sum_{i<16} exp[(q . mu + (V^T q) . c_i) / sqrt(128)]
// from the int8 centroid, int4 rank-8 basis and int8 coefficients of unit
// (page_table[b][j], h / g). No key or value is read.
//
// Design (HBM-bound stream of 776 B per unit):
//  * persistent CTAs, one per SM; a producer warp streams the summaries of
//    64 units per stage (all kv heads of 64/Hkv consecutive logical pages)
//    into a 4-stage shared-memory ring with bulk async copies (TMA engine,
//    L2 evict-first) plus 8-byte LDGSTS for the fp16 scales, completion on
//    mbarriers; a group of 8 consumer warps takes a stage, each warp one kv
//    head and 8 pages; two groups work on alternate stages, or, when the GQA
//    group is > 8, both on every stage with 8 of its query heads each.
//  * V^T q and mu . q run on the tensor cores (mma.sync m16n8k16, f16 in,
//    fp32 accumulate): A = the codes plus their offset (int4 + 8, int8 + 128),
//    read directly as f16 subnormals u * 2^-24 by masking (no conversion
//    arithmetic; codes from the upper nibble come out as 16u and meet query
//    rows pre-divided by 16); B = the query split into an f16 high and low
//    part (about 22 significant bits), so the products match fp32 arithmetic
//    to well below the 1e-3 score tolerance. The offset is taken out with the
//    per-head sum of the query, and the query is pre-scaled by a power of two
//    per head so the f16 parts never overflow.
//  * the per-token reconstruction (V^T q) . c_i is a second MMA (m16n8k8)
//    whose B operand is the first MMA's accumulator, split hi/lo and
//    transposed in registers with movmatrix; the page LSE is a 3-step
//    butterfly over the 8 lanes that hold the 16 token logits.
#include "locks_internal.h"

namespace locks {
namespace {

constexpr int kGroupWarps = 8;          // consumer warps per stage
constexpr int kStages = 4;
constexpr int kStMu = 0;
constexpr int kStBasis = kStMu + kStageUnits * 128;
constexpr int kStCoef = kStBasis + kStageUnits * 512;
constexpr int kStScales = kStCoef + kStageUnits * 128;
constexpr int kStageBytes = kStScales + kStageUnits * 8;   // 49,664 B
constexpr int kSmemBytes = kStages * kStageBytes + 2 * kStages * 8;
// Two consumer groups take alternate stages; with an even ring each group owns
// its own slots, so its parity waits can never see a slot's phase from two fills
// earlier (with an odd ring a group that runs ahead would).
static_assert(kStages % 2 == 0, "the ring must hold an even number of stages");

__device__ __forceinline__ float pow2i(int e) {  // 2^e for |e| <= 126
    return __int_as_float((127 + e) << 23);
}

// Two consumer groups for NT <= 2. HS = 1: they take alternate stages. HS = 2
// (GQA group 16): both take every stage, group i computing heads 8i .. 8i + 7.
template <int NT>
struct Shape {
    static constexpr int kGroups = NT <= 2 ? 2 : 1;
    static constexpr int kConsumerWarps = kGroups * kGroupWarps;
    static constexpr int kThreads = (kConsumerWarps + 1) * 32;
};

template <int HKV, int HS>
constexpr int kSlotWarps = slot_warps(HKV, HS == 2 ? 16 : 8);

template <int HKV, int NT, int HS>
__global__ void __launch_bounds__(Shape<NT>::kThreads, 1) score_kernel(ScoreArgs a, int nchunks, int total_items) {
    constexpr int NP = kStageUnits / HKV;   // pages per stage
    constexpr int kGroups = Shape<NT>::kGroups;
    constexpr int kConsumerWarps = Shape<NT>::kConsumerWarps;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 33);              // 1 expect_tx arrive + 32 LDGSTS arrives
            mbar_init(&empty[s], HS == 2 ? kConsumerWarps : kGroupWarps);
        }
        fence_barrier_init();
    }
    // launched with programmatic stream serialization: the set-up above overlaps
    // the end of the previous kernel; every global access follows
    grid_dependency_wait();
    // The grid is persistent (at most one CTA per SM), so a dependent kernel (the
    // selection) only takes SMs this kernel has left; it may be scheduled as soon
    // as they free up. The trigger follows the wait, so a dependent that reads
    // inputs before its own wait sees everything the kernels before this one wrote.
    allow_dependent_launch();
    __syncthreads();

    const int per = (total_items + gridDim.x - 1) / gridDim.x;
    const int it0 = blockIdx.x * per;
    const int it1 = min(total_items, it0 + per);
    bool failed = false;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer
        // Per stage: each lane owns one page of a 32-page window; pages whose
        // physical ids are consecutive form runs, and the first lane of a run
        // issues one bulk copy per array for the whole run. The fp16 scales
        // go by LDGSTS, at most one 16-byte (or 8-byte for Hkv = 1) copy per
        // lane. The page-table entries of the next stage are loaded before
        // waiting for a free slot.
        const uint64_t pol = policy_evict_first();
        uint32_t k = 0;
        bool bad = false;
        int cur_b = -1, cur_P = 0;
        // page-table prefetch for item `it` (entries of this lane's pages)
        auto load_phys = [&](int it, int w, int nvalid) -> int64_t {
            const int b = it / nchunks, page0 = (it % nchunks) * NP;
            const int pg = w * 32 + lane;
            return pg < nvalid ? static_cast<int64_t>(a.page_table[static_cast<int64_t>(b) * a.max_pages + page0 + pg])
                               : int64_t(-1);
        };
        constexpr int kWindows = (NP + 31) / 32;
        for (int it = it0; it < it1; ++it) {
            const int b = it / nchunks, page0 = (it % nchunks) * NP;
            if (b != cur_b) {
                cur_b = b;
                cur_P = min(a.seq_pages[b], a.max_pages);
            }
            const int nvalid = min(NP, cur_P - page0);
            if (nvalid <= 0) continue;
            int64_t ph[kWindows];
#pragma unroll
            for (int w = 0; w < kWindows; ++w) ph[w] = load_phys(it, w, nvalid);
            const int s = k % kStages;
            if (!mbar_wait_bounded(&empty[s], ((k / kStages) & 1) ^ 1, a.st.wait_limit_ns)) failed = true;
            uint8_t* stg = smem + s * kStageBytes;
            if (lane == 0) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(nvalid * HKV * 768));
            __syncwarp();
#pragma unroll
            for (int w = 0; w < kWindows; ++w) {
                const int pg = w * 32 + lane;
                const int wpages = min(32, nvalid - w * 32);
                if (wpages <= 0) break;
                int64_t phys = ph[w];
                const bool valid = pg < nvalid;
                if (valid && (phys < 0 || phys >= a.num_phys)) {
                    bad = true;
                    phys = 0;
                }
                const int64_t prev = __shfl_up_sync(0xffffffffu, phys, 1);
                const bool start = valid && (lane == 0 || phys != prev + 1);
                const unsigned starts = __ballot_sync(0xffffffffu, start);
                if (start) {
                    const unsigned later = starts & ~((2u << lane) - 1u);   // run starts after this lane
                    const int end = later ? __ffs(later) - 1 : wpages;
                    const uint32_t n = static_cast<uint32_t>((end - lane) * HKV);
                    const int64_t u0 = phys * HKV;
                    bulk_g2s_hint(stg + kStMu + pg * HKV * 128, a.mu + u0 * 128, n * 128, &full[s], pol);
                    bulk_g2s_hint(stg + kStBasis + pg * HKV * 512, a.basis + u0 * 512, n * 512, &full[s], pol);
                    bulk_g2s_hint(stg + kStCoef + pg * HKV * 128, a.coef + u0 * 128, n * 128, &full[s], pol);
                }
                // scales: HKV even -> 16-byte pieces of two units, else one 8-byte unit per lane
                constexpr int kUnitsPerCopy = (HKV % 2 == 0) ? 2 : 1;
                const int pieces = wpages * HKV / kUnitsPerCopy;
                if (lane < pieces) {
                    const int unit_in_window = lane * kUnitsPerCopy;
                    const int wp = unit_in_window / HKV, h = unit_in_window % HKV;
                    const int64_t pphys = __shfl_sync(__activemask(), phys, wp);
                    uint8_t* dst = stg + kStScales + ((w * 32 + wp) * HKV + h) * 8;
                    const uint16_t* src = a.scales + (pphys * HKV + h) * 4;
                    if (kUnitsPerCopy == 2)
                        cp_async_16(dst, src);
                    else
                        cp_async_8(dst, src);
                }
            }
            cp_async_arrive_noinc(&full[s]);
            ++k;
        }
        if (bad) report_error(a.st, LOCKS_ERR_BAD_INDEX);
    } else {
        // ------------------------------------------------------ consumers
        const int group = warp / kGroupWarps, gw = warp % kGroupWarps;
        const int kvh = gw % HKV, blk = gw / HKV;
        const int gid = lane >> 2, t = lane & 3;
        const int g = a.hq / HKV;
        const int hoff = HS == 2 ? group * 4 * NT : 0;   // first head (within the kv group) of this group
        uint32_t bq[8][NT][2];
        float qsum[NT];    // sum of that head's pre-scaled query q' (code-offset correction)
        float qsc[NT];     // 2^e of the output head (4 nt + t) of this thread
        int cur_b = -1, q_b = -1, cur_P = 0;
        // this warp's (max, sum exp) of the scores of its heads over the units it scored of
        // sequence cur_b (lanes 0-3: head hoff + 4 nt + t), written to its slot when the
        // sequence changes and at the end (every sequence of this CTA's range gets a slot)
        float run_m[NT], run_l[NT];
        const int wslot = (HS == 1 ? group * (kGroupWarps / HKV) : 0) + blk;
        const int nslots = gridDim.x * kSlotWarps<HKV, HS>;
        auto flush_partials = [&](int pb) {
            if (a.lse_partials && pb >= 0 && gid == 0) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int hh = hoff + 4 * nt + t;
                    if (hh < g)
                        reinterpret_cast<float2*>(a.lse_partials)
                            [(static_cast<int64_t>(pb) * a.hq + kvh * g + hh) * nslots +
                             blockIdx.x * kSlotWarps<HKV, HS> + wslot] = make_float2(run_m[nt], run_l[nt]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                run_m[nt] = -INFINITY;
                run_l[nt] = 0.f;
            }
        };
        flush_partials(-1);
        uint32_t k = 0;
        for (int it = it0; it < it1; ++it) {
            const int b = it / nchunks, page0 = (it % nchunks) * NP;
            if (b != cur_b) {
                flush_partials(cur_b);
                cur_b = b;
                cur_P = min(a.seq_pages[b], a.max_pages);
            }
            const int nvalid = min(NP, cur_P - page0);
            if (nvalid <= 0) continue;
            if (HS == 1 && static_cast<int>(k % kGroups) != group) {   // the other group's stage
                ++k;
                continue;
            }
            if (b != q_b) {
                // Per-head power-of-two pre-scale: max |q'| < 1.
                int eB[NT], eO[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    eB[nt] = eO[nt] = 0;
                    qsum[nt] = 0.f;
                }
#pragma unroll
                for (int hh = 0; hh < 4 * NT; ++hh) {
                    float mx = 0.f, sm = 0.f;
                    if (hoff + hh < g) {
                        const float4 v = *reinterpret_cast<const float4*>(
                            a.q + (static_cast<int64_t>(b) * a.hq + kvh * g + hoff + hh) * kD + lane * 4);
                        mx = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
                        sm = (v.x + v.y) + (v.z + v.w);
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                        sm += __shfl_xor_sync(0xffffffffu, sm, o);
                    }
                    int e = 0;
                    if (mx > 0.f && mx < INFINITY) e = ilogbf(mx) + 1;
                    e = max(-100, min(100, e));
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (((nt * 8 + gid) >> 1) == hh) eB[nt] = e;
                        if (4 * nt + t == hh) {
                            eO[nt] = e;
                            qsum[nt] = sm * pow2i(-e);
                        }
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    qsc[nt] = pow2i(eO[nt]);
                    const int col = nt * 8 + gid, hh = col >> 1, hl = col & 1;
                    const float inv = pow2i(-eB[nt]);
                    const float* qrow = a.q + (static_cast<int64_t>(b) * a.hq + kvh * g + hoff + hh) * kD;
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        uint32_t r0 = 0, r1 = 0;
                        if (hoff + hh < g) {
                            const float2 x01 = *reinterpret_cast<const float2*>(qrow + 16 * s + 2 * t);
                            const float2 x89 = *reinterpret_cast<const float2*>(qrow + 16 * s + 2 * t + 8);
                            const uint32_t p0 = split_f16_hilo(x01.x * inv), p1 = split_f16_hilo(x01.y * inv);
                            // rows d + 8, d + 9 divided by 16: they meet the 16x-scaled codes
                            const uint32_t p8 = split_f16_hilo(x89.x * inv * 0.0625f),
                                           p9 = split_f16_hilo(x89.y * inv * 0.0625f);
                            // hl = 0: high parts (low halves), hl = 1: low parts (high halves)
                            r0 = hl ? __byte_perm(p0, p1, 0x7632) : __byte_perm(p0, p1, 0x5410);
                            r1 = hl ? __byte_perm(p8, p9, 0x7632) : __byte_perm(p8, p9, 0x5410);
                        }
                        bq[s][nt][0] = r0;
                        bq[s][nt][1] = r1;
                    }
                }
                q_b = b;
            }
            const int s = k % kStages;
            if (!mbar_wait_bounded(&full[s], (k / kStages) & 1, a.st.wait_limit_ns)) failed = true;
            const uint8_t* stg = smem + s * kStageBytes;
            const int nv = min(8, nvalid - 8 * blk);
            if (nv > 0) {
                const int ubase = (8 * blk) * HKV + kvh;   // stage unit index of the warp's unit 0
                // scales of unit `lane` (lanes 0..7); zero for units past the end. The token
                // logits of a unit carry s_V s_C / sqrt(d) (log2 domain): one factor per unit.
                float s_mu = 0.f, s_vc = 0.f;
                if (lane < nv) {
                    const uint2 sc = *reinterpret_cast<const uint2*>(stg + kStScales + (ubase + lane * HKV) * 8);
                    s_mu = __half2float(__ushort_as_half(static_cast<unsigned short>(sc.x & 0xffffu)));
                    s_vc = __half2float(__ushort_as_half(static_cast<unsigned short>(sc.x >> 16))) *
                           __half2float(__ushort_as_half(static_cast<unsigned short>(sc.y & 0xffffu))) *
                           (kInvSqrtD * kLog2e);
                }
                const float smu_row = __shfl_sync(0xffffffffu, s_mu, gid);
                // Per-token logits (log2 domain) of units i and i + 4: MMA1 gives V^T q for both
                // (rows 0-7 and 8-15), MMA2 reconstructs the 16 tokens of each; `use(u, nt, x0, x1)`
                // gets this lane's two tokens (gid, gid + 8) of unit u for head 4 nt + t.
                auto pair_logits = [&](int i, auto&& use) {
                    const uint4 va = *reinterpret_cast<const uint4*>(stg + kStBasis + (ubase + i * HKV) * 512 + lane * 16);
                    const uint4 vb =
                        *reinterpret_cast<const uint4*>(stg + kStBasis + (ubase + (i + 4) * HKV) * 512 + lane * 16);
                    const uint32_t wa[4] = {va.x, va.y, va.z, va.w};
                    const uint32_t wb[4] = {vb.x, vb.y, vb.z, vb.w};
                    float acc[NT][4];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t ra[4], rb[4];
                        int4x8_to_f16x2_sub(wa[j], ra);
                        int4x8_to_f16x2_sub(wb[j], rb);
                        const uint32_t a0[4] = {ra[0], rb[0], ra[1], rb[1]};   // k-step 2j
                        const uint32_t a1[4] = {ra[2], rb[2], ra[3], rb[3]};   // k-step 2j + 1
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma_f16_16816(acc[nt], a0, bq[2 * j][nt][0], bq[2 * j][nt][1]);
                            mma_f16_16816(acc[nt], a1, bq[2 * j + 1][nt][0], bq[2 * j + 1][nt][1]);
                        }
                    }
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int u = i + 4 * half;
                        const float fvc = __shfl_sync(0xffffffffu, s_vc, u);
                        const uint32_t cw =
                            *reinterpret_cast<const uint32_t*>(stg + kStCoef + (ubase + u * HKV) * 128 + lane * 4);
                        uint32_t ca0, ca1;
                        int8x4_to_f16x2(cw, ca0, ca1);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            // W = sum_k (x_k + 8) q'_k - 8 sum_k q'_k (|W| < 3000); the MMA sum carries 2^-24
                            const float raw = half == 0 ? acc[nt][0] + acc[nt][1] : acc[nt][2] + acc[nt][3];
                            const float w = fmaf(raw, 16777216.f, -8.f * qsum[nt]);
                            const uint32_t bw = movmatrix_trans(split_f16_hilo(w));
                            float d2[4] = {0.f, 0.f, 0.f, 0.f};
                            mma_f16_1688(d2, ca0, ca1, bw);
                            const float f = fvc * qsc[nt];
                            use(u, nt, (d2[0] + d2[1]) * f, (d2[2] + d2[3]) * f);
                        }
                    }
                };
                // log2-sum-exp2 over each unit's 16 tokens (8 lanes x 2), taken unshifted: every
                // lane keeps its partial sum for all 8 units, and a reduce-scatter over the 8 lanes
                // of its column (lane bits 2-4 = gid) leaves unit gid's total in lane gid.
                // The first level (lane bit 4) is taken as soon as units i and i + 4 are done.
                const bool b2 = (gid & 4) != 0, b1 = (gid & 2) != 0, b0 = (gid & 1) != 0;
                float y4[NT][4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float zlo[NT], zhi[NT];   // this lane's partial sums of units i and i + 4
                    pair_logits(i, [&](int u, int nt, float x0, float x1) {
                        const float z = fast_exp2(x0) + fast_exp2(x1);
                        if (u == i)
                            zlo[nt] = z;
                        else
                            zhi[nt] = z;
                    });
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        y4[nt][i] = (b2 ? zhi[nt] : zlo[nt]) + __shfl_xor_sync(0xffffffffu, b2 ? zlo[nt] : zhi[nt], 16);
                }
                float lse[NT];
                bool out_of_range = false;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float y2[2];
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        const float send = b1 ? y4[nt][q2] : y4[nt][q2 + 2];
                        y2[q2] = (b1 ? y4[nt][q2 + 2] : y4[nt][q2]) + __shfl_xor_sync(0xffffffffu, send, 8);
                    }
                    const float z = (b0 ? y2[1] : y2[0]) + __shfl_xor_sync(0xffffffffu, b0 ? y2[0] : y2[1], 4);
                    out_of_range |= !(z >= 7.9e-31f && z <= 1.26e30f);
                    lse[nt] = fast_log2(z) * kLn2;
                }
                if (__any_sync(0xffffffffu, out_of_range)) {
                    // some unit's sum left [2^-100, 2^100]: redo every unit with its max factored
                    // out (exact either way up to exp2/log2 rounding)
#pragma unroll 1
                    for (int i = 0; i < 4; ++i)
                        pair_logits(i, [&](int u, int nt, float x0, float x1) {
                            float m = fmaxf(x0, x1);
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                            float z = fast_exp2(x0 - m) + fast_exp2(x1 - m);
                            z += __shfl_xor_sync(0xffffffffu, z, 4);
                            z += __shfl_xor_sync(0xffffffffu, z, 8);
                            z += __shfl_xor_sync(0xffffffffu, z, 16);
                            if (gid == u) lse[nt] = (m + fast_log2(z)) * kLn2;
                        });
                }
                // centroid term: rows = the warp's 8 units, K = 128 dims (taken after the
                // token logits so that its accumulators are not live across them)
                float accmu[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) accmu[nt][0] = accmu[nt][1] = accmu[nt][2] = accmu[nt][3] = 0.f;
                {
                    const uint8_t* mrow = stg + kStMu + (ubase + gid * HKV) * 128 + t * 32;
                    const uint4 m0 = *reinterpret_cast<const uint4*>(mrow);
                    const uint4 m1 = *reinterpret_cast<const uint4*>(mrow + 16);
                    const uint32_t mw[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        uint32_t lo, hi;
                        int8x4_to_f16x2_sub(mw[ks], lo, hi);
                        const uint32_t af[4] = {lo, 0u, hi, 0u};
                        // B rows d + 8, d + 9 back to full size (x16) for the int8 codes
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma_f16_16816(accmu[nt], af, bq[ks][nt][0], hmul2_u32(bq[ks][nt][1], 0x4c004c00u));
                    }
                }
                // score of unit gid, head 4 nt + t: centroid term + token LSE
                float score_out[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float a_raw = fmaf(accmu[nt][0] + accmu[nt][1], 16777216.f, -128.f * qsum[nt]);
                    score_out[nt] = a_raw * smu_row * qsc[nt] * kInvSqrtD + lse[nt];
                }
                if (a.lse_partials) {
                    // (max, sum exp) of this warp's 8 pages for each head, folded into the
                    // warp's running partial of the sequence
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const float sv = gid < nv ? score_out[nt] : -INFINITY;
                        float m = sv;
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                        float z = (sv == -INFINITY || sv != sv) ? 0.f : fast_exp2((sv - m) * kLog2e);
                        z += __shfl_xor_sync(0xffffffffu, z, 4);
                        z += __shfl_xor_sync(0xffffffffu, z, 8);
                        z += __shfl_xor_sync(0xffffffffu, z, 16);
                        if (z > 0.f) {
                            const float M = fmaxf(run_m[nt], m);
                            run_l[nt] = run_l[nt] * fast_exp2((run_m[nt] - M) * kLog2e) + z * fast_exp2((m - M) * kLog2e);
                            run_m[nt] = M;
                        }
                    }
                }
                if (gid < nv) {
                    const int page = page0 + 8 * blk + gid;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int hh = hoff + 4 * nt + t;
                        if (hh < g)
                            a.scores[(static_cast<int64_t>(b) * a.hq + kvh * g + hh) * a.max_pages + page] =
                                score_out[nt];
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            ++k;
        }
        flush_partials(cur_b);
    }
    if (failed) report_error(a.st, LOCKS_ERR_TIMEOUT);
}

template <int HKV, int NT, int HS>
cudaError_t launch_t(const ScoreArgs& a, int num_sms, cudaStream_t stream) {
    constexpr int NP = kStageUnits / HKV;
    const int nchunks = (a.max_pages + NP - 1) / NP;
    const int total = a.batch * nchunks;
    if (total == 0) return cudaSuccess;
    cudaError_t e = ensure_kernel_attrs<score_kernel<HKV, NT, HS>>(kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(score_grid(total, num_sms), 1, 1);
    cfg.blockDim = dim3(Shape<NT>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, score_kernel<HKV, NT, HS>, a, nchunks, total);
}

template <int HKV>
cudaError_t launch_h(const ScoreArgs& a, int num_sms, cudaStream_t stream) {
    const int g = a.hq / a.hkv;
    if (g <= 4) return launch_t<HKV, 1, 1>(a, num_sms, stream);
    if (g <= 8) return launch_t<HKV, 2, 1>(a, num_sms, stream);
    return launch_t<HKV, 2, 2>(a, num_sms, stream);   // g = 9..16: the two groups split the heads
}

}  // namespace

cudaError_t launch_score(const ScoreArgs& a, int num_sms, cudaStream_t stream) {
    switch (a.hkv) {
        case 1: return launch_h<1>(a, num_sms, stream);
        case 2: return launch_h<2>(a, num_sms, stream);
        case 4: return launch_h<4>(a, num_sms, stream);
        case 8: return launch_h<8>(a, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace locks
