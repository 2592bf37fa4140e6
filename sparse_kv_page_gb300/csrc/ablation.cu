// ablation.cu - the selector ablations on the LOCKS pages' synthetic carriers
// (off the decode path):
//   * exact page scores, the selector that reads every key (gist.science Korean
//     summary, sections 1 and 3: the exact, read-all-keys selection LOCKS is
//     measured against): s = log sum_i exp(q . k_i / sqrt(d));
//   * page-local summaries of rank 1..15 with the centroid, basis and
//     coefficients quantised to 2..8 bits or left unquantised, built from the
//     keys and scored in one pass (LOCKS post, "Caveats": the int4 summary
//     loses a few recall points, int2 collapses; Theorem 1 covers the
//     unquantised rank-r summary);
//   * the shared basis of a sequence's keys (the top eigenvectors of the
//     uncentred second moment sum_t k_t k_t^T) and the queries projected on it,
//     so that the shared-basis page score log sum_i exp((W W^T q) . k_i / sqrt(d))
//     runs through the exact scorer (LOCKS post, "Why shared-basis sparse
//     attention is structurally broken"; Proposition 1).
//
// GPU mapping. Exact and variant scores: one warp per (page, kv head) unit,
// 4 warps per CTA, one CTA per (sequence, kv head) and run of 64 pages, the
// group's queries staged in shared memory once per CTA. The exact scorer runs
// its 16 x 128 by 128 x g contraction on the tensor cores (mma.sync bf16). The variant kernel
// keeps the unit's centred keys, Gram matrix, eigenvectors and summary in the
// warp's own shared-memory slice and runs the cyclic Jacobi method in
// round-robin order (8 disjoint rotations per round, 15 rounds per sweep).
// Shared basis: a second-moment kernel (8 x 8 register blocks per thread,
// fp32, one atomic add per entry per CTA) and one CTA per (sequence, kv head)
// running the parallel Jacobi method on the 128 x 128 moment in shared memory
// (64 disjoint rotations per round, 127 rounds per sweep).
#include <cuda_fp16.h>

#include "locks_internal.h"

namespace locks {
namespace {

constexpr int kAbWarps = 4;          // warps per CTA (exact, variant)
constexpr int kAbPagesPerCta = 64;   // pages per CTA (exact, variant)
constexpr int kMomentPages = 128;    // pages per CTA (second moment)
constexpr int kEigThreads = 512;
constexpr int kEigN = 128;
constexpr int kEigStride = 129;
constexpr int kSmallSweeps = 12;     // 16 x 16 Jacobi
constexpr int kLargeSweeps = 30;     // 128 x 128 Jacobi
// A sweep that shrinks the off-diagonal energy by less than 10% has reached the
// fp32 rounding floor (Jacobi converges quadratically until then): stop there.
constexpr float kStallRatio = 0.9f;

__device__ __forceinline__ int seq_len(const AblationArgs& a, int b) {
    const int p = a.seq_pages[b];
    return p < 0 ? 0 : (p > a.max_pages ? a.max_pages : p);
}

// Physical page of logical page j of sequence b; an out-of-range table entry
// records LOCKS_ERR_BAD_INDEX and reads physical page 0 instead.
__device__ __forceinline__ int64_t phys_page(const AblationArgs& a, int b, int j) {
    const int32_t p = a.page_table[static_cast<int64_t>(b) * a.max_pages + j];
    if (p < 0 || p >= a.num_phys) {
        report_error(a.st, LOCKS_ERR_BAD_INDEX);
        return 0;
    }
    return p;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 w, float* out) {
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        out[2 * e] = __uint_as_float(x[e] << 16);
        out[2 * e + 1] = __uint_as_float(x[e] & 0xffff0000u);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// log sum_i exp(t_i) over the 16 lanes of each half-warp, t in log2 units;
// the result (natural log) is returned in every lane.
__device__ __forceinline__ float lse16_log2(float t) {
    float m = t;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = fast_exp2(t - m);
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    return (m + fast_log2(z)) * kLn2;
}

// Symmetric Schur rotation (c, s) that zeroes a_pq (Golub & Van Loan 8.5).
__device__ __forceinline__ float2 schur_rotation(float app, float aqq, float apq) {
    if (apq == 0.f) return make_float2(1.f, 0.f);
    const float tau = (aqq - app) / (2.f * apq);
    const float t = (tau >= 0.f ? 1.f : -1.f) / (fabsf(tau) + sqrtf(1.f + tau * tau));
    const float c = 1.f / sqrtf(1.f + t * t);
    return make_float2(c, t * c);
}

// Stages the g queries of (b, kv head) in shared memory.
__device__ __forceinline__ void stage_queries(const AblationArgs& a, int b, int kvh, float* qs) {
    const int g = a.hq / a.hkv;
    const float* src = a.q + (static_cast<int64_t>(b) * a.hq + kvh * g) * kD;
    for (int i = threadIdx.x; i < g * kD; i += blockDim.x) qs[i] = src[i];
}

// ------------------------------------------------------------ exact scores

constexpr int kExSlot = kPage * kD * 2;   // one unit's 16 keys, 4 KiB

// Byte offset of 16-byte chunk c (0..15) of token row r in a key slot: the chunk
// index is XORed with the row's low bits so that ldmatrix's 8 rows of one
// column block fall in 8 different bank groups.
__device__ __forceinline__ int ex_swz(int r, int c) { return r * 256 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_older() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// x = hi + mid + lo with each part a bf16 value (about 24 significant bits in all).
__device__ __forceinline__ void split3_bf16(float x, float& hi, float& mid, float& lo) {
    hi = __bfloat162float(__float2bfloat16_rn(x));
    const float r = x - hi;
    mid = __bfloat162float(__float2bfloat16_rn(r));
    lo = __bfloat162float(__float2bfloat16_rn(r - mid));
}

// Grid (B * Hkv, runs of 64 pages); HT = ceil(g / 8) tiles of 8 heads. One warp per
// unit: the unit's keys (exactly bf16) are copied into the warp's slot (cp.async,
// double-buffered: the next unit's copy runs while this one is scored) and are the
// A operand of mma.sync m16n8k16 bf16 (rows = the 16 tokens, k = dims, through
// ldmatrix); B = the queries of 8 heads, each split into three bf16 parts that are
// separate MMAs, summed in fp32, so the logits carry fp32-accurate products. The
// page LSE is taken on the accumulator layout (each lane holds two heads' logits
// of tokens gid and gid + 8).
template <int HT>
__global__ void __launch_bounds__(kAbWarps * 32) exact_kernel(AblationArgs a) {
    extern __shared__ __align__(128) unsigned char ex_smem[];
    const int g = a.hq / a.hkv;
    const int b = blockIdx.x / a.hkv, kvh = blockIdx.x % a.hkv;
    const int P = seq_len(a, b);
    const int j0 = blockIdx.y * kAbPagesPerCta;
    if (j0 >= P) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, t = lane & 3;
    uint8_t* slots = ex_smem + warp * 2 * kExSlot;
    float* qs = reinterpret_cast<float*>(ex_smem + kAbWarps * 2 * kExSlot);
    stage_queries(a, b, kvh, qs);
    __syncthreads();
    // B fragments: head ht * 8 + gid, dims 16 ks + 2t (+1) and 16 ks + 2t + 8 (+9)
    uint32_t bq[HT][3][8][2];
#pragma unroll
    for (int ht = 0; ht < HT; ++ht) {
        const int head = ht * 8 + gid;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int d = 16 * ks + 2 * t + 8 * half;
                const float x0 = head < g ? qs[head * kD + d] : 0.f;
                const float x1 = head < g ? qs[head * kD + d + 1] : 0.f;
                float h0, m0, l0, h1, m1, l1;
                split3_bf16(x0, h0, m0, l0);
                split3_bf16(x1, h1, m1, l1);
                bq[ht][0][ks][half] = pack_bf16x2(h0, h1);
                bq[ht][1][ks][half] = pack_bf16x2(m0, m1);
                bq[ht][2][ks][half] = pack_bf16x2(l0, l1);
            }
    }
    const int j1 = min(P, j0 + kAbPagesPerCta);
    auto issue = [&](int j, int slot) {
        const int64_t phys = phys_page(a, b, j);
        const uint8_t* src = reinterpret_cast<const uint8_t*>(a.k_cache + (phys * a.hkv + kvh) * kPage * kD);
        uint8_t* dst = slots + slot * kExSlot;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = lane + 32 * i;   // 16-byte chunk c of the unit: token c / 16, chunk c % 16
            cp_async_16(dst + ex_swz(c >> 4, c & 15), src + c * 16);
        }
    };
    if (j0 + warp < j1) issue(j0 + warp, 0);
    cp_async_commit();
    int slot = 0;
    for (int j = j0 + warp; j < j1; j += kAbWarps) {
        if (j + kAbWarps < j1) issue(j + kAbWarps, slot ^ 1);
        cp_async_commit();
        cp_async_wait_older();   // this unit's copy has landed
        __syncwarp();
        const uint8_t* kb = slots + slot * kExSlot;
        float acc[HT][3][4];
#pragma unroll
        for (int ht = 0; ht < HT; ++ht)
#pragma unroll
            for (int sp = 0; sp < 3; ++sp) acc[ht][sp][0] = acc[ht][sp][1] = acc[ht][sp][2] = acc[ht][sp][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t af[4];   // rows 0-7 / 8-15 x dims 16 ks .. +7 / 16 ks + 8 .. +15
            ldmatrix_x4(af, kb + ex_swz((lane & 7) + 8 * ((lane >> 3) & 1), 2 * ks + (lane >> 4)));
#pragma unroll
            for (int ht = 0; ht < HT; ++ht)
#pragma unroll
                for (int sp = 0; sp < 3; ++sp) mma_bf16_16816(acc[ht][sp], af, bq[ht][sp][ks][0], bq[ht][sp][ks][1]);
        }
#pragma unroll
        for (int ht = 0; ht < HT; ++ht) {
#pragma unroll
            for (int col = 0; col < 2; ++col) {   // head ht * 8 + 2t + col: tokens gid (e = col), gid + 8 (e = col + 2)
                const float xa = ((acc[ht][0][col] + acc[ht][1][col]) + acc[ht][2][col]) * (kInvSqrtD * kLog2e);
                const float xb =
                    ((acc[ht][0][col + 2] + acc[ht][1][col + 2]) + acc[ht][2][col + 2]) * (kInvSqrtD * kLog2e);
                float m = fmaxf(xa, xb);
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                float z = fast_exp2(xa - m) + fast_exp2(xb - m);
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
                const int head = ht * 8 + 2 * t + col;
                if (gid == 0 && head < g)
                    a.scores[(static_cast<int64_t>(b) * a.hq + kvh * g + head) * a.max_pages + j] =
                        (m + fast_log2(z)) * kLn2;
            }
        }
        __syncwarp();   // every lane is done with the slot before it is refilled
        slot ^= 1;
    }
}

// ------------------------------------------------------- query projection

// One CTA of 128 threads per (b, q head): p_r = W_r . q, then q~ = sum_r p_r W_r.
__global__ void __launch_bounds__(128) project_kernel(AblationArgs a) {
    __shared__ float qv[kD], p[kD];
    const int b = blockIdx.x / a.hq, h = blockIdx.x % a.hq;
    const int g = a.hq / a.hkv, kvh = h / g;
    const float* w = a.basis + (static_cast<int64_t>(b) * a.hkv + kvh) * a.rank * kD;
    const int t = threadIdx.x;
    qv[t] = a.q[(static_cast<int64_t>(b) * a.hq + h) * kD + t];
    __syncthreads();
    if (t < a.rank) {
        float s = 0.f;
        for (int c = 0; c < kD; ++c) s = fmaf(w[t * kD + c], qv[c], s);
        p[t] = s;
    }
    __syncthreads();
    float s = 0.f;
    for (int r = 0; r < a.rank; ++r) s = fmaf(p[r], w[r * kD + t], s);
    a.q_proj[(static_cast<int64_t>(b) * a.hq + h) * kD + t] = s;
}

// --------------------------------------------------------- variant scores

// One warp's working set for one unit.
struct alignas(16) VariantWarp {
    float d[kPage][132];     // keys, then the centred keys D (16-byte rows for float4 reads)
    float g[kPage][17];      // Gram matrix D D^T; eigenvalues on the diagonal after the sweeps
    float u[kPage][17];      // eigenvectors (columns)
    float v[15][kD];         // basis: row r is V[:, r]
    float cf[kPage][16];     // coefficients C[token][r]
    float mu[kD];
    float2 cs[8];            // this round's rotations
    int2 pq[8];              // and their index pairs
    int ord[kPage];          // eigenvalue order, descending
};

__host__ __device__ constexpr int variant_qs_bytes(int g) { return (g * kD * 4 + 15) / 16 * 16; }

// x[i * stride + r] for i < rows, r < cols, replaced by its dequantised
// symmetric absmax codes of `bits` bits: scale = fp16(absmax / qmax), qmax =
// 2^(bits-1) - 1, code = clamp(round-half-even(x / scale)); bits 0 keeps x.
__device__ void quant_dequant(float* x, int rows, int cols, int stride, int bits, int lane) {
    if (bits == 0) return;
    const int n = rows * cols;
    float amax = 0.f;
    for (int e = lane; e < n; e += 32) amax = fmaxf(amax, fabsf(x[(e / cols) * stride + e % cols]));
    amax = __shfl_sync(0xffffffffu, warp_max(amax), 0);
    const float qmax = static_cast<float>((1 << (bits - 1)) - 1);
    const float s = __half2float(__double2half(static_cast<double>(amax) / static_cast<double>(qmax)));
    const bool ok = s > 0.f && !isinf(s);
    __syncwarp();
    for (int e = lane; e < n; e += 32) {
        float& y = x[(e / cols) * stride + e % cols];
        const float c = ok ? fminf(fmaxf(rintf(y / s), -qmax), qmax) : 0.f;
        y = c * s;
    }
    __syncwarp();
}

// Grid (B * Hkv, runs of 64 pages); dynamic shared memory = the group's
// queries, then one VariantWarp per warp.
__global__ void __launch_bounds__(kAbWarps * 32, 2) variant_kernel(AblationArgs a) {
    extern __shared__ __align__(16) unsigned char ab_smem[];
    const int g = a.hq / a.hkv;
    float* qs = reinterpret_cast<float*>(ab_smem);
    const int b = blockIdx.x / a.hkv, kvh = blockIdx.x % a.hkv;
    const int P = seq_len(a, b);
    const int j0 = blockIdx.y * kAbPagesPerCta;
    if (j0 >= P) return;
    stage_queries(a, b, kvh, qs);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    VariantWarp& w = reinterpret_cast<VariantWarp*>(ab_smem + variant_qs_bytes(g))[warp];
    const int R = a.rank;
    const int j1 = min(P, j0 + kAbPagesPerCta);
    for (int j = j0 + warp; j < j1; j += kAbWarps) {
        const int64_t phys = phys_page(a, b, j);
        {   // keys to fp32: lane holds token lane / 2, dims [64 (lane % 2), +64)
            const int i = lane >> 1, h = lane & 1;
            const uint4* src = reinterpret_cast<const uint4*>(
                a.k_cache + ((phys * a.hkv + kvh) * kPage + i) * kD + h * 64);
            float* dst = &w.d[i][h * 64];
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                float f[8];
                bf16x8_to_f32(src[v], f);
                reinterpret_cast<float4*>(dst + 8 * v)[0] = make_float4(f[0], f[1], f[2], f[3]);
                reinterpret_cast<float4*>(dst + 8 * v)[1] = make_float4(f[4], f[5], f[6], f[7]);
            }
        }
        __syncwarp();
#pragma unroll
        for (int x = 0; x < 4; ++x) {   // centroid; centring (lane owns dims lane + 32 x)
            const int c = lane + 32 * x;
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < kPage; ++i) s += w.d[i][c];
            const float m = s * (1.f / kPage);
            w.mu[c] = m;
#pragma unroll
            for (int i = 0; i < kPage; ++i) w.d[i][c] -= m;
        }
        __syncwarp();
        {   // Gram matrix (lane: row lane / 2, columns 8 (lane % 2) .. +8) and U = I
            const int i = lane >> 1, jb = (lane & 1) * 8;
            float acc[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) acc[jj] = 0.f;
            for (int c = 0; c < kD; c += 4) {
                const float4 x = *reinterpret_cast<const float4*>(&w.d[i][c]);
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const float4 y = *reinterpret_cast<const float4*>(&w.d[jb + jj][c]);
                    acc[jj] = fmaf(x.x, y.x, acc[jj]);
                    acc[jj] = fmaf(x.y, y.y, acc[jj]);
                    acc[jj] = fmaf(x.z, y.z, acc[jj]);
                    acc[jj] = fmaf(x.w, y.w, acc[jj]);
                }
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                w.g[i][jb + jj] = acc[jj];
                w.u[i][jb + jj] = (i == jb + jj) ? 1.f : 0.f;
            }
        }
        __syncwarp();
        float prev_off = INFINITY;
        for (int sweep = 0; sweep < kSmallSweeps; ++sweep) {   // cyclic Jacobi, round-robin order
            float off = 0.f, tot = 0.f;
            for (int e = lane; e < kPage * kPage; e += 32) {
                const float x = w.g[e >> 4][e & 15];
                tot += x * x;
                if ((e >> 4) != (e & 15)) off += x * x;
            }
            off = __shfl_sync(0xffffffffu, warp_sum(off), 0);
            tot = __shfl_sync(0xffffffffu, warp_sum(tot), 0);
            // converged (also for an all-zero or NaN page), or at the fp32 rounding floor
            if (!(off > 1e-14f * tot) || !(off < kStallRatio * prev_off)) break;
            prev_off = off;
            for (int r = 0; r < 15; ++r) {
                if (lane < 8) {   // round r pairs (r, 15) and ((r + k) mod 15, (r - k) mod 15), k = 1..7
                    const int p = lane == 0 ? r : (r + lane) % 15;
                    const int q = lane == 0 ? 15 : (r + 15 - lane) % 15;
                    w.pq[lane] = make_int2(p, q);
                    w.cs[lane] = schur_rotation(w.g[p][p], w.g[q][q], w.g[p][q]);
                }
                __syncwarp();
#pragma unroll
                for (int x = 0; x < 4; ++x) {   // A <- A J, U <- U J: task (rotation k, row m)
                    const int t = lane + 32 * x, k = t >> 4, m = t & 15;
                    const int2 pq = w.pq[k];
                    const float2 cs = w.cs[k];
                    const float ap = w.g[m][pq.x], aq = w.g[m][pq.y];
                    w.g[m][pq.x] = cs.x * ap - cs.y * aq;
                    w.g[m][pq.y] = cs.y * ap + cs.x * aq;
                    const float up = w.u[m][pq.x], uq = w.u[m][pq.y];
                    w.u[m][pq.x] = cs.x * up - cs.y * uq;
                    w.u[m][pq.y] = cs.y * up + cs.x * uq;
                }
                __syncwarp();
#pragma unroll
                for (int x = 0; x < 4; ++x) {   // A <- J^T A: task (rotation k, column m)
                    const int t = lane + 32 * x, k = t >> 4, m = t & 15;
                    const int2 pq = w.pq[k];
                    const float2 cs = w.cs[k];
                    const float ap = w.g[pq.x][m], aq = w.g[pq.y][m];
                    w.g[pq.x][m] = cs.x * ap - cs.y * aq;
                    w.g[pq.y][m] = cs.y * ap + cs.x * aq;
                }
                __syncwarp();
            }
        }
        if (lane < kPage) w.ord[lane] = lane;
        __syncwarp();
        if (lane < kPage) {   // descending; equal eigenvalues keep the lower index first
            const float li = w.g[lane][lane];
            int rk = 0;
#pragma unroll
            for (int jx = 0; jx < kPage; ++jx) {
                const float lj = w.g[jx][jx];
                rk += (lj > li) || (lj == li && jx < lane);
            }
            w.ord[rk] = lane;
        }
        __syncwarp();
        const float lam1 = w.g[w.ord[0] & 15][w.ord[0] & 15];
        for (int r = 0; r < R; ++r) {   // V[:, r] = D^T u / sigma, C[:, r] = sigma u
            const int col = w.ord[r] & 15;
            const float lam = w.g[col][col];
            const bool keep = lam1 > 0.f && lam > 1e-12f * lam1;
            const float sigma = keep ? sqrtf(lam) : 0.f;
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int c = lane + 32 * x;
                float s = 0.f;
#pragma unroll
                for (int i = 0; i < kPage; ++i) s = fmaf(w.d[i][c], w.u[i][col], s);
                w.v[r][c] = keep ? s / sigma : 0.f;
            }
            if (lane < kPage) w.cf[lane][r] = keep ? sigma * w.u[lane][col] : 0.f;
        }
        __syncwarp();
        quant_dequant(w.mu, 1, kD, kD, a.bits_mu, lane);
        quant_dequant(&w.v[0][0], R, kD, kD, a.bits_v, lane);
        quant_dequant(&w.cf[0][0], kPage, R, 16, a.bits_c, lane);
        for (int hh = 0; hh < g; ++hh) {   // s = LSE_i (q . mu + sum_r (q . V_r) C_ir) / sqrt(d)
            const float* qh = qs + hh * kD;
            float qc[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) qc[x] = qh[lane + 32 * x];
            float am = 0.f;
#pragma unroll
            for (int x = 0; x < 4; ++x) am = fmaf(qc[x], w.mu[lane + 32 * x], am);
            am = warp_sum(am);
            float wr[15];
#pragma unroll
            for (int r = 0; r < 15; ++r) {
                wr[r] = 0.f;
                if (r < R) {
                    float s = 0.f;
#pragma unroll
                    for (int x = 0; x < 4; ++x) s = fmaf(qc[x], w.v[r][lane + 32 * x], s);
                    wr[r] = warp_sum(s);
                }
            }
            const int i = lane & 15;
            float t = am;
#pragma unroll
            for (int r = 0; r < 15; ++r)
                if (r < R) t = fmaf(wr[r], w.cf[i][r], t);
            const float s = lse16_log2(t * (kInvSqrtD * kLog2e));
            if (lane == 0) a.scores[(static_cast<int64_t>(b) * a.hq + kvh * g + hh) * a.max_pages + j] = s;
        }
        __syncwarp();
    }
}

// ------------------------------------------------------------ shared basis

// Grid (B * Hkv, runs of 128 pages), 256 threads: thread (tr, tc) = (t / 16,
// t % 16) accumulates M[8 tr, 8 tr + 8) x [8 tc, 8 tc + 8) over the run's
// tokens, then adds it to the (b, kv head) moment. The next page's keys are
// loaded while the current one is accumulated.
__global__ void __launch_bounds__(256) moment_kernel(AblationArgs a) {
    __shared__ __align__(16) float ks[kPage][kD + 4];
    const int b = blockIdx.x / a.hkv, kvh = blockIdx.x % a.hkv;
    const int P = seq_len(a, b);
    const int j0 = blockIdx.y * kMomentPages;
    if (j0 >= P) return;
    const int j1 = min(P, j0 + kMomentPages);
    const int t = threadIdx.x, tr = t >> 4, tc = t & 15;
    const int li = t >> 4, lc = (t & 15) * 8;   // this thread's 8 keys of a page: token li, dims [lc, lc + 8)
    auto load = [&](int j) -> uint4 {
        const int64_t phys = phys_page(a, b, j);
        return *reinterpret_cast<const uint4*>(a.k_cache + ((phys * a.hkv + kvh) * kPage + li) * kD + lc);
    };
    float acc[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;
    uint4 nxt = load(j0);
    for (int j = j0; j < j1; ++j) {
        float f[8];
        bf16x8_to_f32(nxt, f);
        *reinterpret_cast<float4*>(&ks[li][lc]) = make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4*>(&ks[li][lc + 4]) = make_float4(f[4], f[5], f[6], f[7]);
        __syncthreads();
        if (j + 1 < j1) nxt = load(j + 1);
#pragma unroll 4
        for (int i = 0; i < kPage; ++i) {
            const float4 x0 = *reinterpret_cast<const float4*>(&ks[i][8 * tr]);
            const float4 x1 = *reinterpret_cast<const float4*>(&ks[i][8 * tr + 4]);
            const float4 y0 = *reinterpret_cast<const float4*>(&ks[i][8 * tc]);
            const float4 y1 = *reinterpret_cast<const float4*>(&ks[i][8 * tc + 4]);
            const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            const float ys[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[r][c] = fmaf(xs[r], ys[c], acc[r][c]);
        }
        __syncthreads();
    }
    float* m = a.moment + static_cast<int64_t>(blockIdx.x) * kD * kD;
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) atomicAdd(&m[(8 * tr + r) * kD + 8 * tc + c], acc[r][c]);
}

constexpr int eig_smem_bytes() {
    return 2 * kEigN * kEigStride * 4 + 64 * 8 + 64 * 8 + kEigN * 4 + 36 * 4;   // red: 34 floats used
}

// One CTA per (b, kv head): cyclic Jacobi on the symmetrised moment in
// parallel (round-robin) order; round r pairs (r, 127) and ((r + k) mod 127,
// (r - k) mod 127), k = 1..63, 64 disjoint rotations applied at once. Then the
// eigenvalues in descending order (equal ones keep the lower index first) and
// the top-`rank` eigenvectors, zero where lambda <= 1e-12 lambda_1, the
// largest-magnitude entry made positive.
__global__ void __launch_bounds__(kEigThreads) eig_kernel(AblationArgs a) {
    extern __shared__ __align__(16) unsigned char eig_smem[];
    float* A = reinterpret_cast<float*>(eig_smem);
    float* V = A + kEigN * kEigStride;
    float2* cs = reinterpret_cast<float2*>(V + kEigN * kEigStride);
    int2* pq = reinterpret_cast<int2*>(cs + 64);
    int* ord = reinterpret_cast<int*>(pq + 64);
    float* red = reinterpret_cast<float*>(ord + kEigN);   // [16] off, [16] total, flag, off of the sweep
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int64_t bk = blockIdx.x;
    const float* M = a.moment + bk * kD * kD;
    for (int e = t; e < kD * kD; e += kEigThreads) {
        const int i = e >> 7, j = e & 127;
        A[i * kEigStride + j] = 0.5f * (M[i * kD + j] + M[j * kD + i]);
        V[i * kEigStride + j] = (i == j) ? 1.f : 0.f;
    }
    __syncthreads();
    float prev_off = INFINITY;
    for (int sweep = 0; sweep < kLargeSweeps; ++sweep) {
        float off = 0.f, tot = 0.f;
        for (int e = t; e < kD * kD; e += kEigThreads) {
            const int i = e >> 7, j = e & 127;
            const float x = A[i * kEigStride + j];
            tot += x * x;
            if (i != j) off += x * x;
        }
        off = warp_sum(off);
        tot = warp_sum(tot);
        if (lane == 0) {
            red[warp] = off;
            red[16 + warp] = tot;
        }
        __syncthreads();
        if (t == 0) {   // go on unless converged or at the fp32 rounding floor
            float o = 0.f, s = 0.f;
            for (int x = 0; x < kEigThreads / 32; ++x) {
                o += red[x];
                s += red[16 + x];
            }
            red[32] = (o > 1e-12f * s && o < kStallRatio * prev_off) ? 1.f : 0.f;
            red[33] = o;
        }
        __syncthreads();
        const bool go = red[32] != 0.f;
        __syncthreads();
        if (!go) break;
        prev_off = red[33];
        for (int r = 0; r < kEigN - 1; ++r) {
            if (t < 64) {
                const int p = t == 0 ? r : (r + t) % 127;
                const int q = t == 0 ? 127 : (r + 127 - t) % 127;
                pq[t] = make_int2(p, q);
                cs[t] = schur_rotation(A[p * kEigStride + p], A[q * kEigStride + q], A[p * kEigStride + q]);
            }
            __syncthreads();
            for (int e = t; e < 64 * kEigN; e += kEigThreads) {   // A <- A J, V <- V J: (rotation k, row m)
                const int k = e >> 7, m = e & 127;
                const int2 ij = pq[k];
                const float2 c = cs[k];
                float* ar = A + m * kEigStride;
                const float ap = ar[ij.x], aq = ar[ij.y];
                ar[ij.x] = c.x * ap - c.y * aq;
                ar[ij.y] = c.y * ap + c.x * aq;
                float* vr = V + m * kEigStride;
                const float vp = vr[ij.x], vq = vr[ij.y];
                vr[ij.x] = c.x * vp - c.y * vq;
                vr[ij.y] = c.y * vp + c.x * vq;
            }
            __syncthreads();
            for (int e = t; e < 64 * kEigN; e += kEigThreads) {   // A <- J^T A: (rotation k, column m)
                const int k = e >> 7, m = e & 127;
                const int2 ij = pq[k];
                const float2 c = cs[k];
                float* rp = A + ij.x * kEigStride;
                float* rq = A + ij.y * kEigStride;
                const float ap = rp[m], aq = rq[m];
                rp[m] = c.x * ap - c.y * aq;
                rq[m] = c.y * ap + c.x * aq;
            }
            __syncthreads();
        }
    }
    if (t < kEigN) ord[t] = t;
    __syncthreads();
    if (t < kEigN) {
        const float li = A[t * kEigStride + t];
        int rk = 0;
        for (int j = 0; j < kEigN; ++j) {
            const float lj = A[j * kEigStride + j];
            rk += (lj > li) || (lj == li && j < t);
        }
        ord[rk] = t;
    }
    __syncthreads();
    if (a.eigvals && t < kEigN) {
        const int o = ord[t] & 127;
        a.eigvals[bk * kEigN + t] = A[o * kEigStride + o];
    }
    const int o0 = ord[0] & 127;
    const float lam1 = A[o0 * kEigStride + o0];
    for (int r = warp; r < a.rank; r += kEigThreads / 32) {
        const int col = ord[r] & 127;
        const float lam = A[col * kEigStride + col];
        const bool keep = lam1 > 0.f && lam > 1e-12f * lam1;
        float best = -1.f, bv = 0.f;
        int bi = kEigN;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const int c = lane + 32 * x;
            const float v = V[c * kEigStride + col];
            if (fabsf(v) > best) {
                best = fabsf(v);
                bi = c;
                bv = v;
            }
        }
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) {   // largest magnitude, first index on ties
            const float ob = __shfl_xor_sync(0xffffffffu, best, s);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, s);
            const float ov = __shfl_xor_sync(0xffffffffu, bv, s);
            if (ob > best || (ob == best && oi < bi)) {
                best = ob;
                bi = oi;
                bv = ov;
            }
        }
        const float sgn = bv < 0.f ? -1.f : 1.f;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const int c = lane + 32 * x;
            a.basis[(bk * a.rank + r) * kD + c] = keep ? sgn * V[c * kEigStride + col] : 0.f;
        }
    }
}

}  // namespace

// ---------------------------------------------------------------- launchers

cudaError_t launch_exact_scores(const AblationArgs& a, cudaStream_t stream) {
    if (a.batch == 0 || a.max_pages == 0) return cudaSuccess;
    const int g = a.hq / a.hkv;
    const dim3 grid(a.batch * a.hkv, (a.max_pages + kAbPagesPerCta - 1) / kAbPagesPerCta);
    const int smem = kAbWarps * 2 * kExSlot + g * kD * 4;   // at most 40 KiB (g <= 16)
    if (g <= 8)
        exact_kernel<1><<<grid, kAbWarps * 32, smem, stream>>>(a);
    else
        exact_kernel<2><<<grid, kAbWarps * 32, smem, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_variant_scores(const AblationArgs& a, cudaStream_t stream) {
    if (a.batch == 0 || a.max_pages == 0) return cudaSuccess;
    const int smem = variant_qs_bytes(a.hq / a.hkv) + kAbWarps * static_cast<int>(sizeof(VariantWarp));
    cudaError_t e = ensure_kernel_attrs<variant_kernel>(smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(a.batch * a.hkv, (a.max_pages + kAbPagesPerCta - 1) / kAbPagesPerCta);
    variant_kernel<<<grid, kAbWarps * 32, smem, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_shared_basis(const AblationArgs& a, cudaStream_t stream) {
    if (a.batch == 0) return cudaSuccess;
    const size_t mbytes = static_cast<size_t>(a.batch) * a.hkv * kD * kD * sizeof(float);
    cudaError_t e = cudaMemsetAsync(a.moment, 0, mbytes, stream);
    if (e != cudaSuccess) return e;
    if (a.max_pages > 0) {
        const dim3 grid(a.batch * a.hkv, (a.max_pages + kMomentPages - 1) / kMomentPages);
        moment_kernel<<<grid, 256, 0, stream>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if ((e = ensure_kernel_attrs<eig_kernel>(eig_smem_bytes())) != cudaSuccess) return e;
    eig_kernel<<<a.batch * a.hkv, kEigThreads, eig_smem_bytes(), stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_project_queries(const AblationArgs& a, cudaStream_t stream) {
    if (a.batch == 0) return cudaSuccess;
    project_kernel<<<a.batch * a.hq, 128, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace locks
