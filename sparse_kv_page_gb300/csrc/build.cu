// build.cu - LOCKS page-summary builder (runs when a page fills; off the
// decode critical path).
//
// Per (physical page, kv head) "unit", following the LOCKS post ("How LOCKS
// works": decomposition of the centred key deviations, int8 centroid, int4
// rank-8 basis, int8 coefficients) and the gist.science summary 2.1 (a small
// eigendecomposition of the centred keys):
//   mu = mean of the 16 keys; D = K - mu;
//   G = D D^T (16 x 16), eigenpairs by the cyclic Jacobi method in parallel
//   (round-robin) order; the 8 largest: V[:, r] = D^T u_r / sqrt(lambda_r),
//   C[:, r] = sqrt(lambda_r) u_r (zero if lambda_r <= 1e-12 lambda_1); the
//   largest-magnitude entry of each V column made positive; absmax
//   quantisation to int8 / int4 / int8 with fp16 scales, packed in the
//   scorer's fragment order (see include/locks.h).
//
// GPU mapping: a warp builds two units at a time (four CTAs of four warps per SM; the
// keys stay in bf16 in shared memory and the deviations are formed on the fly). The Gram
// matrix runs on the tensor cores (f16 hi/lo split of the power-of-two-normalised deviations,
// three MMAs per tile, fp32 accumulate); the Jacobi sweeps keep one row of G
// and one row of the eigenvector matrix per lane (lanes 0-15: first unit,
// 16-31: second), 8 disjoint rotations per round on fixed position pairs followed by
// the round-robin permutation of positions, 15 rounds per sweep, register indices
// static, operands exchanged with warp shuffles; the round loop stays rolled.
#include "locks_internal.h"

namespace locks {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kKStride = 136;   // bf16 row stride of the keys in shared memory (conflict-free fragments)
constexpr int kMaxSweeps = 10;
constexpr int64_t kSingleUnitBuild = 512;   // builds of at most this many units: one unit per warp
constexpr int kCtasPerSm = 4;   // 16 warps per SM: 128 registers (no spills), 4 x 56 KB of shared memory

// The keys stay in bf16 (exact) and D = K - mu is formed on the fly in fp32, which keeps
// the per-warp footprint small enough for four CTAs per SM.
struct WarpSmem {
    uint16_t k[2][kPage * kKStride];
    float mu[2][kD];
    float g[2][kPage * kPage];
    float u8[2][kPage * kRank];
    float sig[2][kRank];
    int8_t vcode[kRank * kD];
    int8_t ccode[kPage * kRank];
};

// Symmetric Schur rotation that zeroes a_pq (Golub & Van Loan, section 8.5). The
// quotients may be approximate: c = 1/sqrt(1 + t^2) and s = t c form an orthogonal
// rotation for any t, and t only steers how much of a_pq it removes.
__device__ __forceinline__ void schur(float app, float aqq, float apq, float& c, float& s) {
    if (fabsf(apq) <= 1e-30f || fabsf(apq) <= 1e-9f * sqrtf(fabsf(app * aqq))) {
        c = 1.f;
        s = 0.f;
        return;
    }
    const float tau = __fdividef(aqq - app, 2.f * apq);
    float t;
    if (fabsf(tau) > 1e18f) {
        t = __fdividef(0.5f, tau);
    } else {
        t = __fdividef(tau >= 0.f ? 1.f : -1.f, fabsf(tau) + sqrtf(1.f + tau * tau));
    }
    c = rsqrtf(1.f + t * t);
    s = t * c;
}

// Parallel ordering of the cyclic Jacobi method (the round-robin "circle" schedule): every
// round rotates the fixed position pairs (2k, 2k + 1), then the positions are permuted --
// position 0 stays, the others move one step around the circle of top positions 2k and
// bottom positions 2k + 1 -- so that in 15 rounds every pair of indices meets once. After a
// round position i holds what position rr_src(i) held before.
__host__ __device__ constexpr int rr_src(int i) {
    return i == 0 ? 0 : (i == 2 ? 1 : (i == 15 ? 14 : ((i & 1) ? i + 2 : i - 2)));
}

// One round on a half-warp's matrix: lane i (within the half, base = first lane of the
// half) holds row i of G (gr) and row i of U (ur), columns in registers. Every round runs
// the same code, so the round loop stays rolled and its instructions cached.
__device__ __forceinline__ void jacobi_round(float (&gr)[16], float (&ur)[16], int i, int base) {
    const bool is_p = (i & 1) == 0;   // pair (p, q) = (2k, 2k + 1)
    float dmine = 0.f, doff = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        dmine = m == i ? gr[m] : dmine;
        doff = m == (i ^ 1) ? gr[m] : doff;
    }
    const float dother = __shfl_sync(0xffffffffu, dmine, base + (i ^ 1));
    const float apq = __shfl_sync(0xffffffffu, doff, base + (i & ~1));   // both lanes use row p's
    float cm, sm;
    schur(is_p ? dmine : dother, is_p ? dother : dmine, apq, cm, sm);
    // every lane needs every pair's rotation for the column update
    float c[8], s[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        c[k] = __shfl_sync(0xffffffffu, cm, base + 2 * k);
        s[k] = __shfl_sync(0xffffffffu, sm, base + 2 * k);
    }
    // G <- G J and U <- U J (columns 2k, 2k + 1 of this lane's rows)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float gp = gr[2 * k], gq = gr[2 * k + 1];
        gr[2 * k] = c[k] * gp - s[k] * gq;
        gr[2 * k + 1] = s[k] * gp + c[k] * gq;
        const float up = ur[2 * k], uq = ur[2 * k + 1];
        ur[2 * k] = c[k] * up - s[k] * uq;
        ur[2 * k + 1] = s[k] * up + c[k] * uq;
    }
    // G <- J^T G (rows p, q): combine with the partner row
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const float other = __shfl_sync(0xffffffffu, gr[m], base + (i ^ 1));
        gr[m] = is_p ? (cm * gr[m] - sm * other) : (sm * other + cm * gr[m]);
    }
    // the round-robin permutation: columns of G and U in registers, rows of G across lanes
    float tg[16], tu[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        tg[m] = gr[rr_src(m)];
        tu[m] = ur[rr_src(m)];
    }
    const int src = base + rr_src(i);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        gr[m] = __shfl_sync(0xffffffffu, tg[m], src);
        ur[m] = tu[m];
    }
}

__device__ __forceinline__ float f16_round_scale(float amax, float qmax) {
    return __half2float(__float2half_rn(amax / qmax));
}
__device__ __forceinline__ int quant(float x, float s, int qmax) {
    if (!(s > 0.f) || isinf(s)) return 0;
    float c = rintf(x / s);
    c = fminf(fmaxf(c, -static_cast<float>(qmax)), static_cast<float>(qmax));
    return static_cast<int>(c);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Loads a unit's keys (bf16, kept as they are), their mean mu, and the Gram matrix of the
// centred keys D = K - mu into w.g[slot].
__device__ void load_centre_gram(const BuildArgs& a, int64_t unit, WarpSmem& w, int slot, int lane) {
    uint16_t* k = w.k[slot];
    float* mu = w.mu[slot];
    const int gid = lane >> 2, t = lane & 3;
    if (unit >= 0) {
        const uint16_t* src =
            a.k_cache + (static_cast<int64_t>(a.phys_page_ids[unit / a.hkv]) * a.hkv + unit % a.hkv) * (kPage * kD);
        uint4 v[8];   // all of this lane's loads in flight
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int c = lane + 32 * m;
            v[m] = *reinterpret_cast<const uint4*>(src + (c >> 4) * kD + (c & 15) * 8);
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int c = lane + 32 * m;
            *reinterpret_cast<uint4*>(k + (c >> 4) * kKStride + (c & 15) * 8) = v[m];
        }
    } else {
        // no unit: a zero Gram (its Jacobi ends at once; nothing of it is written out)
        float* g = w.g[slot];
        for (int idx = lane; idx < kPage * kPage; idx += 32) g[idx] = 0.f;
        if (lane == 0) w.sig[slot][0] = __int_as_float(0);
        __syncwarp();
        return;
    }
    __syncwarp();
    // mean over the 16 keys, lane -> dims 4 lane .. 4 lane + 3
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int i = 0; i < kPage; ++i) {
        const uint2 v = *reinterpret_cast<const uint2*>(k + i * kKStride + 4 * lane);
        s4[0] += bf16_lo(v.x);
        s4[1] += bf16_hi(v.x);
        s4[2] += bf16_lo(v.y);
        s4[3] += bf16_hi(v.y);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) s4[q] *= (1.f / kPage);
    *reinterpret_cast<float4*>(mu + 4 * lane) = make_float4(s4[0], s4[1], s4[2], s4[3]);
    float amax = 0.f;
#pragma unroll 4
    for (int i = 0; i < kPage; ++i) {
        const uint2 v = *reinterpret_cast<const uint2*>(k + i * kKStride + 4 * lane);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(v.x) - s4[0]), fabsf(bf16_hi(v.x) - s4[1])),
                                 fmaxf(fabsf(bf16_lo(v.y) - s4[2]), fabsf(bf16_hi(v.y) - s4[3]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    __syncwarp();
    // Gram on the tensor cores: D' = D * 2^-e (max |D'| < 1), split f16 hi/lo.
    int e = 0;
    if (amax > 0.f && amax < INFINITY) e = ilogbf(amax) + 1;
    e = max(-100, min(100, e));
    const float inv = __int_as_float((127 - e) << 23);
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    // once-per-unit loops stay rolled: the code of all phases of the 16 warps of an SM
    // shares the instruction caches with the Jacobi round loop
#pragma unroll 2
    for (int s = 0; s < 8; ++s) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int row = gid + ((r & 1) ? 8 : 0);
            const int col = 16 * s + 2 * t + ((r & 2) ? 8 : 0);
            const uint32_t kv = *reinterpret_cast<const uint32_t*>(k + row * kKStride + col);
            const float2 m2 = *reinterpret_cast<const float2*>(mu + col);
            const uint32_t p0 = split_f16_hilo((bf16_lo(kv) - m2.x) * inv);
            const uint32_t p1 = split_f16_hilo((bf16_hi(kv) - m2.y) * inv);
            hi[r] = __byte_perm(p0, p1, 0x5410);
            lo[r] = __byte_perm(p0, p1, 0x7632);
        }
        // n-tile 0 = tokens 0-7 (B regs = A regs 0, 2), n-tile 1 = tokens 8-15 (A regs 1, 3)
        mma_f16_16816(acc[0], hi, hi[0], hi[2]);
        mma_f16_16816(acc[0], hi, lo[0], lo[2]);
        mma_f16_16816(acc[0], lo, hi[0], hi[2]);
        mma_f16_16816(acc[1], hi, hi[1], hi[3]);
        mma_f16_16816(acc[1], hi, lo[1], lo[3]);
        mma_f16_16816(acc[1], lo, hi[1], hi[3]);
    }
    float* g = w.g[slot];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        g[gid * kPage + nt * 8 + 2 * t] = acc[nt][0];
        g[gid * kPage + nt * 8 + 2 * t + 1] = acc[nt][1];
        g[(gid + 8) * kPage + nt * 8 + 2 * t] = acc[nt][2];
        g[(gid + 8) * kPage + nt * 8 + 2 * t + 1] = acc[nt][3];
    }
    // the normalisation exponent travels in sig[slot][0] (as int bits) until the eigen step
    if (lane == 0) w.sig[slot][0] = __int_as_float(e);
    __syncwarp();
}

// Eigendecomposition of both Gram matrices (half-warp each); writes the
// top-8 eigenvectors (columns) to u8 and sqrt(lambda) (unnormalised) to sig.
__device__ void jacobi_top8(WarpSmem& w, int lane) {
    const int half = lane >> 4, i = lane & 15, base = half * 16;
    const int e = __float_as_int(w.sig[half][0]);
    float gr[16], ur[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        gr[m] = w.g[half][i * kPage + m];
        ur[m] = (m == i) ? 1.f : 0.f;
    }
    float fro2 = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) fro2 += gr[m] * gr[m];
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) fro2 += __shfl_xor_sync(0xffffffffu, fro2, o);
    float prev_off2 = INFINITY;
#pragma unroll 1
    for (int sweep = 0; sweep < kMaxSweeps; ++sweep) {
        float off2 = 0.f, dg = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            off2 += gr[m] * gr[m];
            dg = (m == i) ? gr[m] : dg;
        }
        off2 -= dg * dg;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) off2 += __shfl_xor_sync(0xffffffffu, off2, o);
        // converged: off-diagonal energy <= 1e-7 ||G||^2 (the eigenvectors then move by
        // ~3e-4 ||G|| / gap, far below the int4 basis step of 1/7 of a column's largest
        // entry), or <= 1e-6 ||G||^2 and no longer halving per sweep (the fp32 rounding floor)
        const bool done = off2 <= 1e-7f * fro2 || (off2 <= 1e-6f * fro2 && off2 > 0.5f * prev_off2);
        prev_off2 = off2;
        if (__all_sync(0xffffffffu, done)) break;
#pragma unroll 1
        for (int r = 0; r < 15; ++r) jacobi_round(gr, ur, i, base);
    }
    float lam = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) lam = (m == i) ? gr[m] : lam;
    // rank of this eigenvalue (descending, ties -> lower index)
    int rk = 0;
    float lam1 = lam;
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
        const float lj = __shfl_sync(0xffffffffu, lam, base + j);
        rk += (lj > lam) || (lj == lam && j < i);
        lam1 = fmaxf(lam1, lj);
    }
    const float scale = __int_as_float((127 + e) << 23);   // 2^e: undo the Gram normalisation
#pragma unroll 1
    for (int r = 0; r < kRank; ++r) {
        // column index (lane within the half) holding rank r
        const unsigned bal = __ballot_sync(0xffffffffu, rk == r);
        const int col = __ffs((bal >> base) & 0xffffu) - 1;
        float uv = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) uv = (j == col) ? ur[j] : uv;
        w.u8[half][i * kRank + r] = uv;
        if (i == col) {
            const bool dead = !(lam1 > 0.f) || lam <= 1e-12f * lam1;
            w.sig[half][r] = dead ? 0.f : sqrtf(lam) * scale;
        }
    }
    __syncwarp();
}

// V, C, quantisation and packing for one unit; writes its summary bytes.
__device__ void finish_unit(const BuildArgs& a, int64_t unit, WarpSmem& w, int slot, int lane) {
    const uint16_t* k = w.k[slot];
    const float* u8 = w.u8[slot];
    const float* sig = w.sig[slot];
    const float4 mu4 = *reinterpret_cast<const float4*>(w.mu[slot] + 4 * lane);
    // V[d][r] = sum_i D[i][d] u_r[i] / sigma_r, lane -> dims 4 lane .. +3
    float v[4][kRank];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int r = 0; r < kRank; ++r) v[q][r] = 0.f;
#pragma unroll 2
    for (int i = 0; i < kPage; ++i) {
        const uint2 kv = *reinterpret_cast<const uint2*>(k + i * kKStride + 4 * lane);
        const float4 ua = *reinterpret_cast<const float4*>(u8 + i * kRank);
        const float4 ub = *reinterpret_cast<const float4*>(u8 + i * kRank + 4);
        const float uu[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
        const float dd[4] = {bf16_lo(kv.x) - mu4.x, bf16_hi(kv.x) - mu4.y, bf16_lo(kv.y) - mu4.z,
                             bf16_hi(kv.y) - mu4.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int r = 0; r < kRank; ++r) v[q][r] = fmaf(dd[q], uu[r], v[q][r]);
    }
    float flip[kRank];
    float vmax = 0.f;
#pragma unroll
    for (int r = 0; r < kRank; ++r) {
        const float inv = sig[r] > 0.f ? 1.f / sig[r] : 0.f;
        float best = -1.f;
        int bidx = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            v[q][r] *= inv;
            if (fabsf(v[q][r]) > best) {
                best = fabsf(v[q][r]);
                bidx = 4 * lane + q;
            }
        }
        float bval = v[0][r];
#pragma unroll
        for (int q = 0; q < 4; ++q) bval = (4 * lane + q == bidx) ? v[q][r] : bval;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
            const int i2 = __shfl_xor_sync(0xffffffffu, bidx, o);
            const float v2 = __shfl_xor_sync(0xffffffffu, bval, o);
            if (b2 > best || (b2 == best && i2 < bidx)) {
                best = b2;
                bidx = i2;
                bval = v2;
            }
        }
        flip[r] = bval < 0.f ? -1.f : 1.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            v[q][r] *= flip[r];
            vmax = fmaxf(vmax, fabsf(v[q][r]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    const float sv = f16_round_scale(vmax, 7.f);
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int r = 0; r < kRank; ++r) w.vcode[r * kD + 4 * lane + q] = static_cast<int8_t>(quant(v[q][r], sv, 7));
    // C[i][r] = sigma_r u_r[i] (same sign flip); lane -> 4 of the 128 entries
    float cv[4];
    float cmax = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int idx = 4 * lane + q, i = idx / kRank, r = idx % kRank;
        float fl = 1.f;
#pragma unroll
        for (int rr = 0; rr < kRank; ++rr) fl = (rr == r) ? flip[rr] : fl;
        cv[q] = sig[r] * u8[i * kRank + r] * fl;
        cmax = fmaxf(cmax, fabsf(cv[q]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
    const float sc = f16_round_scale(cmax, 127.f);
#pragma unroll
    for (int q = 0; q < 4; ++q) w.ccode[4 * lane + q] = static_cast<int8_t>(quant(cv[q], sc, 127));
    // centroid
    const float4 m4 = *reinterpret_cast<const float4*>(w.mu[slot] + 4 * lane);
    float mmax = fmaxf(fmaxf(fabsf(m4.x), fabsf(m4.y)), fmaxf(fabsf(m4.z), fabsf(m4.w)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
    const float smu = f16_round_scale(mmax, 127.f);
    __syncwarp();
    if (unit < 0) return;

    // pack: basis byte ob = 64 r + 16 t + 4 j + pb; low nibble h = 0, high h = 1,
    // s = 2 j + pb % 2, e = pb / 2, dim = 16 s + 8 h + 2 t + e
    uint32_t words[4];
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        uint32_t word = 0;
#pragma unroll 1
        for (int bi = 0; bi < 4; ++bi) {
            const int ob = 16 * lane + 4 * wi + bi;
            const int r = ob >> 6, rem = ob & 63, t = rem >> 4, j = (rem & 15) >> 2, pb = rem & 3;
            const int s = 2 * j + (pb & 1), e = pb >> 1;
            const int d0 = 16 * s + 2 * t + e, d1 = d0 + 8;
            const uint32_t byte = (static_cast<uint32_t>(w.vcode[r * kD + d0]) & 0xfu) |
                                  ((static_cast<uint32_t>(w.vcode[r * kD + d1]) & 0xfu) << 4);
            word |= byte << (8 * bi);
        }
        words[wi] = word;
    }
    const int64_t out_unit = static_cast<int64_t>(a.phys_page_ids[unit / a.hkv]) * a.hkv + unit % a.hkv;
    *reinterpret_cast<uint4*>(a.basis + out_unit * 512 + 16 * lane) = make_uint4(words[0], words[1], words[2], words[3]);
    // mu byte o: t = o / 32, s = (o % 32) / 4, h = (o % 4) / 2, e = o % 2
    {
        uint32_t word = 0;
#pragma unroll 1
        for (int bi = 0; bi < 4; ++bi) {
            const int o = 4 * lane + bi;
            const int t = o >> 5, s = (o & 31) >> 2, h = (o & 3) >> 1, e = o & 1;
            const int dim = 16 * s + 8 * h + 2 * t + e;
            const int code = quant(w.mu[slot][dim], smu, 127);
            word |= (static_cast<uint32_t>(code) & 0xffu) << (8 * bi);
        }
        reinterpret_cast<uint32_t*>(a.mu + out_unit * 128)[lane] = word;
    }
    // coef byte o: lane' = o / 4 (gid' = lane' / 4, t' = lane' % 4), i = gid' + 8 ((o % 4) / 2), r = 2 t' + o % 2
    {
        uint32_t word = 0;
#pragma unroll 1
        for (int bi = 0; bi < 4; ++bi) {
            const int o = 4 * lane + bi;
            const int lp = o >> 2, gp = lp >> 2, tp = lp & 3;
            const int i = gp + 8 * ((o & 3) >> 1), r = 2 * tp + (o & 1);
            word |= (static_cast<uint32_t>(w.ccode[i * kRank + r]) & 0xffu) << (8 * bi);
        }
        reinterpret_cast<uint32_t*>(a.coef + out_unit * 128)[lane] = word;
    }
    if (lane == 0) {
        const uint32_t h0 = __half_as_ushort(__float2half_rn(smu));
        const uint32_t h1 = __half_as_ushort(__float2half_rn(sv));
        const uint32_t h2 = __half_as_ushort(__float2half_rn(sc));
        *reinterpret_cast<uint2*>(a.scales + out_unit * 4) = make_uint2(h0 | (h1 << 16), h2);
    }
    __syncwarp();
}

// The unit index, or -1 when it does not exist or its page id is out of range
// (then it is skipped and LOCKS_ERR_BAD_INDEX recorded).
__device__ __forceinline__ int64_t valid_unit(const BuildArgs& a, int64_t u) {
    if (u < 0) return -1;
    const int phys = a.phys_page_ids[u / a.hkv];
    if (phys < 0 || phys >= a.num_phys) {
        if ((threadIdx.x & 31) == 0) report_error(a.st, LOCKS_ERR_BAD_INDEX);
        return -1;
    }
    return u;
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) build_kernel(BuildArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WarpSmem& w = reinterpret_cast<WarpSmem*>(smem)[warp];
    const int64_t n_units = static_cast<int64_t>(a.n_pages) * a.hkv;
    // small builds (a page that just filled) take one unit per warp: its second
    // half-warp's Jacobi is idle, but the unit's set-up and packing are not queued
    // behind another unit's
    const bool single = n_units <= kSingleUnitBuild;
    const int64_t n_pairs = single ? n_units : (n_units + 1) / 2;
    for (int64_t pi = static_cast<int64_t>(blockIdx.x) * kWarps + warp; pi < n_pairs;
         pi += static_cast<int64_t>(gridDim.x) * kWarps) {
        const int64_t u0 = single ? pi : 2 * pi, u1 = (!single && 2 * pi + 1 < n_units) ? 2 * pi + 1 : -1;
        const int64_t v0 = valid_unit(a, u0), v1 = valid_unit(a, u1);
        load_centre_gram(a, v0, w, 0, lane);
        load_centre_gram(a, v1, w, 1, lane);
        jacobi_top8(w, lane);
        finish_unit(a, v0, w, 0, lane);
        if (u1 >= 0) finish_unit(a, v1, w, 1, lane);
    }
}

}  // namespace

cudaError_t launch_build(const BuildArgs& a, int num_sms, cudaStream_t stream) {
    const int64_t n_units = static_cast<int64_t>(a.n_pages) * a.hkv;
    if (n_units == 0) return cudaSuccess;
    const size_t smem = kWarps * sizeof(WarpSmem);
    cudaError_t e = ensure_kernel_attrs<build_kernel>(static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t pairs = n_units <= kSingleUnitBuild ? n_units : (n_units + 1) / 2;
    int64_t grid = (pairs + kWarps - 1) / kWarps;
    const int64_t cap = static_cast<int64_t>(num_sms) * kCtasPerSm;
    if (grid > cap) grid = cap;
    build_kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace locks
