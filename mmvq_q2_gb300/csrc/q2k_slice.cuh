// Activation slices of the Q2_K GEMV/MMVQ kernels: the per-thread K slice
// of the activations held in registers (bf16 as 16-bit fixed point, or
// q8_1), its construction from the staged K chunk, the per-row dot product
// against a Q2_K block held in shared memory, and the lane reduction.
// Shared by q2k_mv.cu (every m <= 8 problem) and q2k_m1.cu (one token over
// long rows).
#pragma once

#include "q2k_common.cuh"
#include "q2k_internal.h"
#include "q2k_q8.cuh"

namespace q2k {

__host__ __device__ constexpr int pow2_ceil(int v) { return v <= 1 ? 1 : 2 * pow2_ceil((v + 1) / 2); }
__host__ __device__ constexpr int log2_exact(int v) { return v <= 1 ? 0 : 1 + log2_exact(v / 2); }

// ---- activation slice ------------------------------------------------------

template <int M, int ACT, int SW>
struct Slice {
    static constexpr int NA = (ACT == ACT_BF16) ? 2 : 1;  // registers per qs word
    static constexpr int NH = (SW == 8) ? 2 : 1;           // sub-block halves covered
    static constexpr int WPH = SW / NH;                    // qs words per half
    uint32_t xa[M][4][SW][NA];
    float xp[M][4][NH];       // scale of the integer sum of pair j (includes 4^-j)
    uint32_t xs16[M][NH][2];  // group sums (j = 0,1 | 2,3) as 16-bit fixed point
    float xsb[M][NH];         // their common power-of-two scale
};

// Pack the four group sums of one (token, half) as 16-bit fixed point with
// a common power-of-two exponent (error below 2^-14 of the largest).  The
// largest lands below 2^14, so rounding can never reach 2^15 and wrap the
// 16-bit field (a sum d*S of a q8_1 scale and an integer can sit within
// half a step of a power of two).
template <int M, int ACT, int SW>
__device__ __forceinline__ void pack_sums(Slice<M, ACT, SW>& sl, int t, int hh, const float (&xs)[4])
{
    const float amax = fmaxf(fmaxf(fabsf(xs[0]), fabsf(xs[1])), fmaxf(fabsf(xs[2]), fabsf(xs[3])));
    const uint32_t eb = (__float_as_uint(amax) >> 23) & 0xFFu;
    if (eb < 27u) {
        sl.xs16[t][hh][0] = sl.xs16[t][hh][1] = 0u;
        sl.xsb[t][hh] = 0.f;
        return;
    }
    const float scale = __uint_as_float((267u - eb) << 23);  // |xs * scale| < 2^14
    int q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        q[j] = __float2int_rn(xs[j] * scale);
    sl.xs16[t][hh][0] = (uint32_t)(q[0] & 0xFFFF) | ((uint32_t)q[1] << 16);
    sl.xs16[t][hh][1] = (uint32_t)(q[2] & 0xFFFF) | ((uint32_t)q[3] << 16);
    sl.xsb[t][hh] = __uint_as_float((eb - 13u) << 23);
}

// 8-word slices: the eight group sums of a token, (j, h) for j = 0..3 and
// h = 0, 1, as 16-bit fixed point with one power-of-two exponent (the
// largest below 2^14, as in pack_sums), packed as
// xs16[t][j >> 1][j & 1] = {sum(j, 0), sum(j, 1)}: the order of the min
// nibbles in the two scale words of a half block.
template <int M, int ACT, int SW>
__device__ __forceinline__ void pack_sums8(Slice<M, ACT, SW>& sl, int t, const float (&xs)[2][4])
{
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        amax = fmaxf(amax, fmaxf(fabsf(xs[0][j]), fabsf(xs[1][j])));
    const uint32_t eb = (__float_as_uint(amax) >> 23) & 0xFFu;
    if (eb < 27u) {
        sl.xs16[t][0][0] = sl.xs16[t][0][1] = sl.xs16[t][1][0] = sl.xs16[t][1][1] = 0u;
        sl.xsb[t][0] = 0.f;
        return;
    }
    const float scale = __uint_as_float((267u - eb) << 23);  // |xs * scale| < 2^14: no wrap
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int q0 = __float2int_rn(xs[0][j] * scale);
        const int q1 = __float2int_rn(xs[1][j] * scale);
        sl.xs16[t][j >> 1][j & 1] = (uint32_t)(q0 & 0xFFFF) | ((uint32_t)q1 << 16);
    }
    sl.xsb[t][0] = __uint_as_float((eb - 13u) << 23);
}

// Bytes of one token's activations per block column in the shared staging
// region: 256 bf16 values, or 8 q8_1 blocks.
template <int ACT>
__host__ __device__ constexpr int x_bytes_per_block() { return ACT == ACT_BF16 ? 512 : 8 * kQ8Bytes; }

// Copy the K chunk of every token's activations for one segment into shared
// memory (all threads of the CTA; coalesced, 16-byte pieces when aligned).
template <int M, int ACT>
__device__ __forceinline__ void stage_x(const uint8_t* xseg, int64_t tok_stride, int kb0, int nbc, int align,
                                        uint8_t* xsm)
{
    const int rowb = nbc * x_bytes_per_block<ACT>();
    const uint8_t* src0 = xseg + (int64_t)kb0 * x_bytes_per_block<ACT>();
    for (int t = 0; t < M; ++t) {
        const uint8_t* src = src0 + t * tok_stride;
        uint8_t* dst = xsm + t * rowb;
        if (align >= 16) {
            for (int o = threadIdx.x * 16; o < rowb; o += blockDim.x * 16)
                *reinterpret_cast<uint4*>(dst + o) = __ldg(reinterpret_cast<const uint4*>(src + o));
        } else if (align >= 4) {
            for (int o = threadIdx.x * 4; o < rowb; o += blockDim.x * 4)
                *reinterpret_cast<uint32_t*>(dst + o) = ldg32_nc(src + o);
        } else {
            for (int o = threadIdx.x * 2; o < rowb; o += blockDim.x * 2)
                *reinterpret_cast<uint16_t*>(dst + o) = *reinterpret_cast<const uint16_t*>(src + o);
        }
    }
}

// bf16 activations for m <= 2 are converted once per CTA, cooperatively:
// 16-bit fixed point with one power-of-two exponent per group of 16 values
// (the group of one Q2_K sub-block's codes in one bit plane).  The packed
// words are stored word-major with an XOR swizzle, so the slice reads of a
// warp fall in 32 different banks (4-word slices: lanes 4 groups apart;
// 8-word slices: lanes 8 groups apart); the exponents follow as one byte
// per group.
template <int M, int ACT, int SW>
__host__ __device__ constexpr bool coop_x() { return ACT == ACT_BF16 && (SW == 4 || SW == 8) && M <= 2; }

template <int SW>
__device__ __forceinline__ int x_group_swz(int G)
{
    if constexpr (SW == 8)
        return G ^ ((G >> 5) & 7);
    else
        return G ^ (((G >> 5) & 3) << 1);
}

// Shared bytes the converted activations of m tokens take (words, then
// exponent bytes).
__host__ __device__ constexpr int coop_x_bytes(int m, int nbc) { return m * nbc * 512 + ((m * nbc * 16 + 15) / 16) * 16; }

constexpr int kCoopGroupsPerThread = 4;  // m * nbc * 16 <= 4 * threads (checked on the host)

template <int M, int SW>
__device__ __forceinline__ void convert_x_bf16(uint8_t* xsm, int nbc)
{
    const int NG = nbc * 16;  // groups of 16 values per token
    uint32_t pk[kCoopGroupsPerThread][8];
    uint32_t ebv[kCoopGroupsPerThread];
#pragma unroll
    for (int k = 0; k < kCoopGroupsPerThread; ++k) {
        const int q = threadIdx.x + k * blockDim.x;
        const bool valid = q < M * NG;  // M * NG is even: pairs are valid together
        ebv[k] = 0u;
#pragma unroll
        for (int w = 0; w < 8; ++w)
            pk[k][w] = 0u;
        float v[16];
        float amax = 0.f;
        if (valid) {
            const uint8_t* src = xsm + (size_t)q * 32;  // token-major, 32 bytes per group
            const uint4 u0 = *reinterpret_cast<const uint4*>(src);
            const uint4 u1 = *reinterpret_cast<const uint4*>(src + 16);
            const uint32_t raw[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v[2 * i] = __uint_as_float(raw[i] << 16);
                v[2 * i + 1] = __uint_as_float(raw[i] & 0xFFFF0000u);
                amax = fmaxf(amax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
            }
        }
        uint32_t eb = (__float_as_uint(amax) >> 23) & 0xFFu;  // biased exponent of amax
        if constexpr (SW == 8) {
            // 8-word slices: the two groups of a 32-value pair (one q8_1-sized
            // block) share the larger exponent (the partner is lane ^ 1)
            eb = max(eb, (uint32_t)__shfl_xor_sync(0xffffffffu, (int)eb, 1));
        }
        if (valid && eb >= 27u) {
            // x16 = x * 2^(XS-eb): |x16| < 2^15 (4-word slices, XS = 141) or
            // 2^14 (8-word slices, XS = 140, so that two sub-block sums add in
            // int32), exact for the group's largest 2^8 range.  Adding 1.5*2^23
            // (ulp 1) rounds to the nearest integer, ties to even, and leaves
            // it in the low mantissa bits as a 16-bit two's complement value.
            const float scale = __uint_as_float(((SW == 8 ? 267u : 268u) - eb) << 23);
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const uint32_t f0 = __float_as_uint(fmaf(v[2 * w], scale, 12582912.0f));
                const uint32_t f1 = __float_as_uint(fmaf(v[2 * w + 1], scale, 12582912.0f));
                pk[k][w] = __byte_perm(f0, f1, 0x5410u);
            }
            ebv[k] = eb;
        }
    }
    __syncthreads();  // every group has been read before any is overwritten
    uint32_t* words = reinterpret_cast<uint32_t*>(xsm);
    uint8_t* ebs = xsm + (size_t)M * NG * 32;
#pragma unroll
    for (int k = 0; k < kCoopGroupsPerThread; ++k) {
        const int q = threadIdx.x + k * blockDim.x;
        if (q < M * NG) {
            const int t = q / NG, G = q - t * NG;
            uint32_t* wt = words + (size_t)t * NG * 8 + x_group_swz<SW>(G);
#pragma unroll
            for (int w = 0; w < 8; ++w)
                wt[w * NG] = pk[k][w];
            ebs[q] = (uint8_t)ebv[k];
        }
    }
    __syncthreads();
}

// Build this thread's activation slice from the staged K chunk.  Slice
// geometry: block b within the chunk, half n, first qs word wi0 (0..7).
// Weight of (j, word w, byte i) is k = b*256 + 128n + 32j + 4w + i.
template <int M, int ACT, int SW>
__device__ __forceinline__ void load_slice(Slice<M, ACT, SW>& sl, const uint8_t* xsm, int nbc, int b, int n, int wi0,
                                           bool active)
{
    using S = Slice<M, ACT, SW>;
    const int rowb = nbc * x_bytes_per_block<ACT>();
#pragma unroll
    for (int t = 0; t < M; ++t) {
        const uint8_t* xt = xsm + t * rowb;
        float xsum[S::NH][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if constexpr (coop_x<M, ACT, SW>()) {
                // converted words of group (b, n, j, h); the thread takes all 16 values
                const int NG = nbc * 16;
#pragma unroll
                for (int hh = 0; hh < S::NH; ++hh) {
                    const int G = b * 16 + 8 * n + 2 * j + (SW == 8 ? hh : (wi0 >> 2));
                    const uint32_t* wt =
                        reinterpret_cast<const uint32_t*>(xsm) + (size_t)t * NG * 8 + x_group_swz<SW>(G);
                    const uint32_t eb = active ? (uint32_t)xsm[(size_t)M * NG * 32 + (size_t)t * NG + G] : 0u;
                    int sum = 0;
#pragma unroll
                    for (int wl = 0; wl < 4; ++wl) {
                        const uint32_t p0 = active ? wt[(2 * wl) * NG] : 0u;
                        const uint32_t p1 = active ? wt[(2 * wl + 1) * NG] : 0u;
                        sum = dp2a_lo_su(p0, 0x0101u, dp2a_lo_su(p1, 0x0101u, sum));
                        sl.xa[t][j][hh * 4 + wl][0] = p0;
                        sl.xa[t][j][hh * 4 + wl][1] = p1;
                    }
                    constexpr uint32_t XO = SW == 8 ? 13u : 14u;  // x16 = x * 2^(127 + XO - eb)
                    sl.xp[t][j][hh] = eb >= 27u ? __uint_as_float((eb - XO - 2u * j) << 23) : 0.f;
                    xsum[hh][j] = eb >= 27u ? (float)sum * __uint_as_float((eb - XO) << 23) : 0.f;
                }
            } else if constexpr (ACT == ACT_BF16) {
#pragma unroll
                for (int hh = 0; hh < S::NH; ++hh) {
                    // S::WPH*4 consecutive bf16 values, 8*WPH bytes, aligned to 8*WPH
                    uint32_t raw[S::WPH * 2];
                    const uint8_t* p = xt + 2 * (b * 256 + 128 * n + 32 * j + 4 * (wi0 + hh * S::WPH));
                    if constexpr (S::WPH >= 2) {
#pragma unroll
                        for (int q = 0; q < S::WPH / 2; ++q) {
                            const uint4 u = *reinterpret_cast<const uint4*>(p + 16 * q);
                            raw[4 * q] = u.x;
                            raw[4 * q + 1] = u.y;
                            raw[4 * q + 2] = u.z;
                            raw[4 * q + 3] = u.w;
                        }
                    } else {
                        const uint2 u = *reinterpret_cast<const uint2*>(p);
                        raw[0] = u.x;
                        raw[1] = u.y;
                    }
                    float v[S::WPH * 4];
                    float amax = 0.f;
#pragma unroll
                    for (int q = 0; q < S::WPH * 2; ++q) {
                        const float lo = active ? __uint_as_float(raw[q] << 16) : 0.f;
                        const float hi = active ? __uint_as_float(raw[q] & 0xFFFF0000u) : 0.f;
                        v[2 * q] = lo;
                        v[2 * q + 1] = hi;
                        amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
                    }
                    const uint32_t eb = (__float_as_uint(amax) >> 23) & 0xFFu;  // biased exponent of amax
                    int sum = 0;
                    if (eb >= 27u) {
                        // x16 = x * 2^(141-eb): |x16| < 2^15, exact for the group's
                        // largest 2^8 range; xp = 2^(eb-141) * 4^-j.
                        const float scale = __uint_as_float((268u - eb) << 23);
                        // round x*scale to an integer by adding 1.5*2^23 (its
                        // ulp is 1; ties to even, as rint): the integer is then
                        // the low mantissa bits, two's complement in 16 bits
#pragma unroll
                        for (int wl = 0; wl < S::WPH; ++wl) {
                            uint32_t f[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                f[i] = __float_as_uint(fmaf(v[wl * 4 + i], scale, 12582912.0f));
                            const uint32_t p0 = __byte_perm(f[0], f[1], 0x5410u);
                            const uint32_t p1 = __byte_perm(f[2], f[3], 0x5410u);
                            sum = dp2a_lo_su(p0, 0x0101u, dp2a_lo_su(p1, 0x0101u, sum));
                            sl.xa[t][j][hh * S::WPH + wl][0] = p0;
                            sl.xa[t][j][hh * S::WPH + wl][1] = p1;
                        }
                        sl.xp[t][j][hh] = __uint_as_float((eb - 14u - 2u * j) << 23);
                        xsum[hh][j] = (float)sum * __uint_as_float((eb - 14u) << 23);
                    } else {
#pragma unroll
                        for (int wl = 0; wl < S::WPH; ++wl) {
                            sl.xa[t][j][hh * S::WPH + wl][0] = 0u;
                            sl.xa[t][j][hh * S::WPH + wl][1] = 0u;
                        }
                        sl.xp[t][j][hh] = 0.f;
                        xsum[hh][j] = 0.f;
                    }
                }
            } else {
                // q8_1 block (b*8 + 4n + j) of the chunk: fp16 d at +0, q[32] at +4.
                const uint8_t* qb = xt + (b * 8 + 4 * n + j) * kQ8Bytes;
                const float d = active ? half_lo_f(lds32(qb)) : 0.f;
#pragma unroll
                for (int hh = 0; hh < S::NH; ++hh) {
                    int sum = 0;
#pragma unroll
                    for (int wl = 0; wl < S::WPH; ++wl) {
                        const int w = wi0 + hh * S::WPH + wl;
                        const uint32_t qv = active ? lds32(qb + 4 + 4 * w) : 0u;
                        sl.xa[t][j][hh * S::WPH + wl][0] = qv;
                        sum = dp4a_us(0x01010101u, qv, sum);
                    }
                    sl.xp[t][j][hh] = d * __uint_as_float((127u - 2u * j) << 23);
                    xsum[hh][j] = d * (float)sum;
                }
            }
        }
        if constexpr (SW == 8) {
            pack_sums8<M, ACT, SW>(sl, t, xsum);
        } else {
#pragma unroll
            for (int hh = 0; hh < S::NH; ++hh)
                pack_sums<M, ACT, SW>(sl, t, hh, xsum[hh]);
        }
    }
}

// One row's contribution of this thread's slice.  blk points at the block
// (in shared memory) holding the slice; n, wi0 as in load_slice.
template <int M, int ACT, int SW>
__device__ __forceinline__ void slice_dot(const Slice<M, ACT, SW>& sl, const uint8_t* blk, int n, int wi0,
                                          float (&acc)[M])
{
    using S = Slice<M, ACT, SW>;
    uint32_t qw[SW];
#pragma unroll
    for (int w = 0; w < SW; ++w)
        qw[w] = lds32(blk + 16 + 32 * n + 4 * (wi0 + w));
    const uint32_t s0 = lds32(blk + 8 * n);
    const uint32_t s1 = lds32(blk + 8 * n + 4);
    const uint32_t dm = lds32(blk + 80);
    const float d = half_lo_f(dm);
    const float dmin = half_hi_f(dm);
    if constexpr (SW == 8) {
        // A whole half block: sub-block 8n + 2j + h has its scale byte at
        // 2j + h of the two scale words.  The two halves h of bit plane j
        // share one activation scale, so their sums meet in int32
        // (|S| * 15 * 2 < 2^31) before the one conversion to float.
        const uint32_t scn[2] = {s0 & 0x0F0F0F0Fu, s1 & 0x0F0F0F0Fu};
        const uint32_t mnn[2] = {(s0 >> 4) & 0x0F0F0F0Fu, (s1 >> 4) & 0x0F0F0F0Fu};
#pragma unroll
        for (int t = 0; t < M; ++t) {
            // min term: the eight group sums against the eight min nibbles
            int Bi = dp2a_lo_su(sl.xs16[t][0][0], mnn[0], 0);
            Bi = dp2a_hi_su(sl.xs16[t][0][1], mnn[0], Bi);
            Bi = dp2a_lo_su(sl.xs16[t][1][0], mnn[1], Bi);
            Bi = dp2a_hi_su(sl.xs16[t][1][1], mnn[1], Bi);
            float A = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                int Sh[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    int Sacc = 0;
#pragma unroll
                    for (int wl = 0; wl < 4; ++wl) {
                        const int w = hh * 4 + wl;
                        const uint32_t c = qw[w] & (0x03030303u << (2 * j));
                        if constexpr (ACT == ACT_BF16) {
                            Sacc = dp2a_lo_su(sl.xa[t][j][w][0], c, Sacc);
                            Sacc = dp2a_hi_su(sl.xa[t][j][w][1], c, Sacc);
                        } else {
                            Sacc = dp4a_us(c, sl.xa[t][j][w][0], Sacc);
                        }
                    }
                    Sh[hh] = Sacc;
                }
                const int sc0 = (int)__byte_perm(scn[j >> 1], 0u, 0x4440u | (uint32_t)((2 * j) & 3));
                const int sc1 = (int)__byte_perm(scn[j >> 1], 0u, 0x4440u | (uint32_t)((2 * j + 1) & 3));
                A = fmaf(sl.xp[t][j][0], (float)(Sh[0] * sc0 + Sh[1] * sc1), A);
            }
            acc[t] = fmaf(d, A, fmaf(-dmin, sl.xsb[t][0] * (float)Bi, acc[t]));
        }
    } else {
#pragma unroll
        for (int hh = 0; hh < S::NH; ++hh) {
            const uint32_t h = (SW == 8) ? (uint32_t)hh : (uint32_t)(wi0 >> 2);
            // scale bytes of sub-blocks 8n + 2j + h, j = 0..3
            const uint32_t sb = __byte_perm(s0, s1, h | ((2u + h) << 4) | ((4u + h) << 8) | ((6u + h) << 12));
            const uint32_t scn = sb & 0x0F0F0F0Fu;
            const uint32_t mnn = (sb >> 4) & 0x0F0F0F0Fu;
            // scale nibbles as integers: the sub-block sum is scaled in int32
            // (|S| * 15 < 2^31) before its one conversion to float
            const int sci[4] = {(int)__byte_perm(scn, 0u, 0x4440u), (int)__byte_perm(scn, 0u, 0x4441u),
                                (int)__byte_perm(scn, 0u, 0x4442u), (int)__byte_perm(scn, 0u, 0x4443u)};
#pragma unroll
            for (int t = 0; t < M; ++t) {
                // min term: sum_j m_j * xsum_j as two 16x8-bit dot products
                const int Bi = dp2a_hi_su(sl.xs16[t][hh][1], mnn, dp2a_lo_su(sl.xs16[t][hh][0], mnn, 0));
                const float B = sl.xsb[t][hh] * (float)Bi;
                float A = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    int Sacc = 0;
#pragma unroll
                    for (int wl = 0; wl < S::WPH; ++wl) {
                        const int w = hh * S::WPH + wl;
                        const uint32_t c = qw[w] & (0x03030303u << (2 * j));
                        if constexpr (ACT == ACT_BF16) {
                            Sacc = dp2a_lo_su(sl.xa[t][j][w][0], c, Sacc);
                            Sacc = dp2a_hi_su(sl.xa[t][j][w][1], c, Sacc);
                        } else {
                            Sacc = dp4a_us(c, sl.xa[t][j][w][0], Sacc);
                        }
                    }
                    A = fmaf(sl.xp[t][j][hh], (float)(Sacc * sci[j]), A);
                }
                acc[t] = fmaf(d, A, fmaf(-dmin, B, acc[t]));
            }
        }
    }
}

// q8_1 activations made inside the kernel from the source rows staged at
// xsm + raw_off (one token): x_prep 1 quantises a bf16 row, x_prep 2 takes
// SwiGLU of an fp32 gate row and an fp32 up row first.  The same encoder and
// SwiGLU as the standalone kernels, so the bits are the same.  All threads.
template <typename Args>
__device__ __forceinline__ void prep_x_q8(const Args& a, uint8_t* xsm, int raw_off, int warp, int lane, int nwarps)
{
    const int nlanes = a.nbc * 8 * 8;  // q8_1 blocks of the chunk x 8 lanes
    const uint8_t* raw = xsm + raw_off;
    for (int wbase = warp * 32; wbase < nlanes; wbase += nwarps * 32) {  // warp-uniform
        const int u = wbase + lane;
        const bool live = u < nlanes;
        const int uu = live ? u : wbase;
        const int lane8 = uu & 7, blk = uu >> 3;
        const int k0 = blk * kQ8Values + 4 * lane8;
        float v[4];
        if (a.x_prep == 1) {
            const uint16_t* xb = reinterpret_cast<const uint16_t*>(raw);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                v[i] = live ? bf16_bits_f(xb[k0 + i]) : 0.f;
        } else {
            const float* g = reinterpret_cast<const float*>(raw);
            const float* up = g + a.nbc * 256;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                v[i] = live ? __bfloat162float(swiglu_bf16(g[k0 + i], up[k0 + i])) : 0.f;
        }
        q8_1_encode_group(v, xsm + blk * kQ8Bytes, lane8, live);
    }
}

// Sum VP values over the 32 lanes of a warp: after the exchanges each lane
// holds the full sum of value index lane >> (5 - log2 VP).
template <int VP>
__device__ __forceinline__ float transpose_reduce(float (&v)[VP], int lane)
{
#pragma unroll
    for (int n = VP / 2, o = 16; n >= 1; n >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float send = up ? v[i] : v[i + n];
            const float keep = up ? v[i + n] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float r = v[0];
#pragma unroll
    for (int o = 16 >> log2_exact(VP); o >= 1; o >>= 1)
        r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

}  // namespace q2k
