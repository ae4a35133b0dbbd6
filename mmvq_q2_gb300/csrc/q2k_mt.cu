// Q2_K projections for several tokens (m = 2..8) on the tensor cores.
//
// The decode pages run m <= 8 projections straight off Q2_K blocks
// (attn_v41/decode.rs, `q_kv_projections`; moe_v41/init.rs, the MMVQ
// kernels).  With more than one token the integer dot products of the
// one-token kernel spend most of their instructions on per-row work, so
// here each 16 x 16 piece of a Q2_K block is turned, in registers, into an
// MMA operand and multiplied against all tokens at once
// (mma.sync m16n8k16, bf16 in, fp32 accumulate):
//
//   A[r][e] = 128 + sc_s(r) * q(r, 16 s + e)      exact small integers in bf16
//   B[e][t] = x_t[256 b + 16 s + e]                bf16 activations (exact)
//
// for sub-block s of block b, row r and token t.  With q8_1 activations both
// operands are fp16 integers instead: A = 1024 + sc*q, B = the q8 values,
// and the accumulator input of a plane's first MMA is -1024 times the sum of
// its 32 q8 values, so the two MMAs of plane c (sub-blocks 2c, 2c+1, one
// q8_1 block) give sum sc*q*q8 exactly; it is scaled by d8 per plane.  Inside a sub-block the
// MMA's k order is permuted the same way on both sides: the thread that
// holds MMA k = 2c, 2c+1, 2c+8, 2c+9 takes weights and activations 4c..4c+3,
// so it reads one aligned qs word and 8 contiguous bytes of activations.  The constant 128 is added
// so that A is built by placing the byte sc*q under the bf16 exponent of
// 128.  It is taken out again with the block sums of B.  The min term uses
// a second MMA: A = 128 + m_s(r), B = the sub-block sums of x split into
// high and low bf16 parts.  Per row and block:
//
//   y_r += d * (acc - 128 X) - dmin * (accm - 128 Xm)
//
// Weights stream through a shared-memory ring of stages (a 16-row tile by a
// K chunk of 16 blocks), each filled by one 2-D tensor copy (rows 16 bytes
// aligned).  Warp w owns one block of every stage's tile and adds its
// partial sums into accumulators of its own in shared memory (per row and
// token), visiting the K chunks in order; after the walk the 16 warps'
// accumulators of each output are added in warp order, so results do not
// depend on timing or on which CTA holds a row.  The last warp out of a
// stage refills its slot; waits sleep in the mbarrier (bounded).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "q2k_common.cuh"
#include "q2k_internal.h"

namespace q2k {

__device__ int g_mt_error = 0;

namespace {

constexpr int kMtThreads = 512;
constexpr int kMtWarps = kMtThreads / 32;
constexpr int kTile = 16;  // weight rows per MMA tile (m16)
constexpr int kTok = 8;    // tokens per MMA (n8)
constexpr int kMtTilesPerCta = 8;  // bounds the warps' accumulators to 64 KB

struct MtArgs {
    const uint8_t* W[2];
    int N[2];              // rows of the two segments, concatenated
    int nb;                // blocks per row
    int64_t row_bytes;
    const uint8_t* x;      // bf16 rows or q8_1 rows
    int64_t x_tok_stride;  // bytes between tokens
    int m;
    int x_al8;             // bf16 rows allow 8-byte loads
    int x_tma;             // activations of each K chunk arrive by bulk copy into shared memory
    uint32_t xcb;          // bytes of one token's activations per full K chunk
    uint32_t xrs;          // their row stride in shared memory
    float* y[2];
    int64_t ldy[2];
    int nbc;               // blocks per K chunk
    int tps;               // tiles per stage (nbc * tps == 16 warps)
    int nchunks;
    int tiles0, tiles_total;
    int tiles_q, tiles_r;  // CTA c owns tiles_q (+1 if c < tiles_r) tiles
    int nst;
    uint32_t nst_magic;    // ceil(2^32 / nst)
    uint32_t stage_bytes;
    uint32_t rstride;      // bytes per row in a stage (nbc * 84)
    int w_aligned;         // every copied row piece is 16-byte aligned
    int yacc_rows;         // rows per warp accumulator: at most kMtTilesPerCta tiles
    uint32_t off_x, off_pl, off_yacc, off_bar, off_cnt;
};

struct Tile {
    int seg, row0, nrows, crow;  // crow: first row in the concatenated order
};

__device__ __forceinline__ Tile tile_at(const MtArgs& a, int T)
{
    if (T < a.tiles0) {
        const int r0 = T * kTile;
        return Tile{0, r0, min(kTile, a.N[0] - r0), r0};
    }
    const int r0 = (T - a.tiles0) * kTile;
    return Tile{1, r0, min(kTile, a.N[1] - r0), a.N[0] + r0};
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1, float c0, float c1, float c2, float c3)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

// 2-D tensor copy of box {x, y} (8-byte elements) into shared memory.
__device__ __forceinline__ void tensor_copy_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                               uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// Loads of the activations keep them in L2 (every CTA reads them, while the
// weights stream through with an evict-first policy).
__device__ __forceinline__ uint2 ldg64_keep(const void* p, uint64_t pol)
{
    uint2 v;
    asm volatile("ld.global.nc.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ uint32_t ldg32_keep(const void* p, uint64_t pol)
{
    uint32_t v;
    asm volatile("ld.global.nc.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ uint16_t bf16_bits(float v)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ float bf16_val(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint32_t pack2(uint16_t lo, uint16_t hi) { return (uint32_t)lo | ((uint32_t)hi << 16); }

// bf16 pairs (128 + byte0, 128 + byte1) and (128 + byte2, 128 + byte3) of v
// (each byte < 128): the byte becomes the mantissa under the exponent of 128.
__device__ __forceinline__ uint32_t lo_pair(uint32_t v) { return __byte_perm(v, 0x43434343u, 0x4140u); }
__device__ __forceinline__ uint32_t hi_pair(uint32_t v) { return __byte_perm(v, 0x43434343u, 0x4342u); }
// The same under the fp16 exponent of 1024 (each byte < 256).
__device__ __forceinline__ uint32_t lo_pair16(uint32_t v) { return __byte_perm(v, 0x64646464u, 0x4140u); }
__device__ __forceinline__ uint32_t hi_pair16(uint32_t v) { return __byte_perm(v, 0x64646464u, 0x4342u); }

// Two q8 values (signed bytes of w picked by SEL) as an exact fp16 pair: the
// bytes, offset by 128, go under the exponent of 1024 and 1152 comes off.
template <uint32_t SEL>
__device__ __forceinline__ uint32_t q8_pair_f16(uint32_t w)
{
    const uint32_t biased = __byte_perm(w ^ 0x80808080u, 0x64646464u, SEL);
    const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&biased),
                              __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
    return *reinterpret_cast<const uint32_t*>(&h);
}


// This warp's operands for block bb (all tokens), read from global memory
// (the activations are small and L2-resident):
//  bx      main MMA B fragments of the 16 sub-blocks: lane 4g + cq gets x_g
//          at 16 s + 4cq .. 4cq+3 (bf16 activations exactly; with q8_1 the
//          q8 values as fp16)
//  bmh/bml min MMA B fragment: sub-block sums of x_g for sub-blocks 4cq..4cq+3,
//          as bf16 high and low parts
//  xa, xm  for tokens 2cq and 2cq+1: what the main (bf16 only) and the min
//          MMA multiply by the constant 128 (the sums of their B operands
//          over the block)
//  pl      q8_1 only, the warp's table in shared memory: pl[4c + cq] for
//          plane c (sub-blocks 2c, 2c+1) holds, for tokens 2cq and 2cq+1,
//          the first MMA's accumulator input -1024 * (sum of the 32 q8
//          values) and d8
// Tokens m..7 (and blocks past the row) are zero.
struct BOps {
    uint2 bx[16];
    uint2 bmh, bml;
    float xa0, xa1, xm0, xm1;
};

// xrow0 / xstride: token 0's activations and the distance between tokens
// (global memory, or a K chunk staged in shared memory when SMEM); kb:
// the block's index from xrow0; live_b: the block exists.
template <int ACT, bool SMEM>
__device__ __forceinline__ void load_b(const MtArgs& a, const uint8_t* xrow0, int64_t xstride, int kb, bool live_b,
                                       int lane, BOps& o, float4* pl)
{
    const int g = lane >> 2, cq = lane & 3;
    const bool live = g < a.m && live_b;
    const uint8_t* xt = xrow0 + (int64_t)(live ? g : 0) * xstride;
    const uint64_t keep = l2_policy_evict_last();
    const int bb = live ? kb : 0;
    float ps[16];      // this lane's share of each sub-block sum of x
    int isum[16];      // q8_1: the same of the q8 values
    float d8c[8];      // q8_1: d8 of each plane
#pragma unroll
    for (int s = 0; s < 16; ++s) {
        const int k0 = bb * kBlockWeights + 16 * s + 4 * cq;  // activations k0..k0+3
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (ACT == ACT_BF16) {
            uint32_t w0 = 0u, w1 = 0u;
            if (live) {
                const uint8_t* p = xt + 2 * (int64_t)k0;
                if (SMEM) {
                    const uint2 u = *reinterpret_cast<const uint2*>(p);
                    w0 = u.x;
                    w1 = u.y;
                } else if (a.x_al8) {
                    const uint2 u = ldg64_keep(p, keep);
                    w0 = u.x;
                    w1 = u.y;
                } else {
                    const unsigned short* p16 = reinterpret_cast<const unsigned short*>(p);
                    w0 = pack2(__ldg(p16), __ldg(p16 + 1));
                    w1 = pack2(__ldg(p16 + 2), __ldg(p16 + 3));
                }
            }
            v[0] = __uint_as_float(w0 << 16);
            v[1] = __uint_as_float(w0 & 0xFFFF0000u);
            v[2] = __uint_as_float(w1 << 16);
            v[3] = __uint_as_float(w1 & 0xFFFF0000u);
            o.bx[s] = make_uint2(w0, w1);
        } else {
            float d8 = 0.f;
            uint32_t qv = 0u;
            if (live) {
                const uint8_t* qb = xt + (int64_t)(k0 >> 5) * kQ8Bytes;
                d8 = half_lo_f(SMEM ? lds32(qb) : ldg32_keep(qb, keep));
                qv = SMEM ? lds32(qb + 4 + (k0 & 31)) : ldg32_keep(qb + 4 + (k0 & 31), keep);
            }
            o.bx[s] = make_uint2(q8_pair_f16<0x4140u>(qv), q8_pair_f16<0x4342u>(qv));
            isum[s] = dp4a_us(0x01010101u, qv, 0);
            d8c[s >> 1] = d8;
        }
        // q8_1: d8 times the exact integer sum (one rounding)
        ps[s] = ACT == ACT_BF16 ? (v[0] + v[1]) + (v[2] + v[3]) : d8c[s >> 1] * (float)isum[s];
    }
    // sub-block sums over the four lanes of token g (same order in every lane)
    float xa = 0.f, xm = 0.f;
    float mine[4] = {0.f, 0.f, 0.f, 0.f};  // sums of sub-blocks 4cq..4cq+3
#pragma unroll
    for (int s = 0; s < 16; ++s) {
        float t = ps[s] + __shfl_xor_sync(0xffffffffu, ps[s], 1);
        t += __shfl_xor_sync(0xffffffffu, t, 2);
        const uint16_t hs = bf16_bits(t);
        xa += t;
        xm += bf16_val(hs) + bf16_val(bf16_bits(t - bf16_val(hs)));
        if ((s >> 2) == cq)  // this lane's min-MMA positions: sub-blocks 4cq..4cq+3
            mine[s & 3] = t;
    }
    uint16_t mh[4], ml[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        mh[i] = bf16_bits(mine[i]);
        ml[i] = bf16_bits(mine[i] - bf16_val(mh[i]));
    }
    o.bmh = make_uint2(pack2(mh[0], mh[1]), pack2(mh[2], mh[3]));
    o.bml = make_uint2(pack2(ml[0], ml[1]), pack2(ml[2], ml[3]));
    // the sums for tokens 2cq and 2cq+1 live in lanes 8cq and 8cq+4
    o.xa0 = __shfl_sync(0xffffffffu, xa, 8 * cq);
    o.xa1 = __shfl_sync(0xffffffffu, xa, 8 * cq + 4);
    o.xm0 = __shfl_sync(0xffffffffu, xm, 8 * cq);
    o.xm1 = __shfl_sync(0xffffffffu, xm, 8 * cq + 4);
    if constexpr (ACT != ACT_BF16) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            int S = isum[2 * c] + isum[2 * c + 1];
            S += __shfl_xor_sync(0xffffffffu, S, 1);
            S += __shfl_xor_sync(0xffffffffu, S, 2);
            const float cs = -1024.f * (float)S;  // exact: |S| <= 4064
            const float4 v = make_float4(__shfl_sync(0xffffffffu, cs, 8 * cq), __shfl_sync(0xffffffffu, cs, 8 * cq + 4),
                                         __shfl_sync(0xffffffffu, d8c[c], 8 * cq),
                                         __shfl_sync(0xffffffffu, d8c[c], 8 * cq + 4));
            if (g == 0)
                pl[4 * c + cq] = v;
        }
        __syncwarp();
    }
}

// One 16-row tile by one Q2_K block (256 weights of each row) against the
// tokens: 16 main MMAs, 2 min MMAs, then the d / dmin (and, with q8_1, the
// per-plane d8) scaling into this thread's four outputs (rows g, g+8;
// tokens 2cq, 2cq+1).
template <int ACT>
__device__ __forceinline__ void mt_block(const uint8_t* blk0, const uint8_t* blk1, const BOps& o,
                                         const float4* pl_tab, int cq, float (&part)[4])
{
    uint32_t sw0[4], sw1[4];  // scale nibbles of sub-blocks 0..15, one per byte
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        sw0[q] = lds32(blk0 + 4 * q) & 0x0F0F0F0Fu;
        sw1[q] = lds32(blk1 + 4 * q) & 0x0F0F0F0Fu;
    }
    const uint32_t dm0 = lds32(blk0 + 80), dm1 = lds32(blk1 + 80);
    // qs bytes 4cq..4cq+3 of each 16-byte quarter (2n + h)
    uint32_t qw0[4], qw1[4];
#pragma unroll
    for (int nh = 0; nh < 4; ++nh) {
        qw0[nh] = lds32(blk0 + 16 + 16 * nh + 4 * cq);
        qw1[nh] = lds32(blk1 + 16 + 16 * nh + 4 * cq);
    }
    // bytes sc*q <= 45 of sub-block s = 8n + 2j + h: codes at bits 2j of
    // quarter 2n + h, times the scale (bytewise, no carries)
    auto scaled = [&](int s, uint32_t& v0, uint32_t& v1) {
        const int nh = ((s >> 3) << 1) | (s & 1);
        const int sh = 2 * ((s >> 1) & 3);
        const uint32_t c0 = (qw0[nh] >> sh) & 0x03030303u;
        const uint32_t c1 = (qw1[nh] >> sh) & 0x03030303u;
        const uint32_t k0 = __byte_perm(sw0[s >> 2], 0u, 0x4440u | (uint32_t)(s & 3));
        const uint32_t k1 = __byte_perm(sw1[s >> 2], 0u, 0x4440u | (uint32_t)(s & 3));
        v0 = c0 * k0;
        v1 = c1 * k1;
    };
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (ACT == ACT_BF16) {
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            uint32_t v0, v1;
            scaled(s, v0, v1);
            mma_bf16(acc, lo_pair(v0), lo_pair(v1), hi_pair(v0), hi_pair(v1), o.bx[s].x, o.bx[s].y);
        }
    } else {
        // plane c: sub-blocks 2c and 2c+1 share one q8_1 block
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 pl = pl_tab[4 * c + cq];
            float d[4];
            uint32_t v0, v1;
            scaled(2 * c, v0, v1);
            mma_f16(d, lo_pair16(v0), lo_pair16(v1), hi_pair16(v0), hi_pair16(v1), o.bx[2 * c].x, o.bx[2 * c].y,
                    pl.x, pl.y, pl.x, pl.y);
            scaled(2 * c + 1, v0, v1);
            mma_f16(d, lo_pair16(v0), lo_pair16(v1), hi_pair16(v0), hi_pair16(v1), o.bx[2 * c + 1].x,
                    o.bx[2 * c + 1].y, d[0], d[1], d[2], d[3]);
            acc[0] = fmaf(pl.z, d[0], acc[0]);
            acc[1] = fmaf(pl.w, d[1], acc[1]);
            acc[2] = fmaf(pl.z, d[2], acc[2]);
            acc[3] = fmaf(pl.w, d[3], acc[3]);
        }
    }
    // min term: A = 128 + m over sub-blocks 4cq..4cq+3 (scale bytes 4cq..4cq+3)
    const uint32_t m0 = (lds32(blk0 + 4 * cq) >> 4) & 0x0F0F0F0Fu;
    const uint32_t m1 = (lds32(blk1 + 4 * cq) >> 4) & 0x0F0F0F0Fu;
    float accm[4] = {0.f, 0.f, 0.f, 0.f};
    mma_bf16(accm, lo_pair(m0), lo_pair(m1), hi_pair(m0), hi_pair(m1), o.bmh.x, o.bmh.y);
    mma_bf16(accm, lo_pair(m0), lo_pair(m1), hi_pair(m0), hi_pair(m1), o.bml.x, o.bml.y);
    const float d0 = half_lo_f(dm0), n0 = half_hi_f(dm0);
    const float d1 = half_lo_f(dm1), n1 = half_hi_f(dm1);
    const float xa0 = ACT == ACT_BF16 ? 128.f * o.xa0 : 0.f, xa1 = ACT == ACT_BF16 ? 128.f * o.xa1 : 0.f;
    const float xm0 = 128.f * o.xm0, xm1 = 128.f * o.xm1;
    part[0] += d0 * (acc[0] - xa0) - n0 * (accm[0] - xm0);
    part[1] += d0 * (acc[1] - xa1) - n0 * (accm[1] - xm1);
    part[2] += d1 * (acc[2] - xa0) - n1 * (accm[2] - xm0);
    part[3] += d1 * (acc[3] - xa1) - n1 * (accm[3] - xm1);
}

template <int ACT>
__global__ void __launch_bounds__(kMtThreads, 1)
    q2k_mt_kernel(const MtArgs a, const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1)
{
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_launch_dependents();  // the next kernel may set itself up meanwhile
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, cq = lane & 3;  // MMA fragment row group and column pair

    uint8_t* ring = smem;
    uint64_t* full_b = reinterpret_cast<uint64_t*>(smem + a.off_bar);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(full_b + a.nst);
    int* done = reinterpret_cast<int*>(smem + a.off_cnt);  // warps finished with the slot's stage
    int* n_issued = done + a.nst;
    int* x_done = n_issued + 1;    // warps holding the current chunk's activations
    int* x_issued = x_done + 1;    // activation chunks copied in
    uint64_t* xbar = full_b + a.nst + 1;
    uint8_t* xs = smem + a.off_x;
    float4* plw = reinterpret_cast<float4*>(smem + a.off_pl) + warp * 32;  // this warp's per-plane q8_1 scalars
    float* yacc = reinterpret_cast<float*>(smem + a.off_yacc);  // [16 warps][rows of this CTA][8 tokens]

    const int cta = blockIdx.x;
    const int tlo = cta * a.tiles_q + min(cta, a.tiles_r);
    const int thi = tlo + a.tiles_q + (cta < a.tiles_r ? 1 : 0);
    const int ngroups = (thi - tlo + a.tps - 1) / a.tps;
    const int nstages = ngroups * a.nchunks;
    const int crow0 = thi > tlo ? tile_at(a, tlo).crow : 0;
    const int pre = min(a.nst, nstages);

    auto ring_pos = [&](int i, int& slot, uint32_t& parity) {
        const int q = (int)__umulhi((uint32_t)i, a.nst_magic);
        slot = i - q * a.nst;
        parity = (uint32_t)q & 1u;
    };

    if (lane == 0) {
        if (tid == 0) {
            *abort_flag = 0;
            for (int s2 = 0; s2 < a.nst; ++s2)
                done[s2] = 0;
            *n_issued = 0;
            *x_done = 0;
            *x_issued = 0;
            mbar_init(smem_u32(xbar), 1);
        }
        for (int s2 = warp; s2 < a.nst; s2 += kMtWarps)
            mbar_init(smem_u32(&full_b[s2]), 1);
        fence_mbar_init();
    }
    for (int i = tid; i < kMtWarps * a.yacc_rows * kTok; i += blockDim.x)
        yacc[i] = 0.f;
    // global memory may still be written by the previous kernel in the stream
    pdl_wait();
    __syncthreads();

    // ---- producer role: stage j (K chunk, tile group) into its ring slot.
    // Lane L copies row piece L (tile L / 16, row L % 16) with a bulk copy;
    // unaligned pieces are copied by the whole warp with 4-byte loads. ----
    auto produce = [&](int j) {
        int slot;
        uint32_t parity;
        ring_pos(j, slot, parity);
        const int cs = j / ngroups;
        const int c = cs;
        const int t0 = tlo + (j - cs * ngroups) * a.tps;
        const int nbc_c = min(a.nbc, a.nb - c * a.nbc);
        const uint32_t piece = (uint32_t)nbc_c * kBlockBytes;  // bytes of a row in this chunk
        uint8_t* dst0 = ring + (size_t)slot * a.stage_bytes;
        const uint32_t fb = smem_u32(&full_b[slot]);
        auto src_of = [&](int L, bool& ok) {
            const int tt = L >> 4, r = L & 15;
            ok = false;
            if (tt >= a.tps || t0 + tt >= thi)
                return (const uint8_t*)nullptr;
            const Tile t = tile_at(a, t0 + tt);
            if (r >= t.nrows)
                return (const uint8_t*)nullptr;
            ok = true;
            return a.W[t.seg] + (int64_t)(t.row0 + r) * a.row_bytes + (int64_t)c * a.nbc * kBlockBytes;
        };
        if (a.w_aligned) {
            // one tensor copy of the tile's rows; rows past the matrix and
            // bytes past the row end are filled with zeros (and counted)
            if (lane == 0) {
                const Tile t = tile_at(a, t0);
                mbar_arrive_expect_tx(fb, a.stage_bytes);
                tensor_copy_2d(smem_u32(dst0), t.seg == 0 ? &tm0 : &tm1, (int)(c * (a.rstride / 8)), t.row0, fb,
                               l2_policy_evict_first());
            }
        } else {
            const uint32_t words = piece >> 2;
            for (int L = 0; L < a.tps * kTile; ++L) {
                bool ok;
                const uint8_t* src = src_of(L, ok);
                if (!ok)
                    continue;
                uint32_t* dst = reinterpret_cast<uint32_t*>(dst0 + (size_t)L * a.rstride);
                for (uint32_t w = lane; w < words; w += 32)
                    dst[w] = ldg32_nc(src + 4 * w);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(fb);
        }
        if (lane == 0)
            atomicAdd(n_issued, 1);
    };
    // Wait for stage data; gives up after ~2 s.
    auto wait_stage = [&](int slot, uint32_t parity) -> bool {
        const bool ok =
            __all_sync(0xffffffffu, !*abort_flag && mbar_wait_bounded(smem_u32(&full_b[slot]), parity, abort_flag));
        if (!ok && lane == 0) {
            atomicOr(&g_mt_error, Q2K_ERR_BIT_WAIT_TIMEOUT);
            *abort_flag = 1;
        }
        return ok;
    };

    // Activations of K chunk c into shared memory (one thread): one bulk copy
    // per token, kept in L2 for the other CTAs.
    auto issue_x = [&](int c) {
        const int nbc_c = min(a.nbc, a.nb - c * a.nbc);
        const uint32_t bytes = (uint32_t)nbc_c * (ACT == ACT_BF16 ? 512u : 8u * kQ8Bytes);
        const uint64_t keep = l2_policy_evict_last();
        mbar_arrive_expect_tx(smem_u32(xbar), bytes * (uint32_t)a.m);
        for (int t = 0; t < a.m; ++t)
            bulk_copy_g2s_hint(smem_u32(xs + (size_t)t * a.xrs), a.x + (int64_t)t * a.x_tok_stride + (int64_t)c * a.xcb,
                               bytes, smem_u32(xbar), keep);
        atomicAdd(x_issued, 1);
    };
    auto wait_x = [&](uint32_t par) -> bool {
        const bool ok = __all_sync(0xffffffffu, !*abort_flag && mbar_wait_bounded(smem_u32(xbar), par, abort_flag));
        if (!ok && lane == 0) {
            atomicOr(&g_mt_error, Q2K_ERR_BIT_WAIT_TIMEOUT);
            *abort_flag = 1;
        }
        return ok;
    };

    if (tid == 0 && a.x_tma)
        issue_x(0);  // the first activations ahead of the weights
    if (warp < pre)
        produce(warp);

    const int tt_w = warp / a.nbc;          // this warp's tile within a stage
    const int bb_w = warp - tt_w * a.nbc;   // and its block within the K chunk
    bool aborted = false;
    float* yw = yacc + (size_t)warp * a.yacc_rows * kTok;  // this warp's accumulators
    BOps ops;  // this warp's B operands for the current K chunk
    int c = 0, gidx = 0, chunk_seq = 0;
    for (int i = 0; i < nstages; ++i) {
        if (gidx == 0) {
            const int kb = c * a.nbc + bb_w;
            if (a.x_tma) {
                // this chunk's activations are in shared memory; the last
                // warp to take its operands copies the next chunk in
                if (!aborted && !wait_x((uint32_t)chunk_seq & 1u))
                    aborted = true;
                load_b<ACT, true>(a, xs, a.xrs, bb_w, kb < a.nb, lane, ops, plw);
                __syncwarp();
                int lastx = 0;
                if (lane == 0) {
                    __threadfence_block();
                    lastx = atomicAdd(x_done, 1) == kMtWarps - 1;
                    if (lastx) {
                        atomicExch(x_done, 0);
                        __threadfence_block();
                        if (chunk_seq + 1 < a.nchunks)
                            issue_x(c + 1 == a.nchunks ? 0 : c + 1);
                    }
                }
            } else {
                load_b<ACT, false>(a, a.x, a.x_tok_stride, kb, kb < a.nb, lane, ops, plw);
            }
            ++chunk_seq;
        }
        int slot;
        uint32_t parity;
        ring_pos(i, slot, parity);
        const int t0 = tlo + gidx * a.tps;
        const int nbc_c = min(a.nbc, a.nb - c * a.nbc);
        if (!aborted && !wait_stage(slot, parity))
            aborted = true;
        if (!aborted && bb_w < nbc_c && t0 + tt_w < thi) {
            const uint8_t* blk0 = ring + (size_t)slot * a.stage_bytes + (size_t)(tt_w * kTile + g) * a.rstride +
                                  (size_t)bb_w * kBlockBytes;
            const uint8_t* blk1 = blk0 + (size_t)8 * a.rstride;
            float part[4] = {0.f, 0.f, 0.f, 0.f};
            mt_block<ACT>(blk0, blk1, ops, plw, cq, part);
            // rows g and g+8 of the tile, tokens 2cq and 2cq+1: this warp's
            // accumulators, added in chunk order
            const Tile t = tile_at(a, t0 + tt_w);
            float* y0 = yw + (size_t)(t.crow - crow0 + g) * kTok + 2 * cq;
            if (g < t.nrows) {
                y0[0] += part[0];
                y0[1] += part[1];
            }
            if (g + 8 < t.nrows) {
                y0[8 * kTok] += part[2];
                y0[8 * kTok + 1] += part[3];
            }
        }
        // release; the last warp out refills the slot
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&done[slot], 1) == kMtWarps - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            if (lane == 0)
                done[slot] = 0;
            __syncwarp();
            if (i + a.nst < nstages && !*abort_flag)
                produce(i + a.nst);
        }
        if (++gidx == ngroups) {
            gidx = 0;
            if (++c == a.nchunks)
                c = 0;
        }
    }

    // every issued copy must have landed before the CTA exits
    __syncthreads();
    if (*abort_flag) {
        if (tid == 0) {
            const int issued = *reinterpret_cast<volatile int*>(n_issued);
            for (int i = max(0, issued - a.nst); i < issued; ++i) {
                int slot;
                uint32_t parity;
                ring_pos(i, slot, parity);
                mbar_wait_bounded(smem_u32(&full_b[slot]), parity, nullptr);
            }
            const int xi = *reinterpret_cast<volatile int*>(x_issued);
            if (xi > 0)
                mbar_wait_bounded(smem_u32(xbar), (uint32_t)(xi - 1) & 1u, nullptr);
        }
        __syncthreads();
        return;
    }
    __syncthreads();
    // ---- outputs: rows of this CTA in order, token-major for coalescing ----
    if (thi > tlo) {
        const Tile tl = tile_at(a, thi - 1);
        const int nrows = tl.crow + tl.nrows - crow0;
        for (int q = tid; q < nrows * a.m; q += blockDim.x) {
            const int t = q / nrows, r = q - t * nrows;
            const int crow = crow0 + r;
            const int seg = crow < a.N[0] ? 0 : 1;
            const int row = seg == 0 ? crow : crow - a.N[0];
            float v = 0.f;
            for (int w = 0; w < kMtWarps; ++w)  // the warps' accumulators in warp order
                v += yacc[((size_t)w * a.yacc_rows + r) * kTok + t];
            a.y[seg][(int64_t)t * a.ldy[seg] + row] = v;
        }
    }
}


size_t mt_align16(size_t v) { return (v + 15) / 16 * 16; }

// cuTensorMapEncodeTiled, found once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Map of a Q2_K matrix as rows of 8-byte elements; box = one tile (16
// rows) by one K chunk.
bool encode_rows(CUtensorMap* map, const void* W, int64_t rows, int64_t row_bytes, uint32_t chunk_bytes)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || rows <= 0)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 8), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {chunk_bytes / 8, (cuuint32_t)kTile};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(W), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int ACT>
cudaError_t launch_mt_one(const MtArgs& a, const CUtensorMap& tm0, const CUtensorMap& tm1, int grid, size_t smem,
                          cudaStream_t s)
{
    auto k = q2k_mt_kernel<ACT>;
    static std::atomic<unsigned long long> smem_devs{0};
    cudaError_t e = allow_max_smem(k, smem_devs);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(k, dim3((unsigned)grid), dim3(kMtThreads), smem, s, a, tm0, tm1);
}

}  // namespace

bool mt_supported(const MvProblem& p)
{
    // from the token counts on where it beats the integer-dot kernel
    const int m_min = p.act == ACT_Q8 ? 5 : 3;
    return p.W_table == nullptr && p.w_seg_stride == 0 && p.m >= m_min && p.m <= kTok &&
           (p.n_seg == 1 || p.x_seg_stride == 0);
}

cudaError_t launch_mt(const MvProblem& p, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess)
        return err;
    if (!mt_supported(p))
        return cudaErrorInvalidValue;
    MtArgs a{};
    a.W[0] = static_cast<const uint8_t*>(p.W[0]);
    a.W[1] = static_cast<const uint8_t*>(p.n_seg > 1 ? p.W[1] : p.W[0]);
    a.N[0] = (int)p.N[0];
    a.N[1] = p.n_seg > 1 ? (int)p.N[1] : 0;
    a.nb = (int)(p.K / kBlockWeights);
    a.row_bytes = (int64_t)a.nb * kBlockBytes;
    a.x = static_cast<const uint8_t*>(p.x);
    a.x_tok_stride = p.x_tok_stride;
    a.m = p.m;
    a.x_al8 = ((reinterpret_cast<uintptr_t>(p.x) | (uintptr_t)p.x_tok_stride) & 7u) == 0 ? 1 : 0;

    for (int e = 0; e < 2; ++e) {
        a.y[e] = p.y[e] ? p.y[e] : p.y[0];
        a.ldy[e] = p.ldy[e];
    }
    const bool q8 = p.act == ACT_Q8;
    a.nbc = kMtWarps;  // one block of the K chunk per warp
    a.tps = 1;
    a.nchunks = (a.nb + a.nbc - 1) / a.nbc;
    a.tiles0 = (a.N[0] + kTile - 1) / kTile;
    a.tiles_total = a.tiles0 + (a.N[1] + kTile - 1) / kTile;
    // one CTA per SM; more CTAs (in waves) when a CTA would own more than
    // kMtTilesPerCta tiles (each warp keeps an accumulator per row and token)
    const int grid = std::min(a.tiles_total,
                              std::max(di.sm_count, (a.tiles_total + kMtTilesPerCta - 1) / kMtTilesPerCta));
    a.tiles_q = a.tiles_total / grid;
    a.tiles_r = a.tiles_total % grid;
    a.rstride = (uint32_t)(a.nbc * kBlockBytes);
    a.xcb = (uint32_t)a.nbc * (q8 ? 8u * kQ8Bytes : 512u);  // a multiple of 16
    a.xrs = a.xcb + 16;                                     // padded: fewer bank conflicts
    a.x_tma = ((reinterpret_cast<uintptr_t>(p.x) | (uintptr_t)p.x_tok_stride) & 15u) == 0 ? 1 : 0;
    a.stage_bytes = (uint32_t)(a.tps * kTile) * a.rstride;
    a.w_aligned = ((reinterpret_cast<uintptr_t>(a.W[0]) | reinterpret_cast<uintptr_t>(a.W[1])) & 15u) == 0 &&
                  a.nb % 4 == 0;
    a.yacc_rows = (a.tiles_q + 1) * kTile;
    const size_t smem_cap = std::min<size_t>((size_t)di.smem_optin, 224 * 1024);
    size_t smem = 0;
    int nst = 8;
    for (; nst >= 2; --nst) {
        a.nst = nst;
        size_t off = (size_t)nst * a.stage_bytes;
        a.off_x = (uint32_t)off;
        off += a.x_tma ? (((size_t)a.m * a.xrs + 127) / 128 * 128) : 0;
        a.off_pl = (uint32_t)off;
        off += q8 ? (size_t)kMtWarps * 32 * sizeof(float4) : 0;
        a.off_yacc = (uint32_t)off;
        off += mt_align16((size_t)kMtWarps * a.yacc_rows * kTok * sizeof(float));
        a.off_bar = (uint32_t)off;
        off += mt_align16((size_t)(nst + 2) * sizeof(uint64_t));
        a.off_cnt = (uint32_t)off;
        off += mt_align16((size_t)(nst + 5) * sizeof(int));
        smem = off;
        if (smem <= smem_cap)
            break;
    }
    if (nst < 2)
        return cudaErrorInvalidConfiguration;
    a.nst_magic = (uint32_t)((0x100000000ull + (uint64_t)a.nst - 1) / (uint64_t)a.nst);
    CUtensorMap tm0{}, tm1{};
    if (a.w_aligned) {
        const bool ok = encode_rows(&tm0, a.W[0], a.N[0], a.row_bytes, a.rstride) &&
                        (a.N[1] == 0 || encode_rows(&tm1, a.W[1], a.N[1], a.row_bytes, a.rstride));
        if (!ok)
            a.w_aligned = 0;  // the warp-copy path
        else if (a.N[1] == 0)
            tm1 = tm0;
    }
    return q8 ? launch_mt_one<ACT_Q8>(a, tm0, tm1, grid, smem, s) : launch_mt_one<ACT_BF16>(a, tm0, tm1, grid, smem, s);
}

cudaError_t mt_error_word(int32_t* out, bool clear)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_mt_error, sizeof(int));
    if (e != cudaSuccess)
        return e;
    *out = v;
    if (clear) {
        int z = 0;
        e = cudaMemcpyToSymbol(g_mt_error, &z, sizeof(int));
    }
    return e;
}

}  // namespace q2k
