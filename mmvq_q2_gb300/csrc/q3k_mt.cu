// Q3_K projections with q8_1 activations for several tokens on the tensor
// cores: the several-token form of the Q3_K MMVQ twin that moe_v41/init.rs
// (`MoeV41::new`) loads beside the Q2_K kernels (`kquant_mmvq_q3_k_w`).
//
// Block (110 bytes, 256 weights): hmask[32] | qs[64] | scales[12] | d (fp16).
// Weight p = 128n + 32j + l has the 2-bit code at bit 2j of qs[32n + l], the
// high bit at bit 4n + j of hmask[l], the 6-bit scale (stored + 32) of
// sub-block 8n + 2j + l/16, and the value d * sc * q with q = code + 4*high
// - 4 in [-4, 3] and sc = stored - 32 in [-32, 31].  All 32 weights of one
// plane c = 4n + j share q8_1 block c of the activations (one d8).
//
// With several tokens the integer dot products of the one-token kernel spend
// their instructions per row and per token pair; here each plane of a
// 16-row tile becomes two mma.sync m16n8k16 (fp16 in, fp32 accumulate)
// against all tokens at once, with exact small integers on both sides:
//
//   A[r][k] = 1152 + sc(r) * q(r, k)    in [1028, 1280]: fp16 0x6480 + sc*q
//   B[k][t] = q8 value of token t        in [-127, 127]
//   C[r][t] = -1152 * (sum of token t's 32 q8 values of the plane)
//
// so the MMA result is sum_k sc*q*q8 exactly (every partial sum is an
// integer below 2^23).  A is built with integer arithmetic on packed 16-bit
// lanes: with u = code + 4*high in [0, 7] in each lane,
// (0x6480 - 4*sc) * 0x00010001 + sc * (u0 | u1 << 16) holds both fp16 bit
// patterns (each lane stays in [0, 2^16), so the 32-bit product is exact).
// Per row, plane and token the result is scaled by d8, and per block by d.
//
// The MMA's k order inside a plane is permuted the same way on A and B: the
// thread holding k = 2cq, 2cq+1, 2cq+8, 2cq+9 of the first MMA takes bytes
// l = 8cq, 8cq+2, 8cq+1, 8cq+3, and of the second MMA 8cq+4 .. 8cq+7 in the
// same pattern, so it reads two consecutive qs and hmask words per row.
//
// Weights stream through a shared-memory ring of stages (a 16-row tile by a
// K chunk of 16 blocks, 1760 bytes a row), each filled by one 2-D tensor
// copy when the rows are 16-byte multiples, else by warp copies.  Warp w
// owns block w of every stage; blocks 110 bytes apart alternate between
// word-aligned and 2 bytes off, so fields are read as aligned words and
// funnel-shifted.  Each warp keeps accumulators of its own per row and
// token, visits the K chunks in order, and after the walk the 16 warps'
// accumulators are added in warp order: the result does not depend on
// timing.  The last warp out of a stage refills its slot; waits are bounded.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "q2k_common.cuh"
#include "q2k_internal.h"

namespace q2k {

__device__ int g_q3mt_error = 0;

namespace {

constexpr int kQ3Bytes = 110;
constexpr int kQtThreads = 512;
constexpr int kQtWarps = kQtThreads / 32;
constexpr int kTile = 16;          // weight rows per MMA tile (m16)
constexpr int kTok = 8;            // tokens per MMA (n8)
constexpr int kChunkBlocks = 16;   // blocks per K chunk: one per warp
constexpr int kTilesPerCta = 8;    // bounds the warps' accumulators
constexpr uint32_t kRowPiece = kChunkBlocks * kQ3Bytes;  // 1760 bytes of a row per stage
constexpr uint32_t kXBlockBytes = 8 * kQ8Bytes;           // q8_1 bytes of one Q3_K block column

struct QtArgs {
    const uint8_t* W;
    int N;
    int nb;                // blocks per row
    int64_t row_bytes;
    const uint8_t* x;      // q8_1 rows
    int64_t x_tok_stride;  // bytes between tokens
    int m;
    int x_tma;             // each K chunk's activations arrive by bulk copy
    uint32_t xcb;          // bytes of one token's activations per full chunk
    uint32_t xrs;          // their row stride in shared memory
    float* y;
    int64_t ldy;
    int nchunks;
    int tiles;
    int tiles_q, tiles_r;  // CTA c owns tiles_q (+1 if c < tiles_r) tiles
    int nst;
    uint32_t nst_magic;    // ceil(2^32 / nst)
    uint32_t stage_bytes;
    int w_tma;             // stages arrive by tensor copy
    int yacc_rows;
    uint32_t off_x, off_ops, off_yacc, off_bar, off_cnt;
};

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1, float c0, float c1, float c2, float c3)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

__device__ __forceinline__ void tensor_copy_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                               uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint32_t ldx32(const uint8_t* p, bool smem)
{
    return smem ? lds32(p) : __ldg(reinterpret_cast<const unsigned int*>(p));
}

// Two q8 values (bytes e0 and e1 of w, signed) as an fp16 pair: each byte,
// offset by 128, becomes the mantissa under the exponent of 1024, and 1152
// is taken off again (exact).
template <uint32_t SEL>
__device__ __forceinline__ uint32_t q8_pair_f16(uint32_t w_flipped)
{
    const uint32_t biased = __byte_perm(w_flipped, 0x64646464u, SEL);
    const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&biased), __halves2half2(__ushort_as_half(0x6480),
                                                                                          __ushort_as_half(0x6480)));
    return *reinterpret_cast<const uint32_t*>(&h);
}

// This warp's B operands for the block at kb (all tokens), and the per-plane
// scalars of the thread's two output tokens, from q8_1 rows starting at
// xrow0 (global memory, or a K chunk staged in shared memory when SMEM):
//  b[c][0..1]  first MMA of plane c: (q8 l=8cq, 8cq+2), (8cq+1, 8cq+3) of token g
//  b[c][2..3]  second MMA: the same at 8cq+4 .. 8cq+7
//  ops[c][cq]  (-1152*S(2cq), -1152*S(2cq+1), d8(2cq), d8(2cq+1)), S the sum
//              of the plane's 32 q8 values, in this warp's shared table
// Tokens m..7 and blocks past the row are zero.
template <bool SMEM>
__device__ __forceinline__ void load_b(const QtArgs& a, const uint8_t* xrow0, int64_t xstride, int kb, bool live_b,
                                       int lane, uint32_t (&b)[8][4], float4* ops)
{
    const int g = lane >> 2, cq = lane & 3;
    const bool live = g < a.m && live_b;
    const uint8_t* xt = xrow0 + (int64_t)(live ? g : 0) * xstride + (int64_t)(live ? kb : 0) * kXBlockBytes;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint8_t* qb = xt + c * kQ8Bytes;
        float d8 = 0.f;
        uint32_t w0 = 0u, w1 = 0u;
        if (live) {
            d8 = half_lo_f(ldx32(qb, SMEM));
            w0 = ldx32(qb + 4 + 8 * cq, SMEM);
            w1 = ldx32(qb + 8 + 8 * cq, SMEM);
        }
        int s = dp4a_us(0x01010101u, w0, 0);
        s = dp4a_us(0x01010101u, w1, s);
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        const uint32_t f0 = w0 ^ 0x80808080u, f1 = w1 ^ 0x80808080u;
        b[c][0] = q8_pair_f16<0x4240u>(f0);
        b[c][1] = q8_pair_f16<0x4341u>(f0);
        b[c][2] = q8_pair_f16<0x4240u>(f1);
        b[c][3] = q8_pair_f16<0x4341u>(f1);
        const float cs = -1152.f * (float)s;  // exact: |s| <= 4064
        // tokens 2cq and 2cq+1 live in lanes 8cq and 8cq+4
        const float cs0 = __shfl_sync(0xffffffffu, cs, 8 * cq);
        const float cs1 = __shfl_sync(0xffffffffu, cs, 8 * cq + 4);
        const float e0 = __shfl_sync(0xffffffffu, d8, 8 * cq);
        const float e1 = __shfl_sync(0xffffffffu, d8, 8 * cq + 4);
        if (g == 0)
            ops[c * 4 + cq] = make_float4(cs0, cs1, e0, e1);
    }
    __syncwarp();
}

// One row's fields for thread cq from the block at blk (2-byte aligned; sh =
// 0 when it starts on a word, 16 when 2 bytes off): hmask and qs bytes
// 8cq .. 8cq+7 (qs of both halves n), the 6-bit scales of the thread's
// sub-blocks 8n + 2j + cq/2 as bytes j of s6[n] in 6-bit two's complement
// (stored value XOR 32 = sc), and d.
struct Q3Row {
    uint32_t q[2][2], h[2], s6[2];
    float d;
};

__device__ __forceinline__ void read_row(const uint8_t* blk, uint32_t sh, uint32_t lsel, uint32_t hsel, int cq,
                                         Q3Row& f)
{
    const uint32_t* pa = reinterpret_cast<const uint32_t*>(reinterpret_cast<uintptr_t>(blk) & ~uintptr_t(3));
    // the two words at byte o of the block (o a multiple of 4): three
    // aligned words and funnel shifts; bytes read stay inside the block
    auto two = [&](int o, uint32_t& lo, uint32_t& hi) {
        const uint32_t w0 = pa[o / 4], w1 = pa[o / 4 + 1], w2 = pa[o / 4 + 2];
        lo = __funnelshift_r(w0, w1, sh);
        hi = __funnelshift_r(w1, w2, sh);
    };
    two(8 * cq, f.h[0], f.h[1]);
    two(32 + 8 * cq, f.q[0][0], f.q[0][1]);
    two(64 + 8 * cq, f.q[1][0], f.q[1][1]);
    // scales[12] at byte 96 (the last aligned word read may hold the 2 bytes
    // after the block: unused, and inside the shared-memory allocation)
    uint32_t w[4], sc[3];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = pa[24 + i];
#pragma unroll
    for (int i = 0; i < 3; ++i)
        sc[i] = __funnelshift_r(w[i], w[i + 1], sh);
    // low nibbles of sub-blocks 2j + hh (bytes j of L), their top two bits
    // from scales[8 + 2(j&1) + hh] at bit 2(2n + j/2)
    const uint32_t L = __byte_perm(sc[0], sc[1], lsel);
    const uint32_t H = __byte_perm(sc[2], 0u, hsel);
    const uint32_t s0 = (L & 0x0F0F0F0Fu) | (((H & 0x00000303u) | ((H >> 2) & 0x03030000u)) << 4);
    const uint32_t s1 = ((L >> 4) & 0x0F0F0F0Fu) | ((((H >> 4) & 0x00000303u) | ((H >> 6) & 0x03030000u)) << 4);
    f.s6[0] = s0 ^ 0x20202020u;
    f.s6[1] = s1 ^ 0x20202020u;
    f.d = __half2float(*reinterpret_cast<const __half*>(blk + 108));
}

// The four A registers of plane c = 4n + j for one row: [2w] the lanes of
// bytes 0 and 2 of word w, [2w + 1] of bytes 1 and 3.
template <int C>
__device__ __forceinline__ void build_a(const Q3Row& f, uint32_t (&A)[4])
{
    constexpr int n = C >> 2, j = C & 3;
    const int sc = (int)(f.s6[n] << (26 - 8 * j)) >> 26;  // sign-extended 6-bit field
    const uint32_t k1 = 0x64806480u - (uint32_t)sc * 0x00040004u;
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        // u = code + 4*high in each byte
        const uint32_t hb = C >= 2 ? (f.h[w] >> (C - 2)) : (f.h[w] << (2 - C));
        const uint32_t u = ((f.q[n][w] >> (2 * j)) & 0x03030303u) | (hb & 0x04040404u);
        A[2 * w] = k1 + (uint32_t)sc * (u & 0x00FF00FFu);
        A[2 * w + 1] = k1 + (uint32_t)sc * ((u >> 8) & 0x00FF00FFu);
    }
}

// One 16-row tile by one Q3_K block against the tokens: 16 MMAs, the d8
// scaling per plane and the d scaling into this thread's four outputs
// (rows g, g+8; tokens 2cq, 2cq+1).
__device__ __forceinline__ void qt_block(const uint8_t* blk0, const uint8_t* blk1, uint32_t sh, uint32_t lsel,
                                         uint32_t hsel, int cq, const uint32_t (&b)[8][4], const float4* ops,
                                         float (&part)[4])
{
    Q3Row r0, r1;
    read_row(blk0, sh, lsel, hsel, cq, r0);
    read_row(blk1, sh, lsel, hsel, cq, r1);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    auto plane = [&](auto cc) {
        constexpr int C = decltype(cc)::value;
        uint32_t A0[4], A1[4];
        build_a<C>(r0, A0);
        build_a<C>(r1, A1);
        const float4 o = ops[C * 4 + cq];
        float d[4];
        mma_f16(d, A0[0], A1[0], A0[1], A1[1], b[C][0], b[C][1], o.x, o.y, o.x, o.y);
        mma_f16(d, A0[2], A1[2], A0[3], A1[3], b[C][2], b[C][3], d[0], d[1], d[2], d[3]);
        acc[0] = fmaf(o.z, d[0], acc[0]);
        acc[1] = fmaf(o.w, d[1], acc[1]);
        acc[2] = fmaf(o.z, d[2], acc[2]);
        acc[3] = fmaf(o.w, d[3], acc[3]);
    };
    plane(std::integral_constant<int, 0>{});
    plane(std::integral_constant<int, 1>{});
    plane(std::integral_constant<int, 2>{});
    plane(std::integral_constant<int, 3>{});
    plane(std::integral_constant<int, 4>{});
    plane(std::integral_constant<int, 5>{});
    plane(std::integral_constant<int, 6>{});
    plane(std::integral_constant<int, 7>{});
    part[0] = fmaf(r0.d, acc[0], part[0]);
    part[1] = fmaf(r0.d, acc[1], part[1]);
    part[2] = fmaf(r1.d, acc[2], part[2]);
    part[3] = fmaf(r1.d, acc[3], part[3]);
}

__global__ void __launch_bounds__(kQtThreads, 1)
    q3k_mt_kernel(const QtArgs a, const __grid_constant__ CUtensorMap tm)
{
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_launch_dependents();  // the next kernel may set itself up meanwhile
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, cq = lane & 3;  // MMA fragment row group and column pair

    uint8_t* ring = smem;
    uint64_t* full_b = reinterpret_cast<uint64_t*>(smem + a.off_bar);
    uint64_t* xbar = full_b + a.nst;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + a.off_cnt);
    int* done = const_cast<int*>(abort_flag) + 1;  // per slot: warps finished with its stage
    int* n_issued = done + a.nst;                  // stages requested
    int* x_done = n_issued + 1;                    // warps holding the current chunk's activations
    int* x_issued = x_done + 1;                    // activation chunks requested
    uint8_t* xs = smem + a.off_x;
    float4* ops = reinterpret_cast<float4*>(smem + a.off_ops) + warp * 32;  // this warp's [plane][cq] scalars
    float* yacc = reinterpret_cast<float*>(smem + a.off_yacc);             // [16 warps][rows of this CTA][8 tokens]

    const int cta = blockIdx.x;
    const int tlo = cta * a.tiles_q + min(cta, a.tiles_r);
    const int thi = tlo + a.tiles_q + (cta < a.tiles_r ? 1 : 0);
    const int ntile = thi - tlo;
    const int nstages = ntile * a.nchunks;  // stage i: chunk i / ntile, tile tlo + i % ntile
    const int pre = min(a.nst, nstages);

    auto ring_pos = [&](int i, int& slot, uint32_t& parity) {
        const int q = (int)__umulhi((uint32_t)i, a.nst_magic);
        slot = i - q * a.nst;
        parity = (uint32_t)q & 1u;
    };

    if (tid == 0) {
        *abort_flag = 0;
        for (int s2 = 0; s2 < a.nst; ++s2)
            done[s2] = 0;
        *n_issued = 0;
        *x_done = 0;
        *x_issued = 0;
        mbar_init(smem_u32(xbar), 1);
        for (int s2 = 0; s2 < a.nst; ++s2)
            mbar_init(smem_u32(&full_b[s2]), 1);
        fence_mbar_init();
    }
    for (int i = tid; i < kQtWarps * a.yacc_rows * kTok; i += blockDim.x)
        yacc[i] = 0.f;
    // global memory may still be written by the previous kernel in the stream
    pdl_wait();
    __syncthreads();

    // ---- producer: stage j (chunk j / ntile, tile tlo + j % ntile) into its
    // slot, by one tensor copy (zero fill past the row end and the last row),
    // or by the whole warp with 2- or 4-byte loads ----
    auto produce = [&](int j) {
        int slot;
        uint32_t parity;
        ring_pos(j, slot, parity);
        const int c = j / ntile;
        const int t = tlo + (j - c * ntile);
        uint8_t* dst0 = ring + (size_t)slot * a.stage_bytes;
        const uint32_t fb = smem_u32(&full_b[slot]);
        if (a.w_tma) {
            if (lane == 0) {
                mbar_arrive_expect_tx(fb, a.stage_bytes);
                tensor_copy_2d(smem_u32(dst0), &tm, (int)(c * (kRowPiece / 8)), t * kTile, fb,
                               l2_policy_evict_first());
            }
        } else {
            const int nbc_c = min(kChunkBlocks, a.nb - c * kChunkBlocks);
            const uint32_t piece = (uint32_t)nbc_c * kQ3Bytes;  // even
            const int nrows = min(kTile, a.N - t * kTile);
            for (int r = 0; r < nrows; ++r) {
                const uint8_t* src = a.W + (int64_t)(t * kTile + r) * a.row_bytes + (int64_t)c * kRowPiece;
                uint8_t* dst = dst0 + (size_t)r * kRowPiece;
                if ((reinterpret_cast<uintptr_t>(src) & 3u) == 0) {
                    for (uint32_t w = lane; w < piece / 4; w += 32)
                        reinterpret_cast<uint32_t*>(dst)[w] = ldg32_nc(src + 4 * w);
                    if ((piece & 2u) && lane == 0)
                        reinterpret_cast<uint16_t*>(dst)[piece / 2 - 1] =
                            __ldg(reinterpret_cast<const unsigned short*>(src) + piece / 2 - 1);
                } else {
                    for (uint32_t w = lane; w < piece / 2; w += 32)
                        reinterpret_cast<uint16_t*>(dst)[w] = __ldg(reinterpret_cast<const unsigned short*>(src) + w);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(fb);
        }
        if (lane == 0)
            atomicAdd(n_issued, 1);
    };
    // Wait for a phase; gives up after ~2 s and raises the abort flag.
    auto wait_bar = [&](uint32_t bar, uint32_t parity) -> bool {
        const bool ok = __all_sync(0xffffffffu, !*abort_flag && mbar_wait_bounded(bar, parity, abort_flag));
        if (!ok && lane == 0) {
            atomicOr(&g_q3mt_error, Q2K_ERR_BIT_WAIT_TIMEOUT);
            *abort_flag = 1;
        }
        return ok;
    };
    // Activations of chunk c into shared memory (one thread): one bulk copy
    // per token, kept in L2 for the other CTAs.
    auto issue_x = [&](int c) {
        const int nbc_c = min(kChunkBlocks, a.nb - c * kChunkBlocks);
        const uint32_t bytes = (uint32_t)nbc_c * kXBlockBytes;
        const uint64_t keep = l2_policy_evict_last();
        mbar_arrive_expect_tx(smem_u32(xbar), bytes * (uint32_t)a.m);
        for (int t = 0; t < a.m; ++t)
            bulk_copy_g2s_hint(smem_u32(xs + (size_t)t * a.xrs), a.x + (int64_t)t * a.x_tok_stride + (int64_t)c * a.xcb,
                               bytes, smem_u32(xbar), keep);
        atomicAdd(x_issued, 1);
    };

    if (tid == 0 && a.x_tma && nstages > 0)
        issue_x(0);  // the first activations ahead of the weights
    if (warp < pre)
        produce(warp);

    // this warp's block of each stage, its word phase, scale selectors
    const int bb = warp;
    const uint32_t sh = (uint32_t)((bb * kQ3Bytes) & 2) * 8;
    const uint32_t lsel = (cq >> 1) ? 0x7531u : 0x6420u;
    const uint32_t hsel = (cq >> 1) ? 0x3131u : 0x2020u;
    bool aborted = false;
    float* yw = yacc + (size_t)warp * a.yacc_rows * kTok;
    uint32_t bops[8][4];
    for (int i = 0, c = 0, ti = 0; i < nstages; ++i) {
        const int nbc_c = min(kChunkBlocks, a.nb - c * kChunkBlocks);
        if (ti == 0) {
            const int kb = c * kChunkBlocks + bb;
            if (a.x_tma) {
                // this chunk's activations are in shared memory; the last
                // warp to take its operands copies the next chunk in
                if (!aborted && !wait_bar(smem_u32(xbar), (uint32_t)c & 1u))
                    aborted = true;
                load_b<true>(a, xs, a.xrs, bb, !aborted && bb < nbc_c, lane, bops, ops);
                int lastx = 0;
                if (lane == 0) {
                    __threadfence_block();
                    lastx = atomicAdd(x_done, 1) == kQtWarps - 1;
                    if (lastx) {
                        atomicExch(x_done, 0);
                        __threadfence_block();
                        if (c + 1 < a.nchunks && !*abort_flag)
                            issue_x(c + 1);
                    }
                }
            } else {
                load_b<false>(a, a.x, a.x_tok_stride, kb, kb < a.nb, lane, bops, ops);
            }
        }
        int slot;
        uint32_t parity;
        ring_pos(i, slot, parity);
        if (!aborted && !wait_bar(smem_u32(&full_b[slot]), parity))
            aborted = true;
        const int t = tlo + ti;
        const int nrows = min(kTile, a.N - t * kTile);
        if (!aborted && bb < nbc_c) {
            const uint8_t* blk0 = ring + (size_t)slot * a.stage_bytes + (size_t)g * kRowPiece + (size_t)bb * kQ3Bytes;
            const uint8_t* blk1 = blk0 + (size_t)8 * kRowPiece;
            float part[4] = {0.f, 0.f, 0.f, 0.f};
            qt_block(blk0, blk1, sh, lsel, hsel, cq, bops, ops, part);
            // rows g and g+8 of the tile, tokens 2cq and 2cq+1: this warp's
            // accumulators, added in chunk order
            float* y0 = yw + (size_t)(ti * kTile + g) * kTok + 2 * cq;
            if (g < nrows) {
                y0[0] += part[0];
                y0[1] += part[1];
            }
            if (g + 8 < nrows) {
                y0[8 * kTok] += part[2];
                y0[8 * kTok + 1] += part[3];
            }
        }
        // release; the last warp out refills the slot
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&done[slot], 1) == kQtWarps - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            if (lane == 0)
                done[slot] = 0;
            __syncwarp();
            if (i + a.nst < nstages && !*abort_flag)
                produce(i + a.nst);
        }
        if (++ti == ntile) {
            ti = 0;
            ++c;
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
    // ---- outputs: rows of this CTA in order, token-major for coalescing ----
    if (ntile > 0) {
        const int r0 = tlo * kTile;
        const int nrows = min(a.N, thi * kTile) - r0;
        for (int q = tid; q < nrows * a.m; q += blockDim.x) {
            const int t = q / nrows, r = q - t * nrows;
            float v = 0.f;
            for (int w = 0; w < kQtWarps; ++w)  // the warps' accumulators in warp order
                v += yacc[((size_t)w * a.yacc_rows + r) * kTok + t];
            a.y[(int64_t)t * a.ldy + r0 + r] = v;
        }
    }
}

size_t qt_align16(size_t v) { return (v + 15) / 16 * 16; }

// cuTensorMapEncodeTiled, found once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 qt_encoder()
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

// Map of a Q3_K matrix as rows of 8-byte elements (rows 16-byte multiples);
// box = one tile (16 rows) by one K chunk (1760 bytes); reads past the row
// end or the last row fill zeros.
bool encode_q3_rows(CUtensorMap* map, const void* W, int64_t rows, int64_t row_bytes)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = qt_encoder();
    if (!enc || rows <= 0 || row_bytes % 16)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 8), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {kRowPiece / 8, (cuuint32_t)kTile};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(W), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool q3mt_supported(const Q3Problem& p)
{
    // from the token count on where it beats the integer-dot kernel
    return p.W_table == nullptr && p.n_seg == 1 && p.m >= kQ3MtMinTokens && p.m <= kTok;
}

cudaError_t launch_q3k_mt(const Q3Problem& p, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess)
        return err;
    if (!q3mt_supported(p))
        return cudaErrorInvalidValue;
    QtArgs a{};
    a.W = static_cast<const uint8_t*>(p.W);
    a.N = (int)p.N;
    a.nb = (int)(p.K / kBlockWeights);
    a.row_bytes = (int64_t)a.nb * kQ3Bytes;
    a.x = static_cast<const uint8_t*>(p.x);
    a.x_tok_stride = p.x_tok_stride;
    a.m = p.m;
    a.y = p.y;
    a.ldy = p.ldy;
    a.nchunks = (a.nb + kChunkBlocks - 1) / kChunkBlocks;
    a.tiles = (a.N + kTile - 1) / kTile;
    // one CTA per SM; more (in waves) when a CTA would own more than
    // kTilesPerCta tiles (each warp keeps an accumulator per row and token)
    const int grid = std::min(a.tiles, std::max(di.sm_count, (a.tiles + kTilesPerCta - 1) / kTilesPerCta));
    a.tiles_q = a.tiles / grid;
    a.tiles_r = a.tiles % grid;
    a.xcb = kChunkBlocks * kXBlockBytes;  // a multiple of 16
    a.xrs = a.xcb + 16;                   // padded: fewer bank conflicts
    a.x_tma = ((reinterpret_cast<uintptr_t>(p.x) | (uintptr_t)p.x_tok_stride) & 15u) == 0 ? 1 : 0;
    a.stage_bytes = kTile * kRowPiece;
    a.w_tma = (reinterpret_cast<uintptr_t>(p.W) & 15u) == 0 && a.row_bytes % 16 == 0;
    a.yacc_rows = (a.tiles_q + (a.tiles_r ? 1 : 0)) * kTile;
    const size_t smem_cap = std::min<size_t>((size_t)di.smem_optin, 224 * 1024);
    size_t smem = 0;
    int nst = 8;
    for (; nst >= 2; --nst) {
        a.nst = nst;
        size_t off = (size_t)nst * a.stage_bytes;
        a.off_x = (uint32_t)off;
        off += a.x_tma ? (((size_t)a.m * a.xrs + 127) / 128 * 128) : 0;
        a.off_ops = (uint32_t)off;
        off += (size_t)kQtWarps * 32 * sizeof(float4);
        a.off_yacc = (uint32_t)off;
        off += qt_align16((size_t)kQtWarps * a.yacc_rows * kTok * sizeof(float));
        a.off_bar = (uint32_t)off;
        off += qt_align16((size_t)(nst + 1) * sizeof(uint64_t));
        a.off_cnt = (uint32_t)off;
        off += qt_align16((size_t)(nst + 4) * sizeof(int));
        smem = off;
        if (smem <= smem_cap)
            break;
    }
    if (nst < 2)
        return cudaErrorInvalidConfiguration;
    a.nst_magic = (uint32_t)((0x100000000ull + (uint64_t)a.nst - 1) / (uint64_t)a.nst);
    CUtensorMap tm{};
    if (a.w_tma && !encode_q3_rows(&tm, a.W, a.N, a.row_bytes))
        a.w_tma = 0;  // the warp-copy path
    static std::atomic<unsigned long long> smem_devs{0};
    if ((err = allow_max_smem(q3k_mt_kernel, smem_devs)) != cudaSuccess)
        return err;
    return launch_pdl(q3k_mt_kernel, dim3((unsigned)grid), dim3(kQtThreads), smem, s, a, tm);
}

cudaError_t q3mt_error_word(int32_t* out, bool clear)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_q3mt_error, sizeof(int));
    if (e != cudaSuccess)
        return e;
    *out = v;
    if (clear) {
        int z = 0;
        e = cudaMemcpyToSymbol(g_q3mt_error, &z, sizeof(int));
    }
    return e;
}

}  // namespace q2k
