// Q3_K MMVQ with q8_1 activations, m <= 8 tokens, straight off the GGUF
// blocks: the Q3_K twins of the single-matrix and experts kernels that
// moe_v41/init.rs (`MoeV41::new`) loads beside the Q2_K ones
// (`kquant_mmvq_q3_k_w`, `kquant_mmvq_q3_k_experts_w*`).
//
// Block (110 bytes, 256 weights; GGUF's layout, the pages give only the
// kernel names): hmask[32] | qs[64] | scales[12] | d (fp16).  Weight
// p = 128n + 32j + l (n < 2, j < 4, l < 32) has its 2-bit code at bit 2j of
// qs[32n + l] and its high bit at bit 4n + j of hmask[l]; it lies in
// sub-block 8n + 2j + l/16, whose 6-bit scale is stored + 32.  Its value is
// d * scale * (code + 4*high - 4).
//
// Design (GB300):
//  * Each lane owns a fixed K-slice: LW consecutive byte positions l of one
//    block column, i.e. 8*LW weights (every n and j).  The q8_1 activations
//    of that slice stay in registers for every row the lane visits, so the
//    per-row traffic is the weight stream alone.
//  * Blocks are 110 bytes, so every other block starts 2 bytes off a word:
//    each field is read with aligned 32-bit loads and a funnel shift.  No
//    staging and no waits: nothing in this kernel can stall on another CTA.
//  * Per (n, j), with c = 4n + j: the codes stay at bit 2j (one AND a word;
//    the 4^j comes off the int32 sum with a shift), the complement of the
//    high bit at bit c (one AND-NOT a word); two DP4A a word give
//    S1 = 4^j * sum(code*q) and S2 = 2^c * sum((1-high)*q), and
//    sum((code + 4*high - 4)*q) = S1 / 4^j - 4 * S2 / 2^c exactly.  The
//    sub-block scale multiplies in int32, the q8_1 scale in fp32.
//  * A warp's lanes cover one chunk of LW block columns; a butterfly
//    shuffle sum gives every lane the chunk's partial for a row, kept in
//    shared memory; after one barrier the chunks are added in chunk order,
//    so the result does not depend on scheduling.
#include "q2k_common.cuh"
#include "q2k_internal.h"

#include <algorithm>

namespace q2k {

__device__ int g_q3_error = 0;

namespace {

constexpr int kQ3Bytes = 110;
constexpr int kQ8Bytes = 36;
constexpr int kQ3Threads = 256;

struct Q3Args {
    const uint8_t* W;            // matrix (segment 0 when W_table is null)
    const void* const* W_table;  // nullable: segment e's matrix
    const uint8_t* x;            // q8_1 rows
    float* y;
    int64_t x_tok_stride;  // bytes between tokens
    int64_t x_seg_stride;  // bytes between segments' inputs (0 = shared)
    int64_t ldy;           // floats between tokens
    int64_t y_seg_stride;  // floats between segments
    int N, nb, nch, rows_per_cta;
};

__device__ __forceinline__ uint32_t ldg_u32(const uint8_t* p) { return __ldg(reinterpret_cast<const unsigned int*>(p)); }

// NW words from a 2-byte aligned address p: aligned loads of NW + 1 words
// and a funnel shift by 0 or 16 bits.  Bytes read: [p - 2, p + 4*NW + 4).
template <int NW>
__device__ __forceinline__ void ldg_words_a2(const uint8_t* p, uint32_t (&out)[NW])
{
    const uintptr_t u = reinterpret_cast<uintptr_t>(p);
    const uint8_t* pa = reinterpret_cast<const uint8_t*>(u & ~uintptr_t(3));
    const uint32_t sh = (uint32_t)(u & 2) * 8;
    uint32_t w[NW + 1];
#pragma unroll
    for (int i = 0; i <= NW; ++i)
        w[i] = ldg_u32(pa + 4 * i);
#pragma unroll
    for (int i = 0; i < NW; ++i)
        out[i] = __funnelshift_r(w[i], w[i + 1], sh);
}

// One lane's share of one block: hmask, both qs halves, the scales, d.
template <int WPL>
struct Q3Slice {
    uint32_t hm[WPL], q0[WPL], q1[WPL], sc[3];
    uint16_t d;
};

template <int WPL>
__device__ __forceinline__ void load_slice(const uint8_t* blk, int l0, Q3Slice<WPL>& s)
{
    ldg_words_a2<WPL>(blk + l0, s.hm);
    ldg_words_a2<WPL>(blk + 32 + l0, s.q0);
    ldg_words_a2<WPL>(blk + 64 + l0, s.q1);
    // scales[12] at byte 96: the four aligned words from byte 92 (block on a
    // word) or 94 (block 2 bytes off), shifted right by 4 or 2 bytes; every
    // byte read lies inside the block
    const uintptr_t u = reinterpret_cast<uintptr_t>(blk) + 94;
    const uint8_t* pa = reinterpret_cast<const uint8_t*>(u & ~uintptr_t(3));
    const uint32_t sh = 16 + (uint32_t)(u & 2) * 8;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = ldg_u32(pa + 4 * i);
#pragma unroll
    for (int i = 0; i < 3; ++i)
        s.sc[i] = __funnelshift_rc(w[i], w[i + 1], sh);
    s.d = __ldg(reinterpret_cast<const unsigned short*>(blk + 108));
}

// Partial dot products of one slice with MG tokens' activations.
// xq[t][4n + j][w]: q8 bytes l0 + 4w.. of q8_1 block 4n + j of this block
// column; d8[t][4n + j] its scale.
template <int MG, int WPL>
__device__ __forceinline__ void dot_slice(const Q3Slice<WPL>& s, uint32_t lsel, uint32_t hsel,
                                          const uint32_t (&xq)[MG][8][WPL], const float (&d8)[MG][8],
                                          float (&out)[MG])
{
    // 6-bit scales of sub-blocks 8n + 2j + hs as bytes j of s6[n]
    const uint32_t L = __byte_perm(s.sc[0], s.sc[1], lsel);
    const uint32_t H = __byte_perm(s.sc[2], 0u, hsel);
    const uint32_t s6_0 = (L & 0x0F0F0F0Fu) | (((H & 0x00000303u) | ((H >> 2) & 0x03030000u)) << 4);
    const uint32_t s6_1 = ((L >> 4) & 0x0F0F0F0Fu) | ((((H >> 4) & 0x00000303u) | ((H >> 6) & 0x03030000u)) << 4);
    float acc[MG];
#pragma unroll
    for (int t = 0; t < MG; ++t)
        acc[t] = 0.f;
#pragma unroll
    for (int n = 0; n < 2; ++n) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = 4 * n + j;
            const int sc = (int)(((n ? s6_1 : s6_0) >> (8 * j)) & 0xFFu) - 32;
            uint32_t a[WPL], h[WPL];
#pragma unroll
            for (int w = 0; w < WPL; ++w) {
                a[w] = (n ? s.q1[w] : s.q0[w]) & (0x03030303u << (2 * j));
                h[w] = ~s.hm[w] & (0x01010101u << c);
            }
#pragma unroll
            for (int t = 0; t < MG; ++t) {
                int s1 = 0, s2 = 0;
#pragma unroll
                for (int w = 0; w < WPL; ++w) {
                    s1 = dp4a_us(a[w], xq[t][c][w], s1);
                    s2 = dp4a_us(h[w], xq[t][c][w], s2);
                }
                const int S = (s1 >> (2 * j)) - (c >= 2 ? (s2 >> (c - 2)) : s2 * (1 << (2 - c)));
                acc[t] = fmaf(d8[t][c], (float)(sc * S), acc[t]);
            }
        }
    }
    const float d = __half2float(__ushort_as_half(s.d));
#pragma unroll
    for (int t = 0; t < MG; ++t)
        out[t] = acc[t] * d;
}

template <int MG>
__device__ __forceinline__ void warp_sum(float (&v)[MG])
{
#pragma unroll
    for (int t = 0; t < MG; ++t)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            v[t] += __shfl_xor_sync(0xFFFFFFFFu, v[t], off);
}

template <int MG, int LW>
__global__ void __launch_bounds__(kQ3Threads, 2) q3k_mv_kernel(const Q3Args a)
{
    constexpr int WPL = LW / 4;    // words per lane per field
    constexpr int LPB = 32 / LW;   // lanes per block column
    constexpr int BPC = 32 / LPB;  // block columns per chunk
    extern __shared__ float part[];  // [rows_per_cta][nch][MG]

    pdl_launch_dependents();
    const int seg = blockIdx.y;
    const int r0 = blockIdx.x * a.rows_per_cta;
    const int nrows = min(a.N - r0, a.rows_per_cta);
    pdl_wait();
    if (nrows <= 0)
        return;
    const uint8_t* W = a.W_table ? static_cast<const uint8_t*>(a.W_table[seg]) : a.W;
    if (reinterpret_cast<uintptr_t>(W) & 3) {  // a table entry off a word: skip it, report
        if (threadIdx.x == 0)
            atomicOr(&g_q3_error, 2);
        return;
    }
    const uint8_t* x = a.x + (int64_t)seg * a.x_seg_stride;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bl = lane / LPB, l0 = (lane % LPB) * LW, hs = l0 >> 4;
    const uint32_t lsel = hs ? 0x7531u : 0x6420u;
    const uint32_t hsel = hs ? 0x3131u : 0x2020u;
    const int nch = a.nch;
    // nch < 8: chunk warp % nch, rows split over 8 / nch warps;
    // nch >= 8: chunks warp, warp + 8, ..., every row
    const int c_step = nch >= 8 ? 8 : nch;
    const int wpc = nch >= 8 ? 1 : 8 / nch;
    const int rg = nch >= 8 ? 0 : warp / nch;
    const int64_t row_bytes = (int64_t)a.nb * kQ3Bytes;

    if (warp < c_step * wpc) {
        for (int c = warp % c_step; c < nch; c += c_step) {
            const int b = c * BPC + bl;
            const bool valid = b < a.nb;
            uint32_t xq[MG][8][WPL];
            float d8[MG][8];
#pragma unroll
            for (int t = 0; t < MG; ++t)
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint8_t* xb = x + (int64_t)t * a.x_tok_stride + ((int64_t)b * 8 + k) * kQ8Bytes;
                    d8[t][k] = valid ? half_lo_f(ldg_u32(xb)) : 0.f;
#pragma unroll
                    for (int w = 0; w < WPL; ++w)
                        xq[t][k][w] = valid ? ldg_u32(xb + 4 + l0 + 4 * w) : 0u;
                }
            const uint8_t* wb = W + (int64_t)r0 * row_bytes + (int64_t)b * kQ3Bytes;
            int r = rg;
            for (; r + wpc < nrows; r += 2 * wpc) {  // two rows at a time: loads in flight
                float v0[MG], v1[MG];
                if (valid) {
                    Q3Slice<WPL> s0, s1;
                    load_slice(wb + (int64_t)r * row_bytes, l0, s0);
                    load_slice(wb + (int64_t)(r + wpc) * row_bytes, l0, s1);
                    dot_slice<MG, WPL>(s0, lsel, hsel, xq, d8, v0);
                    dot_slice<MG, WPL>(s1, lsel, hsel, xq, d8, v1);
                } else {
#pragma unroll
                    for (int t = 0; t < MG; ++t)
                        v0[t] = v1[t] = 0.f;
                }
                warp_sum(v0);
                warp_sum(v1);
                if (lane == 0)
#pragma unroll
                    for (int t = 0; t < MG; ++t) {
                        part[(r * nch + c) * MG + t] = v0[t];
                        part[((r + wpc) * nch + c) * MG + t] = v1[t];
                    }
            }
            if (r < nrows) {
                float v0[MG];
                if (valid) {
                    Q3Slice<WPL> s0;
                    load_slice(wb + (int64_t)r * row_bytes, l0, s0);
                    dot_slice<MG, WPL>(s0, lsel, hsel, xq, d8, v0);
                } else {
#pragma unroll
                    for (int t = 0; t < MG; ++t)
                        v0[t] = 0.f;
                }
                warp_sum(v0);
                if (lane == 0)
#pragma unroll
                    for (int t = 0; t < MG; ++t)
                        part[(r * nch + c) * MG + t] = v0[t];
            }
        }
    }
    __syncthreads();
    float* y = a.y + (int64_t)seg * a.y_seg_stride;
    for (int i = threadIdx.x; i < nrows * MG; i += kQ3Threads) {
        const int r = i / MG, t = i - (i / MG) * MG;
        float s = 0.f;
        for (int c = 0; c < nch; ++c)
            s += part[(r * nch + c) * MG + t];
        y[(int64_t)t * a.ldy + r0 + r] = s;
    }
}

template <int MG, int LW>
cudaError_t launch_q3_tpl(const Q3Args& a, int n_seg, int ctas_x, size_t smem, cudaStream_t s)
{
    return launch_pdl(q3k_mv_kernel<MG, LW>, dim3((unsigned)ctas_x, (unsigned)n_seg), dim3(kQ3Threads), smem, s, a);
}

// Slice width in bytes of l: 16 for one token over rows of 16+ blocks, 8
// for two tokens (registers), 4 otherwise; narrower when the row has fewer
// block columns than a warp chunk.
int q3_lw(int mg, int nb)
{
    const int want = mg == 1 ? 16 : (mg == 2 ? 8 : 4);
    int lw = want;
    while (lw > 4 && nb < lw)
        lw /= 2;
    return lw;
}

}  // namespace

cudaError_t launch_q3k_mv(const Q3Problem& p, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    const int nb = (int)(p.K / 256);
    for (int t0 = 0; t0 < p.m; t0 += 4) {
        const int mg = std::min(4, p.m - t0);
        const int lw = q3_lw(mg, nb);
        Q3Args a{};
        a.W = static_cast<const uint8_t*>(p.W);
        a.W_table = p.W_table;
        a.x = static_cast<const uint8_t*>(p.x) + (int64_t)t0 * p.x_tok_stride;
        a.y = p.y + (int64_t)t0 * p.ldy;
        a.x_tok_stride = p.x_tok_stride;
        a.x_seg_stride = p.x_seg_stride;
        a.ldy = p.ldy;
        a.y_seg_stride = p.y_seg_stride;
        a.N = (int)p.N;
        a.nb = nb;
        a.nch = (nb + lw - 1) / lw;
        // two CTAs per SM over all segments; shared memory for the chunk
        // partials stays within the default 48 KB
        const int64_t target = std::max<int64_t>(1, (2 * (int64_t)di.sm_count + p.n_seg - 1) / p.n_seg);
        int64_t rows = std::max<int64_t>(1, (p.N + target - 1) / target);
        const int64_t max_rows = std::max<int64_t>(1, 49152 / ((int64_t)a.nch * mg * 4));
        rows = std::min(rows, max_rows);
        a.rows_per_cta = (int)rows;
        const int ctas_x = (int)((p.N + rows - 1) / rows);
        const size_t smem = (size_t)rows * a.nch * mg * sizeof(float);
        switch (mg * 100 + lw) {
        case 116: e = launch_q3_tpl<1, 16>(a, p.n_seg, ctas_x, smem, s); break;
        case 108: e = launch_q3_tpl<1, 8>(a, p.n_seg, ctas_x, smem, s); break;
        case 104: e = launch_q3_tpl<1, 4>(a, p.n_seg, ctas_x, smem, s); break;
        case 208: e = launch_q3_tpl<2, 8>(a, p.n_seg, ctas_x, smem, s); break;
        case 204: e = launch_q3_tpl<2, 4>(a, p.n_seg, ctas_x, smem, s); break;
        case 304: e = launch_q3_tpl<3, 4>(a, p.n_seg, ctas_x, smem, s); break;
        case 404: e = launch_q3_tpl<4, 4>(a, p.n_seg, ctas_x, smem, s); break;
        default: return cudaErrorInvalidConfiguration;
        }
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

cudaError_t q3_error_word(int32_t* out, bool clear)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_q3_error, sizeof(int));
    if (e != cudaSuccess)
        return e;
    *out = v;
    if (clear) {
        int z = 0;
        e = cudaMemcpyToSymbol(g_q3_error, &z, sizeof(int));
    }
    return e;
}

}  // namespace q2k
