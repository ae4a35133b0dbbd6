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
//    of that slice (for MG tokens at a time) stay in registers for every row
//    the lane visits, so the per-row traffic is the weight stream alone.
//  * A warp owns one chunk of LW block columns.  It copies each row's chunk
//    (LW*110 bytes, contiguous) into its own shared-memory buffer with
//    coalesced 16-byte loads (4-byte loads when rows are not 16-byte
//    aligned), issued one row ahead so they overlap the arithmetic; the
//    lanes then read their fields from shared memory.  Read straight from
//    global memory, each lane's scattered 32-bit reads cost an L1 wavefront
//    per sector.  The lanes' word reads of 16 blocks 110 bytes apart still
//    meet in the same banks (about 3.6 wavefronts per read), but a layout
//    with half the conflicts ran no faster: the latency of those reads,
//    with 16 warps per SM and issue about two thirds busy, is what binds.
//    Only __syncwarp orders the buffer: no waits between warps or CTAs.
//  * Blocks are 110 bytes, so every other block starts 2 bytes off a word:
//    fields are read as aligned words and funnel-shifted.
//  * Per (n, j), with c = 4n + j: the code stays at bit 2j of each byte
//    (one AND a word) and the high bit is shifted to bit 2j + 2 beside it
//    (one shift and one AND-OR), so a single DP4A a word multiplies
//    4^j * (code + 4*high) (16 * (...) for j = 3, from bit 4); the chain
//    starts at -4 * 4^j * sum(q) of the slice (activations only, made once)
//    and a shift takes the 4^j off exactly: one DP4A per four weights and
//    token, half of what separate code and high-bit products need.  The
//    sub-block scale multiplies in int32 and the product becomes fp32
//    through the 1.5*2^23 bias (one IMAD and one FADD, exact below 2^22),
//    then meets the q8_1 scale in one FFMA.
//  * Two tokens run as a group inside the launch; three to eight go to the
//    tensor-core kernel of q3k_mt.cu, and one or two tokens over long rows
//    to the row-team kernel below (q3k_m1_kernel), both routed in
//    launch_q3k_mv.
//  * A butterfly shuffle sum gives every lane the chunk's partial for a
//    row, kept in shared memory; after one barrier the chunks are added in
//    chunk order, so the result does not depend on scheduling.
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
    int m;      // tokens (groups of MG walk the rows in turn)
    int vec16;  // rows are 16-byte multiples: chunks move in 16-byte pieces
};

// Bytes of a warp's staging buffer for slice width lw: one row's chunk of
// lw blocks plus the 2-byte lead of an unaligned copy, in 16-byte units.
__host__ __device__ constexpr int q3_buf_bytes(int lw) { return ((lw * 110 + 4 + 15) / 16) * 16; }

__device__ __forceinline__ uint32_t ldg_u32(const uint8_t* p) { return __ldg(reinterpret_cast<const unsigned int*>(p)); }

// NW words from a 2-byte aligned shared-memory address p: aligned reads of
// NW + 1 words and a funnel shift by 0 or 16 bits.  Bytes read: [p - 2,
// p + 4*NW + 4), all inside the block that holds p for every field below.
template <int NW>
__device__ __forceinline__ void lds_words_a2(const uint8_t* p, uint32_t (&out)[NW])
{
    const uintptr_t u = reinterpret_cast<uintptr_t>(p);
    const uint32_t* pa = reinterpret_cast<const uint32_t*>(u & ~uintptr_t(3));
    const uint32_t sh = (uint32_t)(u & 2) * 8;
    uint32_t w[NW + 1];
#pragma unroll
    for (int i = 0; i <= NW; ++i)
        w[i] = pa[i];
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
__device__ __forceinline__ void read_slice(const uint8_t* blk, int l0, Q3Slice<WPL>& s)
{
    lds_words_a2<WPL>(blk + l0, s.hm);
    lds_words_a2<WPL>(blk + 32 + l0, s.q0);
    lds_words_a2<WPL>(blk + 64 + l0, s.q1);
    // scales[12] at byte 96: the four aligned words from byte 92 (block on a
    // word) or 94 (block 2 bytes off), shifted right by 4 or 2 bytes
    const uintptr_t u = reinterpret_cast<uintptr_t>(blk) + 94;
    const uint32_t* pa = reinterpret_cast<const uint32_t*>(u & ~uintptr_t(3));
    const uint32_t sh = 16 + (uint32_t)(u & 2) * 8;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = pa[i];
#pragma unroll
    for (int i = 0; i < 3; ++i)
        s.sc[i] = __funnelshift_rc(w[i], w[i + 1], sh);
    s.d = *reinterpret_cast<const uint16_t*>(blk + 108);
}

// Partial dot products of one slice with MG tokens' activations.
// xq[t][4n + j][w]: q8 bytes l0 + 4w.. of q8_1 block 4n + j of this block
// column; d8[t][4n + j] its scale; c4[t][4n + j] = -4 * (sum of those q8
// bytes) * 4^j (16 for j = 3), the start of the (n, j) DP4A chain.
template <int MG, int WPL>
__device__ __forceinline__ void dot_slice(const Q3Slice<WPL>& s, uint32_t lsel, uint32_t hsel,
                                          const uint32_t (&xq)[MG][8][WPL], const float (&d8)[MG][8],
                                          const int (&c4)[MG][8], float (&out)[MG])
{
    // 6-bit scales of sub-blocks 8n + 2j + hs as bytes j of s6_n
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
            // code + 4*high at bits 2j.. of each byte (4j.. for j = 3: 16*(code + 4*high)),
            // so one DP4A per word multiplies the whole 3-bit value
            const int pos = j < 3 ? 2 * j + 2 : 6;  // where the high bit goes
            uint32_t v[WPL];
#pragma unroll
            for (int w = 0; w < WPL; ++w) {
                const uint32_t q = n ? s.q1[w] : s.q0[w];
                const uint32_t lo = j < 3 ? (q & (0x03030303u << (2 * j))) : ((q >> 2) & 0x30303030u);
                const uint32_t hi = c >= pos ? (s.hm[w] >> (c - pos)) : (s.hm[w] << (pos - c));
                v[w] = lo | (hi & (0x01010101u << pos));
            }
#pragma unroll
            for (int t = 0; t < MG; ++t) {
                int s4 = c4[t][c];
#pragma unroll
                for (int w = 0; w < WPL; ++w)
                    s4 = dp4a_us(v[w], xq[t][c][w], s4);
                const int S = s4 >> (j < 3 ? 2 * j : 4);  // exact: every term carries the factor
                // |sc * S| <= 32 * 16*4*128 < 2^22: exact through the bias
                const float f = __int_as_float(0x4B400000 + sc * S) - 12582912.0f;
                acc[t] = fmaf(d8[t][c], f, acc[t]);
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

// One row's chunk in flight: 16-byte pieces (vec16) or words plus a 2-byte
// tail, held in registers between the global loads and the shared stores.
template <int NV>
struct Q3Stage {
    uint32_t v[4 * NV];
    uint32_t tail;
};

// Global loads of the chunk [src, src + span): with vec16, src and span are
// 16-byte multiples; otherwise src is 2-byte aligned and the copy covers
// [src & ~3, src + span) as words (the bytes below src belong to the
// previous block of the matrix) and the last 2 bytes when src + span is 2
// bytes off a word.  No byte at or past src + span is read.
template <int NV>
__device__ __forceinline__ void stage_load(const uint8_t* src, int span, bool vec16, int lane, Q3Stage<NV>& st)
{
    if (vec16) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int k = lane + 32 * i;
            if (k * 16 < span) {
                const uint4 q = __ldg(reinterpret_cast<const uint4*>(src) + k);
                st.v[4 * i] = q.x;
                st.v[4 * i + 1] = q.y;
                st.v[4 * i + 2] = q.z;
                st.v[4 * i + 3] = q.w;
            }
        }
    } else {
        const uintptr_t u = reinterpret_cast<uintptr_t>(src);
        const uint32_t* pa = reinterpret_cast<const uint32_t*>(u & ~uintptr_t(3));
        const int end = (int)(u & 2) + span;  // bytes from pa
        const int nfull = end >> 2;
#pragma unroll
        for (int i = 0; i < 4 * NV; ++i) {
            const int k = lane + 32 * i;
            if (k < nfull)
                st.v[i] = __ldg(pa + k);
        }
        if ((end & 2) && lane == 0)
            st.tail = __ldg(reinterpret_cast<const unsigned short*>(pa + nfull));
    }
}

// The matching shared stores: the chunk's first byte lands at
// buf + (vec16 ? 0 : (src & 2)).
template <int NV>
__device__ __forceinline__ void stage_store(const uint8_t* src, int span, bool vec16, int lane, const Q3Stage<NV>& st,
                                            uint8_t* buf)
{
    if (vec16) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int k = lane + 32 * i;
            if (k * 16 < span)
                reinterpret_cast<uint4*>(buf)[k] = make_uint4(st.v[4 * i], st.v[4 * i + 1], st.v[4 * i + 2],
                                                              st.v[4 * i + 3]);
        }
    } else {
        const int end = (int)(reinterpret_cast<uintptr_t>(src) & 2) + span;
        const int nfull = end >> 2;
#pragma unroll
        for (int i = 0; i < 4 * NV; ++i) {
            const int k = lane + 32 * i;
            if (k < nfull)
                reinterpret_cast<uint32_t*>(buf)[k] = st.v[i];
        }
        if ((end & 2) && lane == 0)
            *reinterpret_cast<uint16_t*>(buf + 4 * nfull) = (uint16_t)st.tail;
    }
}

template <int MG, int LW>
__global__ void __launch_bounds__(kQ3Threads, 2) q3k_mv_kernel(const Q3Args a)
{
    constexpr int WPL = LW / 4;               // words per lane per field
    constexpr int LPB = 32 / LW;              // lanes per block column
    constexpr int BPC = 32 / LPB;             // block columns per chunk
    constexpr int SPAN = BPC * kQ3Bytes;      // bytes of one row's chunk
    constexpr int NV = (SPAN + 511) / 512;    // 16-byte loads per lane
    constexpr int BUF = q3_buf_bytes(LW);     // the warp's staging buffer
    static_assert((SPAN + 2) / 4 <= 32 * 4 * NV, "the word path fits the stage registers");
    extern __shared__ __align__(16) uint8_t q3_smem[];  // 8 buffers, then partials [rows][nch][m]

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
    const bool vec16 = a.vec16 && (reinterpret_cast<uintptr_t>(W) & 15) == 0;
    const uint8_t* x = a.x + (int64_t)seg * a.x_seg_stride;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* buf = q3_smem + warp * BUF;
    float* part = reinterpret_cast<float*>(q3_smem + 8 * BUF);
    const int bl = lane / LPB, l0 = (lane % LPB) * LW, hs = l0 >> 4;
    const uint32_t lsel = hs ? 0x7531u : 0x6420u;
    const uint32_t hsel = hs ? 0x3131u : 0x2020u;
    const int nch = a.nch, m = a.m;
    // nch < 8: chunk warp % nch, rows split over 8 / nch warps;
    // nch >= 8: chunks warp, warp + 8, ..., every row
    const int c_step = nch >= 8 ? 8 : nch;
    const int wpc = nch >= 8 ? 1 : 8 / nch;
    const int rg = nch >= 8 ? 0 : warp / nch;
    const int64_t row_bytes = (int64_t)a.nb * kQ3Bytes;

    if (warp < c_step * wpc && rg < nrows) {
        for (int c = warp % c_step; c < nch; c += c_step) {
            const int b = c * BPC + bl;
            const bool valid = b < a.nb;
            const int span = min(BPC, a.nb - c * BPC) * kQ3Bytes;
            const uint8_t* src0 = W + (int64_t)r0 * row_bytes + (int64_t)c * SPAN;
            for (int t0 = 0; t0 < m; t0 += MG) {
                uint32_t xq[MG][8][WPL];
                float d8[MG][8];
                int c4[MG][8];
#pragma unroll
                for (int t = 0; t < MG; ++t) {
                    const bool on = valid && t0 + t < m;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint8_t* xb = x + (int64_t)(t0 + t) * a.x_tok_stride + ((int64_t)b * 8 + k) * kQ8Bytes;
                        d8[t][k] = on ? half_lo_f(ldg_u32(xb)) : 0.f;
                        int sq = 0;
#pragma unroll
                        for (int w = 0; w < WPL; ++w) {
                            xq[t][k][w] = on ? ldg_u32(xb + 4 + l0 + 4 * w) : 0u;
                            sq = dp4a_us(0x01010101u, xq[t][k][w], sq);
                        }
                        const int j = k & 3;
                        c4[t][k] = -4 * sq * (j < 3 ? (1 << (2 * j)) : 16);
                    }
                }
                int r = rg;
                {
                    Q3Stage<NV> st;
                    stage_load(src0 + (int64_t)r * row_bytes, span, vec16, lane, st);
                    stage_store(src0 + (int64_t)r * row_bytes, span, vec16, lane, st, buf);
                }
                __syncwarp();
                for (; r < nrows; r += wpc) {
                    const int rn = r + wpc;
                    const uint8_t* src = src0 + (int64_t)r * row_bytes;
                    Q3Stage<NV> nx;
                    if (rn < nrows)  // the next row's chunk is in flight during this row's arithmetic
                        stage_load(src0 + (int64_t)rn * row_bytes, span, vec16, lane, nx);
                    float v[MG];
                    if (valid) {
                        const uint8_t* blk = buf + (vec16 ? 0 : (int)(reinterpret_cast<uintptr_t>(src) & 2)) +
                                             bl * kQ3Bytes;
                        Q3Slice<WPL> sl;
                        read_slice(blk, l0, sl);
                        dot_slice<MG, WPL>(sl, lsel, hsel, xq, d8, c4, v);
                    } else {
#pragma unroll
                        for (int t = 0; t < MG; ++t)
                            v[t] = 0.f;
                    }
                    warp_sum(v);
                    if (lane == 0)
#pragma unroll
                        for (int t = 0; t < MG; ++t)
                            if (t0 + t < m)
                                part[(r * nch + c) * m + t0 + t] = v[t];
                    __syncwarp();  // every lane is done with the buffer
                    if (rn < nrows)
                        stage_store(src0 + (int64_t)rn * row_bytes, span, vec16, lane, nx, buf);
                    __syncwarp();  // the next row is in the buffer
                }
            }
        }
    }
    __syncthreads();
    float* y = a.y + (int64_t)seg * a.y_seg_stride;
    for (int i = threadIdx.x; i < nrows * m; i += kQ3Threads) {
        const int r = i / m, t = i - (i / m) * m;
        float s = 0.f;
        for (int c = 0; c < nch; ++c)
            s += part[(r * nch + c) * m + t];
        y[(int64_t)t * a.ldy + r0 + r] = s;
    }
}

template <int MG, int LW>
cudaError_t launch_q3_tpl(const Q3Args& a, int n_seg, int ctas_x, size_t smem, cudaStream_t s)
{
    return launch_pdl(q3k_mv_kernel<MG, LW>, dim3((unsigned)ctas_x, (unsigned)n_seg), dim3(kQ3Threads), smem, s, a);
}

// Slice width in bytes of l: 16 for one token, 8 for a group of two
// (registers); narrower when the row has fewer block columns than a chunk.
int q3_lw(int mg, int nb)
{
    int lw = mg == 1 ? 16 : 8;
    while (lw > 4 && nb < lw)
        lw /= 2;
    return lw;
}

// ---- one or two tokens over long rows: row teams over a ring of whole rows ----
//
// The design of the Q2_K one-token kernel (q2k_m1.cu) with Q3_K blocks.
// One CTA of 16 warps per SM owns a contiguous range of rows.  A row team
// has two lanes per block column for one token (16-byte-position slices,
// 128 weights) or four for two tokens (8-byte slices), the slices that
// read_slice / dot_slice take, so every lane keeps its q8_1 activations in
// registers for every row it visits.  Whole rows arrive
// by 1-D bulk copies into a ring of stages (two rows per team a stage); the
// warp last out of a stage refills its slot one stage later.  A lane's
// partial, the warp's butterfly sum (xor 16, 8, 4, 2, 1) and the sum of the
// team's warps in warp order are, for one token, the same operations, in
// the same order, as q3k_mv_kernel<1, 16> performs (its warp covers the
// same 16 block columns), so both give the same bits: the expert batches,
// which run there, keep equal to single calls.
constexpr int kQm1Threads = 512;
constexpr int kQm1Warps = kQm1Threads / 32;
constexpr int kQm1Rps = 2;   // rows per team in a stage
// byte positions per lane: 16 (128 weights of a block) for one token, 8 for two
__host__ __device__ constexpr int qm1_lw(int mg) { return mg == 1 ? 16 : 8; }
constexpr int kQm1Rows = 4;  // rows per lane between two warp reductions (two stages)

struct Qm1Args {
    const uint8_t* W;              // the matrix, or null with a table
    const void* const* W_table;    // table: matrix e holds rows e*Nm .. e*Nm + Nm - 1 of the row space
    int Nm;                        // rows per matrix of the table
    int64_t y_seg_stride;          // floats between matrices' rows of y (table)
    float* y;
    const uint8_t* x;  // q8_1 rows, one per token
    int64_t x_tok_stride;  // bytes between tokens' rows (a multiple of 16)
    int64_t ldy;           // floats between tokens of y
    int nb;
    int lanes;         // lanes per row team: a power of two >= (32 / LW) * nb, 32..512
    int log_lanes;
    int teams;         // kQm1Threads / lanes
    int wpt;           // warps per team
    int depth;         // stages in the ring
    int rows_q, rows_r;  // CTA c owns rows_q rows (+1 if c < rows_r)
    uint32_t row_bytes, stage_bytes, x_bytes;
    uint32_t off_x, off_bar, off_red;
};

// The warp sums of v[0..VP-1] (VP = 4 or 8): lane L returns the sum of
// v[L / (32 / VP)] over the warp, paired as a butterfly over lane bits 4,
// 3, 2, 1, 0.  The first log2(VP) steps halve the values a lane holds: it
// keeps the half its lane bit selects and adds its partner's copy of it.
template <int VP>
__device__ __forceinline__ float reduce_rows(const float (&v)[VP], int lane)
{
    static_assert(VP == 4 || VP == 8, "four or eight values a lane");
    float a[VP];
#pragma unroll
    for (int i = 0; i < VP; ++i)
        a[i] = v[i];
    int bit = 16;
#pragma unroll
    for (int n = VP; n > 1; n >>= 1, bit >>= 1) {
        const bool up = (lane & bit) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float keep = up ? a[n / 2 + i] : a[i];
            const float send = up ? a[i] : a[n / 2 + i];
            a[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
    }
#pragma unroll
    for (; bit >= 1; bit >>= 1)
        a[0] += __shfl_xor_sync(0xffffffffu, a[0], bit);
    return a[0];
}

template <int MG, bool TAB>
__global__ void __launch_bounds__(kQm1Threads, 1) q3k_m1_kernel(const Qm1Args a)
{
    static_assert(!TAB || MG == 1, "expert tables: one token");
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int LW = qm1_lw(MG);
    constexpr int WPL = LW / 4;
    constexpr int LPB = 32 / LW;            // lanes per block column
    constexpr int VP = kQm1Rows * MG;       // values per lane between two reductions
    pdl_launch_dependents();  // the next kernel may set itself up meanwhile

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int team = tid >> a.log_lanes;
    const int li = tid & (a.lanes - 1);  // lane within the team
    const int wit = li >> 5;             // warp within the team: the chunk of 16 block columns

    uint8_t* ring = smem;
    const uint8_t* xsm = smem + a.off_x;
    uint64_t* full_b = reinterpret_cast<uint64_t*>(smem + a.off_bar);
    uint64_t* xbar = full_b + a.depth;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(xbar + 1);
    int* released = reinterpret_cast<int*>(xbar + 2);  // per slot: warps done, over all its stages
    int* uses = released + a.depth;                      // per slot: copies requested
    float* red = reinterpret_cast<float*>(smem + a.off_red);

    const int cta = (int)blockIdx.x;
    const int lo = cta * a.rows_q + min(cta, a.rows_r);
    const int hi = lo + a.rows_q + (cta < a.rows_r ? 1 : 0);
    const int spr = kQm1Rps * a.teams;          // rows per stage
    const int nst = (hi - lo + spr - 1) / spr;  // stage j: rows lo + spr*j + kQm1Rps*team + q

    if (tid == 0) {
        mbar_init(smem_u32(xbar), 1);
        *abort_flag = 0;
    }
    if (tid < a.depth) {
        mbar_init(smem_u32(&full_b[tid]), 1);
        released[tid] = 0;
        uses[tid] = 0;
    }
    fence_mbar_init();
    __syncthreads();
    // nothing above touched global memory
    pdl_wait();

    // stage j into slot s (one thread): the stage's rows, one bulk copy
    auto issue = [&](int j, int s) {
        const int r0 = lo + spr * j;
        const int r1 = min(hi, r0 + spr);
        const uint32_t fb = smem_u32(&full_b[s]);
        const uint32_t bytes = (uint32_t)(r1 - r0) * a.row_bytes;
        mbar_arrive_expect_tx(fb, bytes);
        bulk_copy_g2s_hint(smem_u32(ring + (size_t)s * a.stage_bytes), a.W + (int64_t)r0 * a.row_bytes, bytes, fb,
                           l2_policy_evict_first());
        atomicAdd(&uses[s], 1);
    };
    // With a table, stage j into slot s by one whole warp: rows of a matrix
    // on a 16-byte boundary arrive by bulk copy, rows of one on a 4-byte
    // boundary are copied by the warp's lanes (words), rows of any other are
    // not read (they are skipped at the end).  One arrival a stage, with the
    // bulk bytes.
    auto issue_tab = [&](int j, int s) {
        const int r0 = lo + spr * j;
        const int r1 = min(hi, r0 + spr);
        uint8_t* dst0 = ring + (size_t)s * a.stage_bytes;
        uint32_t tx = 0;
        for (int r = r0; r < r1;) {
            const int e = r / a.Nm;
            const int re = min(r1, (e + 1) * a.Nm);
            const uint8_t* wp = static_cast<const uint8_t*>(a.W_table[e]);
            const uintptr_t u = reinterpret_cast<uintptr_t>(wp);
            const uint32_t bytes = (uint32_t)(re - r) * a.row_bytes;
            if ((u & 15u) == 0) {
                tx += bytes;
            } else if ((u & 3u) == 0) {
                const uint32_t* src = reinterpret_cast<const uint32_t*>(wp + (int64_t)(r - e * a.Nm) * a.row_bytes);
                uint32_t* dst = reinterpret_cast<uint32_t*>(dst0 + (size_t)(r - r0) * a.row_bytes);
                for (uint32_t w = (uint32_t)lane; w < bytes / 4u; w += 32u)
                    dst[w] = __ldg(src + w);
            }
            r = re;
        }
        __threadfence_block();
        __syncwarp();
        if (lane == 0) {
            const uint32_t fb = smem_u32(&full_b[s]);
            // the slot may hold words the lanes wrote: order them before the copies
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive_expect_tx(fb, tx);
            for (int r = r0; r < r1;) {
                const int e = r / a.Nm;
                const int re = min(r1, (e + 1) * a.Nm);
                const uint8_t* wp = static_cast<const uint8_t*>(a.W_table[e]);
                if ((reinterpret_cast<uintptr_t>(wp) & 15u) == 0)
                    bulk_copy_g2s_hint(smem_u32(dst0 + (size_t)(r - r0) * a.row_bytes),
                                       wp + (int64_t)(r - e * a.Nm) * a.row_bytes, (uint32_t)(re - r) * a.row_bytes,
                                       fb, l2_policy_evict_first());
                r = re;
            }
            atomicAdd(&uses[s], 1);
        }
    };
    if (tid == 0) {
        // the activations first (every CTA reads them: keep them in L2), then
        // the whole ring
        mbar_arrive_expect_tx(smem_u32(xbar), (uint32_t)MG * a.x_bytes);
#pragma unroll
        for (int t = 0; t < MG; ++t)
            bulk_copy_g2s_hint(smem_u32(smem + a.off_x + (size_t)t * a.x_bytes), a.x + (int64_t)t * a.x_tok_stride,
                               a.x_bytes, smem_u32(xbar), l2_policy_evict_last());
        if constexpr (!TAB)
            for (int j = 0; j < min(a.depth, nst); ++j)
                issue(j, j);
    }
    if constexpr (TAB) {
        if (tid < 32)
            for (int j = 0; j < min(a.depth, nst); ++j)
                issue_tab(j, j);
    }
    // every lane waits for itself; gives up after about two seconds
    auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity))
            return true;
        if (mbar_wait_bounded(bar, parity, abort_flag))
            return true;
        atomicOr(&g_q3_error, Q2K_ERR_BIT_WAIT_TIMEOUT);
        *abort_flag = 1;
        return false;
    };

    // this lane's slice: block column b, byte positions l0 .. l0 + LW - 1
    const bool active = li < LPB * a.nb;
    const int b = active ? li / LPB : 0;
    const int l0 = (li % LPB) * LW;
    const uint32_t lsel = (l0 >> 4) ? 0x7531u : 0x6420u;
    const uint32_t hsel = (l0 >> 4) ? 0x3131u : 0x2020u;
    bool aborted = !wait(smem_u32(xbar), 0);
    // per token, q8_1 blocks 8b + 4n + j: d8, the lane's q8 bytes, and the
    // start of the (n, j) chain, -4 * 4^j * (their sum) (16 for j = 3)
    uint32_t xq[MG][8][WPL];
    float d8[MG][8];
    int c4[MG][8];
#pragma unroll
    for (int t = 0; t < MG; ++t) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint8_t* xb = xsm + (size_t)t * a.x_bytes + ((size_t)b * 8 + k) * kQ8Bytes;
            d8[t][k] = active ? half_lo_f(lds32(xb)) : 0.f;
            int sq = 0;
#pragma unroll
            for (int w = 0; w < WPL; ++w) {
                xq[t][k][w] = active ? lds32(xb + 4 + l0 + 4 * w) : 0u;
                sq = dp4a_us(0x01010101u, xq[t][k][w], sq);
            }
            const int j = k & 3;
            c4[t][k] = -4 * sq * (j < 3 ? (1 << (2 * j)) : 16);
        }
    }

    const uint8_t* blk0 = ring + (size_t)team * kQm1Rps * a.row_bytes + (size_t)b * kQ3Bytes;
    // stage j's slot and the parity of its phase there, advanced one stage
    // at a time; the previous stage (its slot, and the count the last warp
    // out of it sees) and, in lane 0, what this warp's atomic returned
    int s = 0, kd = 0;
    uint32_t parity = 0;
    int prev_j = -1, prev_s = 0, prev_last = 0, prev_count = 0;
    auto stage = [&](int j, float* v) {
        if (!aborted && !wait(smem_u32(&full_b[s]), parity))
            aborted = true;
#pragma unroll
        for (int q = 0; q < kQm1Rps; ++q) {
            float out[MG];
#pragma unroll
            for (int t = 0; t < MG; ++t)
                out[t] = 0.f;
            if (!aborted && active && lo + spr * j + kQm1Rps * team + q < hi) {
                Q3Slice<WPL> sl;
                read_slice<WPL>(blk0 + (size_t)s * a.stage_bytes + (size_t)q * a.row_bytes, l0, sl);
                dot_slice<MG, WPL>(sl, lsel, hsel, xq, d8, c4, out);
            }
#pragma unroll
            for (int t = 0; t < MG; ++t)
                v[q * MG + t] = out[t];
        }
        __syncwarp();
        if constexpr (TAB) {
            int refill = 0;
            if (lane == 0) {
                __threadfence_block();
                const int c = atomicAdd(&released[s], 1);
                // the warp that was last out of the previous stage refills its slot
                refill = prev_count == prev_last && prev_j >= 0 && prev_j + a.depth < nst && !*abort_flag;
                prev_count = c;
            }
            if (__shfl_sync(0xffffffffu, refill, 0))
                issue_tab(prev_j + a.depth, prev_s);
        } else {
            if (lane == 0) {
                __threadfence_block();
                const int c = atomicAdd(&released[s], 1);
                // the warp that was last out of the previous stage refills its slot
                if (prev_count == prev_last && prev_j >= 0 && prev_j + a.depth < nst && !*abort_flag)
                    issue(prev_j + a.depth, prev_s);
                prev_count = c;
            }
        }
        prev_j = j;
        prev_s = s;
        prev_last = kQm1Warps * (kd + 1) - 1;
        if (++s == a.depth) {
            s = 0;
            parity ^= 1u;
            ++kd;
        }
    };
    constexpr int kSpg = kQm1Rows / kQm1Rps;  // stages per reduction
    constexpr int kGl = 32 / VP;  // lanes that end with each value
    for (int j0 = 0; j0 < nst; j0 += kSpg) {
        float v[VP];
#pragma unroll
        for (int g = 0; g < kSpg; ++g) {
            if (j0 + g < nst) {
                stage(j0 + g, v + kQm1Rps * MG * g);
            } else {
#pragma unroll
                for (int q = 0; q < kQm1Rps * MG; ++q)
                    v[kQm1Rps * MG * g + q] = 0.f;
            }
        }
        // lanes kGl*k .. kGl*k + kGl-1 hold the warp's sum for value k:
        // token k % MG of row (k / MG) % Rps of the team in stage
        // j0 + k / (Rps * MG)
        const int k = lane / kGl;
        const int kr = k / MG, t = k - kr * MG;
        const int rl = spr * (j0 + kr / kQm1Rps) + kQm1Rps * team + kr % kQm1Rps;  // row within the CTA's range
        const float r = reduce_rows<VP>(v, lane);
        if ((lane & (kGl - 1)) == 0 && lo + rl < hi)
            red[((size_t)rl * MG + t) * a.wpt + wit] = r;
    }

    __syncthreads();
    if (*abort_flag) {
        // every copy issued must land before the CTA's shared memory goes away
        // (the u-th copy into a slot completes the slot's phase u - 1)
        if (tid < a.depth && uses[tid] > 0)
            mbar_wait_bounded(smem_u32(&full_b[tid]), (uint32_t)(uses[tid] - 1) & 1u, nullptr);
        if (tid == 0)
            mbar_wait_bounded(smem_u32(xbar), 0, nullptr);
        __syncthreads();
        return;
    }
    // the team's warps (the chunks) of each (row, token), added in order
    for (int i = tid; i < (hi - lo) * MG; i += blockDim.x) {
        const int r = i / MG, t = i - r * MG;
        if constexpr (TAB) {
            // a matrix off a 4-byte boundary was not read: its rows of y stay
            if (reinterpret_cast<uintptr_t>(a.W_table[(lo + r) / a.Nm]) & 3u) {
                atomicOr(&g_q3_error, 2);
                continue;
            }
        }
        float v = 0.f;
        for (int w = 0; w < a.wpt; ++w)
            v += red[(size_t)i * a.wpt + w];
        if constexpr (TAB) {
            const int e = (lo + r) / a.Nm;
            a.y[(int64_t)e * a.y_seg_stride + (lo + r - e * a.Nm)] = v;
        } else {
            a.y[(int64_t)t * a.ldy + lo + r] = v;
        }
    }
}

// The launch plan of q3k_m1_kernel; false when the problem is not its: one
// or two tokens on one matrix, rows of 16..128 blocks in 16-byte multiples
// (K a multiple of 2048), W, x and the tokens' rows on 16-byte boundaries.
bool plan_q3m1(const Q3Problem& p, const DeviceInfo& di, Qm1Args& a, int& grid, size_t& smem)
{
    // a table: one token, one input row shared by every matrix
    const bool tab = p.W_table != nullptr;
    const int64_t rows = tab ? p.N * p.n_seg : p.N;
    if ((p.m != 1 && p.m != 2) || p.N < 1 || rows > (int64_t(1) << 30))
        return false;
    if (tab ? (p.m != 1 || p.x_seg_stride != 0 || p.n_seg < 1) : p.n_seg != 1)
        return false;
    if (p.K % 2048 || p.K < 16 * 256 || p.K > 128 * 256)
        return false;
    if (((tab ? 0u : reinterpret_cast<uintptr_t>(p.W)) | reinterpret_cast<uintptr_t>(p.x)) & 15u ||
        (p.m > 1 && (p.x_tok_stride & 15)))
        return false;
    a = Qm1Args{};
    a.nb = (int)(p.K / 256);
    const int lpb = 32 / qm1_lw(p.m);
    a.lanes = 32;
    a.log_lanes = 5;
    while (a.lanes < lpb * a.nb) {
        a.lanes *= 2;
        ++a.log_lanes;
    }
    if (a.lanes > kQm1Threads)
        return false;
    a.teams = kQm1Threads / a.lanes;
    a.wpt = a.lanes / 32;
    a.row_bytes = (uint32_t)(a.nb * kQ3Bytes);
    a.stage_bytes = (uint32_t)(kQm1Rps * a.teams) * a.row_bytes;
    a.x_bytes = (uint32_t)(a.nb * 8 * kQ8Bytes);
    a.W = tab ? nullptr : static_cast<const uint8_t*>(p.W);
    a.W_table = p.W_table;
    a.Nm = (int)p.N;
    a.y_seg_stride = p.y_seg_stride;
    a.x = static_cast<const uint8_t*>(p.x);
    a.x_tok_stride = p.x_tok_stride;
    a.y = p.y;
    a.ldy = p.ldy;
    grid = (int)std::min<int64_t>(di.sm_count, rows);
    a.rows_q = (int)(rows / grid);
    a.rows_r = (int)(rows % grid);
    const size_t cap = std::min<size_t>((size_t)di.smem_optin, 227 * 1024);
    const size_t red_bytes = (size_t)(a.rows_q + 1) * p.m * a.wpt * sizeof(float);
    for (int depth = 8; depth >= 2; --depth) {
        a.depth = depth;
        a.off_x = (uint32_t)((size_t)depth * a.stage_bytes);
        a.off_bar = a.off_x + (uint32_t)p.m * a.x_bytes;  // x_bytes is a multiple of 16
        a.off_red = (uint32_t)(((size_t)a.off_bar + (size_t)(depth + 2) * sizeof(uint64_t) +
                                (size_t)(2 * depth) * sizeof(int) + 15) / 16 * 16);
        smem = ((size_t)a.off_red + red_bytes + 15) / 16 * 16;
        if (smem <= cap)
            return true;
    }
    return false;
}

template <int MG, bool TAB>
cudaError_t launch_q3m1_tpl(const Qm1Args& a, int grid, size_t smem, cudaStream_t s)
{
    static std::atomic<unsigned long long> smem_devs{0};
    cudaError_t e = allow_max_smem(q3k_m1_kernel<MG, TAB>, smem_devs);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(q3k_m1_kernel<MG, TAB>, dim3((unsigned)grid), dim3(kQm1Threads), smem, s, a);
}

}  // namespace

cudaError_t launch_q3k_mv(const Q3Problem& p, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    if (q3mt_supported(p))  // several tokens: the tensor-core kernel
        return launch_q3k_mt(p, s);
    {
        Qm1Args a1;
        int grid1;
        size_t smem1;
        if (plan_q3m1(p, di, a1, grid1, smem1))  // one or two tokens over long rows: row teams
            return p.W_table ? launch_q3m1_tpl<1, true>(a1, grid1, smem1, s)
                   : p.m == 1 ? launch_q3m1_tpl<1, false>(a1, grid1, smem1, s)
                              : launch_q3m1_tpl<2, false>(a1, grid1, smem1, s);
    }
    const int nb = (int)(p.K / 256);
    // tokens per walk over the rows: one, or pairs (groups of four tokens
    // in 4-byte slices measured slower: 188 vs 103 us for m = 4 at 16384^2)
    const int mg = p.m == 1 ? 1 : 2;
    const int lw = q3_lw(mg, nb);
    Q3Args a{};
    a.W = static_cast<const uint8_t*>(p.W);
    a.W_table = p.W_table;
    a.x = static_cast<const uint8_t*>(p.x);
    a.y = p.y;
    a.x_tok_stride = p.x_tok_stride;
    a.x_seg_stride = p.x_seg_stride;
    a.ldy = p.ldy;
    a.y_seg_stride = p.y_seg_stride;
    a.N = (int)p.N;
    a.nb = nb;
    a.nch = (nb + lw - 1) / lw;
    a.m = p.m;
    // row bytes and chunk bytes 16-byte multiples (the base is checked per
    // matrix); a 4-byte slice makes 440-byte chunks, which take the word path
    a.vec16 = nb % 8 == 0 && (lw * kQ3Bytes) % 16 == 0;
    // two CTAs per SM over all segments; staging buffers and chunk partials
    // stay within the default 48 KB of shared memory
    const int64_t bufs = 8 * (int64_t)q3_buf_bytes(lw);
    const int64_t target = std::max<int64_t>(1, (2 * (int64_t)di.sm_count + p.n_seg - 1) / p.n_seg);
    int64_t rows = std::max<int64_t>(1, (p.N + target - 1) / target);
    const int64_t max_rows = std::max<int64_t>(1, (49152 - bufs) / ((int64_t)a.nch * p.m * 4));
    rows = std::min(rows, max_rows);
    a.rows_per_cta = (int)rows;
    const int ctas_x = (int)((p.N + rows - 1) / rows);
    const size_t smem = (size_t)(bufs + rows * a.nch * p.m * (int64_t)sizeof(float));
    switch (mg * 100 + lw) {
    case 116: return launch_q3_tpl<1, 16>(a, p.n_seg, ctas_x, smem, s);
    case 108: return launch_q3_tpl<1, 8>(a, p.n_seg, ctas_x, smem, s);
    case 104: return launch_q3_tpl<1, 4>(a, p.n_seg, ctas_x, smem, s);
    case 208: return launch_q3_tpl<2, 8>(a, p.n_seg, ctas_x, smem, s);
    case 204: return launch_q3_tpl<2, 4>(a, p.n_seg, ctas_x, smem, s);
    default: return cudaErrorInvalidConfiguration;
    }
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
