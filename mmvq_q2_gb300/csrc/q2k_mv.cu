// Q2_K GEMV / MMVQ for m <= 8 tokens, straight off the GGUF blocks.
//
// Follows engram_v41/apply.rs (single-token `wkv` projection off
// `wkv_q2k`), attn_v41/decode.rs (`kquant_mmvq_pair_w`: two matrices, one
// q8_1 input, one launch) and moe_v41/init.rs (`kquant_mmvq_q2_k_experts_w8`
// batches, `moe_v41_accumulate` route-weighted sum).
//
// Design (GB300):
//  * Weight rows stream into a ring of shared-memory stages with 1-D bulk
//    asynchronous copies (cp.async.bulk, the TMA engine) signalled on
//    mbarriers.  Lane 0 of warp 0 issues them: the ring is primed up front
//    and each slot is refilled once every warp has released it (one
//    mbarrier arrival per warp).  Rows that are not 16-byte aligned are
//    copied by warp 0's lanes instead.  Every wait is bounded.
//  * Each consumer thread owns a fixed K-slice of every row (SW words of a
//    block's qs, i.e. 16*SW weights spread over 4 sub-blocks) and keeps the
//    matching activations in registers for all rows it visits, so the only
//    per-row traffic is the weight stream itself.
//  * Codes are extracted four at a time with one AND per register (the code
//    of pair j stays at bit 2j of each byte, i.e. scaled by 4^j; the 4^-j is
//    folded into the per-sub-block activation scale) and multiplied by
//    DP4A (q8_1 activations) or two DP2A (bf16 activations as 16-bit fixed
//    point with one exponent per group).
//  * Per sub-block: y += d*sc*xscale*S - dmin*m*sum(x), with the scale and
//    min nibbles converted to float once per sub-block and shared by all
//    tokens.  Row partial sums are reduced with warp shuffles and, when a
//    row spans several warps, through shared memory in a fixed order.
#include "q2k_common.cuh"
#include "q2k_internal.h"

#include <algorithm>

namespace q2k {

__device__ int g_mv_error = 0;

// Row slots per thread per stage: fewer for more tokens (registers).
__host__ __device__ constexpr int rpt_max(int m) { return m <= 2 ? 4 : (m <= 4 ? 2 : 1); }

struct MvArgs {
    int n_seg;
    int table;  // 1: W_table segments, stacked over one row range
    const void* const* W_table;
    const uint8_t* W[2];
    int64_t N[2];
    int64_t row_bytes;  // bytes of a full weight row
    int kb0;            // first block column of this K chunk
    int nbc;            // blocks in this K chunk
    const uint8_t* x;
    int64_t x_tok_stride;
    int64_t x_seg_stride;
    float* y[2];
    int64_t ldy[2];
    float* y_exp;
    const float* route_w;
    float* y_sum;
    int accumulate;
    // decomposition
    int rpt;         // row slots per thread per stage (<= rpt_max(M))
    int s_real;      // slices per row
    int s_pad;       // lanes per row group
    int groups;      // row groups
    int tc;          // consumer threads
    int rps;         // rows per stage (multiple of groups)
    int nst;         // stages in the ring
    uint32_t rstride;   // shared-memory row stride (16-byte multiple)
    uint32_t stage_bytes;
    int64_t rows_total;  // concat: N0 + N1; table: N
    int ysum_cap;
};

struct Stage {
    int e;
    int64_t row0;
    int nrows;
};

// Rows [lo, hi) of this CTA.
__device__ __forceinline__ void cta_range(const MvArgs& a, int64_t& lo, int64_t& hi)
{
    lo = (a.rows_total * (int64_t)blockIdx.x) / gridDim.x;
    hi = (a.rows_total * (int64_t)(blockIdx.x + 1)) / gridDim.x;
}

__device__ __forceinline__ int stage_count(const MvArgs& a, int64_t lo, int64_t hi)
{
    if (hi <= lo)
        return 0;
    if (a.table) {
        int per = (int)((hi - lo + a.rps - 1) / a.rps);
        return per * a.n_seg;
    }
    int64_t n0 = a.N[0];
    int64_t l0 = max((int64_t)0, min(hi, n0) - lo);
    int64_t l1 = max((int64_t)0, hi - max(lo, n0));
    return (int)((l0 + a.rps - 1) / a.rps + (l1 + a.rps - 1) / a.rps);
}

__device__ __forceinline__ Stage stage_at(const MvArgs& a, int64_t lo, int64_t hi, int i)
{
    Stage s;
    if (a.table) {
        int per = (int)((hi - lo + a.rps - 1) / a.rps);
        s.e = i / per;
        int c = i - s.e * per;
        s.row0 = lo + (int64_t)c * a.rps;
        s.nrows = (int)min((int64_t)a.rps, hi - s.row0);
        return s;
    }
    int64_t n0 = a.N[0];
    int64_t b0 = lo, e0 = min(hi, n0);
    int c0 = e0 > b0 ? (int)((e0 - b0 + a.rps - 1) / a.rps) : 0;
    if (i < c0) {
        s.e = 0;
        s.row0 = b0 + (int64_t)i * a.rps;
        s.nrows = (int)min((int64_t)a.rps, e0 - s.row0);
    } else {
        int64_t b1 = max(lo, n0);
        s.e = 1;
        s.row0 = (b1 - n0) + (int64_t)(i - c0) * a.rps;
        s.nrows = (int)min((int64_t)a.rps, (hi - n0) - s.row0);
    }
    return s;
}

__device__ __forceinline__ const uint8_t* seg_weights(const MvArgs& a, int e)
{
    if (a.table) {
        const void* p;
        asm volatile("ld.global.nc.u64 %0, [%1];" : "=l"(p) : "l"(a.W_table + e));
        return static_cast<const uint8_t*>(p);
    }
    return a.W[e];
}

// ---- activation slice ------------------------------------------------------

template <int M, int ACT, int SW>
struct Slice {
    static constexpr int NA = (ACT == ACT_BF16) ? 2 : 1;  // registers per qs word
    static constexpr int NH = (SW == 8) ? 2 : 1;           // sub-block halves covered
    static constexpr int WPH = SW / NH;                    // qs words per half
    uint32_t xa[M][4][SW][NA];
    float xp[M][4][NH];
    float xs[M][4][NH];
};

// Load and convert this thread's activation slice.  Slice geometry: block
// column bcol (absolute), half n, first qs word wi0 (0..7) within the half.
// Weight of (j, word w, byte i) is k = bcol*256 + 128n + 32j + 4w + i.
template <int M, int ACT, int SW>
__device__ __forceinline__ void load_slice(Slice<M, ACT, SW>& sl, const uint8_t* xseg, int64_t tok_stride,
                                           int bcol, int n, int wi0, bool active)
{
    using S = Slice<M, ACT, SW>;
#pragma unroll
    for (int t = 0; t < M; ++t) {
        const uint8_t* xt = xseg + t * tok_stride;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if constexpr (ACT == ACT_BF16) {
                const uint16_t* xv = reinterpret_cast<const uint16_t*>(xt);
#pragma unroll
                for (int hh = 0; hh < S::NH; ++hh) {
                    float v[S::WPH * 4];
                    float amax = 0.f;
#pragma unroll
                    for (int wl = 0; wl < S::WPH; ++wl)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            int64_t k = (int64_t)bcol * 256 + 128 * n + 32 * j + 4 * (wi0 + hh * S::WPH + wl) + i;
                            float f = active ? bf16_bits_f(xv[k]) : 0.f;
                            v[wl * 4 + i] = f;
                            amax = fmaxf(amax, fabsf(f));
                        }
                    uint32_t eb = (__float_as_uint(amax) >> 23) & 0xFFu;  // biased exponent of amax
                    int sum = 0;
                    if (eb >= 27u) {
                        // x16 = x * 2^(141-eb): |x16| < 2^15, exact for the group's
                        // largest 2^8 range; xp = 2^(eb-141) * 4^-j.
                        float scale = __uint_as_float((268u - eb) << 23);
#pragma unroll
                        for (int wl = 0; wl < S::WPH; ++wl) {
                            int q[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                q[i] = __float2int_rn(v[wl * 4 + i] * scale);
                                sum += q[i];
                            }
                            sl.xa[t][j][hh * S::WPH + wl][0] = (uint32_t)(q[0] & 0xFFFF) | ((uint32_t)q[1] << 16);
                            sl.xa[t][j][hh * S::WPH + wl][1] = (uint32_t)(q[2] & 0xFFFF) | ((uint32_t)q[3] << 16);
                        }
                        sl.xp[t][j][hh] = __uint_as_float((eb - 14u - 2u * j) << 23);
                        sl.xs[t][j][hh] = (float)sum * __uint_as_float((eb - 14u) << 23);
                    } else {
#pragma unroll
                        for (int wl = 0; wl < S::WPH; ++wl) {
                            sl.xa[t][j][hh * S::WPH + wl][0] = 0u;
                            sl.xa[t][j][hh * S::WPH + wl][1] = 0u;
                        }
                        sl.xp[t][j][hh] = 0.f;
                        sl.xs[t][j][hh] = 0.f;
                    }
                }
            } else {
                // q8_1 block (bcol*8 + 4n + j): fp16 d at +0, q[32] at +4.
                const uint8_t* qb = xt + ((int64_t)bcol * 8 + 4 * n + j) * kQ8Bytes;
                float d = active ? half_lo_f(ldg32_nc(qb)) : 0.f;
#pragma unroll
                for (int hh = 0; hh < S::NH; ++hh) {
                    int sum = 0;
#pragma unroll
                    for (int wl = 0; wl < S::WPH; ++wl) {
                        int w = wi0 + hh * S::WPH + wl;
                        uint32_t qv = active ? ldg32_nc(qb + 4 + 4 * w) : 0u;
                        sl.xa[t][j][hh * S::WPH + wl][0] = qv;
                        sum = dp4a_us(0x01010101u, qv, sum);
                    }
                    sl.xp[t][j][hh] = d * __uint_as_float((127u - 2u * j) << 23);
                    sl.xs[t][j][hh] = d * (float)sum;
                }
            }
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
#pragma unroll
    for (int hh = 0; hh < S::NH; ++hh) {
        const uint32_t h = (SW == 8) ? (uint32_t)hh : (uint32_t)(wi0 >> 2);
        // scale bytes of sub-blocks 8n + 2j + h, j = 0..3
        const uint32_t sb = __byte_perm(s0, s1, h | ((2u + h) << 4) | ((4u + h) << 8) | ((6u + h) << 12));
        const uint32_t scn = sb & 0x0F0F0F0Fu;
        const uint32_t mnn = (sb >> 4) & 0x0F0F0F0Fu;
        const float sc[4] = {byte_as_float<0>(scn), byte_as_float<1>(scn), byte_as_float<2>(scn),
                             byte_as_float<3>(scn)};
        const float mn[4] = {byte_as_float<0>(mnn), byte_as_float<1>(mnn), byte_as_float<2>(mnn),
                             byte_as_float<3>(mnn)};
#pragma unroll
        for (int t = 0; t < M; ++t) {
            float A = 0.f, B = 0.f;
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
                A = fmaf(sc[j], sl.xp[t][j][hh] * (float)Sacc, A);
                B = fmaf(mn[j], sl.xs[t][j][hh], B);
            }
            acc[t] = fmaf(d, A, fmaf(-dmin, B, acc[t]));
        }
    }
}

__device__ __forceinline__ void flag_error(volatile int* abort_flag)
{
    atomicOr(&g_mv_error, Q2K_ERR_BIT_WAIT_TIMEOUT);
    *abort_flag = 1;
}

template <int M, int ACT, int SW, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB) q2k_mv_kernel(const MvArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    using S = Slice<M, ACT, SW>;
    constexpr int SPB = 16 / SW;  // slices per block
    constexpr int RPT = rpt_max(M);

    // shared layout: [stages][ mbarriers full/empty, abort ][ reduction x2 ][ ysum ]
    uint8_t* ring = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)a.nst * a.stage_bytes);
    const int wpg = a.s_pad >= 32 ? a.s_pad / 32 : 1;  // warps per row group
    float* red = reinterpret_cast<float*>(bars + 2 * a.nst + 2);
    const int red_one = a.groups * RPT * M * wpg;
    float* ysum = red + 2 * red_one;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * a.nst);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int nwarps = a.tc >> 5;

    int64_t lo, hi;
    cta_range(a, lo, hi);
    const int nstages = stage_count(a, lo, hi);

    if (tid == 0) {
        for (int s = 0; s < a.nst; ++s) {
            mbar_init(smem_u32(&bars[s]), 1);
            mbar_init(smem_u32(&bars[a.nst + s]), nwarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (a.table && a.y_sum) {
        for (int r = tid; r < a.ysum_cap; r += blockDim.x) {
            int64_t row = lo + r;
            ysum[r] = (a.accumulate && row < hi) ? a.y_sum[row] : 0.f;
        }
    }
    __syncthreads();

    // Producer role (warp 0): fill stage i into its ring slot.  Bulk copies
    // when every row start and length is 16-byte aligned, else warp-wide
    // 4-byte copies.  Called by all lanes of warp 0.
    const uint32_t chunk = (uint32_t)a.nbc * kBlockBytes;
    auto produce = [&](int i) {
        const int slot = i % a.nst;
        const Stage st = stage_at(a, lo, hi, i);
        const uint8_t* src0 = seg_weights(a, st.e) + st.row0 * a.row_bytes + (int64_t)a.kb0 * kBlockBytes;
        uint8_t* dst0 = ring + (size_t)slot * a.stage_bytes;
        const uint32_t full = smem_u32(&bars[slot]);
        const bool tma = ((reinterpret_cast<uintptr_t>(src0) | (uintptr_t)a.row_bytes | chunk) & 15u) == 0;
        if (tma) {
            if (lane == 0) {
                mbar_arrive_expect_tx(full, chunk * st.nrows);
                for (int r = 0; r < st.nrows; ++r)
                    bulk_copy_g2s(smem_u32(dst0 + (size_t)r * a.rstride), src0 + r * a.row_bytes, chunk, full);
            }
        } else {
            const uint32_t words = chunk >> 2;
            for (int r = 0; r < st.nrows; ++r) {
                const uint8_t* src = src0 + r * a.row_bytes;
                uint32_t* dst = reinterpret_cast<uint32_t*>(dst0 + (size_t)r * a.rstride);
                for (uint32_t w = lane; w < words; w += 32)
                    dst[w] = ldg32_nc(src + 4 * w);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(full);
        }
    };
    int issued = 0;
    if (warp == 0) {
        const int pre = min(a.nst, nstages);
        for (; issued < pre; ++issued)
            produce(issued);
    }

    const int g = tid / a.s_pad;           // row group
    const int sl_idx = tid - g * a.s_pad;  // slice within the row
    const bool active = sl_idx < a.s_real;
    const int b = active ? sl_idx / SPB : 0;          // block within chunk
    const int w0 = (active ? sl_idx % SPB : 0) * SW;  // first qs word, 0..15
    const int n = w0 >> 3;
    const int wi0 = w0 & 7;
    const int wig = sl_idx >> 5;  // warp index within the group

    S sl;
    int cur_e = -1;
    float racc[RPT][M];

    for (int i = 0; i < nstages; ++i) {
        const int slot = i % a.nst;
        const Stage st = stage_at(a, lo, hi, i);
        if (st.e != cur_e && (cur_e < 0 || a.x_seg_stride != 0)) {
            load_slice<M, ACT, SW>(sl, a.x + (int64_t)st.e * a.x_seg_stride, a.x_tok_stride, a.kb0 + b, n, wi0,
                                   active);
        }
        cur_e = st.e;
        bool ok = !*abort_flag;
        if (ok) {
            if (lane == 0)
                ok = mbar_wait_bounded(smem_u32(&bars[slot]), (i / a.nst) & 1, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok && lane == 0)
                flag_error(abort_flag);
        }
#pragma unroll
        for (int k = 0; k < RPT; ++k)
#pragma unroll
            for (int t = 0; t < M; ++t)
                racc[k][t] = 0.f;
        if (ok) {
            const uint8_t* base = ring + (size_t)slot * a.stage_bytes + (size_t)b * kBlockBytes;
#pragma unroll
            for (int k = 0; k < RPT; ++k) {
                const int rr = g + k * a.groups;
                if (k < a.rpt && rr < st.nrows && active)
                    slice_dot<M, ACT, SW>(sl, base + (size_t)rr * a.rstride, n, wi0, racc[k]);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bars[a.nst + slot]));
        }
        // refill this slot with stage i + nst once every warp has released it
        if (warp == 0 && issued < nstages) {
            bool ok2 = !*abort_flag;
            if (ok2) {
                if (lane == 0)
                    ok2 = mbar_wait_bounded(smem_u32(&bars[a.nst + slot]), (i / a.nst) & 1, abort_flag);
                ok2 = __shfl_sync(0xffffffffu, ok2, 0);
                if (!ok2 && lane == 0)
                    flag_error(abort_flag);
            }
            if (ok2) {
                produce(issued);
                ++issued;
            }
        }
        // reduce every (row slot, token) over the row group's lanes
        const int width = a.s_pad < 32 ? a.s_pad : 32;
#pragma unroll
        for (int k = 0; k < RPT; ++k)
#pragma unroll
            for (int t = 0; t < M; ++t) {
                float v = racc[k][t];
                if (k < a.rpt)
                    for (int o = width >> 1; o > 0; o >>= 1)
                        v += __shfl_xor_sync(0xffffffffu, v, o);
                racc[k][t] = v;
            }
        float* rbuf = red + (i & 1) * red_one;
        if (wpg > 1) {
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < RPT; ++k)
#pragma unroll
                    for (int t = 0; t < M; ++t)
                        rbuf[((g * RPT + k) * M + t) * wpg + wig] = racc[k][t];
            }
            __syncthreads();
        }
        // writer: thread (k*M + t) of the group (several warps), or the
        // group's slice-0 lane (group within one warp)
        if (ok) {
#pragma unroll
            for (int k = 0; k < RPT; ++k)
#pragma unroll
                for (int t = 0; t < M; ++t) {
                    const int rr = g + k * a.groups;
                    if (k >= a.rpt || rr >= st.nrows)
                        continue;
                    float v;
                    if (wpg > 1) {
                        if (sl_idx != k * M + t)
                            continue;
                        v = 0.f;
                        const float* rp = rbuf + ((g * RPT + k) * M + t) * wpg;
                        for (int q = 0; q < wpg; ++q)
                            v += rp[q];
                    } else {
                        if (sl_idx != 0)
                            continue;
                        v = racc[k][t];
                    }
                    const int64_t row = st.row0 + rr;
                    if (a.table) {
                        if (a.y_exp) {
                            float* yp = a.y_exp + (int64_t)st.e * a.N[0] + row;
                            *yp = a.accumulate ? *yp + v : v;
                        }
                        if (a.y_sum)
                            ysum[row - lo] = fmaf(a.route_w[st.e], v, ysum[row - lo]);
                    } else {
                        float* yp = a.y[st.e] + (int64_t)t * a.ldy[st.e] + row;
                        *yp = a.accumulate ? *yp + v : v;
                    }
                }
        }
    }
    // every issued copy must have landed before the CTA exits
    if (*abort_flag && warp == 0 && lane == 0) {
        for (int i = max(0, issued - a.nst); i < issued; ++i)
            mbar_wait_bounded(smem_u32(&bars[i % a.nst]), (i / a.nst) & 1, nullptr);
    }
    __syncthreads();
    if (a.table && a.y_sum) {
        for (int r = tid; r < (int)(hi - lo); r += a.tc)
            a.y_sum[lo + r] = ysum[r];
    }
}

// ---- host side ----------------------------------------------------------------

namespace {

template <int M, int ACT, int SW, int MAXT, int MINB>
cudaError_t launch_one(const MvArgs& a, int grid, size_t smem, cudaStream_t s)
{
    auto k = q2k_mv_kernel<M, ACT, SW, MAXT, MINB>;
    static int configured_for = -1;  // device id the attribute was set for
    static size_t configured_smem = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (configured_for != dev || configured_smem < smem) {
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        configured_for = dev;
        configured_smem = smem;
    }
    k<<<grid, a.tc, smem, s>>>(a);
    return cudaGetLastError();
}

int sw_for(int act, int m)
{
    if (act == ACT_Q8)
        return m <= 4 ? 4 : 2;
    return m <= 2 ? 4 : (m <= 4 ? 2 : 1);
}

int mchunk_max(int act) { return act == ACT_Q8 ? 8 : 8; }

int nbc_max(int sw) { return sw == 4 ? 64 : (sw == 2 ? 64 : 32); }

template <int ACT, int SW>
cudaError_t dispatch_m(int m, const MvArgs& a, int grid, size_t smem, cudaStream_t s)
{
    constexpr int MAXT = SW == 4 ? 256 : 512;
    constexpr int MINB = SW == 4 ? 2 : 1;
    switch (m) {
#define Q2K_CASE(MM)                                                        \
    case MM:                                                                \
        if constexpr ((SW == 4 && (ACT == ACT_Q8 ? MM <= 4 : MM <= 2)) ||   \
                      (SW == 2 && (ACT == ACT_Q8 ? MM >= 5 : (MM >= 3 && MM <= 4))) || \
                      (SW == 1 && ACT == ACT_BF16 && MM >= 5))              \
            return launch_one<MM, ACT, SW, MAXT, MINB>(a, grid, smem, s);   \
        break;
        Q2K_CASE(1) Q2K_CASE(2) Q2K_CASE(3) Q2K_CASE(4) Q2K_CASE(5) Q2K_CASE(6) Q2K_CASE(7) Q2K_CASE(8)
#undef Q2K_CASE
    }
    return cudaErrorInvalidValue;
}

cudaError_t dispatch(int act, int sw, int m, const MvArgs& a, int grid, size_t smem, cudaStream_t s)
{
    if (act == ACT_Q8) {
        if (sw == 4)
            return dispatch_m<ACT_Q8, 4>(m, a, grid, smem, s);
        return dispatch_m<ACT_Q8, 2>(m, a, grid, smem, s);
    }
    if (sw == 4)
        return dispatch_m<ACT_BF16, 4>(m, a, grid, smem, s);
    if (sw == 2)
        return dispatch_m<ACT_BF16, 2>(m, a, grid, smem, s);
    return dispatch_m<ACT_BF16, 1>(m, a, grid, smem, s);
}

}  // namespace

cudaError_t launch_mv(const MvProblem& p, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess)
        return err;
    const int64_t nb = p.K / kBlockWeights;
    const int64_t act_bytes_per_k = 0;  // (documentation only)
    (void)act_bytes_per_k;
    const bool table = p.W_table != nullptr;

    // token chunks (all tokens in one chunk: the kernel family covers m <= 8)
    for (int t0 = 0; t0 < p.m; t0 += mchunk_max(p.act)) {
        const int mc = std::min(p.m - t0, mchunk_max(p.act));
        const int sw = sw_for(p.act, mc);
        const int spb = 16 / sw;
        const int64_t nbcm = nbc_max(sw);
        for (int64_t kb0 = 0; kb0 < nb; kb0 += nbcm) {
            const int nbc = (int)std::min(nbcm, nb - kb0);
            MvArgs a{};
            a.n_seg = p.n_seg;
            a.table = table ? 1 : 0;
            a.W_table = p.W_table;
            a.W[0] = static_cast<const uint8_t*>(p.W[0]);
            a.W[1] = static_cast<const uint8_t*>(p.W[1]);
            a.N[0] = p.N[0];
            a.N[1] = p.N[1];
            a.row_bytes = nb * kBlockBytes;
            a.kb0 = (int)kb0;
            a.nbc = nbc;
            a.x = static_cast<const uint8_t*>(p.x) + (int64_t)t0 * p.x_tok_stride;
            a.x_tok_stride = p.x_tok_stride;
            a.x_seg_stride = p.x_seg_stride;
            for (int e = 0; e < 2; ++e) {
                a.y[e] = p.y[e] ? p.y[e] + (int64_t)t0 * p.ldy[e] : nullptr;
                a.ldy[e] = p.ldy[e];
            }
            a.y_exp = p.y_exp;
            a.route_w = p.route_w;
            a.y_sum = p.y_sum;
            a.accumulate = kb0 > 0 ? 1 : 0;

            a.s_real = nbc * spb;
            if (a.s_real <= 32) {
                int sp = 1;
                while (sp < a.s_real)
                    sp <<= 1;
                a.s_pad = sp;
            } else {
                a.s_pad = (a.s_real + 31) / 32 * 32;
            }
            const int tc_target = 256;
            a.groups = std::max(1, tc_target / a.s_pad);
            a.tc = a.groups * a.s_pad;
            const int64_t chunk = (int64_t)nbc * kBlockBytes;
            a.rstride = (uint32_t)((chunk + 15) / 16 * 16);
            const int stage_target = 16384;
            const int rmax = rpt_max(mc);
            int rpt = (int)std::max<int64_t>(1, std::min<int64_t>(rmax, stage_target / ((int64_t)a.groups * a.rstride)));
            a.rpt = rpt;
            a.rps = a.groups * rpt;
            a.stage_bytes = (uint32_t)a.rps * a.rstride;

            const bool big = sw == 4;
            const int ctas_per_sm = big ? 2 : 1;
            const size_t smem_cap = std::min<size_t>((size_t)di.smem_optin, big ? 110 * 1024 : 220 * 1024);
            a.rows_total = table ? p.N[0] : p.N[0] + (p.n_seg > 1 ? p.N[1] : 0);
            int64_t grid = (int64_t)di.sm_count * ctas_per_sm;
            // at least a couple of rows per CTA
            grid = std::min<int64_t>(grid, std::max<int64_t>(1, a.rows_total / 2));
            if (grid < 1)
                grid = 1;
            const int64_t rows_per_cta = (a.rows_total + grid - 1) / grid;
            a.ysum_cap = (table && p.y_sum) ? (int)rows_per_cta : 0;

            const int wpg = a.s_pad >= 32 ? a.s_pad / 32 : 1;
            const size_t red_bytes = 2 * sizeof(float) * (size_t)a.groups * rmax * mc * wpg;
            const size_t fixed = red_bytes + sizeof(float) * (size_t)a.ysum_cap;
            int nst = (int)std::min<int64_t>(16, (int64_t)((smem_cap - fixed - 256) / (a.stage_bytes + 16)));
            // no more stages than this CTA will ever fill
            const int64_t max_stages = ((rows_per_cta + a.rps - 1) / a.rps) * (table ? p.n_seg : 2);
            nst = (int)std::min<int64_t>(nst, std::max<int64_t>(2, max_stages));
            if (nst < 2)
                return cudaErrorInvalidConfiguration;
            a.nst = nst;
            const size_t smem = (size_t)nst * a.stage_bytes + (2 * nst + 2) * sizeof(uint64_t) + fixed;
            err = dispatch(p.act, sw, mc, a, (int)grid, smem, s);
            if (err != cudaSuccess)
                return err;
        }
    }
    return cudaSuccess;
}

cudaError_t mv_error_word(int32_t* out, bool clear)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_mv_error, sizeof(int));
    if (e != cudaSuccess)
        return e;
    *out = v;
    if (clear) {
        int z = 0;
        e = cudaMemcpyToSymbol(g_mv_error, &z, sizeof(int));
    }
    return e;
}

}  // namespace q2k
