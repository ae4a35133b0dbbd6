// Q2_K GEMV / MMVQ for m <= 8 tokens, straight off the GGUF blocks.
//
// Follows engram_v41/apply.rs (single-token `wkv` projection off
// `wkv_q2k`), attn_v41/decode.rs (`kquant_mmvq_pair_w`: two matrices, one
// q8_1 input, one launch) and moe_v41/init.rs (`kquant_mmvq_q2_k_experts_w8`
// batches, `moe_v41_accumulate` route-weighted sum).
//
// Design (GB300, one CTA of 16 warps per SM):
//  * Weight rows stream into a ring of shared-memory stages (one or more
//    reduction units of rows, up to ~86 KB) with 1-D bulk asynchronous
//    copies (cp.async.bulk, the TMA engine) signalled on mbarriers.  Warp w
//    primes slot w; afterwards any warp may claim the refill of a slot that
//    every warp has released (a compare-and-swap on the next stage to
//    issue), so no warp is dedicated to producing.  Rows that are not
//    16-byte aligned are copied with 4-byte loads instead.  Every wait is
//    bounded.
//  * The activations of the CTA's K chunk are staged once in shared memory
//    (or made there: q8_1 of a bf16 row, or of SwiGLU of fp32 gate/up rows);
//    each thread then owns a fixed K-slice of every row (SW words of a
//    block's qs: 16*SW weights over 4 sub-blocks; 8 words, a whole half
//    block, for one token over long rows) and keeps the matching
//    activations in registers for all rows it visits, so the only per-row
//    traffic is the weight stream itself.
//  * Codes are extracted four at a time with one AND per register (the code
//    of pair j stays at bit 2j of each byte, i.e. scaled by 4^j; the 4^-j is
//    folded into the activation scale) and multiplied by DP4A (q8_1
//    activations) or two DP2A (bf16 activations as 16-bit fixed point with
//    one exponent per group of 16, or per 32 for 8-word slices).
//  * Per sub-block: y += d*sc*xscale*S - dmin*m*sum(x).  S*sc is formed in
//    int32 (with 8-word slices the two halves of a bit plane meet in int32
//    too); the min term is a dot product of the min nibbles with the group
//    sums (16-bit fixed point, one exponent per slice).
//  * Partial sums: a transpose-reduce across each warp's lanes deposits one
//    (row, token) sum per warp in shared memory; after the stage loop the
//    warps' sums are added in a fixed order (deterministic), which also
//    fuses the experts' route-weighted sum when one CTA walks every expert
//    of its rows.  With per-expert outputs each expert gets CTAs of its own
//    instead (segment-major), and the weighted sum is a separate pass.
//  * The kernel is a programmatic dependent launch: it touches no global
//    memory before griddepcontrol.wait, so its setup overlaps the previous
//    kernel in the stream.
#include "q2k_common.cuh"
#include "q2k_internal.h"
#include "q2k_q8.cuh"
#include "q2k_slice.cuh"

#include <algorithm>

namespace q2k {

__device__ int g_mv_error = 0;

constexpr int kThreads = 512;  // one CTA of 16 warps per SM

// Rows per thread per reduction unit (fewer for more tokens: registers).
__host__ __device__ constexpr int rpt_for(int m) { return m <= 2 ? 4 : (m <= 4 ? 2 : 1); }

struct MvArgs {
    // read by every thread in the prologue: kept together at the front
    int rows_q, rows_r;  // rows_total = rows_q * grid + rows_r: CTA c owns rows_q (+1 if c < rows_r) rows
    int rps;             // rows per stage = groups * RPT * sub
    int nst;             // stages in the ring
    uint32_t nst_magic;  // ceil(2^32 / nst): i / nst == umulhi(i, nst_magic) for i < 2^24
    int n_seg;
    int table;      // 1: W_table segments, stacked over one row range
    int seg_major;  // table only: CTA c works on segment c / cps alone, rows
                    // split cps ways (per-segment activations staged once)
    int cps;        // CTAs per segment (seg_major)
    int x_prep;     // 0: activations as given; 1: bf16 x quantised to q8_1 here;
                    // 2: q8_1 of SwiGLU(gu[e], gu[gu_E + e]) made here
    int N[2];
    int x_bulk;     // 1: the first segment's activations arrive by bulk copy
    int x_in_ring;  // 1: they arrive in the last ring slot, which the
                    // weights take over once every warp holds its slice
    int kb0;        // first block column of this K chunk
    int nbc;        // blocks in this K chunk
    int tc;         // threads
    uint32_t rstride;  // shared-memory row stride (16-byte multiple)
    uint32_t stage_bytes;
    // shared-memory layout (byte offsets, each 16-byte aligned)
    uint32_t off_x, off_bar, off_tab, off_cnt, off_red;
    int64_t row_bytes;  // bytes of a full weight row
    const uint8_t* x;
    int64_t x_tok_stride;
    int64_t x_seg_stride;
    const uint8_t* W[2];
    const void* const* W_table;
    int64_t w_seg_stride;  // table without W_table: segment e is W[0] + e * w_seg_stride
    int64_t ldy_exp;       // token stride of y_exp (table outputs for several tokens)
    const float* gu;  // x_prep 2: fp32 gate rows [gu_E][gu_ld], then up rows
    uint8_t* x_out;   // x_prep: the prepared q8_1 rows are also stored here
    int64_t gu_ld;    // floats per gu row
    int gu_E;
    // decomposition
    int s_real;         // slices per row
    int s_pad;          // lanes per row group
    int groups;         // row groups
    int sub;            // reduction units per stage
    int rows_total;     // concat: N0 + N1; table: N
    int max_stages;     // stages of the largest CTA
    int x_align;        // 16, 4 or 2: widest copy the activation addresses allow
    int accumulate;
    float* y[2];
    int64_t ldy[2];
    float* y_exp;
    const float* route_w;
    float* y_sum;
};

struct Stage {
    int e;
    int row0;
    int nrows;
};

__device__ __forceinline__ int stage_count(const MvArgs& a, int lo, int hi)
{
    if (hi <= lo)
        return 0;
    if (a.table)
        return ((hi - lo + a.rps - 1) / a.rps) * (a.seg_major ? 1 : a.n_seg);
    const int n0 = a.N[0];
    const int l0 = max(0, min(hi, n0) - lo);
    const int l1 = max(0, hi - max(lo, n0));
    return (l0 + a.rps - 1) / a.rps + (l1 + a.rps - 1) / a.rps;
}

// Stage i of the CTA owning rows [lo, hi): the rows split at the segment
// end (concat: both matrices' rows one after the other), repeated for every
// segment (table), or of the CTA's one segment seg (table, seg_major), in
// chunks of rps rows.
__device__ __forceinline__ Stage stage_at(const MvArgs& a, int lo, int hi, int i, int seg)
{
    if (a.table) {
        if (a.seg_major) {
            const int r = lo + i * a.rps;
            return Stage{seg, r, min(a.rps, hi - r)};
        }
        const int per = (hi - lo + a.rps - 1) / a.rps;
        const int e = i / per, c = i - e * per;
        const int r = lo + c * a.rps;
        return Stage{e, r, min(a.rps, hi - r)};
    }
    const int e0 = min(hi, a.N[0]);
    const int c0 = e0 > lo ? (e0 - lo + a.rps - 1) / a.rps : 0;
    if (i < c0) {
        const int r = lo + i * a.rps;
        return Stage{0, r, min(a.rps, e0 - r)};
    }
    const int r = max(lo, a.N[0]) - a.N[0] + (i - c0) * a.rps;
    return Stage{1, r, min(a.rps, hi - a.N[0] - r)};
}

__device__ __forceinline__ const uint8_t* seg_weights(const MvArgs& a, int e)
{
    if (a.table) {
        if (!a.W_table)  // row blocks of one matrix at a fixed stride
            return a.W[0] + (int64_t)e * a.w_seg_stride;
        const void* p;
        asm volatile("ld.global.nc.u64 %0, [%1];" : "=l"(p) : "l"(a.W_table + e));
        return static_cast<const uint8_t*>(p);
    }
    return a.W[e];
}

__device__ __forceinline__ void flag_error(volatile int* abort_flag)
{
    atomicOr(&g_mv_error, Q2K_ERR_BIT_WAIT_TIMEOUT);
    *abort_flag = 1;
}

// All lanes wait on the barrier (no divergence); the warp proceeds only if
// every lane saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int lane)
{
    const bool ok = __all_sync(0xffffffffu, !*abort_flag && mbar_wait_bounded(bar, parity, abort_flag));
    if (!ok && lane == 0)
        flag_error(abort_flag);
    return ok;
}

template <int M, int ACT, int SW>
__global__ void __launch_bounds__(kThreads, 1) q2k_mv_kernel(const MvArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    using S = Slice<M, ACT, SW>;
    constexpr int SPB = 16 / SW;  // slices per block
    constexpr int RPT = rpt_for(M);
    constexpr int V = RPT * M;        // partial sums per thread per unit
    constexpr int VP = pow2_ceil(V);  // padded to a power of two (<= 32)

    // Read one field from every 32 bytes of the parameter block up front:
    // their first (cold) reads then overlap instead of queuing one after
    // another behind the dependent index arithmetic below.
    asm volatile("" ::"r"(a.rows_q), "r"(a.x_bulk), "r"(a.off_x), "l"(a.x), "l"(a.W[1]), "r"(a.rows_total),
                 "l"(a.ldy[0]), "l"(a.y_sum));
    pdl_launch_dependents();  // the next kernel may set itself up meanwhile
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int nwarps = a.tc >> 5;
    const int wpg = a.s_pad >= 32 ? a.s_pad / 32 : 1;  // warps per row group
    const int red_one = a.groups * wpg * VP;           // floats per reduction unit
    const int unit_rows = a.groups * RPT;              // rows of one reduction unit

    // shared layout (offsets from the host, 16-byte aligned): weight ring |
    // staged activations | full barriers, abort flag | stage table |
    // release counters, copies issued, next stage to issue | partial sums
    // of every unit
    uint8_t* ring = smem;
    uint8_t* xsm = a.x_in_ring ? ring + (size_t)(a.nst - 1) * a.stage_bytes : smem + a.off_x;
    uint64_t* full_b = reinterpret_cast<uint64_t*>(smem + a.off_bar);
    uint64_t* xbar = full_b + a.nst;  // the first activation chunk landed
    volatile int* abort_flag = reinterpret_cast<volatile int*>(full_b + a.nst + 1);
    int4* tab = reinterpret_cast<int4*>(smem + a.off_tab);  // {e, row0, nrows, -} per stage
    int* cnt = reinterpret_cast<int*>(smem + a.off_cnt);    // warps done with each slot's stage
    int* n_issued = cnt + a.nst;
    int* next_issue = cnt + a.nst + 1;  // the next stage to copy in
    float* red = reinterpret_cast<float*>(smem + a.off_red);

    // seg_major: CTAs [e * cps, (e + 1) * cps) split the rows of segment e
    const int seg = a.seg_major ? (int)blockIdx.x / a.cps : 0;
    const int cta = (int)blockIdx.x - seg * (a.seg_major ? a.cps : 0);
    const int lo = cta * a.rows_q + min(cta, a.rows_r);
    const int hi = lo + a.rows_q + (cta < a.rows_r ? 1 : 0);
    const int nstages = stage_count(a, lo, hi);
    const int pre = min(a.x_in_ring ? a.nst - 1 : a.nst, nstages);  // stages copied in by the prologue
    // ring slot and phase parity of stage i, without a division
    auto ring_pos = [&](int i, int& slot, uint32_t& parity) {
        const int q = (int)__umulhi((uint32_t)i, a.nst_magic);
        slot = i - q * a.nst;
        parity = (uint32_t)q & 1u;
    };
    const bool x_first_bulk = a.x_bulk && nstages > 0;
    const int x_rowb = a.nbc * x_bytes_per_block<ACT>();
    const int x_rowb16 = (x_rowb + 15) & ~15;  // prepared activations: the source rows follow

    const uint32_t chunk = (uint32_t)a.nbc * kBlockBytes;
    // Bulk copy of stage st into a ring slot (lane 0 only; the source rows
    // start on 16-byte boundaries).
    auto copy_stage = [&](int slot, const int4 st, const uint8_t* src0) {
        uint8_t* dst0 = ring + (size_t)slot * a.stage_bytes;
        const uint32_t fb = smem_u32(&full_b[slot]);
        const uint64_t pol = l2_policy_evict_first();  // the weights are read once
        mbar_arrive_expect_tx(fb, chunk * st.z);
        if (chunk == a.rstride && (int64_t)chunk == a.row_bytes) {
            // whole rows, contiguous in global and in the ring: one copy
            bulk_copy_g2s_hint(smem_u32(dst0), src0, chunk * st.z, fb, pol);
        } else {
            for (int r = 0; r < st.z; ++r)
                bulk_copy_g2s_hint(smem_u32(dst0 + (size_t)r * a.rstride), src0 + r * a.row_bytes, chunk, fb, pol);
        }
    };
    auto stage_src = [&](const int4 st) {
        return seg_weights(a, st.x) + (int64_t)st.y * a.row_bytes + (int64_t)a.kb0 * kBlockBytes;
    };
    auto src_aligned = [&](const uint8_t* src0) {
        return ((reinterpret_cast<uintptr_t>(src0) | (uintptr_t)a.row_bytes | chunk) & 15u) == 0;
    };

    // Prologue, before the first barrier: lane 0 of warp w sets up slot w's
    // barrier and copies in stage w at once (warp 0 first the activations),
    // so the first bytes are requested as early as possible.
    bool early = false;  // this warp's prologue stage went out here
    if (lane == 0) {
        if (tid == 0) {
            mbar_init(smem_u32(xbar), 1);
            *abort_flag = 0;
            for (int s = 0; s <= a.nst; ++s)
                cnt[s] = 0;
            *next_issue = pre;
        }
        for (int s = warp; s < a.nst; s += nwarps)
            mbar_init(smem_u32(&full_b[s]), 1);
        fence_mbar_init();
    }
    // Everything above reads only parameters and shared memory; global
    // memory may still be written by the previous kernel in the stream.
    pdl_wait();
    if (tid == 0) {
        if (x_first_bulk) {
            // the activations first, ahead of the weight prefetch
            const int e0 = stage_at(a, lo, hi, 0, seg).e;
            const uint64_t pol = l2_policy_evict_last();  // every CTA reads them
            if (ACT == ACT_Q8 && a.x_prep == 1) {
                // the bf16 row, quantised to q8_1 below
                const uint32_t raw = (uint32_t)a.nbc * 512u;
                mbar_arrive_expect_tx(smem_u32(xbar), raw);
                bulk_copy_g2s_hint(smem_u32(xsm + x_rowb16), a.x + (int64_t)a.kb0 * 512, raw, smem_u32(xbar), pol);
            } else if (ACT == ACT_Q8 && a.x_prep == 2) {
                // the fp32 gate and up rows of segment e0, SwiGLU + q8_1 below
                const uint32_t raw = (uint32_t)a.nbc * 1024u;
                mbar_arrive_expect_tx(smem_u32(xbar), 2 * raw);
                const float* g0 = a.gu + (int64_t)e0 * a.gu_ld + (int64_t)a.kb0 * 256;
                const float* u0 = a.gu + (int64_t)(a.gu_E + e0) * a.gu_ld + (int64_t)a.kb0 * 256;
                bulk_copy_g2s_hint(smem_u32(xsm + x_rowb16), g0, raw, smem_u32(xbar), pol);
                bulk_copy_g2s_hint(smem_u32(xsm + x_rowb16 + raw), u0, raw, smem_u32(xbar), pol);
            } else {
                const uint8_t* xs0 =
                    a.x + (int64_t)e0 * a.x_seg_stride + (int64_t)a.kb0 * x_bytes_per_block<ACT>();
                mbar_arrive_expect_tx(smem_u32(xbar), (uint32_t)(M * x_rowb));
                for (int t = 0; t < M; ++t)
                    bulk_copy_g2s_hint(smem_u32(xsm + t * x_rowb), xs0 + t * a.x_tok_stride, (uint32_t)x_rowb,
                                       smem_u32(xbar), pol);
            }
        }
    }
    // The first stage goes out right behind the activations; the other
    // prologue stages wait until the activations have landed, so that the
    // copy engine serves the bytes needed first, first.
    const bool issue_now = warp < pre && (warp == 0 || !x_first_bulk);
    if (issue_now) {
        const Stage st0 = stage_at(a, lo, hi, warp, seg);
        const int4 st = make_int4(st0.e, st0.row0, st0.nrows, 0);
        const uint8_t* src0 = stage_src(st);
        early = src_aligned(src0);  // uniform within the warp
        if (early && lane == 0)
            copy_stage(warp, st, src0);
    }
    for (int i = tid; i < nstages; i += blockDim.x) {
        const Stage st = stage_at(a, lo, hi, i, seg);
        tab[i] = make_int4(st.e, st.row0, st.nrows, 0);
    }
    __syncthreads();

    // ---- producer role: stage i into slot i % nst.  Bulk copies are issued
    // by lane 0; the 4-byte fallback uses the whole warp. ----
    auto produce = [&](int i) {
        int slot;
        uint32_t parity;
        ring_pos(i, slot, parity);
        const int4 st = tab[i];
        const uint8_t* src0 = stage_src(st);
        uint8_t* dst0 = ring + (size_t)slot * a.stage_bytes;
        const uint32_t fb = smem_u32(&full_b[slot]);
        if (src_aligned(src0)) {
            if (lane == 0)
                copy_stage(slot, st, src0);
        } else {
            const uint32_t words = chunk >> 2;
            for (int r = 0; r < st.z; ++r) {
                const uint8_t* src = src0 + r * a.row_bytes;
                uint32_t* dst = reinterpret_cast<uint32_t*>(dst0 + (size_t)r * a.rstride);
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
    // Refills are claimed by whichever warp gets there first, so the cost of
    // issuing a copy does not settle on one warp: a stage can be copied in
    // once every warp has released its slot's previous stage.
    auto try_issue = [&]() {
        int claim = -1;
        if (lane == 0) {
            const int j = *reinterpret_cast<volatile int*>(next_issue);
            if (j < nstages) {
                int sj;  // a.nst >= 2
                uint32_t pj;
                ring_pos(j, sj, pj);
                if (*reinterpret_cast<volatile int*>(&cnt[sj]) == nwarps && atomicCAS(next_issue, j, j + 1) == j) {
                    atomicExch(&cnt[sj], 0);
                    __threadfence_block();
                    claim = j;
                }
            }
        }
        claim = __shfl_sync(0xffffffffu, claim, 0);
        if (claim >= 0)
            produce(claim);
    };
    // Wait for a weight stage.  A waiting warp polls (a short sleep between
    // polls) and claims refills meanwhile, so slots freed by slower warps
    // are refilled by the warps that are ahead.  Gives up (and raises the
    // abort flag) after about two seconds.
    auto wait_stage = [&](int slot, uint32_t parity) -> bool {
        const uint32_t bar = smem_u32(&full_b[slot]);
        uint64_t t0 = 0;
        for (uint32_t it = 0;; ++it) {
            if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity)))
                return true;
            try_issue();
            __nanosleep(64);
            if ((it & 15u) == 15u) {
                if (*abort_flag)
                    return false;
                const uint64_t now = global_timer_ns();
                if (t0 == 0) {
                    t0 = now;
                } else if (now - t0 > 2000000000ull) {
                    if (lane == 0)
                        flag_error(abort_flag);
                    return false;
                }
            }
        }
    };
    // prologue stages issued before the barrier are counted now; those whose
    // rows are not 16-byte aligned go out now (whole-warp copies)
    if (issue_now) {
        if (early) {
            if (lane == 0)
                atomicAdd(n_issued, 1);
        } else {
            produce(warp);
        }
    }

    // ---- this thread's slice ----
    const int g = tid / a.s_pad;           // row group
    const int sl_idx = tid - g * a.s_pad;  // slice within the row
    const bool active = sl_idx < a.s_real;
    const int b = active ? sl_idx / SPB : 0;          // block within chunk
    const int w0 = (active ? sl_idx % SPB : 0) * SW;  // first qs word, 0..15
    const int n = w0 >> 3;
    const int wi0 = w0 & 7;
    const int wig = sl_idx >> 5;  // warp index within the group
    const int wl = a.s_pad < 32 ? a.s_pad : 32;

    S sl;
    int cur_e = -1;
    bool aborted = false;  // after a wait gave up: keep walking the stages
                           // (segment-change barriers stay matched) but skip work
    if (x_first_bulk) {
        aborted = !warp_wait(smem_u32(xbar), 0, abort_flag, lane);
        if (warp > 0 && warp < pre)
            produce(warp);  // the rest of the prologue stages, now the activations are in
        if constexpr (ACT == ACT_Q8 && M == 1) {
            if (a.x_prep) {  // uniform across the CTA
                prep_x_q8(a, xsm, x_rowb16, warp, lane, nwarps);
                __syncthreads();
                // the prepared rows also go out (the first CTA of each
                // segment; a shared row is written once)
                if (a.x_out && cta == 0 && (a.x_prep == 2 || seg == 0)) {
                    uint8_t* dst = a.x_out + (int64_t)seg * a.x_seg_stride + (int64_t)a.kb0 * 8 * kQ8Bytes;
                    for (int o = tid * 4; o < x_rowb; o += blockDim.x * 4)
                        *reinterpret_cast<uint32_t*>(dst + o) = *reinterpret_cast<const uint32_t*>(xsm + o);
                }
            }
        }
        if constexpr (coop_x<M, ACT, SW>())
            convert_x_bf16<M, SW>(xsm, a.nbc);  // every thread (the condition is uniform)
        load_slice<M, ACT, SW>(sl, xsm, a.nbc, b, n, wi0, active);
        cur_e = tab[0].x;
        if (a.x_in_ring) {
            // the activations now sit in registers: release their slot
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                atomicAdd(&cnt[a.nst - 1], 1);
            }
        }
    }

    bool released_last = false;  // this warp freed a slot last time round
    for (int i = 0; i < nstages; ++i) {
        int slot;
        uint32_t parity;
        ring_pos(i, slot, parity);
        const int4 st4 = tab[i];
        const Stage st{st4.x, st4.y, st4.z};
        if (st.e != cur_e && (cur_e < 0 || a.x_seg_stride != 0)) {
            // uniform across the CTA: every warp walks the same stages
            __syncthreads();  // everyone is done with the previous chunk
            stage_x<M, ACT>(a.x + (int64_t)st.e * a.x_seg_stride, a.x_tok_stride, a.kb0, a.nbc, a.x_align, xsm);
            __syncthreads();
            if constexpr (coop_x<M, ACT, SW>())
                convert_x_bf16<M, SW>(xsm, a.nbc);
            load_slice<M, ACT, SW>(sl, xsm, a.nbc, b, n, wi0, active);
        }
        cur_e = st.e;
        // the warp that freed a slot last is the one behind: leave the
        // refill to a warp that is ahead (or waiting)
        if (!aborted && !released_last)
            try_issue();
        if (aborted || !wait_stage(slot, parity)) {
            aborted = true;
            continue;
        }
        const uint8_t* base = ring + (size_t)slot * a.stage_bytes + (size_t)b * kBlockBytes;

        for (int s = 0; s < a.sub; ++s) {
            const int rr0 = s * unit_rows;
            if (rr0 >= st.nrows)
                break;  // uniform: every warp skips the same units
            const int u = i * a.sub + s;
            float v[VP];
#pragma unroll
            for (int q = 0; q < VP; ++q)
                v[q] = 0.f;
#pragma unroll
            for (int k = 0; k < RPT; ++k) {
                const int rr = rr0 + g + k * a.groups;
                if (rr < st.nrows) {  // uniform within a row group
                    float acc[M];
#pragma unroll
                    for (int t = 0; t < M; ++t)
                        acc[t] = 0.f;
                    slice_dot<M, ACT, SW>(sl, base + (size_t)rr * a.rstride, n, wi0, acc);
#pragma unroll
                    for (int t = 0; t < M; ++t)
                        v[k * M + t] = acc[t];
                }
            }
            // reduce over the row group's lanes and deposit the warp's sums;
            // they are added across warps once, after the stage loop
            float* rb = red + (size_t)u * red_one;
            if (wl == 32) {
                const float r = transpose_reduce<VP>(v, lane);
                constexpr int SH = 5 - log2_exact(VP);
                if ((lane & ((1 << SH) - 1)) == 0)
                    rb[(g * wpg + wig) * VP + (lane >> SH)] = r;
            } else {
#pragma unroll
                for (int q = 0; q < V; ++q)
                    for (int o = wl >> 1; o > 0; o >>= 1)
                        v[q] += __shfl_xor_sync(0xffffffffu, v[q], o);
                if (sl_idx == 0) {
#pragma unroll
                    for (int q = 0; q < V; ++q)
                        rb[g * VP + q] = v[q];
                }
            }
        }
        // release the slot (its refill is claimed by the next warp to look)
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&cnt[slot], 1) == nwarps - 1;
        }
        released_last = __shfl_sync(0xffffffffu, last, 0) != 0;
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
            if (x_first_bulk)
                mbar_wait_bounded(smem_u32(xbar), 0, nullptr);
        }
        __syncthreads();
        return;
    }

    // ---- outputs: add the warps' partial sums of every (row, token) ----
    // Unit u = i*sub + s holds rows s*unit_rows + g + k*groups of stage i,
    // value index k*M + t, one partial per warp of the row group.
    const int per_stage = a.sub * a.groups * V;
    for (int q = tid; q < nstages * per_stage; q += blockDim.x) {
        const int i = q / per_stage, p = q - i * per_stage;
        {
            const int4 st4 = tab[i];
            const Stage st{st4.x, st4.y, st4.z};
            const int s2 = p / (a.groups * V);
            const int rem = p - s2 * (a.groups * V);
            const int g2 = rem / V, idx = rem - g2 * V;
            const int k = idx / M, t = idx - k * M;
            const int rr = s2 * unit_rows + g2 + k * a.groups;
            if (rr >= st.nrows)
                continue;
            const float* rb = red + (size_t)(i * a.sub + s2) * red_one + g2 * wpg * VP + idx;
            float v = 0.f;
            for (int q = 0; q < wpg; ++q)
                v += rb[q * VP];
            const int row = st.row0 + rr;
            if (a.table) {
                if (a.y_exp) {
                    float* yp = a.y_exp + (int64_t)t * a.ldy_exp + (int64_t)st.e * a.N[0] + row;
                    *yp = a.accumulate ? *yp + v : v;
                }
            } else {
                float* yp = a.y[st.e] + (int64_t)t * a.ldy[st.e] + row;
                *yp = a.accumulate ? *yp + v : v;
            }
        }
    }
    // fused route-weighted sum over the segments, in segment order
    if (a.table && a.y_sum) {
        const int per = (hi - lo + a.rps - 1) / a.rps;  // stages per segment
        for (int r = tid; r < hi - lo; r += blockDim.x) {
            const int c = r / a.rps, rin = r - c * a.rps;  // stage within a segment, row within it
            const int s2 = rin / unit_rows, rem = rin - s2 * unit_rows;
            const int k = rem / a.groups, g2 = rem - k * a.groups;
            const int idx = k * M;  // token 0 (experts run m = 1)
            float acc = a.accumulate ? a.y_sum[lo + r] : 0.f;
            for (int e = 0; e < a.n_seg; ++e) {
                const float* rb = red + (size_t)((e * per + c) * a.sub + s2) * red_one + g2 * wpg * VP + idx;
                float v = 0.f;
                for (int q = 0; q < wpg; ++q)
                    v += rb[q * VP];
                acc = fmaf(a.route_w[e], v, acc);
            }
            a.y_sum[lo + r] = acc;
        }
    }
}

// ---- host side ----------------------------------------------------------------

namespace {

template <int M, int ACT, int SW>
cudaError_t launch_one(const MvArgs& a, int grid, size_t smem, cudaStream_t s)
{
    auto k = q2k_mv_kernel<M, ACT, SW>;
    static std::atomic<unsigned long long> smem_devs{0};
    cudaError_t e = allow_max_smem(k, smem_devs);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(k, dim3((unsigned)grid), dim3((unsigned)a.tc), smem, s, a);
}

// Qs words per thread slice.  One token over a row of 16 blocks or more
// takes 8-word slices (128 weights: the per-row scale, min and load work is
// spread over twice the weights; the single-call kernel of q2k_m1.cu walks
// such rows the same way, and the two must give the same bits), and so does
// one q8_1 token over 8 to 15 blocks (the routed experts' down matrices:
// the MoE step went from 25.8 to 22.8 us; bf16 rows of 8 blocks were slower
// that way, 12.1 -> 13.4 us for the engram projection).  Shorter rows keep
// 4-word slices, so enough threads share each row.  The choice depends on
// the activation type, token count and row length alone, so an expert's row
// and a single call give the same bits.
int sw_for(int act, int m, int64_t nb)
{
    if (m == 1 && (nb >= 16 || (act == ACT_Q8 && nb >= 8)))
        return 8;
    if (act == ACT_Q8)
        return m <= 4 ? 4 : 2;
    return m <= 2 ? 4 : (m <= 4 ? 2 : 1);
}

template <int ACT, int SW>
cudaError_t dispatch_m(int m, const MvArgs& a, int grid, size_t smem, cudaStream_t s)
{
    switch (m) {
#define Q2K_CASE(MM)                                                                   \
    case MM:                                                                           \
        if constexpr ((SW == 8 && MM == 1) || (SW == 4 && (ACT == ACT_Q8 ? MM <= 4 : MM <= 2)) || \
                      (SW == 2 && (ACT == ACT_Q8 ? MM >= 5 : (MM >= 3 && MM <= 4))) || \
                      (SW == 1 && ACT == ACT_BF16 && MM >= 5))                         \
            return launch_one<MM, ACT, SW>(a, grid, smem, s);                          \
        break;
        Q2K_CASE(1) Q2K_CASE(2) Q2K_CASE(3) Q2K_CASE(4) Q2K_CASE(5) Q2K_CASE(6) Q2K_CASE(7) Q2K_CASE(8)
#undef Q2K_CASE
    }
    return cudaErrorInvalidValue;
}

cudaError_t dispatch(int act, int sw, int m, const MvArgs& a, int grid, size_t smem, cudaStream_t s)
{
    if (sw == 8)
        return act == ACT_Q8 ? dispatch_m<ACT_Q8, 8>(m, a, grid, smem, s) : dispatch_m<ACT_BF16, 8>(m, a, grid, smem, s);
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

size_t align16(size_t v) { return (v + 15) / 16 * 16; }

}  // namespace

namespace {

// Plan (and, unless dry, launch) every K chunk of a problem for
// q2k_mv_kernel.  A dry run makes no CUDA call besides the device query, so
// every chunk's plan is checked before the first launch.
cudaError_t run_mv(const MvProblem& p, cudaStream_t s, bool dry)
{
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess)
        return err;
    const int64_t nb = p.K / kBlockWeights;
    const bool table = p.W_table != nullptr || p.w_seg_stride != 0;  // segments of one shape
    if (p.N[0] > (1 << 30) || p.N[1] > (1 << 30) || (int64_t)p.N[0] + p.N[1] > (1 << 30))
        return cudaErrorInvalidValue;

    const int mc = p.m;  // the kernel family covers m <= 8 in one pass
    const int sw = sw_for(p.act, mc, nb);
    const int spb = 16 / sw;
    const int rpt = rpt_for(mc);
    const int vp = pow2_ceil(rpt * mc);
    const int xbpb = p.act == ACT_BF16 ? 512 : 8 * kQ8Bytes;  // staged bytes per token and block column
    // blocks per K chunk: the slices of a row fit the CTA, and the staged
    // activations take at most half of the shared memory
    int64_t nbcm = kThreads * sw / 16;
    while (nbcm > 1 && (int64_t)mc * nbcm * xbpb > 112 * 1024)
        nbcm /= 2;
    const size_t smem_cap = std::min<size_t>((size_t)di.smem_optin, 224 * 1024);

    for (int64_t kb0 = 0; kb0 < nb; kb0 += nbcm) {
        const int nbc = (int)std::min(nbcm, nb - kb0);
        MvArgs a{};
        a.n_seg = p.n_seg;
        a.table = table ? 1 : 0;
        a.W_table = p.W_table;
        a.W[0] = static_cast<const uint8_t*>(p.W[0]);
        a.W[1] = static_cast<const uint8_t*>(p.W[1]);
        a.N[0] = (int)p.N[0];
        a.N[1] = (int)p.N[1];
        a.row_bytes = nb * kBlockBytes;
        a.kb0 = (int)kb0;
        a.nbc = nbc;
        a.x = static_cast<const uint8_t*>(p.x);
        a.x_tok_stride = p.x_tok_stride;
        a.x_seg_stride = p.x_seg_stride;
        {
            const uintptr_t bits = (reinterpret_cast<uintptr_t>(p.x) + (uintptr_t)(kb0 * xbpb)) |
                                   (uintptr_t)(mc > 1 ? p.x_tok_stride : 0) | (uintptr_t)p.x_seg_stride;
            a.x_align = (bits & 15u) == 0 ? 16 : ((bits & 3u) == 0 ? 4 : 2);
            a.x_bulk = a.x_align == 16 ? 1 : 0;
        }
        a.x_prep = p.x_prep;
        a.gu = p.gu;
        a.gu_E = (int)p.gu_E;
        a.gu_ld = p.K;
        a.x_out = static_cast<uint8_t*>(p.x_out);
        if (p.x_prep) {
            // prepared activations: one token, q8_1, sources a bulk copy can read
            const uintptr_t src = p.x_prep == 1 ? reinterpret_cast<uintptr_t>(p.x) : reinterpret_cast<uintptr_t>(p.gu);
            if (p.act != ACT_Q8 || mc != 1 || (p.x_prep == 2 && (!p.gu || !table || p.gu_E < p.n_seg)) ||
                (src & 15u) != 0)
                return cudaErrorInvalidValue;
            a.x_align = 16;
            a.x_bulk = 1;
        }
        for (int e = 0; e < 2; ++e) {
            a.y[e] = p.y[e];
            a.ldy[e] = p.ldy[e];
        }
        a.y_exp = p.y_exp;
        a.ldy_exp = p.ldy_exp;
        a.w_seg_stride = p.w_seg_stride;
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
        a.groups = std::max(1, kThreads / a.s_pad);
        a.tc = a.groups * a.s_pad;  // <= kThreads, a multiple of 32
        const int64_t chunk = (int64_t)nbc * kBlockBytes;
        a.rstride = (uint32_t)((chunk + 15) / 16 * 16);
        const int unit_rows = a.groups * rpt;
        // stages of about 40 KB: several reduction units each
        a.sub = (int)std::max<int64_t>(1, std::min<int64_t>(16, 40 * 1024 / ((int64_t)unit_rows * a.rstride)));

        a.rows_total = table ? (int)p.N[0] : (int)(p.N[0] + (p.n_seg > 1 ? p.N[1] : 0));
        const int wpg = a.s_pad >= 32 ? a.s_pad / 32 : 1;
        // seg_major: CTAs per segment (one segment per CTA), else one row
        // range per CTA over every segment
        a.seg_major = (table && p.seg_major) ? 1 : 0;
        if (a.seg_major && p.y_sum)
            return cudaErrorInvalidValue;  // the route-weighted sum is a separate pass
        const int nseg_cta = (table && !a.seg_major) ? p.n_seg : 1;  // segments each CTA walks
        int64_t splits = a.seg_major ? std::max<int64_t>(1, di.sm_count / p.n_seg)
                                     : std::min<int64_t>(di.sm_count, std::max<int64_t>(1, a.rows_total / 2));
        if (a.seg_major)
            splits = std::min<int64_t>(splits, std::max<int64_t>(1, a.rows_total / 2));
        int64_t rows_per_cta = (a.rows_total + splits - 1) / splits;
        // more CTAs (in waves) when one CTA's partial sums would not fit
        const int64_t per_row = (int64_t)wpg * vp * nseg_cta * (int64_t)sizeof(float) / rpt + 1;
        while (rows_per_cta * per_row > 48 * 1024 && rows_per_cta > (int64_t)unit_rows * a.sub) {
            splits += a.seg_major ? splits : di.sm_count;
            rows_per_cta = (a.rows_total + splits - 1) / splits;
        }
        const int64_t grid = a.seg_major ? splits * p.n_seg : splits;
        a.cps = (int)splits;
        // a stage never holds more rows than the CTA owns
        while (a.sub > 1 && (int64_t)unit_rows * a.sub / 2 >= rows_per_cta)
            a.sub = (a.sub + 1) / 2;
        a.rps = unit_rows * a.sub;
        a.stage_bytes = (uint32_t)(a.rps * (int64_t)a.rstride);

        a.rows_q = (int)(a.rows_total / splits);
        a.rows_r = (int)(a.rows_total % splits);
        const int64_t stages_per_cta = ((rows_per_cta + a.rps - 1) / a.rps) * (table ? nseg_cta : 2);
        a.max_stages = (int)stages_per_cta;
        const bool coop = p.act == ACT_BF16 && (sw == 4 || sw == 8) && mc <= 2;
        if (coop && (int64_t)mc * nbc * 16 > (int64_t)kCoopGroupsPerThread * a.tc)
            return cudaErrorInvalidConfiguration;  // not reached: tc >= 4 * nbc and groups >= 2 for m = 2
        size_t x_bytes = coop ? align16((size_t)coop_x_bytes(mc, nbc)) : align16((size_t)mc * nbc * xbpb);
        if (p.x_prep)  // the source rows follow the q8_1 rows
            x_bytes += (size_t)nbc * (p.x_prep == 1 ? 512 : 2048);
        // a single activation chunk, read once: stage it in the last ring slot
        a.x_in_ring = (a.x_bulk && (p.x_seg_stride == 0 || p.n_seg == 1 || a.seg_major) && x_bytes <= a.stage_bytes) ? 1 : 0;
        const size_t red_bytes = sizeof(float) * (size_t)stages_per_cta * a.sub * a.groups * wpg * vp;
        size_t smem = 0;
        int nst = 8;
        for (; nst >= 2; --nst) {
            a.nst = (int)std::min<int64_t>(nst, std::max<int64_t>(2, stages_per_cta + a.x_in_ring));
            a.off_x = (uint32_t)((size_t)a.nst * a.stage_bytes);
            a.off_bar = (uint32_t)(a.off_x + (a.x_in_ring ? 0 : x_bytes));
            a.off_tab = (uint32_t)align16(a.off_bar + (size_t)(a.nst + 2) * sizeof(uint64_t));
            a.off_cnt = (uint32_t)align16(a.off_tab + (size_t)a.max_stages * sizeof(int4));
            a.off_red = (uint32_t)align16(a.off_cnt + (size_t)(a.nst + 2) * sizeof(int));
            smem = align16(a.off_red + red_bytes);
            if (smem <= smem_cap)
                break;
        }
        if (nst < 2)
            return cudaErrorInvalidConfiguration;
        a.nst_magic = (uint32_t)((0x100000000ull + (uint64_t)a.nst - 1) / (uint64_t)a.nst);
        if (dry)
            continue;
        err = dispatch(p.act, sw, mc, a, (int)grid, smem, s);
        if (err != cudaSuccess)
            return err;
    }
    return cudaSuccess;
}

}  // namespace

bool mv_plan_ok(const MvProblem& p)
{
    if (m1_supported(p) || mt_supported(p))
        return true;
    return run_mv(p, nullptr, true) == cudaSuccess;
}

cudaError_t launch_mv(const MvProblem& p, cudaStream_t s)
{
    if (m1_supported(p))
        return launch_m1(p, s);  // one token over long rows: per-team rings
    if (mt_supported(p))
        return launch_mt(p, s);  // several tokens: the tensor-core kernel
    cudaError_t err = run_mv(p, s, true);  // every chunk planned before any launch
    if (err != cudaSuccess)
        return err;
    return run_mv(p, s, false);
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
