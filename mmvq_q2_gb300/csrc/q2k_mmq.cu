// Q2_K matmul for many tokens, y = x W^T with W read as Q2_K blocks
// (moe_v41/init.rs, `MoeV41::new`: the `metrale_q2_k_mmq128_*` kernels and
// their q8_1 activation quantisers for more than 8 tokens; the prefill side
// of the path).  On the 5th-generation tensor cores, one persistent CTA per
// SM, 16 warps, a pipeline of 128-K stages:
//
//   warp 0       streams the weights as raw Q2_K bytes: 128 rows x 4 blocks
//                (1024 K, 43 KB) per 2-D tensor copy into a ring of two
//                "raw" stages (84 bytes per 256 weights, not 512 as bf16);
//   warps 4-11   expand them into the MMA's A operand in TENSOR memory: a
//                ring of up to 4 slots of 128 lanes x 64 columns (128 K of
//                bf16).  Thread (warp w, lane l) owns weight row 32(w%4) + l,
//                the TMEM lane its warp may store to; warps 4-7 take the even
//                stages, warps 8-11 the odd ones.  Each weight is
//                d*sc*q - dmin*m in fp32 rounded once to bf16 (the value
//                q2k_dequant_rows gives it): the thread makes the four
//                possible values of each 16-weight sub-block and picks them
//                with byte permutes keyed by the 2-bit codes, and stores its
//                row's 64-weight halves with tcgen05.st;
//   warp 2       copies the activation tile of each stage (bf16, the token
//                tile x 128 K as two 128-byte-swizzled 64-K boxes) with 2-D
//                tensor copies into shared memory, one stage per A slot;
//   warp 1       allocates tensor memory and issues tcgen05.mma (M = 128,
//                N = token tile, K = 16; A from tensor memory, B from shared
//                memory): for token tiles up to 64 the whole warp walks the
//                stages and one elected lane issues, wider tiles from one
//                thread;
//   warps 12-15  read a finished accumulator back (tcgen05.ld) and store or
//                add it into y while the next one fills (two accumulators
//                when the token tile is at most 128 wide).
// Measured on this GPU, and the reasons for the shape:
//   * the tensor work of a tcgen05.mma of M = 128, K = 16 is about N/2
//     cycles (128 at N = 256), while one thread issuing alone spends about
//     50 cycles per MMA (about 20 with the whole warp walking the loop):
//     narrow token tiles gain little, so one token tile of up to 256 serves
//     every token count up to 256, and the expansion goes to tensor memory
//     (its stores do not compete with the MMA's operand reads in shared
//     memory);
//   * the issuing thread's own mbarrier waits, commits and MMA issues cost
//     about 100, 70 and 64 cycles each, even when nothing is pending.  So a
//     stage is 128 K (8 MMAs) behind ONE barrier: "full" completes when the
//     four converter warps of the stage have arrived and the activation
//     boxes have landed (their bytes), and ONE commit to "empty" frees both
//     the A slot and the activation stage.  At 64 K per stage with separate
//     A and B barriers the thread took about 860 cycles per 512 tensor
//     cycles.
// Work is dealt as (128-row tile, 1024-K stage) units, a contiguous run of
// them per CTA, so every SM gets the same share; a tile split between CTAs
// adds its partial sums into y with fp32 atomics after a clear.
// Every wait is bounded: on a timeout the kernel raises its error word,
// lets its issued copies and MMAs finish, frees its tensor memory and
// returns.
#include <algorithm>
#include <mutex>

#include "q2k_common.cuh"
#include "q2k_internal.h"
#include "q2k_umma.cuh"

#include <cudaTypedefs.h>

namespace q2k {

__device__ int g_mmq_error = 0;

namespace {

constexpr int kMqThreads = 512;       // 16 warps
constexpr int kMqConvWarp0 = 4;       // converters: warps 4..11
constexpr int kMqEpiWarp0 = 12;       // epilogue: warps 12..15
constexpr int kMqBlocks = 4;          // Q2_K blocks per raw stage (1024 K)
constexpr uint32_t kRawBytes = kBM * kMqBlocks * kBlockBytes;  // 43008
constexpr uint32_t kRawRowBytes = kMqBlocks * kBlockBytes;     // 336
constexpr int kSK = 2 * kBK;          // K per stage of the A/B pipeline: 128
constexpr int kMqStages = kMqBlocks * 256 / kSK;            // pipeline stages per raw stage: 8
constexpr int kBoxes = kSK / kBK;     // 64-K activation boxes per stage
constexpr uint32_t kACols = kSK / 2;  // A slot: 128 bf16 per lane
constexpr int kMaxStages = 4;         // A ring in tensor memory: 4 x 64 columns
constexpr uint32_t kTmemCols = 512;   // accumulators + A ring (one CTA per SM)

struct MqArgs {
    int m, N;
    int64_t ldy;
    float* y;
    int ntok;         // token tile (MMA N): multiple of 16, <= 256
    int nacc;         // accumulators in tensor memory (1 or 2)
    uint32_t acc_stride;  // columns between accumulators
    uint32_t a_col0;  // first column of the A ring
    int nst;          // pipeline stages (A slots = activation stages)
    int nraw;         // raw ring stages
    int nrs;          // raw stages (1024 K) over the whole K
    int64_t units;    // (tile, raw stage) units of one token tile
    int ctas;         // CTAs sharing the units of one token tile
    int atomic;       // partial tiles add into y
    int warp_issue;   // the instance whose MMA issuer's loop runs on its whole warp (token tiles up to 64)
    uint32_t b_box;   // bytes of one 64-K activation box: ntok x 128
    uint32_t off_raw, off_bar;
};

// The eight bf16 values of one 16-byte chunk: positions 8c .. 8c+7 of plane
// j, from the two qs words w0, w1, through the four-entry table {lo, hi}
// (value of code q at bytes 2q, 2q+1).
__device__ __forceinline__ uint4 expand_chunk(uint32_t w0, uint32_t w1, int j, uint32_t lo, uint32_t hi)
{
    // codes c of four positions, one per byte; the byte-permute selector of
    // two values {T[c_a], T[c_b]} is nibbles 2c_a, 2c_a+1, 2c_b, 2c_b+1
    const uint32_t s0 = ((w0 >> (2 * j)) & 0x03030303u) * 0x22u + 0x10101010u;
    const uint32_t s1 = ((w1 >> (2 * j)) & 0x03030303u) * 0x22u + 0x10101010u;
    uint4 o;
    o.x = __byte_perm(lo, hi, s0);
    o.y = __byte_perm(lo, hi, s0 >> 16);
    o.z = __byte_perm(lo, hi, s1);
    o.w = __byte_perm(lo, hi, s1 >> 16);
    return o;
}

// bf16 values of codes 0..3 of a sub-block with scale byte sc: fp32
// d*(sc&15)*q - dmin*(sc>>4), rounded once to bf16, as {T0,T1} and {T2,T3}.
__device__ __forceinline__ void subblock_table(float d, float dmin, uint32_t sc, uint32_t& lo, uint32_t& hi)
{
    const float dl = d * (float)(sc & 15u);
    const float ml = dmin * (float)(sc >> 4);
    const __nv_bfloat162 a = __floats2bfloat162_rn(fmaf(dl, 0.f, -ml), fmaf(dl, 1.f, -ml));
    const __nv_bfloat162 b = __floats2bfloat162_rn(fmaf(dl, 2.f, -ml), fmaf(dl, 3.f, -ml));
    lo = *reinterpret_cast<const uint32_t*>(&a);
    hi = *reinterpret_cast<const uint32_t*>(&b);
}

// The 64 weights of one row in 64-wide K step s16 (0..15) of a raw stage,
// as 32 bf16 pairs (K 2i in the low half of r[i]).  Step s16 is block s16/4
// of the stage, quarter qq = s16%4: half qq/2 of the block, bit planes
// 2(qq%2) (K 0..31 of the step) and 2(qq%2)+1 (K 32..63), sub-blocks
// 4qq .. 4qq+3.
__device__ __forceinline__ void expand_row_step(const uint8_t* rrow, int s16, uint32_t (&r)[32])
{
    const uint8_t* blk = rrow + (s16 >> 2) * kBlockBytes;
    const int qq = s16 & 3;
    const uint8_t* qs = blk + 16 + 32 * (qq >> 1);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        w[i] = lds32(qs + 4 * i);
    const uint32_t sc4 = lds32(blk + 4 * qq);
    const uint32_t dm = lds32(blk + 80);
    const float d = half_lo_f(dm), dmin = half_hi_f(dm);
#pragma unroll
    for (int pj = 0; pj < 2; ++pj) {
        const int j = 2 * (qq & 1) + pj;
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // sub-block 4qq + 2pj + h: plane positions 16h .. 16h+15
            uint32_t lo, hi;
            subblock_table(d, dmin, (sc4 >> (8 * (2 * pj + h))) & 0xFFu, lo, hi);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * h + cc;  // positions 8c .. 8c+7 of the plane
                const uint4 o = expand_chunk(w[2 * c], w[2 * c + 1], j, lo, hi);
                r[16 * pj + 4 * c + 0] = o.x;
                r[16 * pj + 4 * c + 1] = o.y;
                r[16 * pj + 4 * c + 2] = o.z;
                r[16 * pj + 4 * c + 3] = o.w;
            }
        }
    }
}

// A CTA's units [u0, u0 + nu), walked as (tile, raw stage) with 32-bit
// counters; a piece of work ends after a unit that is the CTA's last or the
// last stage of its tile.
struct UnitWalk {
    int tile, st;
    __device__ UnitWalk(int64_t u0, int nrs) : tile((int)(u0 / nrs)), st((int)(u0 % nrs)) {}
    __device__ void next(int nrs)
    {
        if (++st == nrs) {
            st = 0;
            ++tile;
        }
    }
};

// WI: the MMA issuer's loop runs on its whole warp (token tiles up to 64);
// otherwise on one thread.  Two instances, so each holds one issuer loop.
template <bool WI>
__global__ void __launch_bounds__(kMqThreads, 1)
    q2k_mmq_kernel(const MqArgs a, const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tx)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    pdl_launch_dependents();  // the next kernel may set itself up meanwhile
    // the 128-byte swizzle repeats every 1024 bytes: stages start on 1024
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.y * a.ntok;  // first token of the tile
    const int64_t u0 = a.units * blockIdx.x / a.ctas;
    const int nu = (int)(a.units * (blockIdx.x + 1) / a.ctas - u0);
    const int nss = nu * kMqStages;  // pipeline stages of this CTA
    const uint32_t b_bytes = kBoxes * a.b_box;

    uint8_t* bring = smem;
    uint8_t* rring = smem + a.off_raw;
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem + a.off_bar);
    uint64_t* raw_empty = raw_full + a.nraw;
    uint64_t* full = raw_empty + a.nraw;  // A slot written and activation box landed
    uint64_t* empty = full + kMaxStages;  // the MMAs reading both are done
    uint64_t* acc_full = empty + kMaxStages;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* mma_done = acc_empty + 2;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(mma_done + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 2);
    volatile int* raw_issued = reinterpret_cast<volatile int*>(mma_done + 3);
    volatile int* b_issued = raw_issued + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.nraw; ++s) {
            mbar_init(smem_u32(&raw_full[s]), 1);
            mbar_init(smem_u32(&raw_empty[s]), 8);  // one arrival per converter warp
        }
        for (int s = 0; s < a.nst; ++s) {
            mbar_init(smem_u32(&full[s]), 5);  // the four warps of the stage + the copy issuer
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&acc_full[s]), 1);
            mbar_init(smem_u32(&acc_empty[s]), 4);  // the four epilogue warps
        }
        mbar_init(smem_u32(mma_done), 1);
        *abort_flag = 0;
        *raw_issued = 0;
        *b_issued = 0;
        fence_mbar_init();
    }
    if (warp == 1) {  // accumulators and the A ring: 128 lanes x 512 columns
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // global memory may still be written by the previous kernel in the stream
    pdl_wait();
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    auto give_up = [&]() {
        atomicOr(&g_mmq_error, Q2K_ERR_BIT_WAIT_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp == 0) {
        if (lane == 0) {  // raw Q2_K stages: 128 rows x 336 bytes (84 words)
            const uint64_t pol = l2_policy_evict_first();
            UnitWalk w(u0, a.nrs);
            for (int i = 0; i < nu && !*abort_flag; ++i, w.next(a.nrs)) {
                const int r = i % a.nraw, u = i / a.nraw;
                if (u > 0 && !mbar_wait_bounded(smem_u32(&raw_empty[r]), (uint32_t)(u - 1) & 1u, abort_flag)) {
                    give_up();
                    break;
                }
                mbar_arrive_expect_tx(smem_u32(&raw_full[r]), kRawBytes);
                tma_load_2d(smem_u32(rring + (size_t)r * kRawBytes), &tq, w.st * (int)(kRawRowBytes / 4), w.tile * kBM,
                            smem_u32(&raw_full[r]), pol);
                *raw_issued = i + 1;
            }
        }
    } else if (warp == 2) {
        if (lane == 0) {  // activation tiles: the token tile x 128 K as two swizzled 64-K boxes
            const uint64_t pol = l2_policy_evict_last();  // every weight tile reads them
            UnitWalk w(u0, a.nrs);
            int s = 0, k8 = 0;
            uint32_t ph = 0;
            for (int g = 0; g < nss && !*abort_flag; ++g) {
                if (g >= a.nst && !mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u, abort_flag)) {
                    give_up();
                    break;
                }
                const int k = w.st * (kMqStages * kSK) + k8 * kSK;
                const uint32_t dst = smem_u32(bring + (size_t)s * b_bytes);
                mbar_arrive_expect_tx(smem_u32(&full[s]), b_bytes);
#pragma unroll
                for (int bx = 0; bx < kBoxes; ++bx)
                    tma_load_2d(dst + bx * a.b_box, &tx, k + bx * kBK, t0, smem_u32(&full[s]), pol);
                *b_issued = g + 1;
                if (++s == a.nst) {
                    s = 0;
                    ph ^= 1u;
                }
                if (++k8 == kMqStages) {
                    k8 = 0;
                    w.next(a.nrs);
                }
            }
        }
    } else if (WI && warp == 1) {
        // MMA issuer for token tiles up to 128: the whole warp walks the
        // stages (one wait and one commit per stage), one elected lane issues
        const uint32_t idesc = instr_desc(a.ntok);
        const uint32_t box16 = a.b_box >> 4;  // descriptor address units
        bool ok = true;
        int s = 0, pc = 0;
        uint32_t ph = 0;
        UnitWalk w(u0, a.nrs);
        for (int i = 0; i < nu && ok; ++i, w.next(a.nrs)) {
            const bool fresh = i == 0 || w.st == 0;  // first unit of a piece
            const int buf = pc % a.nacc;
            if (fresh && pc >= a.nacc &&
                !__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&acc_empty[buf]), (uint32_t)(pc / a.nacc - 1) & 1u,
                                                           abort_flag))) {
                ok = false;
                break;
            }
            const uint32_t dt = tmem + (uint32_t)buf * a.acc_stride;
            for (int k8 = 0; k8 < kMqStages; ++k8) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&full[s]), ph, abort_flag))) {
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t at = tmem + a.a_col0 + (uint32_t)s * kACols;
                const uint64_t bd = smem_desc_sw128(smem_u32(bring + (size_t)s * b_bytes));
#pragma unroll
                for (int k = 0; k < kSK / 16; ++k) {  // K = 16 per MMA: 8 A columns; 32 bytes along B's row
                    if (elect_one())
                        umma_f16_tmem_a(dt, at + 8 * k, bd + (uint64_t)((k >> 2) * box16 + 2 * (k & 3)), idesc,
                                        !(fresh && k8 == 0 && k == 0));
                }
                if (elect_one())
                    umma_commit(smem_u32(&empty[s]));  // the slot and the stage are free once these MMAs are done
                __syncwarp();
                if (++s == a.nst) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (ok && (i + 1 == nu || w.st + 1 == a.nrs)) {
                if (elect_one())
                    umma_commit(smem_u32(&acc_full[buf]));  // this accumulator is complete
                __syncwarp();
                ++pc;
            }
        }
        if (!ok && lane == 0)
            give_up();
        // every MMA issued so far has finished once this arrives
        if (elect_one())
            umma_commit(smem_u32(mma_done));
        __syncwarp();
        mbar_wait_bounded(smem_u32(mma_done), 0u, nullptr);
        __syncwarp();
    } else if (!WI && warp == 1) {
        if (lane == 0) {  // MMA issuer (wider tiles): one thread, one wait and one commit per stage
            const uint32_t idesc = instr_desc(a.ntok);
            const uint32_t box16 = a.b_box >> 4;  // descriptor address units
            bool ok = true;
            int s = 0, pc = 0;
            uint32_t ph = 0;
            UnitWalk w(u0, a.nrs);
            for (int i = 0; i < nu && ok; ++i, w.next(a.nrs)) {
                const bool fresh = i == 0 || w.st == 0;  // first unit of a piece
                const int buf = pc % a.nacc;
                if (fresh && pc >= a.nacc &&
                    !mbar_wait_bounded(smem_u32(&acc_empty[buf]), (uint32_t)(pc / a.nacc - 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t dt = tmem + (uint32_t)buf * a.acc_stride;
                for (int k8 = 0; k8 < kMqStages; ++k8) {
                    if (!mbar_wait_bounded(smem_u32(&full[s]), ph, abort_flag)) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t at = tmem + a.a_col0 + (uint32_t)s * kACols;
                    const uint64_t bd = smem_desc_sw128(smem_u32(bring + (size_t)s * b_bytes));
#pragma unroll
                    for (int k = 0; k < kSK / 16; ++k)  // K = 16 per MMA: 8 A columns; 32 bytes along B's row
                        umma_f16_tmem_a(dt, at + 8 * k, bd + (uint64_t)((k >> 2) * box16 + 2 * (k & 3)), idesc,
                                        !(fresh && k8 == 0 && k == 0));
                    umma_commit(smem_u32(&empty[s]));  // the slot and the stage are free once these MMAs are done
                    if (++s == a.nst) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (ok && (i + 1 == nu || w.st + 1 == a.nrs)) {
                    umma_commit(smem_u32(&acc_full[buf]));  // this accumulator is complete
                    ++pc;
                }
            }
            if (!ok)
                give_up();
            // every MMA issued so far has finished once this arrives
            umma_commit(smem_u32(mma_done));
            mbar_wait_bounded(smem_u32(mma_done), 0u, nullptr);
        }
        __syncwarp();
    } else if (warp >= kMqConvWarp0 && warp < kMqEpiWarp0) {
        // ---- converters: warp w stores TMEM lanes 32(w%4) .. +31; group
        // (w-4)/4 takes the pipeline stages of its parity ----
        const int q = warp & 3, grp = (warp - kMqConvWarp0) >> 2;
        const int row = 32 * q + lane;
        const uint32_t tlane = tmem + ((uint32_t)(32 * q) << 16) + a.a_col0;
        int s = grp % a.nst;
        uint32_t ph = (uint32_t)(grp / a.nst) & 1u;  // stage g = grp uses slot grp % nst
        for (int i = 0; i < nu; ++i) {
            const int r = i % a.nraw;
            if (*abort_flag || !mbar_wait_bounded(smem_u32(&raw_full[r]), (uint32_t)(i / a.nraw) & 1u, abort_flag)) {
                give_up();
                break;
            }
            const uint8_t* rrow = rring + (size_t)r * kRawBytes + (size_t)row * kRawRowBytes;
            bool stop = false;
            for (int k8 = grp; k8 < kMqStages; k8 += 2) {
                const int g = i * kMqStages + k8;
                if (g >= a.nst && !mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u, abort_flag)) {
                    give_up();
                    stop = true;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
                for (int bx = 0; bx < kBoxes; ++bx) {
                    uint32_t v[32];
                    expand_row_step(rrow, kBoxes * k8 + bx, v);
                    tmem_st32(tlane + (uint32_t)s * kACols + 32 * bx, v);
                }
                tmem_wait_st();
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&full[s]));
                // this group's next stage is g + 2
                s += 2;
                while (s >= a.nst) {
                    s -= a.nst;
                    ph ^= 1u;
                }
            }
            if (stop)
                break;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&raw_empty[r]));  // this warp is done with the raw stage
        }
    } else if (warp >= kMqEpiWarp0) {
        // ---- epilogue: warp w reads TMEM lanes 32(w%4) .. +31 ----
        const int q = warp & 3;
        int pc = 0;
        UnitWalk w(u0, a.nrs);
        for (int i = 0; i < nu; ++i, w.next(a.nrs)) {
            if (!(i + 1 == nu || w.st + 1 == a.nrs))
                continue;
            const int buf = pc % a.nacc;
            const bool ok =
                __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&acc_full[buf]), (uint32_t)(pc / a.nacc) & 1u,
                                                          abort_flag));
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (!ok) {
                if (lane == 0)
                    give_up();
                break;
            }
            const int wrow = w.tile * kBM + 32 * q + lane;
            const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)buf * a.acc_stride;
            for (int c = 0; c < a.ntok; c += 16) {
                float v[16];
                tmem_ld16(ta + (uint32_t)c, v);
                if (wrow < a.N) {
#pragma unroll
                    for (int jx = 0; jx < 16; ++jx) {
                        const int tok = t0 + c + jx;
                        if (tok < a.m) {
                            float* yp = a.y + (int64_t)tok * a.ldy + wrow;
                            if (a.atomic)
                                atomicAdd(yp, v[jx]);
                            else
                                *yp = v[jx];
                        }
                    }
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&acc_empty[buf]));
            ++pc;
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        // let the copies that were issued land before the CTA exits (a stage
        // whose converters gave up never completes: its wait runs out)
        const int ri = *raw_issued, bi = *b_issued;
        for (int i = max(0, ri - a.nraw); i < ri; ++i)
            mbar_wait_bounded(smem_u32(&raw_full[i % a.nraw]), (uint32_t)(i / a.nraw) & 1u, nullptr);
        for (int g = max(0, bi - a.nst); g < bi; ++g)
            mbar_wait_bounded(smem_u32(&full[g % a.nst]), (uint32_t)(g / a.nst) & 1u, nullptr);
    }
    __syncthreads();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// q8_1 rows -> bf16 rows: x = bf16(f32(d) * q), the values the q8_1 row
// encodes rounded once to bf16 (the MMQ's activation operand).
__global__ void __launch_bounds__(256) q8_1_to_bf16_kernel(const uint8_t* __restrict__ xq, int64_t m, int64_t K,
                                                           __nv_bfloat16* __restrict__ out)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t nblk = K / kQ8Values;
    const int64_t total = m * nblk * 8;  // 4 values per thread
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t blk = u >> 3;
        const int part = (int)(u & 7);
        const uint8_t* b = xq + blk * kQ8Bytes;
        const float d = __half2float(*reinterpret_cast<const __half*>(b));
        const uint32_t q4 = *reinterpret_cast<const uint32_t*>(b + 4 + 4 * part);
        const __nv_bfloat162 v0 =
            __floats2bfloat162_rn(d * (float)(int8_t)(q4 & 0xFF), d * (float)(int8_t)((q4 >> 8) & 0xFF));
        const __nv_bfloat162 v1 =
            __floats2bfloat162_rn(d * (float)(int8_t)((q4 >> 16) & 0xFF), d * (float)(int8_t)(q4 >> 24));
        __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(out + blk * kQ8Values + 4 * part);
        o[0] = v0;
        o[1] = v1;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 mq_encoder()
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

struct MqPlan {
    MqArgs a;
    dim3 grid;
    size_t smem;
};

bool plan_mmq(int64_t m, int64_t N, int64_t K, const DeviceInfo& di, MqPlan& p)
{
    if (m < 1 || N < 1 || K % (kMqBlocks * 256) || K < 1024)
        return false;
    MqArgs& a = p.a;
    a = MqArgs{};
    a.m = (int)m;
    a.N = (int)N;
    a.ntok = (int)std::min<int64_t>(256, (m + 15) / 16 * 16);
    a.nacc = a.ntok <= 128 ? 2 : 1;
    // whole-warp issue: 63.1 / 65.4 us at m = 16 / 64 (16384^2) against
    // 67.1 / 69.0 from one thread; mixed at 128-wide tiles, slower at 256
    a.warp_issue = a.ntok <= 64 ? 1 : 0;
    a.acc_stride = 128;
    a.a_col0 = 256;
    a.b_box = (uint32_t)a.ntok * kBK * 2;
    a.nrs = (int)(K / (kMqBlocks * 256));
    const int64_t tiles = (N + kBM - 1) / kBM;
    const int gy = (int)((m + a.ntok - 1) / a.ntok);
    a.units = tiles * a.nrs;
    a.ctas = (int)std::min<int64_t>(a.units, std::max(1, di.sm_count / gy));
    // a CTA's share is whole tiles only when the units divide evenly into
    // tile-aligned runs; otherwise partial tiles add into y
    a.atomic = (a.units % a.ctas != 0 || (a.units / a.ctas) % a.nrs != 0) ? 1 : 0;
    const size_t cap = std::min<size_t>((size_t)di.smem_optin, 227 * 1024);
    const size_t bars = 1024;  // barriers, flags: well inside 1 KB
    a.nraw = 2;
    for (a.nst = kMaxStages; a.nst >= 2; --a.nst) {
        a.off_raw = (uint32_t)((size_t)a.nst * kBoxes * a.b_box);
        a.off_bar = (uint32_t)(a.off_raw + (size_t)a.nraw * kRawBytes);
        p.smem = 1024 + (size_t)a.off_bar + bars;
        if (p.smem <= cap)
            break;
    }
    if (a.nst < 2)
        return false;
    // at least 120 KB of shared memory (over half an SM's 228 KB) keeps this
    // CTA alone on its SM, so its 512-column tensor-memory allocation never
    // waits for another CTA's
    p.smem = std::max<size_t>(p.smem, 120 * 1024);
    if (p.smem > cap)
        return false;
    p.grid = dim3((unsigned)a.ctas, (unsigned)gy, 1);
    return true;
}

}  // namespace

size_t mmq_q8_1_workspace(int64_t m, int64_t K) { return (size_t)m * (size_t)K * 2; }

bool mmq_supported(int64_t m, int64_t N, int64_t K)
{
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess || !mq_encoder())
        return false;
    MqPlan p;
    return plan_mmq(m, N, K, di, p);
}

cudaError_t launch_mmq_bf16(const void* W, int64_t N, int64_t K, const uint16_t* x, int64_t m, int64_t ldx, float* y,
                            int64_t ldy, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    PFN_cuTensorMapEncodeTiled_v12000 enc = mq_encoder();
    MqPlan p;
    if (!enc || !plan_mmq(m, N, K, di, p))
        return cudaErrorInvalidValue;
    MqArgs& a = p.a;
    a.ldy = ldy;
    a.y = y;
    const int64_t row_bytes = K / 256 * kBlockBytes;
    CUtensorMap tq{}, tx{};
    {
        // the weights as 4-byte words: [N rows, row_bytes / 4], a box of 84
        // words (4 blocks) x 128 rows
        const cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 4), (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
        const cuuint32_t box[2] = {kRawRowBytes / 4, (cuuint32_t)kBM};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(W), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)m};
        const cuuint64_t strides[1] = {(cuuint64_t)(ldx * 2)};
        const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)a.ntok};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    auto kern = a.warp_issue ? q2k_mmq_kernel<true> : q2k_mmq_kernel<false>;
    static std::atomic<unsigned long long> smem_devs[2] = {{0}, {0}};
    if ((e = allow_max_smem(kern, smem_devs[a.warp_issue ? 1 : 0])) != cudaSuccess)
        return e;
    if (a.atomic) {
        e = cudaMemset2DAsync(y, (size_t)ldy * sizeof(float), 0, (size_t)N * sizeof(float), (size_t)m, s);
        if (e != cudaSuccess)
            return e;
    }
    return launch_pdl(kern, p.grid, dim3(kMqThreads), p.smem, s, a, tq, tx);
}

cudaError_t launch_q8_1_to_bf16(const void* xq, int64_t m, int64_t K, uint16_t* out, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    const int64_t total = m * (K / kQ8Values) * 8;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, (int64_t)di.sm_count * 8));
    return launch_pdl(q8_1_to_bf16_kernel, dim3((unsigned)grid), dim3(256), 0, s, static_cast<const uint8_t*>(xq), m,
                      K, reinterpret_cast<__nv_bfloat16*>(out));
}

cudaError_t mmq_error_word(int32_t* out, bool clear)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_mmq_error, sizeof(int));
    if (e != cudaSuccess)
        return e;
    *out = v;
    if (clear) {
        int z = 0;
        e = cudaMemcpyToSymbol(g_mmq_error, &z, sizeof(int));
    }
    return e;
}

}  // namespace q2k
