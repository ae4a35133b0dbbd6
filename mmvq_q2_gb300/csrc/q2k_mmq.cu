// Q2_K matmul for many tokens, y = x W^T with W read as Q2_K blocks
// (moe_v41/init.rs, `MoeV41::new`: the `metrale_q2_k_mmq128_*` kernels and
// their q8_1 activation quantisers for more than 8 tokens; the prefill side
// of the path).  On the 5th-generation tensor cores:
//
//   warp 0      streams the weights as raw Q2_K bytes: 128 rows x 4 blocks
//               (1024 K, 43 KB) per 2-D tensor copy into a ring of "raw"
//               stages (the weight stream is 84 bytes per 256 weights, not
//               512 as bf16);
//   warps 3-10  expand them on-chip into the MMA's A operand: bf16 tiles of
//               128 rows x 64 K in the 128-byte-swizzled K-major layout.
//               Each weight is d*sc*q - dmin*m computed in fp32 and rounded
//               once to bf16 (the value q2k_dequant_rows gives it); a
//               thread makes the four possible values of a 16-weight
//               sub-block and picks them with byte permutes keyed by the
//               2-bit codes;
//   warp 2      copies the activation tiles (bf16, 64 K x the token tile,
//               same swizzle) with 2-D tensor copies;
//   warp 1      allocates the fp32 accumulator in tensor memory and issues
//               tcgen05.mma (M = 128, N = token tile, K = 16) from one
//               thread, freeing each A/B stage with tcgen05.commit;
//   warps 4-7   read the accumulator back (tcgen05.ld) and store y.
// K is split across CTAs (in 1024-wide pieces) when the tiles are too few to
// fill the GPU; the splits then add into y with fp32 atomics after a clear.
// Every wait is bounded: on a timeout the kernel raises its error word,
// lets its issued copies land, frees its tensor memory and returns.
#include <algorithm>
#include <mutex>

#include "q2k_common.cuh"
#include "q2k_internal.h"
#include "q2k_umma.cuh"

#include <cudaTypedefs.h>

namespace q2k {

__device__ int g_mmq_error = 0;

namespace {

constexpr int kMqThreads = 352;       // 11 warps
constexpr int kMqConv0 = 96;          // first converter thread (warp 3)
constexpr int kMqConv = 256;          // converter threads (warps 3..10)
constexpr int kMqBlocks = 4;          // Q2_K blocks per raw stage (1024 K)
constexpr int kMqSteps = kMqBlocks * 256 / kBK;           // 64-wide K steps per raw stage: 16
constexpr uint32_t kRawBytes = kBM * kMqBlocks * kBlockBytes;  // 43008
constexpr uint32_t kRawRowBytes = kMqBlocks * kBlockBytes;     // 336

struct MqArgs {
    int m, N;
    int64_t ldy;
    float* y;
    int ntok;         // token tile (MMA N): multiple of 16, <= 256
    int nsa;          // A/B ring stages
    int nraw;         // raw ring stages
    int rs_per_split; // raw stages (1024 K each) per CTA
    int nrs;          // raw stages over the whole K
    int atomic;       // splits add into y
    int tmem_cols;
    uint32_t b_bytes;
    uint32_t off_b, off_raw, off_bar;
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

__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__global__ void __launch_bounds__(kMqThreads, 1)
    q2k_mmq_kernel(const MqArgs a, const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tx)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    pdl_launch_dependents();  // the next kernel may set itself up meanwhile
    // the 128-byte swizzle repeats every 1024 bytes: stages start on 1024
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kBM;     // first W row of the tile
    const int t0 = blockIdx.y * a.ntok;  // first token of the tile
    const int rs0 = blockIdx.z * a.rs_per_split;
    const int nr = min(a.nrs, rs0 + a.rs_per_split) - rs0;  // raw stages of this CTA
    const int ng = nr * kMqSteps;                           // 64-wide K steps of this CTA

    uint8_t* aring = smem;
    uint8_t* bring = smem + a.off_b;
    uint8_t* rring = smem + a.off_raw;
    uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem + a.off_bar);
    uint64_t* raw_empty = raw_full + a.nraw;
    uint64_t* a_full = raw_empty + a.nraw;
    uint64_t* b_full = a_full + a.nsa;
    uint64_t* ab_empty = b_full + a.nsa;
    uint64_t* acc_b = ab_empty + a.nsa;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(acc_b + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_b + 2);
    volatile int* raw_issued = reinterpret_cast<volatile int*>(acc_b + 3);
    volatile int* b_issued = raw_issued + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.nraw; ++s) {
            mbar_init(smem_u32(&raw_full[s]), 1);
            mbar_init(smem_u32(&raw_empty[s]), kMqConv);
        }
        for (int s = 0; s < a.nsa; ++s) {
            mbar_init(smem_u32(&a_full[s]), kMqConv);
            mbar_init(smem_u32(&b_full[s]), 1);
            mbar_init(smem_u32(&ab_empty[s]), 1);
        }
        mbar_init(smem_u32(acc_b), 1);
        *abort_flag = 0;
        *raw_issued = 0;
        *b_issued = 0;
        fence_mbar_init();
    }
    if (warp == 1) {  // the accumulator: 128 lanes x tmem_cols fp32 columns
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"((uint32_t)a.tmem_cols)
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
            for (int i = 0; i < nr && !*abort_flag; ++i) {
                const int r = i % a.nraw, u = i / a.nraw;
                if (u > 0 && !mbar_wait_bounded(smem_u32(&raw_empty[r]), (uint32_t)(u - 1) & 1u, abort_flag)) {
                    give_up();
                    break;
                }
                mbar_arrive_expect_tx(smem_u32(&raw_full[r]), kRawBytes);
                tma_load_2d(smem_u32(rring + (size_t)r * kRawBytes), &tq, (rs0 + i) * (int)(kRawRowBytes / 4), n0,
                            smem_u32(&raw_full[r]), pol);
                *raw_issued = i + 1;
            }
        }
    } else if (warp == 2) {
        if (lane == 0) {  // activation tiles: the token tile x 64 K, swizzled
            const uint64_t pol = l2_policy_evict_last();  // every weight tile reads them
            const int k0 = rs0 * kMqSteps;
            for (int g = 0; g < ng && !*abort_flag; ++g) {
                const int s = g % a.nsa, u = g / a.nsa;
                if (u > 0 && !mbar_wait_bounded(smem_u32(&ab_empty[s]), (uint32_t)(u - 1) & 1u, abort_flag)) {
                    give_up();
                    break;
                }
                mbar_arrive_expect_tx(smem_u32(&b_full[s]), a.b_bytes);
                tma_load_2d(smem_u32(bring + (size_t)s * a.b_bytes), &tx, (k0 + g) * kBK, t0, smem_u32(&b_full[s]),
                            pol);
                *b_issued = g + 1;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            const uint32_t idesc = instr_desc(a.ntok);
            bool ok = true;
            for (int g = 0; g < ng; ++g) {
                const int s = g % a.nsa, u = g / a.nsa;
                if (!mbar_wait_bounded(smem_u32(&a_full[s]), (uint32_t)u & 1u, abort_flag) ||
                    !mbar_wait_bounded(smem_u32(&b_full[s]), (uint32_t)u & 1u, abort_flag)) {
                    give_up();
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t sa = smem_u32(aring + (size_t)s * kATileBytes);
                const uint32_t sb = smem_u32(bring + (size_t)s * a.b_bytes);
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)  // K = 16 per MMA: 32 bytes along the swizzled row
                    umma_f16(tmem, smem_desc_sw128(sa + 32 * k), smem_desc_sw128(sb + 32 * k), idesc, g > 0 || k > 0);
                umma_commit(smem_u32(&ab_empty[s]));  // A and B of the stage are free once these MMAs are done
            }
            if (ok)
                umma_commit(smem_u32(acc_b));  // the accumulator is complete
        }
        __syncwarp();
    } else {
        // ---- converters: thread ct owns W row `row` of the tile and, in
        // every 64-wide step, one bit plane of it (32 weights, 4 chunks) ----
        const int ct = threadIdx.x - kMqConv0;
        const int row = ct & (kBM - 1);
        const int jj = ct >> 7;  // which of the step's two bit planes
        uint8_t* arow = aring + (size_t)row * 128;
        for (int i = 0; i < nr; ++i) {
            const int r = i % a.nraw;
            if (*abort_flag || !mbar_wait_bounded(smem_u32(&raw_full[r]), (uint32_t)(i / a.nraw) & 1u, abort_flag)) {
                give_up();
                break;
            }
            const uint8_t* rrow = rring + (size_t)r * kRawBytes + (size_t)row * kRawRowBytes;
            bool stop = false;
            for (int s16 = 0; s16 < kMqSteps; ++s16) {
                const int g = i * kMqSteps + s16;
                const int s = g % a.nsa, u = g / a.nsa;
                if (u > 0 && !mbar_wait_bounded(smem_u32(&ab_empty[s]), (uint32_t)(u - 1) & 1u, abort_flag)) {
                    give_up();
                    stop = true;
                    break;
                }
                // step s16: block s16/4 of the stage, quarter qq (64 weights:
                // half qq/2, bit planes 2(qq&1) and 2(qq&1)+1)
                const uint8_t* blk = rrow + (s16 >> 2) * kBlockBytes;
                const int qq = s16 & 3;
                const int j = 2 * (qq & 1) + jj;
                const uint8_t* qs = blk + 16 + 32 * (qq >> 1);
                const uint32_t sc2 = *reinterpret_cast<const uint16_t*>(blk + 4 * qq + 2 * jj);  // its two sub-blocks
                const uint32_t dm = lds32(blk + 80);
                const float d = half_lo_f(dm), dmin = half_hi_f(dm);
                uint32_t lo0, hi0, lo1, hi1;
                subblock_table(d, dmin, sc2 & 0xFFu, lo0, hi0);
                subblock_table(d, dmin, sc2 >> 8, lo1, hi1);
                uint8_t* at = arow + (size_t)s * kATileBytes;
#pragma unroll
                for (int c = 0; c < 4; ++c) {  // positions 8c .. 8c+7 of the plane: K = 32 jj + 8c ..
                    const uint32_t w0 = lds32(qs + 8 * c), w1 = lds32(qs + 8 * c + 4);
                    const uint4 o = c < 2 ? expand_chunk(w0, w1, j, lo0, hi0) : expand_chunk(w0, w1, j, lo1, hi1);
                    *reinterpret_cast<uint4*>(at + 16 * ((4 * jj + c) ^ (row & 7))) = o;
                }
                fence_proxy_async_smem();  // the tensor cores read what the threads wrote
                mbar_arrive(smem_u32(&a_full[s]));
            }
            if (stop)
                break;
            mbar_arrive(smem_u32(&raw_empty[r]));  // this thread is done with the raw stage
        }
        // ---- epilogue: warps 4..7 read TMEM lanes 32q .. 32q+31 ----
        if (warp >= 4 && warp <= 7) {
            const int q = warp & 3;
            const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(acc_b), 0u, abort_flag));
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (!ok) {
                if (lane == 0)
                    give_up();
            } else {
                const int wrow = n0 + 32 * q + lane;
                for (int c = 0; c < a.ntok; c += 16) {
                    float v[16];
                    tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c, v);
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
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        // let the copies that were issued land before the CTA exits
        const int ri = *raw_issued, bi = *b_issued;
        for (int i = max(0, ri - a.nraw); i < ri; ++i)
            mbar_wait_bounded(smem_u32(&raw_full[i % a.nraw]), (uint32_t)(i / a.nraw) & 1u, nullptr);
        for (int g = max(0, bi - a.nsa); g < bi; ++g)
            mbar_wait_bounded(smem_u32(&b_full[g % a.nsa]), (uint32_t)(g / a.nsa) & 1u, nullptr);
    }
    __syncthreads();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)a.tmem_cols)
                     : "memory");
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
    a.tmem_cols = 32;
    while (a.tmem_cols < a.ntok)
        a.tmem_cols *= 2;
    a.b_bytes = (uint32_t)a.ntok * kBK * 2;
    a.nrs = (int)(K / (kMqBlocks * 256));
    const int gx = (int)((N + kBM - 1) / kBM);
    const int gy = (int)((m + a.ntok - 1) / a.ntok);
    int splits = 1;
    while ((int64_t)gx * gy * splits * 2 <= di.sm_count && a.nrs / (splits * 2) >= 2)
        splits *= 2;
    a.rs_per_split = (a.nrs + splits - 1) / splits;
    splits = (a.nrs + a.rs_per_split - 1) / a.rs_per_split;
    a.atomic = splits > 1 ? 1 : 0;
    const size_t cap = std::min<size_t>((size_t)di.smem_optin, 227 * 1024);
    const size_t bars = 1024;  // barriers, flags: well inside 1 KB
    for (a.nraw = 2; a.nraw >= 1; --a.nraw) {
        for (a.nsa = 4; a.nsa >= 2; --a.nsa) {
            a.off_b = (uint32_t)(a.nsa * kATileBytes);
            a.off_raw = (uint32_t)(a.off_b + (size_t)a.nsa * a.b_bytes);
            a.off_bar = (uint32_t)(a.off_raw + (size_t)a.nraw * kRawBytes);
            p.smem = 1024 + (size_t)a.off_bar + bars;
            if (p.smem <= cap) {
                p.grid = dim3((unsigned)gx, (unsigned)gy, (unsigned)splits);
                return true;
            }
        }
    }
    return false;
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
    static int configured_dev = -1;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess)
        return e;
    if (configured_dev != dev) {
        e = cudaFuncSetAttribute(q2k_mmq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(227 * 1024));
        if (e != cudaSuccess)
            return e;
        configured_dev = dev;
    }
    if (a.atomic) {
        e = cudaMemset2DAsync(y, (size_t)ldy * sizeof(float), 0, (size_t)N * sizeof(float), (size_t)m, s);
        if (e != cudaSuccess)
            return e;
    }
    return launch_pdl(q2k_mmq_kernel, p.grid, dim3(kMqThreads), p.smem, s, a, tq, tx);
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
