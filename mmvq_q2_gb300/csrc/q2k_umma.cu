// Dense bf16 GEMM y = x W^T on the 5th-generation tensor cores (tcgen05),
// for the multi-token rows of the engram projection (engram_v41/apply.rs,
// `ops::dense_gemm` when tokens > 1) and the dense GEMMs of the sweep.
//
// One CTA computes a 128-row tile of W against a tile of up to 256 tokens:
//   warp 0      copies W and x tiles (64 K values each, 128-byte swizzled)
//               into a ring of shared-memory stages with TMA tensor copies;
//   warp 1      allocates the accumulator in tensor memory and issues
//               tcgen05.mma (M = 128, N = token tile, K = 16, bf16 in,
//               fp32 accumulate) from one thread, freeing each stage with
//               tcgen05.commit;
//   warps 2..5  read the accumulator back (tcgen05.ld, one TMEM lane per
//               W row) and store y, coalesced along N.
// K is split across CTAs when there are too few tiles to fill the GPU; the
// splits then add into y with fp32 atomics (y is cleared first).  When the
// tiles outnumber the SMs the ring is capped so that two CTAs share an SM
// (no second wave for the few tiles past one per SM).
// Every wait is bounded: on a timeout the kernel raises its error word,
// still frees its tensor memory and returns.  The kernel is a programmatic
// dependent launch: barriers and tensor memory are set up before it waits
// for the previous grid.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "q2k_common.cuh"
#include "q2k_internal.h"
#include "q2k_umma.cuh"

namespace q2k {

__device__ int g_umma_error = 0;

namespace {

constexpr int kUmThreads = 192;

struct UmArgs {
    int m, N, K;
    int64_t ldy;
    float* y;
    int ntok;          // token tile (MMA N): multiple of 16, <= 256
    int nst;           // ring stages
    int kt_per_split;  // 64-wide K steps per CTA
    int nkt;           // 64-wide K steps in total
    int atomic;        // splits add into y
    int tmem_cols;     // power of two >= ntok, >= 32
    uint32_t stage_bytes, b_bytes;
};

__global__ void __launch_bounds__(kUmThreads, 1)
    umma_gemm_kernel(const UmArgs a, const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    pdl_launch_dependents();  // the next kernel may set itself up meanwhile
    // the 128-byte swizzle repeats every 1024 bytes: stages start on 1024
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kBM;     // first W row of the tile
    const int t0 = blockIdx.y * a.ntok;  // first token of the tile
    const int kt0 = blockIdx.z * a.kt_per_split;
    const int nk = min(a.nkt, kt0 + a.kt_per_split) - kt0;

    uint8_t* ring = smem;
    uint64_t* full_b = reinterpret_cast<uint64_t*>(smem + (size_t)a.nst * a.stage_bytes);
    uint64_t* empty_b = full_b + a.nst;
    uint64_t* acc_b = empty_b + a.nst;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(acc_b + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_b + 2);
    volatile int* n_issued = reinterpret_cast<volatile int*>(acc_b + 3);

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.nst; ++s) {
            mbar_init(smem_u32(&full_b[s]), 1);
            mbar_init(smem_u32(&empty_b[s]), 1);
        }
        mbar_init(smem_u32(acc_b), 1);
        *abort_flag = 0;
        *n_issued = 0;
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
        atomicOr(&g_umma_error, Q2K_ERR_BIT_WAIT_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp == 0) {
        if (lane == 0) {  // producer
            const uint64_t wpol = l2_policy_evict_first(), xpol = l2_policy_evict_last();
            for (int i = 0; i < nk; ++i) {
                const int s = i % a.nst, u = i / a.nst;
                if (u > 0 && !mbar_wait_bounded(smem_u32(&empty_b[s]), (uint32_t)(u - 1) & 1u, abort_flag)) {
                    give_up();
                    break;
                }
                const uint32_t sa = smem_u32(ring + (size_t)s * a.stage_bytes);
                mbar_arrive_expect_tx(smem_u32(&full_b[s]), a.stage_bytes);
                tma_load_2d(sa, &tw, (kt0 + i) * kBK, n0, smem_u32(&full_b[s]), wpol);
                tma_load_2d(sa + kATileBytes, &tx, (kt0 + i) * kBK, t0, smem_u32(&full_b[s]), xpol);
                *n_issued = i + 1;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            const uint32_t idesc = instr_desc(a.ntok);
            bool ok = true;
            for (int i = 0; i < nk; ++i) {
                const int s = i % a.nst, u = i / a.nst;
                if (!mbar_wait_bounded(smem_u32(&full_b[s]), (uint32_t)u & 1u, abort_flag)) {
                    give_up();
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t sa = smem_u32(ring + (size_t)s * a.stage_bytes);
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)  // K = 16 per MMA: 32 bytes along the swizzled row
                    umma_f16(tmem, smem_desc_sw128(sa + 32 * k), smem_desc_sw128(sa + kATileBytes + 32 * k), idesc,
                             i > 0 || k > 0);
                umma_commit(smem_u32(&empty_b[s]));  // the stage is free once these MMAs are done
            }
            if (ok)
                umma_commit(smem_u32(acc_b));  // the accumulator is complete
        }
        __syncwarp();
    } else {
        // epilogue: this warp reads TMEM lanes 32q..32q+31 (W rows n0 + 32q + lane)
        const int q = warp & 3;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(acc_b), 0u, abort_flag));
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (!ok) {
            if (lane == 0)
                give_up();
        } else {
            const int row = n0 + 32 * q + lane;
            for (int c = 0; c < a.ntok; c += 16) {
                float v[16];
                tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c, v);
                if (row < a.N) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int tok = t0 + c + j;
                        if (tok < a.m) {
                            float* yp = a.y + (int64_t)tok * a.ldy + row;
                            if (a.atomic)
                                atomicAdd(yp, v[j]);
                            else
                                *yp = v[j];
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
        const int issued = *n_issued;
        for (int i = max(0, issued - a.nst); i < issued; ++i)
            mbar_wait_bounded(smem_u32(&full_b[i % a.nst]), (uint32_t)(i / a.nst) & 1u, nullptr);
    }
    __syncthreads();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)a.tmem_cols)
                     : "memory");
}

PFN_cuTensorMapEncodeTiled_v12000 um_encoder()
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

// bf16 matrix [rows, K] with row stride ld (elements), box 64 x box_rows,
// 128-byte swizzle.
bool encode_bf16(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int64_t ld, int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = um_encoder();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool umma_supported(int64_t m, int64_t K, int64_t N)
{
    return m >= 16 && K >= 1 && N >= 1 && um_encoder() != nullptr;
}

cudaError_t launch_dense_gemm_tc(const uint16_t* x, int64_t m, int64_t K, int64_t ldx, const uint16_t* W, int64_t N,
                                 float* y, int64_t ldy, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    UmArgs a{};
    a.m = (int)m;
    a.N = (int)N;
    a.K = (int)K;
    a.ldy = ldy;
    a.y = y;
    a.ntok = (int)std::min<int64_t>(256, (m + 15) / 16 * 16);
    a.tmem_cols = 32;
    while (a.tmem_cols < a.ntok)
        a.tmem_cols *= 2;
    a.b_bytes = (uint32_t)a.ntok * kBK * 2;
    a.stage_bytes = (uint32_t)kATileBytes + a.b_bytes;
    a.nkt = (int)((K + kBK - 1) / kBK);
    const int gx = (int)((N + kBM - 1) / kBM);
    const int gy = (int)((m + a.ntok - 1) / a.ntok);
    int splits = 1;
    while (gx * gy * splits * 2 <= di.sm_count && a.nkt / (splits * 2) >= 8)
        splits *= 2;
    a.kt_per_split = (a.nkt + splits - 1) / splits;
    splits = (a.nkt + a.kt_per_split - 1) / a.kt_per_split;
    a.atomic = splits > 1 ? 1 : 0;
    const size_t smem_cap = std::min<size_t>((size_t)di.smem_optin, 224 * 1024);
    const size_t fixed = 1024 + 64 + 16 * 8;
    // more tiles than SMs: two CTAs per SM rather than a second wave
    const size_t cap2 = (gx * gy * splits > di.sm_count) ? std::min<size_t>(smem_cap, 112 * 1024) : smem_cap;
    a.nst = (int)std::min<size_t>(8, (cap2 - fixed) / a.stage_bytes);
    if (a.nst < 2)
        return cudaErrorInvalidConfiguration;
    const size_t smem = fixed + (size_t)a.nst * a.stage_bytes;
    CUtensorMap tw{}, tx{};
    if (!encode_bf16(&tw, W, N, K, K, kBM) || !encode_bf16(&tx, x, m, K, ldx, a.ntok))
        return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> smem_devs{0};
    if ((e = allow_max_smem(umma_gemm_kernel, smem_devs)) != cudaSuccess)
        return e;
    if (a.atomic) {
        e = cudaMemset2DAsync(y, (size_t)ldy * sizeof(float), 0, (size_t)N * sizeof(float), (size_t)m, s);
        if (e != cudaSuccess)
            return e;
    }
    return launch_pdl(umma_gemm_kernel, dim3(gx, gy, splits), dim3(kUmThreads), smem, s, a, tw, tx);
}

cudaError_t umma_error_word(int32_t* out, bool clear)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_umma_error, sizeof(int));
    if (e != cudaSuccess)
        return e;
    *out = v;
    if (clear) {
        int z = 0;
        e = cudaMemcpyToSymbol(g_umma_error, &z, sizeof(int));
    }
    return e;
}

}  // namespace q2k
