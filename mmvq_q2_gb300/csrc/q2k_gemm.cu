// Dense bf16 GEMM y = x W^T, fp32 accumulate and output, for the
// multi-token rows (engram_v41/apply.rs, `ops::dense_gemm` when tokens > 1).
// Sixteen tokens or more go to the tcgen05 kernel (q2k_umma.cu); this
// mma.sync kernel takes fewer, below that kernel's smallest MMA width.
//
// Weights are streamed once per token tile: a CTA owns 64 weight rows and a
// tile of up to 64 tokens, stages W and x tiles through a 4-deep cp.async
// ring with an XOR swizzle (conflict-free ldmatrix), and multiplies on the
// tensor cores with m16n8k16 bf16 MMAs (weight rows on the MMA's M side,
// tokens on its N side).  Short N is split over K across CTAs; the partial
// sums then meet in y through fp32 atomics.
#include "q2k_common.cuh"
#include "q2k_internal.h"

#include <algorithm>

namespace q2k {

__device__ int g_gemm_error = 0;

namespace {

constexpr int kBN = 64, kBK = 64, kStages = 4;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
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

// byte offset of 16-byte chunk ch of row r in a [rows][128 B] swizzled tile
__device__ __forceinline__ uint32_t swz(int r, int ch) { return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4)); }

template <int BT>
__global__ void __launch_bounds__(128) dense_gemm_kernel(const uint16_t* __restrict__ x, int m, int K, int64_t ldx,
                                                         const uint16_t* __restrict__ W, int N, float* __restrict__ y,
                                                         int64_t ldy, int k_per_split, int atomic)
{
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int W_BYTES = kBN * kBK * 2;
    constexpr int X_BYTES = BT * kBK * 2;
    constexpr int STAGE = W_BYTES + X_BYTES;
    constexpr int NT = BT / 8;  // n8 tiles per warp

    pdl_launch_dependents();
    pdl_wait();
    const int n0 = blockIdx.x * kBN;
    const int t0 = blockIdx.y * BT;
    const int kbeg = blockIdx.z * k_per_split;
    const int kend = min(K, kbeg + k_per_split);
    const int nk = kend > kbeg ? (kend - kbeg + kBK - 1) / kBK : 0;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    auto load = [&](int s, int kt) {
        const int kk = kbeg + kt * kBK;
        uint8_t* sw = smem + s * STAGE;
        uint8_t* sx = sw + W_BYTES;
#pragma unroll
        for (int c = tid; c < kBN * 8; c += 128) {
            const int r = c >> 3, ch = c & 7;
            const int gk = kk + ch * 8, gn = n0 + r;
            const bool ok = gn < N && gk < kend;
            cp_async16(smem_u32(sw + swz(r, ch)), ok ? (const void*)(W + (int64_t)gn * K + gk) : (const void*)W,
                       ok ? 16 : 0);
        }
#pragma unroll
        for (int c = tid; c < BT * 8; c += 128) {
            const int r = c >> 3, ch = c & 7;
            const int gk = kk + ch * 8, gt = t0 + r;
            const bool ok = gt < m && gk < kend;
            cp_async16(smem_u32(sx + swz(r, ch)), ok ? (const void*)(x + (int64_t)gt * ldx + gk) : (const void*)x,
                       ok ? 16 : 0);
        }
    };

    float acc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i)
        acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < nk)
            load(s, s);
        cp_async_commit();
    }
    for (int kt = 0; kt < nk; ++kt) {
        cp_async_wait<kStages - 2>();
        __syncthreads();
        const int nxt = kt + kStages - 1;
        if (nxt < nk)
            load(nxt % kStages, nxt);
        cp_async_commit();

        const uint8_t* sw = smem + (kt % kStages) * STAGE;
        const uint8_t* sx = sw + W_BYTES;
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks) {
            uint32_t a0, a1, a2, a3;
            {
                const int q = lane >> 3;
                const int r = warp * 16 + (q & 1) * 8 + (lane & 7);
                const int ch = 2 * ks + (q >> 1);
                ldsm_x4(smem_u32(sw + swz(r, ch)), a0, a1, a2, a3);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                uint32_t b0, b1;
                const int q = (lane >> 3) & 1;
                const int r = nt * 8 + (lane & 7);
                ldsm_x2(smem_u32(sx + swz(r, 2 * ks + q)), b0, b1);
                mma_bf16(acc[nt], a0, a1, a2, a3, b0, b1);
            }
        }
    }
    cp_async_wait<0>();

    // epilogue: c0,c1 -> weight row g, tokens 2*tig, 2*tig+1; c2,c3 -> row g+8
    const int g = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = n0 + warp * 16 + g + (i >= 2 ? 8 : 0);
            const int tok = t0 + nt * 8 + 2 * tig + (i & 1);
            if (row < N && tok < m) {
                float* yp = y + (int64_t)tok * ldy + row;
                if (atomic)
                    atomicAdd(yp, acc[nt][i]);
                else
                    *yp = acc[nt][i];
            }
        }
}

template <int BT>
cudaError_t launch_bt(const uint16_t* x, int m, int K, int64_t ldx, const uint16_t* W, int N, float* y, int64_t ldy,
                      int sm_count, cudaStream_t s)
{
    constexpr int SMEM = kStages * (kBN * kBK * 2 + BT * kBK * 2);
    static std::atomic<unsigned long long> smem_devs{0};
    cudaError_t e = allow_max_smem(dense_gemm_kernel<BT>, smem_devs);
    if (e != cudaSuccess)
        return e;
    const int gx = (N + kBN - 1) / kBN;
    const int gy = (m + BT - 1) / BT;
    const int nkt = (K + kBK - 1) / kBK;
    int splits = 1;
    const int target = 2 * sm_count;
    while (gx * gy * splits < target && nkt / (splits * 2) >= 4)
        splits *= 2;
    const int kps = ((nkt + splits - 1) / splits) * kBK;
    splits = (K + kps - 1) / kps;
    if (splits > 1) {
        e = cudaMemset2DAsync(y, (size_t)ldy * sizeof(float), 0, (size_t)N * sizeof(float), (size_t)m, s);
        if (e != cudaSuccess)
            return e;
    }
    dim3 grid(gx, gy, splits);
    return launch_pdl(dense_gemm_kernel<BT>, grid, dim3(128), (size_t)SMEM, s, x, m, K, ldx, W, N, y, ldy, kps,
                      splits > 1 ? 1 : 0);
}

}  // namespace

cudaError_t launch_dense_gemm(const uint16_t* x, int64_t m, int64_t K, int64_t ldx, const uint16_t* W, int64_t N,
                              float* y, int64_t ldy, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    if (umma_supported(m, K, N))
        return launch_dense_gemm_tc(x, m, K, ldx, W, N, y, ldy, s);  // tcgen05 / TMEM
    if (m <= 16)
        return launch_bt<16>(x, (int)m, (int)K, ldx, W, (int)N, y, ldy, di.sm_count, s);
    if (m <= 32)
        return launch_bt<32>(x, (int)m, (int)K, ldx, W, (int)N, y, ldy, di.sm_count, s);
    return launch_bt<64>(x, (int)m, (int)K, ldx, W, (int)N, y, ldy, di.sm_count, s);
}

cudaError_t gemm_error_word(int32_t* out, bool clear)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(int));
    if (e != cudaSuccess)
        return e;
    *out = v;
    if (clear) {
        int z = 0;
        e = cudaMemcpyToSymbol(g_gemm_error, &z, sizeof(int));
    }
    return e;
}

}  // namespace q2k
