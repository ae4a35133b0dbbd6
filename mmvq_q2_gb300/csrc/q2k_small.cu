// Small memory-bound kernels around the projections:
//  - gather + dequantise Q2_K rows to bf16 (engram_v41.rs, `rows_from_q2k`,
//    `dequant_q2_k_to_bf16`), with the row gather moved onto the device;
//  - bf16 -> q8_1 rows (attn_v41/decode.rs, `kquant_q8_1_rows`);
//  - SwiGLU fused with q8_1 requantisation (moe_v41/init.rs,
//    `kquant_swiglu_q8_1_rows_bf16`);
//  - the engram n-gram hash (engram_v41.rs, `EngramHasher::hash`) and the
//    engram gate (engram_v41.rs module doc, step 4).
#include "q2k_common.cuh"
#include "q2k_internal.h"
#include "q2k_q8.cuh"

#include <algorithm>

namespace q2k {

// ---- dequant ----------------------------------------------------------------
// One thread per 8 consecutive weights p = 8l..8l+7 of a block (l = 0..31):
// they share half n = l/16, pair j = (l%16)/4, sub-block l/2, and take qs
// bytes 32n + 8(l%4) .. +7 at bit shift 2j.
template <bool VEC16>
__global__ void __launch_bounds__(256) q2k_dequant_kernel(const uint8_t* __restrict__ table, int64_t n_table_rows,
                                                          int nb, const int32_t* __restrict__ ids, int64_t n_rows,
                                                          uint16_t* __restrict__ out, int32_t* err_flag)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t total = n_rows * nb * 32;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += (int64_t)gridDim.x * blockDim.x) {
        const int l = (int)(u & 31);
        const int64_t bi = u >> 5;
        const int64_t r = bi / nb;
        const int b = (int)(bi - r * nb);
        const int64_t src = ids ? (int64_t)ids[r] : r;
        uint16_t* o = out + (r * nb + b) * kBlockWeights + 8 * l;
        uint32_t packed[4];
        if (src < 0 || src >= n_table_rows) {
            packed[0] = packed[1] = packed[2] = packed[3] = 0u;
            if (err_flag && l == 0)
                atomicExch(err_flag, 1);
        } else {
            const uint8_t* blk = table + (src * nb + b) * kBlockBytes;
            const int n = l >> 4, j = (l & 15) >> 2, sb = l >> 1;
            const uint32_t dm = ldg32_nc(blk + 80);
            const uint32_t scw = ldg32_nc(blk + (sb & ~3));
            const uint32_t scb = (scw >> (8 * (sb & 3))) & 0xFFu;
            const float dl = half_lo_f(dm) * (float)(scb & 15u);  // exact
            const float ml = half_hi_f(dm) * (float)(scb >> 4);   // exact
            const uint8_t* qp = blk + 16 + 32 * n + 8 * (l & 3);
            const uint32_t q0 = ldg32_nc(qp), q1 = ldg32_nc(qp + 4);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t w = i < 2 ? q0 : q1;
                const int bA = (2 * i) & 3, bB = (2 * i + 1) & 3;
                const float qa = (float)((w >> (8 * bA + 2 * j)) & 3u);
                const float qb = (float)((w >> (8 * bB + 2 * j)) & 3u);
                // one rounding to fp32 (dl*q is exact), then one to bf16
                const __nv_bfloat16 ha = __float2bfloat16_rn(fmaf(dl, qa, -ml));
                const __nv_bfloat16 hb = __float2bfloat16_rn(fmaf(dl, qb, -ml));
                packed[i] = (uint32_t)__bfloat16_as_ushort(ha) | ((uint32_t)__bfloat16_as_ushort(hb) << 16);
            }
        }
        if constexpr (VEC16) {
            *reinterpret_cast<uint4*>(o) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                o[2 * i] = (uint16_t)(packed[i] & 0xFFFFu);
                o[2 * i + 1] = (uint16_t)(packed[i] >> 16);
            }
        }
    }
}

cudaError_t launch_dequant_rows(const void* table, int64_t n_table_rows, int64_t K, const int32_t* ids,
                                int64_t n_rows, uint16_t* out, int32_t* err_flag, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    const int nb = (int)(K / kBlockWeights);
    const int64_t threads = n_rows * nb * 32;
    const int64_t grid = std::min<int64_t>((threads + 255) / 256, (int64_t)di.sm_count * 8);
    const bool vec = (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
    const uint8_t* tb = static_cast<const uint8_t*>(table);
    if (vec)
        return launch_pdl(q2k_dequant_kernel<true>, dim3((unsigned)grid), dim3(256), 0, s, tb, n_table_rows, nb, ids,
                          n_rows, out, err_flag);
    return launch_pdl(q2k_dequant_kernel<false>, dim3((unsigned)grid), dim3(256), 0, s, tb, n_table_rows, nb, ids,
                      n_rows, out, err_flag);
}

// ---- q8_1 ---------------------------------------------------------------------
__global__ void __launch_bounds__(256) q8_1_quantize_kernel(const uint16_t* __restrict__ x, int64_t m, int nblk,
                                                            int64_t ldx, uint8_t* __restrict__ out)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t total = m * nblk * 8;  // lanes
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    // every lane of a warp must reach the shuffles: iterate a warp-uniform count
    const int64_t base0 = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31);
    for (int64_t wbase = base0; wbase < total; wbase += stride) {
        const int64_t u = wbase + (threadIdx.x & 31);
        const bool live = u < total;
        const int64_t uu = live ? u : wbase;
        const int lane8 = (int)(uu & 7);
        const int64_t bi = uu >> 3;
        const int64_t t = bi / nblk;
        const int b = (int)(bi - t * nblk);
        const uint16_t* xp = x + t * ldx + (int64_t)b * kQ8Values + 4 * lane8;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            v[i] = live ? bf16_bits_f(xp[i]) : 0.f;
        q8_1_encode_group(v, out + (t * nblk + b) * kQ8Bytes, lane8, live);
    }
}

cudaError_t launch_q8_1_quantize(const uint16_t* x, int64_t m, int64_t K, int64_t ldx, void* out, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    const int nblk = (int)(K / kQ8Values);
    const int64_t lanes = m * nblk * 8;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((lanes + 255) / 256, (int64_t)di.sm_count * 8));
    return launch_pdl(q8_1_quantize_kernel, dim3((unsigned)grid), dim3(256), 0, s, x, m, nblk, ldx,
                      static_cast<uint8_t*>(out));
}

// ---- SwiGLU + q8_1 --------------------------------------------------------------
__global__ void __launch_bounds__(256) swiglu_q8_1_kernel(const float* __restrict__ gate_up, int64_t E, int64_t N,
                                                          uint8_t* __restrict__ h_q8, uint16_t* __restrict__ h_bf16)
{
    pdl_launch_dependents();
    pdl_wait();
    const int nblk = (int)(N / kQ8Values);
    const int64_t total = E * nblk * 8;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t base0 = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31);
    for (int64_t wbase = base0; wbase < total; wbase += stride) {
        const int64_t u = wbase + (threadIdx.x & 31);
        const bool live = u < total;
        const int64_t uu = live ? u : wbase;
        const int lane8 = (int)(uu & 7);
        const int64_t bi = uu >> 3;
        const int64_t e = bi / nblk;
        const int b = (int)(bi - e * nblk);
        const int64_t k0 = (int64_t)b * kQ8Values + 4 * lane8;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float hv = 0.f;
            if (live) {
                // g, u rounded to bf16 first (bf16 expert buffers), then
                // h = silu(g) * u in fp32, rounded to bf16.
                const __nv_bfloat16 hb = swiglu_bf16(gate_up[e * N + k0 + i], gate_up[(E + e) * N + k0 + i]);
                hv = __bfloat162float(hb);
                if (h_bf16)
                    h_bf16[e * N + k0 + i] = __bfloat16_as_ushort(hb);
            }
            v[i] = hv;
        }
        q8_1_encode_group(v, h_q8 + (e * nblk + b) * kQ8Bytes, lane8, live);
    }
}

cudaError_t launch_swiglu_q8_1(const float* gate_up, int64_t E, int64_t N, void* h_q8, uint16_t* h_bf16,
                               cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    const int64_t lanes = E * (N / kQ8Values) * 8;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((lanes + 255) / 256, (int64_t)di.sm_count * 8));
    return launch_pdl(swiglu_q8_1_kernel, dim3((unsigned)grid), dim3(256), 0, s, gate_up, E, N,
                      static_cast<uint8_t*>(h_q8), h_bf16);
}

// ---- route-weighted sum of per-expert outputs ----------------------------------
// y_sum[n] = sum_e route_w[e] * y_exp[e][n] (moe_v41/init.rs,
// `moe_v41_accumulate`), one fp32 fmaf per expert in expert order from 0:
// the same chain as the sum fused into the expert GEMV, so both give the
// same bits.
__global__ void __launch_bounds__(256) expert_sum_kernel(const float* __restrict__ y_exp,
                                                         const float* __restrict__ route_w, int E, int64_t N,
                                                         float* __restrict__ y_sum)
{
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; n < N; n += (int64_t)gridDim.x * blockDim.x) {
        float acc = 0.f;
        for (int e = 0; e < E; ++e)
            acc = fmaf(route_w[e], y_exp[(int64_t)e * N + n], acc);
        y_sum[n] = acc;
    }
}

cudaError_t launch_expert_sum(const float* y_exp, const float* route_w, int64_t E, int64_t N, float* y_sum,
                              cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((N + 255) / 256, (int64_t)di.sm_count * 4));
    return launch_pdl(expert_sum_kernel, dim3((unsigned)grid), dim3(256), 0, s, y_exp, route_w, (int)E, N, y_sum);
}

// ---- engram n-gram hash ---------------------------------------------------------
// engram_v41.rs, `EngramHasher::hash`, on the device: the input tokens are
// mapped through token_map into the sequence cache at start_pos.., then for
// each position and layer the n-gram chain rolling_i = (t_0*m_0) ^ ... ^
// (t_i*m_i) (wrapping i64 products) gives, per n-gram length i and head h,
// rem_euclid(rolling_i, prime) + offset.  A token before the sequence start,
// or at or past an unmapped one (-1), reads as pad_id.
constexpr int kHashMaxNgram = 16;

// Mapped token at sequence position pos: this call's tokens are read through
// token_map directly (so no thread waits for another's cache write), earlier
// ones from the cache.  An id outside token_map reads as unmapped (-1).
__device__ __forceinline__ int64_t hash_token_at(const int64_t* token_map, int64_t vocab, const int64_t* cache,
                                                 const uint32_t* input_ids, int64_t start_pos, int64_t pos)
{
    if (pos < start_pos)
        return cache[pos];
    const uint32_t id = input_ids[pos - start_pos];
    return (int64_t)id < vocab ? token_map[id] : -1;
}

__global__ void __launch_bounds__(256) engram_hash_kernel(
    const int64_t* __restrict__ token_map, int64_t vocab, int64_t* __restrict__ cache,
    const uint32_t* __restrict__ input_ids, int64_t seqlen, int64_t start_pos, int ng, int nl, int nh,
    const int64_t* __restrict__ mults, const int64_t* __restrict__ primes, const int64_t* __restrict__ offsets,
    int64_t pad_id, int64_t* __restrict__ out, int32_t* __restrict__ layer_ids, int layer_index,
    int32_t* __restrict__ err_flag)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // this call's tokens into the cache (read by later calls)
    for (int64_t s = t0; s < seqlen; s += stride) {
        const uint32_t id = input_ids[s];
        if ((int64_t)id >= vocab && err_flag)
            atomicOr(err_flag, 1);  // outside token_map: the position reads as unmapped
        cache[start_pos + s] = (int64_t)id < vocab ? token_map[id] : -1;
    }
    // one thread per output id (position s, layer li, column col = (i-1)*nh + h)
    const int cols = (ng - 1) * nh;
    for (int64_t u = t0; u < seqlen * nl * cols; u += stride) {
        const int64_t s = u / ((int64_t)nl * cols);
        const int rem = (int)(u - s * nl * cols);
        const int li = rem / cols, col = rem - li * cols;
        const int i = col / nh + 1, h = col - (i - 1) * nh;  // n-gram of the token and the i before it
        const int64_t pos = start_pos + s;
        const int64_t* m = mults + (int64_t)li * ng;
        bool blocked = false;
        uint64_t rolling = 0;
#pragma unroll
        for (int shift = 0; shift < kHashMaxNgram; ++shift) {
            if (shift <= i) {
                int64_t t = -1;
                if (pos >= shift)
                    t = hash_token_at(token_map, vocab, cache, input_ids, start_pos, pos - shift);
                blocked = blocked || pos < shift || t == -1;
                rolling ^= (uint64_t)(blocked ? pad_id : t) * (uint64_t)m[shift];
            }
        }
        const int64_t p = primes[((int64_t)li * (ng - 1) + (i - 1)) * nh + h];
        int64_t v = 0;
        if (p > 0) {
            const int64_t r = (int64_t)rolling % p;
            v = (r < 0 ? r + p : r) + offsets[(int64_t)li * cols + col];
        } else if (err_flag) {
            atomicOr(err_flag, 2);  // a modulus that is not positive: id 0
        }
        out[u] = v;
        if (layer_ids && li == layer_index)
            layer_ids[s * cols + col] = (int32_t)v;
    }
}

cudaError_t launch_engram_hash(const int64_t* token_map, int64_t vocab, int64_t* cache, const uint32_t* input_ids,
                               int64_t seqlen, int64_t start_pos, int ng, int nl, int nh, const int64_t* mults,
                               const int64_t* primes, const int64_t* offsets, int64_t pad_id, int64_t* out,
                               int32_t* layer_ids, int layer_index, int32_t* err_flag, cudaStream_t s)
{
    const int64_t work = std::max<int64_t>(seqlen, seqlen * nl * (int64_t)(ng - 1) * nh);
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((work + 255) / 256, 1024));
    return launch_pdl(engram_hash_kernel, dim3((unsigned)grid), dim3(256), 0, s, token_map, vocab, cache, input_ids, seqlen,
                      start_pos, ng, nl, nh, mults, primes, offsets, pad_id, out, layer_ids, layer_index, err_flag);
}

// ---- engram gate ----------------------------------------------------------------
// engram_v41.rs, module doc, step 4, and engram_v41/apply.rs, `apply` (the
// `gate_k` launch over [tokens, hc]): one CTA per (token, stream).  The
// stream h (fp32, dim values), its key k and the shared value v (kv row t:
// keys 0..hc-1, then the value; each kv value rounded to bf16, the page's
// kv buffer being bf16) give
//   s = sum_i qk_i h_i k_i / (rms(h) rms(k) sqrt(dim)),
//   rms(z) = sqrt(mean(z^2) + eps),  g = sigmoid(sign(s) sqrt(|s|)),
// and h += g v in place.  The three sums are reduced in a fixed order, so a
// call repeats bit for bit.
__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

__global__ void __launch_bounds__(256) engram_gate_kernel(float* __restrict__ streams, const float* __restrict__ kv,
                                                          int64_t ld_kv, const float* __restrict__ qk, int hc, int dim,
                                                          float eps, float* __restrict__ gates)
{
    pdl_launch_dependents();
    pdl_wait();
    const int t = (int)blockIdx.x, c = (int)blockIdx.y;
    float* h = streams + ((int64_t)t * hc + c) * dim;
    const float* k = kv + (int64_t)t * ld_kv + (int64_t)c * dim;
    const float* v = kv + (int64_t)t * ld_kv + (int64_t)hc * dim;
    const float* q = qk + (int64_t)c * dim;
    float shh = 0.f, skk = 0.f, shk = 0.f;
    for (int i = threadIdx.x; i < dim; i += blockDim.x) {
        const float hv = h[i];
        const float kk = bf16_round(k[i]);
        shh = fmaf(hv, hv, shh);
        skk = fmaf(kk, kk, skk);
        shk = fmaf(q[i] * hv, kk, shk);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        shh += __shfl_xor_sync(0xffffffffu, shh, o);
        skk += __shfl_xor_sync(0xffffffffu, skk, o);
        shk += __shfl_xor_sync(0xffffffffu, shk, o);
    }
    __shared__ float part[3][8];
    __shared__ float gate;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        part[0][warp] = shh;
        part[1][warp] = skk;
        part[2][warp] = shk;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = 0.f, b = 0.f, d = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
            a += part[0][w];
            b += part[1][w];
            d += part[2][w];
        }
        const float rh = sqrtf(a / (float)dim + eps);
        const float rk = sqrtf(b / (float)dim + eps);
        const float sc = d / (rh * rk * sqrtf((float)dim));
        const float ss = copysignf(sqrtf(fabsf(sc)), sc);
        gate = 1.f / (1.f + expf(-ss));
        if (gates)
            gates[(int64_t)t * hc + c] = gate;
    }
    __syncthreads();
    const float g = gate;
    for (int i = threadIdx.x; i < dim; i += blockDim.x)
        h[i] = fmaf(g, bf16_round(v[i]), h[i]);
}

// The same gate with every operand in registers: for dim <= 4096, a multiple
// of 4, with 16-byte aligned rows.  Each thread loads its float4s of the
// stream, key, qk and value at once (one memory round trip instead of one
// per strided step), reduces, and updates the stream from its registers.
constexpr int kGateVec = 4;  // float4s per thread: 256 x 4 x 4 = 4096 values

__global__ void __launch_bounds__(256) engram_gate_vec_kernel(float* __restrict__ streams,
                                                              const float* __restrict__ kv, int64_t ld_kv,
                                                              const float* __restrict__ qk, int hc, int dim,
                                                              float eps, float* __restrict__ gates)
{
    pdl_launch_dependents();
    pdl_wait();
    const int t = (int)blockIdx.x, c = (int)blockIdx.y;
    float4* h = reinterpret_cast<float4*>(streams + ((int64_t)t * hc + c) * dim);
    const float4* k = reinterpret_cast<const float4*>(kv + (int64_t)t * ld_kv + (int64_t)c * dim);
    const float4* v = reinterpret_cast<const float4*>(kv + (int64_t)t * ld_kv + (int64_t)hc * dim);
    const float4* q = reinterpret_cast<const float4*>(qk + (int64_t)c * dim);
    const int n4 = dim >> 2;
    float4 hv[kGateVec], kk[kGateVec], qv[kGateVec], vv[kGateVec];
#pragma unroll
    for (int j = 0; j < kGateVec; ++j) {
        const int u = (int)threadIdx.x + 256 * j;
        if (u < n4) {
            hv[j] = h[u];
            kk[j] = k[u];
            qv[j] = q[u];
            vv[j] = v[u];
        }
    }
    float shh = 0.f, skk = 0.f, shk = 0.f;
#pragma unroll
    for (int j = 0; j < kGateVec; ++j) {
        if ((int)threadIdx.x + 256 * j < n4) {
            const float hx[4] = {hv[j].x, hv[j].y, hv[j].z, hv[j].w};
            const float kx[4] = {bf16_round(kk[j].x), bf16_round(kk[j].y), bf16_round(kk[j].z), bf16_round(kk[j].w)};
            const float qx[4] = {qv[j].x, qv[j].y, qv[j].z, qv[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                shh = fmaf(hx[e], hx[e], shh);
                skk = fmaf(kx[e], kx[e], skk);
                shk = fmaf(qx[e] * hx[e], kx[e], shk);
            }
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        shh += __shfl_xor_sync(0xffffffffu, shh, o);
        skk += __shfl_xor_sync(0xffffffffu, skk, o);
        shk += __shfl_xor_sync(0xffffffffu, shk, o);
    }
    __shared__ float part[3][8];
    __shared__ float gate;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        part[0][warp] = shh;
        part[1][warp] = skk;
        part[2][warp] = shk;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = 0.f, b = 0.f, d = 0.f;
        for (int w = 0; w < 8; ++w) {
            a += part[0][w];
            b += part[1][w];
            d += part[2][w];
        }
        const float rh = sqrtf(a / (float)dim + eps);
        const float rk = sqrtf(b / (float)dim + eps);
        const float sc = d / (rh * rk * sqrtf((float)dim));
        const float ss = copysignf(sqrtf(fabsf(sc)), sc);
        gate = 1.f / (1.f + expf(-ss));
        if (gates)
            gates[(int64_t)t * hc + c] = gate;
    }
    __syncthreads();
    const float g = gate;
#pragma unroll
    for (int j = 0; j < kGateVec; ++j) {
        const int u = (int)threadIdx.x + 256 * j;
        if (u < n4) {
            float4 o;
            o.x = fmaf(g, bf16_round(vv[j].x), hv[j].x);
            o.y = fmaf(g, bf16_round(vv[j].y), hv[j].y);
            o.z = fmaf(g, bf16_round(vv[j].z), hv[j].z);
            o.w = fmaf(g, bf16_round(vv[j].w), hv[j].w);
            h[u] = o;
        }
    }
}

cudaError_t launch_engram_gate(float* streams, const float* kv, int64_t ld_kv, const float* qk, int64_t tokens,
                               int hc, int dim, float eps, float* gates, cudaStream_t s)
{
    const bool vec = dim % 4 == 0 && dim <= 256 * 4 * kGateVec && ld_kv % 4 == 0 &&
                     (reinterpret_cast<uintptr_t>(streams) & 15u) == 0 && (reinterpret_cast<uintptr_t>(kv) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(qk) & 15u) == 0;
    if (vec)
        return launch_pdl(engram_gate_vec_kernel, dim3((unsigned)tokens, (unsigned)hc), dim3(256), 0, s, streams, kv,
                          ld_kv, qk, hc, dim, eps, gates);
    return launch_pdl(engram_gate_kernel, dim3((unsigned)tokens, (unsigned)hc), dim3(256), 0, s, streams, kv, ld_kv, qk,
                      hc, dim, eps, gates);
}

}  // namespace q2k
