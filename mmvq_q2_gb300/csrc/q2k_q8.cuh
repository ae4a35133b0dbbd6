// q8_1 block encoding and the SwiGLU element, shared by the standalone
// kernels (q8_1_quantize_rows, swiglu_q8_1_rows) and the GEMV kernel's fused
// activation staging, so that both give the same bits.
#pragma once

#include "q2k_common.cuh"

namespace q2k {

// Eight lanes per 32-value block, four values per lane.  amax, d32 = amax/127
// and q = round(x/d32) use IEEE fp32 division (explicit __fdiv_rn) and
// round-half-away-from-zero, so q and d are bit-exact to the encoding.
// Every lane of the warp calls this (dead lanes with live == false and
// zeros) so that the shuffles stay converged; only live lanes store.
__device__ __forceinline__ void q8_1_encode_group(const float (&v)[4], uint8_t* blk, int lane8, bool live)
{
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float d32 = __fdiv_rn(amax, 127.0f);
    int q[4];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        q[i] = amax == 0.0f ? 0 : (int)roundf(__fdiv_rn(v[i], d32));
        sum += q[i];
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1)
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const __half dh = __float2half_rn(d32);
    const __half sh = __float2half_rn(__fmul_rn(__half2float(dh), (float)sum));
    const uint32_t qw = (uint32_t)(q[0] & 0xFF) | ((uint32_t)(q[1] & 0xFF) << 8) | ((uint32_t)(q[2] & 0xFF) << 16) |
                        ((uint32_t)(q[3] & 0xFF) << 24);
    if (!live)
        return;
    *reinterpret_cast<uint32_t*>(blk + 4 + 4 * lane8) = qw;
    if (lane8 == 0)
        *reinterpret_cast<uint32_t*>(blk) =
            (uint32_t)__half_as_ushort(dh) | ((uint32_t)__half_as_ushort(sh) << 16);
}

// SwiGLU of one element (moe_v41/init.rs, `kquant_swiglu_q8_1_rows_bf16`):
// g and u rounded to bf16 first (the page's expert buffers are bf16), then
// h = silu(g) * u in fp32 (silu(z) = z / (1 + e^-z), expf), rounded to bf16.
__device__ __forceinline__ __nv_bfloat16 swiglu_bf16(float g_in, float u_in)
{
    const float g = __bfloat162float(__float2bfloat16_rn(g_in));
    const float uv = __bfloat162float(__float2bfloat16_rn(u_in));
    const float silu = __fdiv_rn(g, 1.0f + expf(-g));
    return __float2bfloat16_rn(__fmul_rn(silu, uv));
}

}  // namespace q2k
