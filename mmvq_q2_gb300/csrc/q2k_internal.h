// Host-side interface between the C-ABI layer (q2k_api.cu) and the kernel
// translation units.  Shapes arrive here already validated.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace q2k {

enum Act : int { ACT_BF16 = 0, ACT_Q8 = 1 };

// Let `kernel` take up to the device's opt-in shared memory per block, once
// per device (devs: a bit per device id below 64 that has it).  The limit
// is only ever raised to that maximum, so concurrent callers with different
// needs cannot lower it under one another; a repeated first call is
// harmless.
template <typename Kernel>
inline cudaError_t allow_max_smem(Kernel kernel, std::atomic<unsigned long long>& devs)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit && (devs.load(std::memory_order_acquire) & bit))
        return cudaSuccess;
    int optin = 0;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin)) != cudaSuccess)
        return e;
    devs.fetch_or(bit, std::memory_order_acq_rel);
    return cudaSuccess;
}

// Per-device facts read once (multiprocessor count, shared memory limit).
struct DeviceInfo {
    int sm_count;
    int smem_optin;  // max dynamic shared memory per block (bytes)
    int cc_major, cc_minor;
};
cudaError_t device_info(DeviceInfo* out);

// One GEMV/MMVQ problem.  Segments are weight matrices sharing K.
//  - explicit segments (n_seg 1 or 2): W[e], N[e], y[e] + t*ldy[e]
//  - table segments (W_table != null, experts): n_seg matrices of N[0] rows,
//    y_exp [n_seg, N], optional route-weighted y_sum [N]; m == 1.
struct MvProblem {
    int act;  // Act
    int m;
    int64_t K;
    int n_seg;
    const void* const* W_table;
    const void* W[2];
    int64_t N[2];
    float* y[2];
    int64_t ldy[2];
    float* y_exp;
    const float* route_w;
    float* y_sum;
    const void* x;           // bf16 elements or q8_1 bytes
    int64_t x_tok_stride;    // bytes between tokens
    int64_t x_seg_stride;    // bytes between segments' inputs (0 = shared)
    int seg_major;           // table, per-segment inputs, no y_sum: each CTA
                             // works on one segment (its input staged once)
    // q8_1 activations prepared inside the GEMV (m = 1, q8_1, bulk-copyable
    // sources): 1 = x is a bf16 row, quantised per CTA; 2 = segment e's input
    // is SwiGLU(gu[e], gu[gu_E + e]) of fp32 rows of length K, quantised per
    // CTA.  x_out, when set, receives the q8_1 rows (row e at e * x_seg_stride).
    int x_prep;
    // segments as row blocks of one matrix W[0] (table mode without a
    // pointer table): segment e starts at W[0] + e * w_seg_stride bytes
    int64_t w_seg_stride;
    int64_t ldy_exp;  // token stride of y_exp, in floats (several tokens)
    const float* gu;
    int64_t gu_E;
    void* x_out;
};

cudaError_t launch_mv(const MvProblem& p, cudaStream_t s);
// True when every K chunk of the problem has a launch plan that fits the
// device (shared memory for the ring and the partial sums); no CUDA call
// besides the cached device query.
bool mv_plan_ok(const MvProblem& p);
// One token (bf16 or q8_1) over rows of 16..128 blocks, or two tokens, or
// four q8_1 tokens over rows of 8..128 blocks (K % 1024 == 0, 16-byte
// aligned weights and activations), one or two explicit segments: row teams
// fed by ~43 KB stages (q2k_m1.cu).
bool m1_supported(const MvProblem& p);
cudaError_t launch_m1(const MvProblem& p, cudaStream_t s);
// Several tokens (bf16 m = 3..8, q8_1 m = 5..8; explicit segments) on the
// tensor cores (q2k_mt.cu).
bool mt_supported(const MvProblem& p);
cudaError_t launch_mt(const MvProblem& p, cudaStream_t s);

cudaError_t launch_dequant_rows(const void* table, int64_t n_table_rows, int64_t K, const int32_t* ids,
                                int64_t n_rows, uint16_t* out, int32_t* err_flag, cudaStream_t s);
cudaError_t launch_q8_1_quantize(const uint16_t* x, int64_t m, int64_t K, int64_t ldx, void* out,
                                 cudaStream_t s);
cudaError_t launch_swiglu_q8_1(const float* gate_up, int64_t E, int64_t N, void* h_q8, uint16_t* h_bf16,
                               cudaStream_t s);
cudaError_t launch_engram_hash(const int64_t* token_map, int64_t vocab, int64_t* cache, const uint32_t* input_ids,
                               int64_t seqlen, int64_t start_pos, int ng, int nl, int nh, const int64_t* mults,
                               const int64_t* primes, const int64_t* offsets, int64_t pad_id, int64_t* out,
                               int32_t* layer_ids, int layer_index, int32_t* err_flag, cudaStream_t s);
// The engram gate over [tokens, hc] (q2k.h, q2k_engram_gate).
cudaError_t launch_engram_gate(float* streams, const float* kv, int64_t ld_kv, const float* qk, int64_t tokens,
                               int hc, int dim, float eps, float* gates, cudaStream_t s);
// y_sum[n] = sum_e route_w[e] * y_exp[e][n], fp32 fmaf in e order from 0.
cudaError_t launch_expert_sum(const float* y_exp, const float* route_w, int64_t E, int64_t N, float* y_sum,
                              cudaStream_t s);
cudaError_t launch_dense_gemm(const uint16_t* x, int64_t m, int64_t K, int64_t ldx, const uint16_t* W,
                              int64_t N, float* y, int64_t ldy, cudaStream_t s);
// The tcgen05 (tensor memory) GEMM for m >= 16 when the tensor-map encoder is there.
bool umma_supported(int64_t m, int64_t K, int64_t N);
cudaError_t launch_dense_gemm_tc(const uint16_t* x, int64_t m, int64_t K, int64_t ldx, const uint16_t* W,
                                 int64_t N, float* y, int64_t ldy, cudaStream_t s);

// Q2_K matmul for many tokens on tcgen05 (q2k_mmq.cu): y = x W^T with the
// weights expanded from Q2_K to bf16 on-chip.  K % 1024 == 0, W and x
// 16-byte aligned, ldx % 8 == 0.
bool mmq_supported(int64_t m, int64_t N, int64_t K);
cudaError_t launch_mmq_bf16(const void* W, int64_t N, int64_t K, const uint16_t* x, int64_t m, int64_t ldx, float* y,
                            int64_t ldy, cudaStream_t s);
// q8_1 rows -> bf16 rows of the values they encode (rounded once to bf16).
cudaError_t launch_q8_1_to_bf16(const void* xq, int64_t m, int64_t K, uint16_t* out, cudaStream_t s);
size_t mmq_q8_1_workspace(int64_t m, int64_t K);

// Q3_K MMVQ with q8_1 activations (m = 1..8): one matrix, or n_seg matrices
// from W_table (N rows each, y row block e at y + e * y_seg_stride).
struct Q3Problem {
    const void* W;
    const void* const* W_table;
    int n_seg;
    int64_t N, K;
    int m;
    const void* x;
    int64_t x_tok_stride;  // bytes between tokens
    int64_t x_seg_stride;  // bytes between segments' inputs (0 = shared)
    float* y;
    int64_t ldy;           // floats between tokens
    int64_t y_seg_stride;  // floats between segments
};
cudaError_t launch_q3k_mv(const Q3Problem& p, cudaStream_t s);
// The same for m >= kQ3MtMinTokens tokens on one matrix, on the tensor
// cores (q3k_mt.cu); launch_q3k_mv routes those problems here.
constexpr int kQ3MtMinTokens = 3;
bool q3mt_supported(const Q3Problem& p);
cudaError_t launch_q3k_mt(const Q3Problem& p, cudaStream_t s);

// Read (and optionally clear) this translation unit's device error word.
cudaError_t mv_error_word(int32_t* out, bool clear);
cudaError_t m1_error_word(int32_t* out, bool clear);
cudaError_t mmq_error_word(int32_t* out, bool clear);
cudaError_t gemm_error_word(int32_t* out, bool clear);
cudaError_t mt_error_word(int32_t* out, bool clear);
cudaError_t umma_error_word(int32_t* out, bool clear);
cudaError_t q3_error_word(int32_t* out, bool clear);
cudaError_t q3mt_error_word(int32_t* out, bool clear);

}  // namespace q2k
