// C ABI entry points (include/q2k.h): argument validation before any CUDA
// call, then dispatch to the kernel translation units.  Validation mirrors
// the pages' `ensure!` checks that run before any launch
// (engram_v41/apply.rs `apply`, engram_v41.rs `rows_from_q2k`,
// moe_v41/init.rs `MoeV41::new`).
#include "../../include/q2k.h"
#include "q2k_common.cuh"
#include "q2k_internal.h"

#include <mutex>

namespace q2k {

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
bool g_info_ok[kMaxDevices];
std::mutex g_info_mu;
thread_local int t_last_cuda_error = 0;

int fail_cuda(cudaError_t e)
{
    t_last_cuda_error = (int)e;
    return Q2K_ERR_CUDA;
}
}  // namespace

cudaError_t device_info(DeviceInfo* out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lk(g_info_mu);
        if (g_info_ok[dev]) {
            *out = g_info[dev];
            return cudaSuccess;
        }
    }
    DeviceInfo d{};
    if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lk(g_info_mu);
    g_info[dev] = d;
    g_info_ok[dev] = true;
    *out = d;
    return cudaSuccess;
}

}  // namespace q2k

using namespace q2k;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Device check: compute capability 10.3 (the library carries sm_103a code only).
int check_device()
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return fail_cuda(e);
    if (di.cc_major != 10 || di.cc_minor != 3)
        return Q2K_ERR_UNSUPPORTED;
    return Q2K_OK;
}

int finish(cudaError_t e) { return e == cudaSuccess ? Q2K_OK : fail_cuda(e); }

// Largest K the library accepts (weights rows up to 1 MiB of blocks).
constexpr int64_t kMaxK = 1 << 20;

}  // namespace

extern "C" {

size_t q2k_row_bytes(int64_t K)
{
    if (K <= 0 || K % kBlockWeights)
        return 0;
    return (size_t)(K / kBlockWeights) * kBlockBytes;
}

size_t q3k_row_bytes(int64_t K)
{
    if (K <= 0 || K % kBlockWeights)
        return 0;
    return (size_t)(K / kBlockWeights) * 110;
}

size_t q8_1_row_bytes(int64_t K)
{
    if (K <= 0 || K % kQ8Values)
        return 0;
    return (size_t)(K / kQ8Values) * kQ8Bytes;
}

const char* q2k_status_string(int status)
{
    switch (status) {
    case Q2K_OK: return "ok";
    case Q2K_ERR_NULL_ARG: return "null argument";
    case Q2K_ERR_BAD_SHAPE: return "bad shape";
    case Q2K_ERR_MISALIGNED: return "misaligned pointer";
    case Q2K_ERR_CUDA: return "cuda runtime error";
    case Q2K_ERR_UNSUPPORTED: return "unsupported device (needs compute capability 10.3)";
    case Q2K_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
    }
}

int q2k_last_cuda_error(void) { return t_last_cuda_error; }

int q2k_device_error(int32_t* host_out, int clear)
{
    if (!host_out)
        return Q2K_ERR_NULL_ARG;
    int32_t a = 0, b = 0, c = 0, d = 0, q = 0, o = 0, mq = 0, q3t = 0;
    cudaError_t e = mv_error_word(&a, clear != 0);
    if (e == cudaSuccess)
        e = m1_error_word(&o, clear != 0);
    if (e == cudaSuccess)
        e = mmq_error_word(&mq, clear != 0);
    if (e == cudaSuccess)
        e = gemm_error_word(&b, clear != 0);
    if (e == cudaSuccess)
        e = mt_error_word(&c, clear != 0);
    if (e == cudaSuccess)
        e = umma_error_word(&d, clear != 0);
    if (e == cudaSuccess)
        e = q3_error_word(&q, clear != 0);
    if (e == cudaSuccess)
        e = q3mt_error_word(&q3t, clear != 0);
    if (e != cudaSuccess)
        return fail_cuda(e);
    *host_out = a | b | c | d | q | o | mq | q3t;
    return Q2K_OK;
}

int q2k_dequant_rows(const void* table, int64_t n_table_rows, int64_t K, const int32_t* ids, int64_t n_rows,
                     uint16_t* out_bf16, int32_t* err_flag, q2k_stream_t stream)
{
    if (!table || !out_bf16)
        return Q2K_ERR_NULL_ARG;
    if (K <= 0 || K % kBlockWeights || K > kMaxK || n_rows < 0 || n_table_rows <= 0)
        return Q2K_ERR_BAD_SHAPE;
    if (!ids && n_rows > n_table_rows)
        return Q2K_ERR_BAD_SHAPE;
    if (!aligned(table, 4) || !aligned(out_bf16, 2) || (ids && !aligned(ids, 4)) || (err_flag && !aligned(err_flag, 4)))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    if (n_rows == 0)
        return Q2K_OK;
    return finish(launch_dequant_rows(table, n_table_rows, K, ids, n_rows, out_bf16, err_flag,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

int q2k_engram_hash(const int64_t* token_map, int64_t vocab, int64_t* cache, int64_t max_seq,
                    const uint32_t* input_ids, int64_t seqlen, int64_t start_pos, int64_t max_ngram,
                    int64_t n_layers, int64_t n_heads, const int64_t* multipliers, const int64_t* primes,
                    const int64_t* offsets, int64_t pad_id, int64_t* out, int32_t* layer_ids,
                    int64_t layer_index, int32_t* err_flag, q2k_stream_t stream)
{
    if (!token_map || !cache || (seqlen > 0 && !input_ids) || !multipliers || !primes || !offsets ||
        (seqlen > 0 && !out))
        return Q2K_ERR_NULL_ARG;
    if (vocab <= 0 || max_seq <= 0 || seqlen < 0 || start_pos < 0 || start_pos + seqlen > max_seq ||
        max_ngram < 2 || max_ngram > 16 || n_layers < 1 || n_layers > 1024 || n_heads < 1 || n_heads > 1024 ||
        (layer_ids && (layer_index < 0 || layer_index >= n_layers)))
        return Q2K_ERR_BAD_SHAPE;
    if (!aligned(token_map, 8) || !aligned(cache, 8) || !aligned(input_ids, 4) || !aligned(multipliers, 8) ||
        !aligned(primes, 8) || !aligned(offsets, 8) || !aligned(out, 8) || !aligned(layer_ids, 4) ||
        !aligned(err_flag, 4))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    if (seqlen == 0)
        return Q2K_OK;
    return finish(launch_engram_hash(token_map, vocab, cache, input_ids, seqlen, start_pos, (int)max_ngram,
                                     (int)n_layers, (int)n_heads, multipliers, primes, offsets, pad_id, out, layer_ids,
                                     (int)layer_index, err_flag, reinterpret_cast<cudaStream_t>(stream)));
}

int q2k_engram_gate(float* streams, const float* kv, int64_t ld_kv, const float* qk, int64_t tokens, int64_t hc,
                    int64_t dim, float eps, float* gates, q2k_stream_t stream)
{
    if (tokens > 0 && (!streams || !kv || !qk))
        return Q2K_ERR_NULL_ARG;
    if (tokens < 0 || tokens > (1 << 30) || hc < 1 || hc > 4 || dim < 1 || dim > kMaxK || ld_kv < (hc + 1) * dim ||
        !(eps >= 0.f) || eps > 3.0e38f)
        return Q2K_ERR_BAD_SHAPE;
    if (!aligned(streams, 4) || !aligned(kv, 4) || !aligned(qk, 4) || (gates && !aligned(gates, 4)))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    if (tokens == 0)
        return Q2K_OK;
    return finish(launch_engram_gate(streams, kv, ld_kv, qk, tokens, (int)hc, (int)dim, eps, gates,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int q8_1_quantize_rows(const uint16_t* x_bf16, int64_t m, int64_t K, int64_t ldx, void* out_q8_1,
                       q2k_stream_t stream)
{
    if (!x_bf16 || !out_q8_1)
        return Q2K_ERR_NULL_ARG;
    if (m < 0 || K <= 0 || K % kQ8Values || ldx < K || K > kMaxK)
        return Q2K_ERR_BAD_SHAPE;
    if (!aligned(x_bf16, 2) || !aligned(out_q8_1, 4))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    if (m == 0)
        return Q2K_OK;
    return finish(launch_q8_1_quantize(x_bf16, m, K, ldx, out_q8_1, reinterpret_cast<cudaStream_t>(stream)));
}

int q2k_gemv_bf16(const void* W, int64_t N, int64_t K, const uint16_t* x, int64_t m, int64_t ldx, float* y,
                  int64_t ldy, q2k_stream_t stream)
{
    if (!W || !x || !y)
        return Q2K_ERR_NULL_ARG;
    if (N <= 0 || K <= 0 || K % kBlockWeights || K > kMaxK || m < 1 || m > 8 || ldx < K || ldy < N)
        return Q2K_ERR_BAD_SHAPE;
    if (!aligned(W, 4) || !aligned(x, 2) || !aligned(y, 4))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    MvProblem p{};
    p.act = ACT_BF16;
    p.m = (int)m;
    p.K = K;
    p.n_seg = 1;
    p.W[0] = W;
    p.N[0] = N;
    p.y[0] = y;
    p.ldy[0] = ldy;
    p.x = x;
    p.x_tok_stride = ldx * 2;
    return finish(launch_mv(p, reinterpret_cast<cudaStream_t>(stream)));
}

int q2k_mmvq_q8_1(const void* W, int64_t N, int64_t K, const void* xq, int64_t m, float* y, int64_t ldy,
                  q2k_stream_t stream)
{
    if (!W || !xq || !y)
        return Q2K_ERR_NULL_ARG;
    if (N <= 0 || K <= 0 || K % kBlockWeights || K > kMaxK || m < 1 || m > 8 || ldy < N)
        return Q2K_ERR_BAD_SHAPE;
    if (!aligned(W, 4) || !aligned(xq, 4) || !aligned(y, 4))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    MvProblem p{};
    p.act = ACT_Q8;
    p.m = (int)m;
    p.K = K;
    p.n_seg = 1;
    p.W[0] = W;
    p.N[0] = N;
    p.y[0] = y;
    p.ldy[0] = ldy;
    p.x = xq;
    p.x_tok_stride = (int64_t)q8_1_row_bytes(K);
    return finish(launch_mv(p, reinterpret_cast<cudaStream_t>(stream)));
}

int q2k_mmvq_pair(const void* Wa, int64_t Na, float* ya, const void* Wb, int64_t Nb, float* yb, int64_t K,
                  const void* xq, int64_t m, q2k_stream_t stream)
{
    if (!Wa || !Wb || !ya || !yb || !xq)
        return Q2K_ERR_NULL_ARG;
    if (Na <= 0 || Nb <= 0 || K <= 0 || K % kBlockWeights || K > kMaxK || m < 1 || m > 8)
        return Q2K_ERR_BAD_SHAPE;
    if (!aligned(Wa, 4) || !aligned(Wb, 4) || !aligned(ya, 4) || !aligned(yb, 4) || !aligned(xq, 4))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    MvProblem p{};
    p.act = ACT_Q8;
    p.m = (int)m;
    p.K = K;
    p.n_seg = 2;
    p.W[0] = Wa;
    p.W[1] = Wb;
    p.N[0] = Na;
    p.N[1] = Nb;
    p.y[0] = ya;
    p.y[1] = yb;
    p.ldy[0] = Na;
    p.ldy[1] = Nb;
    p.x = xq;
    p.x_tok_stride = (int64_t)q8_1_row_bytes(K);
    return finish(launch_mv(p, reinterpret_cast<cudaStream_t>(stream)));
}

int q2k_mmvq_pair_bf16(const void* Wa, int64_t Na, float* ya, const void* Wb, int64_t Nb, float* yb, int64_t K,
                       const uint16_t* x_bf16, int64_t m, void* xq_out, q2k_stream_t stream)
{
    if (!Wa || !Wb || !ya || !yb || !x_bf16 || !xq_out)
        return Q2K_ERR_NULL_ARG;
    if (Na <= 0 || Nb <= 0 || K <= 0 || K % kBlockWeights || K > kMaxK || m < 1 || m > 8)
        return Q2K_ERR_BAD_SHAPE;
    if (!aligned(Wa, 4) || !aligned(Wb, 4) || !aligned(ya, 4) || !aligned(yb, 4) || !aligned(x_bf16, 2) ||
        !aligned(xq_out, 4))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    MvProblem p{};
    p.act = ACT_Q8;
    p.m = (int)m;
    p.K = K;
    p.n_seg = 2;
    p.W[0] = Wa;
    p.W[1] = Wb;
    p.N[0] = Na;
    p.N[1] = Nb;
    p.y[0] = ya;
    p.y[1] = yb;
    p.ldy[0] = Na;
    p.ldy[1] = Nb;
    p.x_tok_stride = (int64_t)q8_1_row_bytes(K);
    p.x = xq_out;
    if (m == 1 && aligned(x_bf16, 16) && !m1_supported(p)) {
        // one launch: every CTA encodes the row, the first also stores it.
        // (Where the row-team kernel takes the pair, a separate encoding
        // launch ahead of it measured faster: 4.5 vs 6.0 us at cfg2.)
        p.x = x_bf16;
        p.x_prep = 1;
        p.x_out = xq_out;
        return finish(launch_mv(p, s));
    }
    cudaError_t e = launch_q8_1_quantize(x_bf16, m, K, K, xq_out, s);
    if (e != cudaSuccess)
        return fail_cuda(e);
    p.x = xq_out;
    return finish(launch_mv(p, s));
}

int q2k_mmvq_grouped(const void* W, int64_t groups, int64_t rows_per_group, int64_t K_group, const void* xq,
                     int64_t m, float* y, q2k_stream_t stream)
{
    if (!W || !xq || !y)
        return Q2K_ERR_NULL_ARG;
    if (groups <= 0 || groups > 4096 || rows_per_group <= 0 || K_group <= 0 || K_group % kBlockWeights ||
        K_group > kMaxK || m < 1 || m > 8 || groups * rows_per_group > (1 << 30))
        return Q2K_ERR_BAD_SHAPE;
    if (!aligned(W, 4) || !aligned(xq, 4) || !aligned(y, 4))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    MvProblem p{};
    p.act = ACT_Q8;
    p.m = (int)m;
    p.K = K_group;
    p.n_seg = (int)groups;
    p.W[0] = W;  // group g: rows g*rows_per_group.. of W
    p.w_seg_stride = rows_per_group * (int64_t)q2k_row_bytes(K_group);
    p.N[0] = rows_per_group;
    p.y_exp = y;  // y[t, g*rows_per_group + r]
    p.ldy_exp = groups * rows_per_group;
    p.seg_major = 1;  // each group gets CTAs of its own, its slice staged once
    p.x = xq;
    p.x_tok_stride = (int64_t)q8_1_row_bytes(groups * K_group);
    p.x_seg_stride = (int64_t)q8_1_row_bytes(K_group);  // group g's blocks of each token's row
    return finish(launch_mv(p, reinterpret_cast<cudaStream_t>(stream)));
}

int q2k_mmvq_experts(const void* const* W_table, int64_t n_mat, int64_t N, int64_t K, const void* xq,
                     int x_per_matrix, float* y, const float* route_w, float* y_sum, q2k_stream_t stream)
{
    if (!W_table || !xq || (!y && !y_sum) || (y_sum && !route_w))
        return Q2K_ERR_NULL_ARG;
    if (n_mat <= 0 || n_mat > 4096 || N <= 0 || K <= 0 || K % kBlockWeights || K > kMaxK ||
        (x_per_matrix != 0 && x_per_matrix != 1))
        return Q2K_ERR_BAD_SHAPE;
    if (!aligned(W_table, 8) || !aligned(xq, 4) || (y && !aligned(y, 4)) || (route_w && !aligned(route_w, 4)) ||
        (y_sum && !aligned(y_sum, 4)))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    MvProblem p{};
    p.act = ACT_Q8;
    p.m = 1;
    p.K = K;
    p.n_seg = (int)n_mat;
    p.W_table = W_table;
    p.N[0] = N;
    p.y_exp = y;
    p.route_w = route_w;
    p.y_sum = y_sum;
    p.x = xq;
    p.x_tok_stride = (int64_t)q8_1_row_bytes(K);
    p.x_seg_stride = x_per_matrix ? (int64_t)q8_1_row_bytes(K) : 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (y) {
        // each matrix gets CTAs of its own (full reduction units, its input
        // row staged once); the route-weighted sum, if asked for, is a
        // second pass over y
        p.seg_major = 1;
        p.y_sum = nullptr;
        cudaError_t e = launch_mv(p, s);
        if (e != cudaSuccess || !y_sum)
            return e != cudaSuccess ? fail_cuda(e) : finish(e);
        return finish(launch_expert_sum(y, route_w, n_mat, N, y_sum, s));
    }
    // the fused sum keeps every matrix's partial sums of a CTA's rows in
    // shared memory: refuse, before any launch, a problem whose partials do
    // not fit (per-matrix outputs in y are then the workspace it needs)
    if (!mv_plan_ok(p))
        return Q2K_ERR_WORKSPACE;
    return finish(launch_mv(p, s));
}

int q3k_mmvq_q8_1(const void* W, int64_t N, int64_t K, const void* xq, int64_t m, float* y, int64_t ldy,
                  q2k_stream_t stream)
{
    if (!W || !xq || !y)
        return Q2K_ERR_NULL_ARG;
    if (N <= 0 || N > (1 << 30) || K <= 0 || K % kBlockWeights || K > kMaxK || m < 1 || m > 8 || ldy < N)
        return Q2K_ERR_BAD_SHAPE;
    if (!aligned(W, 4) || !aligned(xq, 4) || !aligned(y, 4))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    Q3Problem p{};
    p.W = W;
    p.n_seg = 1;
    p.N = N;
    p.K = K;
    p.m = (int)m;
    p.x = xq;
    p.x_tok_stride = (int64_t)q8_1_row_bytes(K);
    p.y = y;
    p.ldy = ldy;
    return finish(launch_q3k_mv(p, reinterpret_cast<cudaStream_t>(stream)));
}

int q3k_mmvq_experts(const void* const* W_table, int64_t n_mat, int64_t N, int64_t K, const void* xq,
                     int x_per_matrix, float* y, const float* route_w, float* y_sum, q2k_stream_t stream)
{
    if (!W_table || !xq || !y || (y_sum && !route_w))
        return Q2K_ERR_NULL_ARG;
    if (n_mat <= 0 || n_mat > 4096 || N <= 0 || N > (1 << 30) || K <= 0 || K % kBlockWeights || K > kMaxK ||
        (x_per_matrix != 0 && x_per_matrix != 1))
        return Q2K_ERR_BAD_SHAPE;
    if (!aligned(W_table, 8) || !aligned(xq, 4) || !aligned(y, 4) || (route_w && !aligned(route_w, 4)) ||
        (y_sum && !aligned(y_sum, 4)))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    Q3Problem p{};
    p.W_table = W_table;
    p.n_seg = (int)n_mat;
    p.N = N;
    p.K = K;
    p.m = 1;
    p.x = xq;
    p.x_tok_stride = (int64_t)q8_1_row_bytes(K);
    p.x_seg_stride = x_per_matrix ? (int64_t)q8_1_row_bytes(K) : 0;
    p.y = y;
    p.ldy = N;
    p.y_seg_stride = N;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_q3k_mv(p, s);
    if (e != cudaSuccess || !y_sum)
        return e != cudaSuccess ? fail_cuda(e) : finish(e);
    return finish(launch_expert_sum(y, route_w, n_mat, N, y_sum, s));
}

int swiglu_q8_1_rows(const float* gate_up, int64_t E, int64_t N, void* h_q8, uint16_t* h_bf16, q2k_stream_t stream)
{
    if (!gate_up || !h_q8)
        return Q2K_ERR_NULL_ARG;
    if (E <= 0 || N <= 0 || N % kQ8Values || N > kMaxK)
        return Q2K_ERR_BAD_SHAPE;
    if (!aligned(gate_up, 4) || !aligned(h_q8, 4) || (h_bf16 && !aligned(h_bf16, 2)))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    return finish(launch_swiglu_q8_1(gate_up, E, N, h_q8, h_bf16, reinterpret_cast<cudaStream_t>(stream)));
}

static size_t round256(size_t v) { return (v + 255) / 256 * 256; }

size_t q2k_moe_m1_workspace_bytes(int64_t E, int64_t dim, int64_t inter)
{
    if (E <= 0 || dim <= 0 || inter <= 0 || dim % kBlockWeights || inter % kBlockWeights)
        return 0;
    return round256(q8_1_row_bytes(dim)) + round256((size_t)2 * E * inter * sizeof(float)) +
           round256((size_t)E * q8_1_row_bytes(inter)) + round256((size_t)E * dim * sizeof(float));
}

int q2k_moe_m1(const void* const* ptrs, int64_t E, int64_t dim, int64_t inter, const uint16_t* x_bf16,
               const float* route_w, float* y, void* workspace, size_t workspace_bytes, q2k_stream_t stream)
{
    if (!ptrs || !x_bf16 || !route_w || !y)
        return Q2K_ERR_NULL_ARG;
    if (E <= 0 || E > 1024 || dim <= 0 || inter <= 0 || dim % kBlockWeights || inter % kBlockWeights ||
        dim > kMaxK || inter > kMaxK)
        return Q2K_ERR_BAD_SHAPE;
    const size_t need = q2k_moe_m1_workspace_bytes(E, dim, inter);
    if (!workspace || workspace_bytes < need)
        return Q2K_ERR_WORKSPACE;
    if (!aligned(ptrs, 8) || !aligned(x_bf16, 2) || !aligned(route_w, 4) || !aligned(y, 4) || !aligned(workspace, 256))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* xq = ws;
    float* gate_up = reinterpret_cast<float*>(ws + round256(q8_1_row_bytes(dim)));
    void* h_q8 = ws + round256(q8_1_row_bytes(dim)) + round256((size_t)2 * E * inter * sizeof(float));
    float* down_out = reinterpret_cast<float*>(static_cast<uint8_t*>(h_q8) + round256((size_t)E * q8_1_row_bytes(inter)));
    // A 16-byte aligned x is quantised inside the gate/up GEMV (each CTA
    // encodes it; the first also stores it in the workspace), and SwiGLU +
    // q8_1 of h run inside the down GEMV the same way: three launches, the
    // same bits as the five separate steps.
    const bool fuse_x = aligned(x_bf16, 16);
    cudaError_t e = cudaSuccess;
    if (!fuse_x && (e = launch_q8_1_quantize(x_bf16, 1, dim, dim, xq, s)) != cudaSuccess)
        return fail_cuda(e);
    MvProblem p{};
    p.act = ACT_Q8;
    p.m = 1;
    p.K = dim;
    p.n_seg = (int)(2 * E);
    p.W_table = ptrs;
    p.N[0] = inter;
    p.y_exp = gate_up;
    p.seg_major = 1;  // each gate/up matrix gets CTAs of its own
    p.x = fuse_x ? static_cast<const void*>(x_bf16) : xq;
    p.x_tok_stride = (int64_t)q8_1_row_bytes(dim);
    p.x_seg_stride = 0;
    if (fuse_x) {
        p.x_prep = 1;
        p.x_out = xq;
    }
    if ((e = launch_mv(p, s)) != cudaSuccess)
        return fail_cuda(e);
    MvProblem d{};
    d.act = ACT_Q8;
    d.m = 1;
    d.K = inter;
    d.n_seg = (int)E;
    d.W_table = ptrs + 2 * E;
    d.N[0] = dim;
    d.y_exp = down_out;  // one expert per CTA, then the route-weighted sum
    d.seg_major = 1;
    d.x = h_q8;
    d.x_tok_stride = (int64_t)q8_1_row_bytes(inter);
    d.x_seg_stride = (int64_t)q8_1_row_bytes(inter);
    d.x_prep = 2;  // h = SwiGLU(gate, up) -> q8_1 per CTA, also stored in h_q8
    d.gu = gate_up;
    d.gu_E = E;
    d.x_out = h_q8;
    if ((e = launch_mv(d, s)) != cudaSuccess)
        return fail_cuda(e);
    return finish(launch_expert_sum(down_out, route_w, E, dim, y, s));
}

size_t q2k_mmq_q8_1_workspace_bytes(int64_t m, int64_t K)
{
    if (m < 1 || m > (1 << 24) || K <= 0 || K % 1024 || K > kMaxK)
        return 0;
    return mmq_q8_1_workspace(m, K);
}

int q2k_mmq_bf16(const void* W, int64_t N, int64_t K, const uint16_t* x, int64_t m, int64_t ldx, float* y,
                 int64_t ldy, q2k_stream_t stream)
{
    if (!W || !x || !y)
        return Q2K_ERR_NULL_ARG;
    if (N < 1 || N > (1 << 30) || K <= 0 || K % 1024 || K > kMaxK || m < 1 || m > (1 << 24) || ldx < K || ldx % 8 ||
        ldy < N)
        return Q2K_ERR_BAD_SHAPE;
    if (!aligned(W, 16) || !aligned(x, 16) || !aligned(y, 4))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    if (!mmq_supported(m, N, K))
        return Q2K_ERR_UNSUPPORTED;  // no tensor-map encoder in this driver
    return finish(launch_mmq_bf16(W, N, K, x, m, ldx, y, ldy, reinterpret_cast<cudaStream_t>(stream)));
}

int q2k_mmq_q8_1(const void* W, int64_t N, int64_t K, const void* xq, int64_t m, float* y, int64_t ldy,
                 void* workspace, size_t workspace_bytes, q2k_stream_t stream)
{
    if (!W || !xq || !y)
        return Q2K_ERR_NULL_ARG;
    if (N < 1 || N > (1 << 30) || K <= 0 || K % 1024 || K > kMaxK || m < 1 || m > (1 << 24) || ldy < N)
        return Q2K_ERR_BAD_SHAPE;
    if (!workspace || workspace_bytes < q2k_mmq_q8_1_workspace_bytes(m, K))
        return Q2K_ERR_WORKSPACE;
    if (!aligned(W, 16) || !aligned(xq, 4) || !aligned(y, 4) || !aligned(workspace, 16))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    if (!mmq_supported(m, N, K))
        return Q2K_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint16_t* xb = static_cast<uint16_t*>(workspace);
    cudaError_t e = launch_q8_1_to_bf16(xq, m, K, xb, s);
    if (e != cudaSuccess)
        return fail_cuda(e);
    return finish(launch_mmq_bf16(W, N, K, xb, m, K, y, ldy, s));
}

int dense_gemm_bf16(const uint16_t* x, int64_t m, int64_t K, int64_t ldx, const uint16_t* W, int64_t N, float* y,
                    int64_t ldy, q2k_stream_t stream)
{
    if (!x || !W || !y)
        return Q2K_ERR_NULL_ARG;
    if (m < 1 || K <= 0 || K % 8 || N <= 0 || ldx < K || ldx % 8 || ldy < N || K > (1 << 30) / 2 ||
        N > (1 << 30) || m > (1 << 24))
        return Q2K_ERR_BAD_SHAPE;
    if (!aligned(x, 16) || !aligned(W, 16) || !aligned(y, 4))
        return Q2K_ERR_MISALIGNED;
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    return finish(launch_dense_gemm(x, m, K, ldx, W, N, y, ldy, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---- routed experts without any allocation -------------------------------------
//
// Some callers cannot hand the library a workspace: a host program that links
// only this library and has no device allocator of its own, or a decode loop
// whose memory is planned once up front and must not allocate (or make its
// allocator grow) between steps.  For them this entry point runs the same
// launches as q2k_moe_m1 on a fixed scratch buffer that lives in the
// library's own device image.  The scratch is a file-scope __device__ array,
// so it is reserved when the module loads: nothing is allocated or freed here.
//
// Every byte of the scratch is written before it is read within one call
// (the q8_1 x, the fp32 gate/up outputs and the q8_1 h are produced in full
// by their launches), so nothing has to be cleared.  Calls that overlap on
// one device (two streams, or two threads) share this buffer and race; keep
// them on one stream.

namespace {
__device__ __align__(256) unsigned char g_moe_scratch[Q2K_MOE_M1_STATIC_SCRATCH_BYTES];

void* g_moe_scratch_ptr[kMaxDevices];
std::mutex g_moe_scratch_mu;

// The scratch's device address on the current device, looked up once per
// device (the first call on a device does this; it may load the module).
// The cached address belongs to the device's context at that time: after a
// cudaDeviceReset the module loads again, possibly elsewhere, and the cached
// address is stale, so a process that resets a device must not call this
// entry point on it afterwards.
cudaError_t moe_scratch(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_moe_scratch_mu);
    if (!g_moe_scratch_ptr[dev]) {
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_moe_scratch)) != cudaSuccess)
            return e;
        g_moe_scratch_ptr[dev] = p;
    }
    *out = g_moe_scratch_ptr[dev];
    return cudaSuccess;
}
}  // namespace

extern "C" int q2k_moe_m1_static_scratch(const void* const* ptrs, int64_t E, int64_t dim, int64_t inter,
                                         const uint16_t* x_bf16, const float* route_w, float* y,
                                         q2k_stream_t stream)
{
    if (!ptrs || !x_bf16 || !route_w || !y)
        return Q2K_ERR_NULL_ARG;
    // the shapes q2k_moe_m1 refuses are refused here the same way; only a
    // valid problem that needs more than the fixed scratch is a WORKSPACE error
    if (E <= 0 || E > 1024 || dim <= 0 || inter <= 0 || dim % kBlockWeights || inter % kBlockWeights ||
        dim > kMaxK || inter > kMaxK)
        return Q2K_ERR_BAD_SHAPE;
    const size_t need = q2k_moe_m1_workspace_bytes(E, dim, inter);
    if (need > (size_t)Q2K_MOE_M1_STATIC_SCRATCH_BYTES)
        return Q2K_ERR_WORKSPACE;  // the problem does not fit the fixed scratch
    int st = check_device();
    if (st != Q2K_OK)
        return st;
    void* ws = nullptr;
    cudaError_t e = moe_scratch(&ws);
    if (e != cudaSuccess)
        return fail_cuda(e);
    return q2k_moe_m1(ptrs, E, dim, inter, x_bf16, route_w, y, ws, (size_t)Q2K_MOE_M1_STATIC_SCRATCH_BYTES, stream);
}

