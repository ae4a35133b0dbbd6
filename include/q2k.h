/*
 * q2k.h -- C ABI of the Q2_K decode-projection library (libq2k.so).
 *
 * Decode-time projections read straight off GGUF Q2_K weight blocks, for
 * m <= 8 tokens, with bf16 or q8_1 activations, on one NVIDIA GB300
 * (sm_103a).  Sources are the metrale docs pages (engram_v41.rs,
 * engram_v41/apply.rs, attn_v41/decode.rs, moe_v41/init.rs); each entry
 * point cites the item it follows.
 *
 * Conventions (engram_v41/apply.rs `apply` and attn_v41/decode.rs
 * `q_kv_projections`: raw device pointers, integer shapes, a stream; every
 * check before any launch):
 *  - Every pointer argument is a DEVICE pointer unless its comment says
 *    otherwise.  The caller owns every buffer; the library never allocates,
 *    frees or synchronises, and keeps no state besides per-device launch
 *    tuning read from the device once.  All work is enqueued on `stream`
 *    (NULL = the legacy default stream); calls return before it runs.
 *  - Arguments are validated before anything is enqueued.  A non-zero
 *    status means nothing was launched (Q2K_ERR_CUDA: a launch was refused
 *    by the runtime; its error is reported by q2k_last_cuda_error()).
 *  - Weights: row-major [N, K] as GGUF ships them, K/256 super-blocks per
 *    row (engram_v41.rs, `wkv_q2k`: `[out, in / 256]` blocks).  y = x W^T.
 *  - Activations: bf16 (raw uint16 bit patterns) or q8_1 rows.
 *  - Outputs: fp32 unless stated.
 *
 * Q2_K super-block, 84 bytes, 256 weights (engram_v41.rs,
 * `ENGRAM_ROW_BYTES`), read as the GGUF Q2_K layout:
 *     bytes  0..15  scales[16]: sub-block j = p/16; low nibble = scale,
 *                   high nibble = min
 *     bytes 16..79  qs[64]: weight p's 2-bit code q_p is bits
 *                   2*((p%128)/32)..+1 of qs[32*(p/128) + p%32]
 *     bytes 80..81  d    (fp16, little endian)
 *     bytes 82..83  dmin (fp16, little endian)
 *     w_p = d * (scales[j] & 15) * q_p - dmin * (scales[j] >> 4)
 *
 * q8_1 block, 36 bytes, 32 values (the library's own layout; attn_v41 and
 * moe_v41 name the format only):
 *     bytes 0..1 d (fp16), bytes 2..3 s (fp16), bytes 4..35 q[32] (int8)
 *     d32 = amax/127 (fp32 divide), q = round_half_away(x/d32),
 *     d = fp16(d32), s = fp16(f32(d) * sum(q)).  Rows are K/32 blocks,
 *     contiguous, rows back to back.
 *
 * Alignment: weights and q8_1 rows must be 4-byte aligned, bf16 arrays
 * 2-byte aligned, fp32 arrays 4-byte aligned (Q2K_ERR_MISALIGNED).
 * Weight rows that start on 16-byte boundaries (K % 1024 == 0 and a 16-byte
 * aligned base) are streamed with bulk asynchronous copies; other rows take
 * a slower copy path with identical results.
 */
#ifndef Q2K_H
#define Q2K_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st* q2k_stream_t;

enum q2k_status {
    Q2K_OK = 0,
    Q2K_ERR_NULL_ARG = 1,    /* a required pointer is NULL */
    Q2K_ERR_BAD_SHAPE = 2,   /* K % 256 != 0, m outside 1..8, N <= 0, ... */
    Q2K_ERR_MISALIGNED = 3,  /* a pointer below its required alignment */
    Q2K_ERR_CUDA = 4,        /* the CUDA runtime refused a query or launch */
    Q2K_ERR_UNSUPPORTED = 5, /* current device is not compute capability 10.3 */
    Q2K_ERR_WORKSPACE = 6    /* workspace NULL or smaller than required */
};

/* Bytes of one Q2_K row of K weights: K/256*84, or 0 when K % 256 != 0. */
size_t q2k_row_bytes(int64_t K);

/* Bytes of one Q3_K row of K weights: K/256*110, or 0 when K % 256 != 0. */
size_t q3k_row_bytes(int64_t K);

/* Bytes of one q8_1 row of K values: K/32*36, or 0 when K % 32 != 0
 * (moe_v41/init.rs, `kquant_q8_1_rows_bytes`). */
size_t q8_1_row_bytes(int64_t K);

/* Gather + dequantise Q2_K rows to bf16 (engram_v41.rs, `rows_from_q2k`
 * and `dequant_q2_k_to_bf16`; the gather of rows by id is done on the
 * device instead of on the host).
 *   table         Q2_K rows, [n_table_rows, K/256] blocks
 *   ids           int32 [n_rows] row ids into table, or NULL for rows
 *                 0..n_rows-1 (then n_rows <= n_table_rows)
 *   out_bf16      [n_rows, K] bf16, row r = decode(table[ids[r]]), each
 *                 weight computed in fp32 and rounded once to bf16 (RN)
 *   err_flag      int32, nullable: set to 1 when an id is outside
 *                 [0, n_table_rows); that row is written as zeros
 * Engram rows are K = 256 (one block per row) in [token][col] order. */
int q2k_dequant_rows(const void* table, int64_t n_table_rows, int64_t K, const int32_t* ids,
                     int64_t n_rows, uint16_t* out_bf16, int32_t* err_flag, q2k_stream_t stream);

/* Engram n-gram hash on the device (engram_v41.rs, `EngramHasher::hash`):
 * the ids of the engram table rows for a run of tokens, so that the rows can
 * be gathered (q2k_dequant_rows) and projected without a host round trip.
 *   token_map    int64 [vocab]: token id -> engram token (-1: unmapped)
 *   cache        int64 [max_seq]: the sequence's mapped tokens; positions
 *                start_pos .. start_pos+seqlen-1 are written, earlier ones
 *                are read (the caller keeps it across calls, as the page's
 *                hasher keeps its cache)
 *   input_ids    uint32 [seqlen]
 *   multipliers  int64 [n_layers, max_ngram]
 *   primes       int64 [n_layers, max_ngram-1, n_heads] (positive)
 *   offsets      int64 [n_layers, (max_ngram-1)*n_heads]
 *   out          int64 [seqlen, n_layers, cols], cols = (max_ngram-1)*n_heads:
 *                rolling_i = (t_0*m_0) ^ ... ^ (t_i*m_i) over the current
 *                token and the i before it (wrapping i64 products; a token
 *                before the start, or at or past an unmapped one, reads as
 *                pad_id); out[s, l, (i-1)*n_heads + h] =
 *                rem_euclid(rolling_i, primes[l, i-1, h]) + offsets[l, col]
 *   layer_ids    int32 [seqlen, cols], nullable: layer layer_index's ids in
 *                [token][col] order (`layer_row_ids`), ready for
 *                q2k_dequant_rows
 *   err_flag     int32, nullable: bit 0 set when an input id is outside
 *                token_map (that position then reads as unmapped; the page
 *                stops with an error instead), bit 1 when a prime is not
 *                positive (its ids are 0)
 * 2 <= max_ngram <= 16; start_pos + seqlen <= max_seq.  One launch. */
int q2k_engram_hash(const int64_t* token_map, int64_t vocab, int64_t* cache, int64_t max_seq,
                    const uint32_t* input_ids, int64_t seqlen, int64_t start_pos, int64_t max_ngram,
                    int64_t n_layers, int64_t n_heads, const int64_t* multipliers, const int64_t* primes,
                    const int64_t* offsets, int64_t pad_id, int64_t* out, int32_t* layer_ids,
                    int64_t layer_index, int32_t* err_flag, q2k_stream_t stream);

/* Engram gate (engram_v41.rs, module doc, step 4; engram_v41/apply.rs,
 * `apply`, the `gate_k` launch over [tokens, hc] with streams, kv, qk, dim,
 * hc, eps): a normalised dot of each stream against its key, a signed-sqrt
 * sigmoid, and h += gate * value, in place on the fp32 streams.
 *   streams  fp32 [tokens, hc, dim], contiguous; updated in place
 *   kv       fp32 [tokens, ld_kv]: row t holds hc keys of dim values, then
 *            the shared value (dim values): the projection's output
 *            (engram_v41.rs, `out_features` = dim * (hc + 1)); every kv
 *            value is rounded to bf16 before use, as the page's kv buffer
 *            is bf16
 *   ld_kv    floats between kv rows, >= (hc + 1) * dim
 *   qk       fp32 [hc, dim]: q_weight * k_weight, elementwise
 *            (engram_v41.rs, `EngramV41::upload_qk`)
 *   gates    fp32 [tokens, hc], nullable: receives each gate
 * For stream c of token t, with h the stream, k its key and v the value:
 *   s = sum_i qk[c,i] h_i k_i / (rms(h) rms(k) sqrt(dim)),
 *   rms(z) = sqrt(mean(z^2) + eps),  g = 1 / (1 + exp(-sign(s) sqrt(|s|))),
 *   h_i += g v_i.
 * The pages name these steps without their arithmetic; the 1/sqrt(dim)
 * scale and the key/value order are this library's reading.  fp32, sums in
 * a fixed order (a call repeats bit for bit).  1 <= hc <= 4 (the page's
 * limit), 1 <= dim <= 2^20, eps >= 0.  One launch; tokens == 0 is a no-op. */
int q2k_engram_gate(float* streams, const float* kv, int64_t ld_kv, const float* qk, int64_t tokens, int64_t hc,
                    int64_t dim, float eps, float* gates, q2k_stream_t stream);

/* Quantise bf16 rows to q8_1 (attn_v41/decode.rs, `kquant_q8_1_rows`;
 * moe_v41/init.rs, `kquant_q8_1_rows_bf16`).
 *   x_bf16   [m, K] with row stride ldx elements (ldx >= K); K % 32 == 0
 *   out_q8_1 m * q8_1_row_bytes(K) bytes
 * q and d are bit-exact to the encoding in this header's preamble. */
int q8_1_quantize_rows(const uint16_t* x_bf16, int64_t m, int64_t K, int64_t ldx, void* out_q8_1,
                       q2k_stream_t stream);

/* Q2_K GEMV with bf16 activations, m = 1..8 tokens (engram_v41/apply.rs,
 * the single-token `engram_v41_wkv_q2k_gemv` off `wkv_q2k`).
 *   W  Q2_K [N, K];  x  bf16 [m, K], row stride ldx;  y  fp32 [m, N], row
 *   stride ldy.  y[t, n] = sum_k w[n, k] x[t, k].  One and two tokens:
 *   exact int32 dot products of the 2-bit codes with fixed-point
 *   activations per sub-block, scaled by d, the sub-block scales and the
 *   activation exponents and summed in fp32 (the bf16 values are not
 *   multiplied as floats).
 * The activations enter the integer dot products as 16-bit fixed point
 * with one power-of-two exponent per 16 values (exact unless a group spans
 * more than 2^7 in magnitude; then the smallest lose bits below 2^-15 of
 * the group maximum).  One token over rows of K >= 4096 uses one exponent
 * per 32 values and a 2^14 range (exact within 2^6 of the group maximum,
 * bits below 2^-14 of it lost).  Groups below 2^-100 count as zero.
 * Three to eight tokens run on the tensor cores instead: the bf16 values
 * enter exactly, against the integers 128 + sc*q of each sub-block (fp32
 * accumulation), and the min term's sub-block sums of x enter as a bf16
 * high and low pair. */
int q2k_gemv_bf16(const void* W, int64_t N, int64_t K, const uint16_t* x, int64_t m, int64_t ldx,
                  float* y, int64_t ldy, q2k_stream_t stream);

/* Q2_K x q8_1 MMVQ, m = 1..8 (moe_v41/init.rs, `kquant_mmvq_q2_k_w`).
 *   W Q2_K [N, K];  xq  m q8_1 rows of K values;  y fp32 [m, N], stride ldy.
 * Per sub-block: d*sc*d8*sum(q*q8) - dmin*m*d8*sum(q8), in fp32. */
int q2k_mmvq_q8_1(const void* W, int64_t N, int64_t K, const void* xq, int64_t m, float* y,
                  int64_t ldy, q2k_stream_t stream);

/* Two Q2_K matrices over one q8_1 input in a single launch (attn_v41/
 * decode.rs, `kquant_mmvq_pair_w`: `wq_a` -> `qr_raw`, `wkv` -> `kv_raw`).
 *   Wa [Na, K] -> ya fp32 [m, Na];  Wb [Nb, K] -> yb fp32 [m, Nb]
 * Each output equals q2k_mmvq_q8_1 of its matrix bit for bit. */
int q2k_mmvq_pair(const void* Wa, int64_t Na, float* ya, const void* Wb, int64_t Nb, float* yb,
                  int64_t K, const void* xq, int64_t m, q2k_stream_t stream);

/* The pair over bf16 activations: the q8_1 quantisation of x
 * (q8_1_quantize_rows) and q2k_mmvq_pair as one call (attn_v41/decode.rs,
 * `q_kv_projections`: one q8_1 quantisation feeds one launch for both).
 *   x_bf16  [m, K] bf16 rows back to back
 *   xq_out  m q8_1 rows; receives q8_1_quantize_rows(x) in every case
 *   Wa, Na, ya, Wb, Nb, yb, K, m  as for q2k_mmvq_pair
 * For m = 1, a 16-byte aligned x and rows outside 16..128 blocks (K %
 * 1024 == 0) the encoding runs inside the pair launch (each CTA encodes the
 * row; one launch).  Otherwise it is a launch of its own, then the pair
 * (rows of 16..128 blocks run a kernel for which that is faster).  Either
 * way xq_out, ya and yb equal the two separate calls bit for bit. */
int q2k_mmvq_pair_bf16(const void* Wa, int64_t Na, float* ya, const void* Wb, int64_t Nb, float* yb,
                       int64_t K, const uint16_t* x_bf16, int64_t m, void* xq_out, q2k_stream_t stream);

/* Grouped (block-diagonal) MMVQ, m = 1..8 (attn_v41/decode.rs,
 * `attend_and_project`: og[t, g*o_rank + r] = o_g . wo_a[g*o_rank + r], the
 * Q2_K `wo_a_grouped` path for m <= 8).
 *   W       Q2_K [groups * rows_per_group, K_group]: group g owns rows
 *           g*rows_per_group .. (g+1)*rows_per_group - 1
 *   xq      m q8_1 rows of groups * K_group values; group g's input is
 *           values g*K_group .. (g+1)*K_group - 1 of each row
 *   y       fp32 [m, groups * rows_per_group]:
 *           y[t, g*rows_per_group + r] = sum_k W[g*rows_per_group + r, k] *
 *           x_t[g*K_group + k]
 * One launch; each group's output equals q2k_mmvq_q8_1 of its row block and
 * its input slice bit for bit (m = 1). */
int q2k_mmvq_grouped(const void* W, int64_t groups, int64_t rows_per_group, int64_t K_group,
                     const void* xq, int64_t m, float* y, q2k_stream_t stream);

/* Batched single-token MMVQ over n_mat Q2_K matrices of one shape, with an
 * optional fused route-weighted sum (moe_v41/init.rs,
 * `kquant_mmvq_q2_k_experts_w8`, `moe_v41_accumulate`).
 *   W_table      device array of n_mat device pointers, each Q2_K [N, K]
 *   xq           q8_1 input: one row shared by every matrix
 *                (x_per_matrix == 0) or row e for matrix e (x_per_matrix
 *                == 1, rows back to back)
 *   y            fp32 [n_mat, N], nullable when y_sum is given; row e
 *                equals q2k_mmvq_q8_1(W_table[e], xq row) bit for bit
 *   route_w      fp32 [n_mat], required with y_sum
 *   y_sum        fp32 [N], nullable: y_sum[n] = sum_e route_w[e]*y[e,n],
 *                added in e order (deterministic).  With y given, each
 *                matrix gets CTAs of its own and the sum is a second
 *                launch over y; the bits are the same.
 *                Without y the sum is fused: each CTA keeps the partial
 *                sums of all n_mat matrices for its rows in shared memory;
 *                a problem whose partials do not fit returns
 *                Q2K_ERR_WORKSPACE before any launch (pass y, which then
 *                holds the per-matrix outputs, for many small matrices).
 * Gate and up run as one batch of 2*topk matrices; down as topk matrices
 * with x_per_matrix = 1 (moe_v41/init.rs, the `gate_out` comment). */
int q2k_mmvq_experts(const void* const* W_table, int64_t n_mat, int64_t N, int64_t K,
                     const void* xq, int x_per_matrix, float* y, const float* route_w,
                     float* y_sum, q2k_stream_t stream);

/* Q3_K twins (moe_v41/init.rs, `MoeV41::new`, loads `kquant_mmvq_q3_k_w`
 * and `kquant_mmvq_q3_k_experts_w*` beside the Q2_K kernels; the pages give
 * no Q3_K layout, so the block is GGUF's Q3_K, 110 bytes per 256 weights:
 * hmask[32] | qs[64] | scales[12] | d (fp16 LE).  Weight p of a block is
 * d * s_j * (code_p - 4 * (1 - high_p)), with j = p/16, s_j the signed
 * 6-bit sub-block scale (stored + 32: low nibble in scales[j] for j < 8 or
 * the high nibble of scales[j-8], top two bits at bit 2*(j/4) of
 * scales[8 + j%4]), code_p the 2-bit field at bit 2*((p%128)/32) of
 * qs[32*(p/128) + p%32] and high_p bit p/32 of hmask[p%32]).
 *
 * Single matrix, m = 1..8 tokens:
 *   W    Q3_K [N, K], row-major blocks, 4-byte aligned
 *   xq   m q8_1 rows of K values, back to back, 4-byte aligned
 *   y    fp32, y[t*ldy + n] = sum_k W[n, k] * x_t[k], ldy >= N
 * Errors before any launch: NULL_ARG, BAD_SHAPE (K % 256, K > 2^20, N < 1,
 * m outside 1..8, ldy < N), MISALIGNED.  The sum is deterministic: the same
 * inputs give the same bits on every call. */
int q3k_mmvq_q8_1(const void* W, int64_t N, int64_t K, const void* xq, int64_t m, float* y, int64_t ldy,
                  q2k_stream_t stream);

/* Batched single-token Q3_K MMVQ over n_mat matrices of one shape.
 *   W_table   device array of n_mat device pointers, each Q3_K [N, K]; an
 *             entry that is not 4-byte aligned is skipped (its rows of y
 *             are left as they were) and sets bit 1 of the device error word
 *   xq        q8_1 input: one row shared by every matrix (x_per_matrix ==
 *             0) or row e for matrix e (x_per_matrix == 1)
 *   y         fp32 [n_mat, N], required; row e equals
 *             q3k_mmvq_q8_1(W_table[e], its input row) bit for bit
 *   route_w   fp32 [n_mat], required with y_sum
 *   y_sum     fp32 [N], nullable: sum_e route_w[e]*y[e, n] in e order, a
 *             second launch over y */
int q3k_mmvq_experts(const void* const* W_table, int64_t n_mat, int64_t N, int64_t K, const void* xq,
                     int x_per_matrix, float* y, const float* route_w, float* y_sum, q2k_stream_t stream);

/* SwiGLU fused with q8_1 requantisation (moe_v41/init.rs,
 * `kquant_swiglu_q8_1_rows_bf16`).
 *   gate_up  fp32 [2E, N]: gate rows 0..E-1, up rows E..2E-1 (the layout
 *            q2k_mmvq_experts writes for a 2E gate+up batch)
 *   h_q8     E q8_1 rows of N values;  h_bf16 [E, N] bf16, nullable
 * g and u are first rounded to bf16 (the page's expert buffers are bf16),
 * h = silu(g)*u in fp32 (silu(z) = z/(1+e^-z), expf) rounded to bf16, then
 * q8_1-encoded.  N % 32 == 0. */
int swiglu_q8_1_rows(const float* gate_up, int64_t E, int64_t N, void* h_q8, uint16_t* h_bf16,
                     q2k_stream_t stream);

/* Workspace bytes q2k_moe_m1 needs for E experts (256-byte aligned parts). */
size_t q2k_moe_m1_workspace_bytes(int64_t E, int64_t dim, int64_t inter);

/* The routed-expert step for one token as one call (moe_v41/init.rs): q8_1
 * of x, the 2E gate+up batch, SwiGLU + q8_1 of h, the E down batch, the
 * route-weighted sum.  Three launches on `stream`: the q8_1 of x (when x is
 * 16-byte aligned; a separate launch otherwise) runs inside the gate/up
 * batch and SwiGLU + q8_1 of h inside the down batch, with the same bits as
 * the separate steps.
 *   ptrs      device array of 3E device pointers: gate_0..gate_{E-1}
 *             ([inter, dim] each), up_0..up_{E-1} ([inter, dim]),
 *             down_0..down_{E-1} ([dim, inter]) (moe_v41/init.rs, `ptrs_dev`)
 *   x_bf16    [dim];  route_w fp32 [E];  y fp32 [dim]
 *   workspace at least q2k_moe_m1_workspace_bytes(E, dim, inter) bytes,
 *             256-byte aligned; its contents on return are the q8_1 x, the
 *             fp32 gate/up outputs, the q8_1 h and the fp32 down outputs
 *             [E, dim] (before the route weights), in that order. */
int q2k_moe_m1(const void* const* ptrs, int64_t E, int64_t dim, int64_t inter,
               const uint16_t* x_bf16, const float* route_w, float* y, void* workspace,
               size_t workspace_bytes, q2k_stream_t stream);

/* Size of the fixed device scratch behind q2k_moe_m1_static_scratch. */
#define Q2K_MOE_M1_STATIC_SCRATCH_BYTES (1u << 20)

/* q2k_moe_m1 without a caller workspace.  The pages have no counterpart:
 * this is a library convenience for callers that cannot allocate device
 * memory (no device allocator of their own, or memory planned once that
 * must not grow between decode steps).
 *   ptrs, E, dim, inter, x_bf16, route_w, y   as for q2k_moe_m1
 * The workspace is a fixed Q2K_MOE_M1_STATIC_SCRATCH_BYTES (1 MiB) buffer
 * in the library's device image; nothing is allocated or freed.  Problems
 * with q2k_moe_m1_workspace_bytes(E, dim, inter) above that size return
 * Q2K_ERR_WORKSPACE before anything is enqueued (E = 8, dim = 4096,
 * inter = 2048 needs 285,184 bytes).  The first call on each device looks
 * the scratch's address up (cudaGetSymbolAddress, which may load the
 * module) and keeps it for the life of the process; make that first call
 * before any stream capture.  A cudaDeviceReset invalidates the kept
 * address: do not call this entry point on a device after resetting it.
 * Shapes q2k_moe_m1 refuses return Q2K_ERR_BAD_SHAPE here too.  Calls that
 * overlap on one device share the scratch and race: issue them on one
 * stream.  Results equal q2k_moe_m1's bit for bit. */
int q2k_moe_m1_static_scratch(const void* const* ptrs, int64_t E, int64_t dim, int64_t inter,
                              const uint16_t* x_bf16, const float* route_w, float* y,
                              q2k_stream_t stream);

/* Q2_K matmul for many tokens (moe_v41/init.rs, `MoeV41::new`: the
 * `metrale_q2_k_mmq128_*` kernels with their q8_1 activation quantisers take
 * the rows of more than 8 tokens; the prefill side of the path).
 *   W   Q2_K [N, K], 16-byte aligned; K % 1024 == 0 (rows on 16-byte
 *       boundaries, streamed four blocks at a time)
 *   x   bf16 [m, K], row stride ldx (ldx % 8 == 0), 16-byte aligned
 *   y   fp32 [m, N], row stride ldy: y = x W^T
 * The weights are read as Q2_K (84 bytes per 256 weights) and expanded on
 * the chip to bf16: each weight is d*sc*q - dmin*m in fp32 rounded once to
 * bf16, the values q2k_dequant_rows gives; the products run on the tensor
 * cores with fp32 accumulation.  So y equals dense_gemm_bf16(x, the
 * dequantised W) up to the order of the fp32 sums.  Any m >= 1 (tokens in
 * tiles of up to 256); for m <= 8 the GEMV/MMVQ calls read the weights
 * once per call too and are the faster route.  When the library splits K
 * across thread blocks (few weight tiles), partial sums are added with fp32
 * atomics, so the last bits may differ between runs.
 * Q2K_ERR_UNSUPPORTED when the CUDA driver offers no tensor-map encoder. */
int q2k_mmq_bf16(const void* W, int64_t N, int64_t K, const uint16_t* x, int64_t m, int64_t ldx, float* y,
                 int64_t ldy, q2k_stream_t stream);

/* Workspace bytes q2k_mmq_q8_1 needs: m * K * 2 (0 for a bad shape). */
size_t q2k_mmq_q8_1_workspace_bytes(int64_t m, int64_t K);

/* The Q2_K matmul over q8_1 activations: xq holds m q8_1 rows of K values
 * (back to back).  The values they encode, f32(d) * q, are rounded once to
 * bf16 into `workspace` (a launch of its own), then q2k_mmq_bf16 runs on
 * them.  workspace: at least q2k_mmq_q8_1_workspace_bytes(m, K) bytes,
 * 16-byte aligned.  Two launches. */
int q2k_mmq_q8_1(const void* W, int64_t N, int64_t K, const void* xq, int64_t m, float* y, int64_t ldy,
                 void* workspace, size_t workspace_bytes, q2k_stream_t stream);

/* Dense bf16 GEMM on the tensor cores, any m >= 1 (engram_v41/apply.rs,
 * `ops::dense_gemm` for several tokens; moe_v41/init.rs `dense_gemm_bf16`).
 *   x bf16 [m, K], row stride ldx;  W bf16 [N, K] row-major;
 *   y fp32 [m, N], row stride ldy.  K % 8 == 0; x, W 16-byte aligned and
 *   ldx % 8 == 0.  fp32 accumulation.  When the library splits K across
 *   thread blocks (small N), partial sums are added with fp32 atomics, so
 *   the last bits may differ between runs. */
int dense_gemm_bf16(const uint16_t* x, int64_t m, int64_t K, int64_t ldx, const uint16_t* W,
                    int64_t N, float* y, int64_t ldy, q2k_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* q2k_status_string(int status);

/* The last CUDA runtime error code a call returned as Q2K_ERR_CUDA in
 * this thread (0 if none). */
int q2k_last_cuda_error(void);

/* Diagnostics, synchronous (not for use inside stream capture): reads the
 * device's library error word into *host_out (0 = none; bit 0 = a bounded
 * wait in a kernel gave up and that kernel returned early, outputs
 * incomplete; bit 1 = a Q3_K table entry off a 4-byte boundary was
 * skipped) and clears it when clear != 0. */
int q2k_device_error(int32_t* host_out, int clear);

#ifdef __cplusplus
}
#endif

#endif /* Q2K_H */
