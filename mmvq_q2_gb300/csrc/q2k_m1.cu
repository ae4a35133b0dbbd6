// Q2_K GEMV / MMVQ for one, two or four tokens over long rows
// (engram_v41/apply.rs, the single-token `engram_v41_wkv_q2k_gemv` off
// `wkv_q2k`; attn_v41/decode.rs, `kquant_mmvq_pair_w` for the pair; the
// m <= 8 MMVQ of moe_v41/init.rs).
//
// One CTA of 16 warps per SM owns a contiguous range of output rows.  The
// CTA's lanes are split into row teams: a team has one lane per half block
// of a row for one token (8-word slices: 2*K/256 lanes, rounded up to a
// power of two), or per quarter block for two or four tokens (4-word
// slices, 4*K/256 lanes: the same registers for the activations), so each
// lane owns a fixed slice of every row and keeps the matching activations
// of every token in registers (q2k_slice.cuh).
//
// Weight stream.  A stage is 16/SW rows per team (two rows with 8-word
// slices, four with 4-word ones): about 43 KB of consecutive rows of the
// CTA's range, so it arrives with a single 1-D bulk copy.  The
// copy size is what sets the stream rate on this part: rings of 1.3 KB or
// 5 KB copies stream the 16384^2 matrix at 3.6 and 4.3 TB/s, 21 KB and
// 43 KB copies at 6.3 and 6.4 TB/s (plain 16-byte loads: 6.15).  Two rows
// per team also halve the per-row cost of waiting for and releasing a
// stage.  The weights do not depend on the activations, so the whole ring
// (4 stages, about 170 KB) is requested right after the launch's dependency
// wait, before the activations are staged, and covers the activation
// prologue.
//
// Release and refill.  A warp done with a stage counts itself out on the
// slot's counter in shared memory (lane 0, one atomic add); the warp that
// brings the count to 16 refills the slot.  It reads the atomic's result
// one stage later, so the atomic's latency never stalls it; the refill then
// leaves one stage after the release, well inside the 8-stage ring.  (A
// single polling producer refills only when it looks, and a ring refilled
// on demand waits the whole copy latency at every stage; a 17th, producer
// warp would cap the 16 consumer warps at 96 registers, below what the
// bf16 slice needs.)  Waits use mbarrier try_wait (the thread sleeps in
// hardware), bounded by the global timer.
//
// Each lane accumulates four rows, then one transpose-reduce across the
// warp leaves each row's warp partial in shared memory; after the walk the
// partials of a row's warps are added in warp order, so the output is
// deterministic and equal for every call.
#include "q2k_slice.cuh"

#include <algorithm>

namespace q2k {

__device__ int g_m1_error = 0;

namespace {

constexpr int kM1Threads = 512;  // 16 warps of row teams
constexpr int kM1Warps = kM1Threads / 32;
// rows per team in a stage: a stage of about 43 KB whatever the slice width
__host__ __device__ constexpr int m1_rps(int sw) { return 16 / sw; }
// rows per lane between two reductions: at least 4, and whole stages
__host__ __device__ constexpr int m1_rpt(int sw) { return m1_rps(sw) > 4 ? m1_rps(sw) : 4; }

struct M1Args {
    const uint8_t* W[2];  // row space: rows [0, N0) of W[0], then rows of W[1]
    float* y[2];
    int64_t ldy[2];       // floats between tokens of y
    int N0;
    int rows_total;
    int rows_q, rows_r;  // CTA c owns rows_q rows (+1 if c < rows_r)
    int nb;              // Q2_K blocks per row
    int lanes;           // lanes per row team: a power of two >= 2 * nb, 32..512
    int log_lanes;
    int teams;           // kM1Threads / lanes
    int wpt;             // warps per team (lanes / 32)
    int depth;           // stages in the ring
    uint32_t row_bytes;  // nb * 84, a multiple of 16
    uint32_t stage_bytes;  // kM1Rps * teams * row_bytes
    const uint8_t* x;    // bf16 rows or q8_1 rows, one per token
    int64_t x_tok_stride;  // bytes between tokens (a multiple of 16)
    uint32_t x_bytes;    // bytes of one token's row
    uint32_t off_x, off_bar, off_red;
};

__device__ __forceinline__ void m1_flag_error(volatile int* abort_flag)
{
    atomicOr(&g_m1_error, Q2K_ERR_BIT_WAIT_TIMEOUT);
    *abort_flag = 1;
}

template <int ACT, int M, int SW>
__global__ void __launch_bounds__(kM1Threads, 1) q2k_m1_kernel(const M1Args a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    using S = Slice<M, ACT, SW>;
    constexpr int kM1Rps = m1_rps(SW);
    constexpr int kM1Rpt = m1_rpt(SW);
    constexpr int VP = kM1Rpt * M;  // values per lane between two reductions
    static_assert(VP <= 32, "one (row, token) value per lane at most");
    pdl_launch_dependents();  // the next kernel may set itself up meanwhile

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int team = tid >> a.log_lanes;
    const int li = tid & (a.lanes - 1);  // lane within the team = slice of the row
    const int wit = li >> 5;             // warp within the team

    uint8_t* ring = smem;
    uint8_t* xsm = smem + a.off_x;
    uint64_t* full_b = reinterpret_cast<uint64_t*>(smem + a.off_bar);
    uint64_t* xbar = full_b + a.depth;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(xbar + 1);
    int* released = reinterpret_cast<int*>(xbar + 2);  // per slot: warps done, over all its stages
    int* uses = released + a.depth;                      // per slot: copies requested
    float* red = reinterpret_cast<float*>(smem + a.off_red);

    const int cta = (int)blockIdx.x;
    const int lo = cta * a.rows_q + min(cta, a.rows_r);
    const int hi = lo + a.rows_q + (cta < a.rows_r ? 1 : 0);
    const int spr = kM1Rps * a.teams;        // rows per stage
    const int nst = (hi - lo + spr - 1) / spr;  // stage j: rows lo + spr*j + Rps*t + q

    if (tid == 0) {
        mbar_init(smem_u32(xbar), 1);
        *abort_flag = 0;
    }
    if (tid < a.depth) {
        mbar_init(smem_u32(&full_b[tid]), 1);
        released[tid] = 0;
        uses[tid] = 0;
    }
    fence_mbar_init();
    __syncthreads();
    // Nothing above touched global memory: the previous kernel in the
    // stream may still be writing it until this wait returns.
    pdl_wait();

    // ---- stage j into slot s = j % depth (one thread) ----
    auto issue = [&](int j, int s) {
        const int r0 = lo + spr * j;
        const int r1 = min(hi, r0 + spr);
        const uint32_t fb = smem_u32(&full_b[s]);
        uint8_t* dst = ring + (size_t)s * a.stage_bytes;
        const uint64_t pol = l2_policy_evict_first();  // the weights are read once
        mbar_arrive_expect_tx(fb, (uint32_t)(r1 - r0) * a.row_bytes);
        // rows of the first matrix, then of the second (the pair)
        const int m0 = min(r1, a.N0);
        if (m0 > r0)
            bulk_copy_g2s_hint(smem_u32(dst), a.W[0] + (int64_t)r0 * a.row_bytes, (uint32_t)(m0 - r0) * a.row_bytes,
                               fb, pol);
        const int s1 = max(r0, a.N0);
        if (r1 > s1)
            bulk_copy_g2s_hint(smem_u32(dst + (size_t)(s1 - r0) * a.row_bytes),
                               a.W[1] + (int64_t)(s1 - a.N0) * a.row_bytes, (uint32_t)(r1 - s1) * a.row_bytes, fb, pol);
        atomicAdd(&uses[s], 1);
    };
    if (tid == 0) {
        // the activations first (every CTA reads them: keep them in L2), then
        // the whole ring, before any arithmetic
        mbar_arrive_expect_tx(smem_u32(xbar), (uint32_t)M * a.x_bytes);
#pragma unroll
        for (int t = 0; t < M; ++t)
            bulk_copy_g2s_hint(smem_u32(xsm + (size_t)t * a.x_bytes), a.x + (int64_t)t * a.x_tok_stride, a.x_bytes,
                               smem_u32(xbar), l2_policy_evict_last());
        for (int j = 0; j < min(a.depth, nst); ++j)
            issue(j, j);
    }

    // Wait for a phase.  Every lane waits for itself (they see the same
    // barrier); the common case is one try_wait.  Gives up after about two
    // seconds and raises the abort flag.
    auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity))
            return true;
        if (mbar_wait_bounded(bar, parity, abort_flag))
            return true;
        m1_flag_error(abort_flag);
        return false;
    };

    // ---- this lane's activation slice: block b, half n, first qs word wi0 ----
    constexpr int kLanesPerBlock = 16 / SW;  // 2, 4 or 8 (2 halves x 8/SW slices)
    const bool active = li < kLanesPerBlock * a.nb;
    const int b = active ? li / kLanesPerBlock : 0;
    const int n = (li / (kLanesPerBlock / 2)) & 1;
    const int wi0 = SW * (li & (kLanesPerBlock / 2 - 1));
    S sl;
    bool aborted = !wait(smem_u32(xbar), 0);
    // bf16 rows of one or two tokens are converted in place, cooperatively
    // (their region is sized for it); four tokens convert per thread inside
    // load_slice, from the raw rows
    if constexpr (coop_x<M, ACT, SW>())
        convert_x_bf16<M, SW>(xsm, a.nb);  // every thread (two CTA barriers inside)

    {
        load_slice<M, ACT, SW>(sl, xsm, a.nb, b, n, wi0, active);

        const uint8_t* blk0 = ring + (size_t)team * kM1Rps * a.row_bytes + (size_t)b * kBlockBytes;
        // stage j's slot, the parity of its phase there, j / depth and this
        // team's first row, advanced one stage at a time (no divisions)
        int s = 0, kd = 0, row = lo + kM1Rps * team;
        uint32_t parity = 0;
        // the previous stage (its slot, and the count the last warp out of it
        // sees) and, in lane 0, what this warp's atomic returned for it
        int prev_j = -1, prev_s = 0, prev_last = 0, prev_count = 0;
        // One stage: wait, this team's rows, count the warp out; the
        // previous stage's count has come back by now, and the warp that was
        // last out of it refills its slot.  TAIL: the stage may lack rows for
        // this team (the CTA's last stage).
        auto stage = [&](int j, bool tail, float* v) {
            if (!aborted && !wait(smem_u32(&full_b[s]), parity))
                aborted = true;
#pragma unroll
            for (int q = 0; q < kM1Rps; ++q) {
                float acc[M];
#pragma unroll
                for (int t = 0; t < M; ++t)
                    acc[t] = 0.f;
                if (!aborted && (!tail || row + q < hi))
                    slice_dot<M, ACT, SW>(sl, blk0 + (size_t)s * a.stage_bytes + (size_t)q * a.row_bytes, n, wi0, acc);
#pragma unroll
                for (int t = 0; t < M; ++t)
                    v[q * M + t] = acc[t];
            }
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                const int c = atomicAdd(&released[s], 1);
                if (prev_count == prev_last && prev_j >= 0 && prev_j + a.depth < nst && !*abort_flag)
                    issue(prev_j + a.depth, prev_s);
                prev_count = c;
            }
            prev_j = j;
            prev_s = s;
            prev_last = kM1Warps * (kd + 1) - 1;
            row += spr;
            if (++s == a.depth) {
                s = 0;
                parity ^= 1u;
                ++kd;
            }
        };
        // value i = k*M + t of v is token t of row Rps*team + (k % Rps) of
        // stage j0 + k / Rps; each lane group of 32/VP ends up with one
        // (row, token) warp partial
        constexpr int SPG = kM1Rpt / kM1Rps;  // stages per reduction group
        constexpr int kGroupLanes = 32 / VP;
        auto deposit = [&](int j0, float (&v)[VP]) {
            const float r = transpose_reduce<VP>(v, lane);
            const int i = lane / kGroupLanes;
            const int k = i / M, t = i - k * M;
            const int rl = spr * (j0 + k / kM1Rps) + kM1Rps * team + k % kM1Rps;  // row within the CTA's range
            if ((lane & (kGroupLanes - 1)) == 0 && lo + rl < hi)
                red[((size_t)rl * M + t) * a.wpt + wit] = r;
        };
        const int nst_full = (hi - lo) / spr;  // stages with every row present
        int j0 = 0;
        for (; j0 + SPG <= nst_full; j0 += SPG) {
            float v[VP];
#pragma unroll
            for (int g = 0; g < SPG; ++g)
                stage(j0 + g, false, v + g * kM1Rps * M);
            deposit(j0, v);
        }
        for (; j0 < nst; j0 += SPG) {
            float v[VP];
#pragma unroll
            for (int g = 0; g < SPG; ++g) {
                if (j0 + g < nst) {
                    stage(j0 + g, true, v + g * kM1Rps * M);
                } else {
#pragma unroll
                    for (int q = 0; q < kM1Rps * M; ++q)
                        v[g * kM1Rps * M + q] = 0.f;
                }
            }
            deposit(j0, v);
        }
        // the last stage's count needs no refill: nothing is left to load
    }

    __syncthreads();
    if (*abort_flag) {
        // every copy issued must land before the CTA's shared memory goes away
        // (the u-th copy into a slot completes the slot's phase u - 1)
        if (tid < a.depth && uses[tid] > 0)
            mbar_wait_bounded(smem_u32(&full_b[tid]), (uint32_t)(uses[tid] - 1) & 1u, nullptr);
        if (tid == 0)
            mbar_wait_bounded(smem_u32(xbar), 0, nullptr);
        __syncthreads();
        return;
    }
    // the warps' partials of each (row, token), added in warp order
    for (int i = tid; i < (hi - lo) * M; i += blockDim.x) {
        const int r = i / M, t = i - r * M;
        float v = 0.f;
        for (int w = 0; w < a.wpt; ++w)
            v += red[(size_t)i * a.wpt + w];
        const int row = lo + r;
        if (row < a.N0)
            a.y[0][(int64_t)t * a.ldy[0] + row] = v;
        else
            a.y[1][(int64_t)t * a.ldy[1] + row - a.N0] = v;
    }
}

size_t align16(size_t v) { return (v + 15) / 16 * 16; }

int log2i(int v)
{
    int l = 0;
    while ((1 << l) < v)
        ++l;
    return l;
}

// The launch plan; false when the problem is not this kernel's.
bool plan_m1(const MvProblem& p, const DeviceInfo& di, M1Args& a, int& grid, size_t& smem)
{
    // one token (8-word slices), two or four (4-word slices; four only with
    // q8_1: four bf16 tokens in 2-word slices were slower here than the
    // tensor-core kernel, 22.8 vs 20.2 us at 8192^2)
    const bool tokens_ok = p.m == 1 || p.m == 2 || (p.m == 4 && p.act == ACT_Q8);
    if (!tokens_ok || p.W_table || p.w_seg_stride || p.x_prep || p.n_seg < 1 || p.n_seg > 2)
        return false;
    // One token: rows of 16..128 blocks, the rows the general kernel also
    // walks with 128-weight slices and the same reduction, so the two give
    // the same bits (the pair from bf16 and the expert batches run there and
    // promise equality with this one).  Several tokens: rows of 8..128
    // blocks (no other path promises their bits).
    const int64_t kmin = (p.m == 1 ? 16 : 8) * (int64_t)kBlockWeights;
    if (p.K % 1024 || p.K < kmin || p.K > 128 * kBlockWeights)
        return false;
    const int nseg = p.n_seg;
    for (int e = 0; e < nseg; ++e)
        if ((reinterpret_cast<uintptr_t>(p.W[e]) & 15u) || p.N[e] <= 0)
            return false;
    if ((reinterpret_cast<uintptr_t>(p.x) & 15u) || (p.m > 1 && (p.x_tok_stride & 15)))
        return false;
    const int64_t rows = p.N[0] + (nseg > 1 ? p.N[1] : 0);
    if (rows > (1 << 30))
        return false;
    const int sw = p.m == 1 ? 8 : 4;
    // bf16 activations of one or two tokens are converted cooperatively:
    // every 16-value group of every token needs a thread slot
    if (p.act == ACT_BF16 && p.m <= 2 && p.m * (p.K / 16) > kCoopGroupsPerThread * kM1Threads)
        return false;
    a = M1Args{};
    a.nb = (int)(p.K / kBlockWeights);
    a.lanes = std::max(32, 1 << log2i((16 / sw) * a.nb));
    if (a.lanes > kM1Threads)
        return false;
    a.log_lanes = log2i(a.lanes);
    a.teams = kM1Threads / a.lanes;
    a.wpt = a.lanes / 32;
    a.row_bytes = (uint32_t)(a.nb * kBlockBytes);
    a.stage_bytes = (uint32_t)(m1_rps(sw) * a.teams) * a.row_bytes;
    a.W[0] = static_cast<const uint8_t*>(p.W[0]);
    a.W[1] = static_cast<const uint8_t*>(nseg > 1 ? p.W[1] : p.W[0]);
    a.y[0] = p.y[0];
    a.y[1] = nseg > 1 ? p.y[1] : p.y[0];
    a.ldy[0] = p.ldy[0];
    a.ldy[1] = nseg > 1 ? p.ldy[1] : p.ldy[0];
    a.x_tok_stride = p.x_tok_stride;
    a.N0 = (int)p.N[0];
    a.rows_total = (int)rows;
    a.x = static_cast<const uint8_t*>(p.x);
    a.x_bytes = p.act == ACT_BF16 ? (uint32_t)(p.K * 2) : (uint32_t)(p.K / kQ8Values * kQ8Bytes);
    grid = (int)std::min<int64_t>(di.sm_count, rows);
    a.rows_q = (int)(rows / grid);
    a.rows_r = (int)(rows % grid);
    const int rows_cta = a.rows_q + (a.rows_r ? 1 : 0);
    const size_t x_region = p.act == ACT_BF16 && p.m <= 2 ? align16((size_t)coop_x_bytes(p.m, a.nb))
                                                           : align16((size_t)p.m * a.x_bytes);
    const size_t cap = std::min<size_t>((size_t)di.smem_optin, 227 * 1024);
    for (int depth = 8; depth >= 2; --depth) {
        a.depth = depth;
        a.off_x = (uint32_t)((size_t)depth * a.stage_bytes);
        a.off_bar = (uint32_t)(a.off_x + x_region);
        a.off_red = (uint32_t)align16(a.off_bar + (size_t)(depth + 2) * sizeof(uint64_t) +
                                      (size_t)(2 * depth) * sizeof(int));
        const int spr = m1_rps(sw) * a.teams;
        smem = align16(a.off_red + (size_t)spr * ((rows_cta + spr - 1) / spr) * p.m * a.wpt * sizeof(float));
        if (smem <= cap)
            return true;
    }
    return false;
}

template <int ACT, int M, int SW>
cudaError_t launch_m1_act(const M1Args& a, int grid, size_t smem, cudaStream_t s)
{
    auto k = q2k_m1_kernel<ACT, M, SW>;
    static std::atomic<unsigned long long> smem_devs{0};
    cudaError_t e = allow_max_smem(k, smem_devs);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(k, dim3((unsigned)grid), dim3(kM1Threads), smem, s, a);
}

}  // namespace

bool m1_supported(const MvProblem& p)
{
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess)
        return false;
    M1Args a;
    int grid;
    size_t smem;
    return plan_m1(p, di, a, grid, smem);
}

cudaError_t launch_m1(const MvProblem& p, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess)
        return e;
    M1Args a;
    int grid;
    size_t smem;
    if (!plan_m1(p, di, a, grid, smem))
        return cudaErrorInvalidValue;
    if (p.act == ACT_BF16)
        return p.m == 1 ? launch_m1_act<ACT_BF16, 1, 8>(a, grid, smem, s) : launch_m1_act<ACT_BF16, 2, 4>(a, grid, smem, s);
    if (p.m == 1)
        return launch_m1_act<ACT_Q8, 1, 8>(a, grid, smem, s);
    return p.m == 2 ? launch_m1_act<ACT_Q8, 2, 4>(a, grid, smem, s) : launch_m1_act<ACT_Q8, 4, 4>(a, grid, smem, s);
}

cudaError_t m1_error_word(int32_t* out, bool clear)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_m1_error, sizeof(int));
    if (e != cudaSuccess)
        return e;
    *out = v;
    if (clear) {
        int z = 0;
        e = cudaMemcpyToSymbol(g_m1_error, &z, sizeof(int));
    }
    return e;
}

}  // namespace q2k
