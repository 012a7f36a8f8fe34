// kda_segment_scan.cu -- incoming state of every segment of a segmented prefill.
//
// A segment's tokens act on the state as one affine map S -> M S + S~ (the composition of the
// tokens' maps; "Kimi K3: architecture, derivations and a pinned-source audit", section 4.5, and
// the KDA context-parallel decomposition of the "Kimi K3" reading notes, section 7:
// S_t = S~_t + M_{t<-1} S_in).  With (M_k, S~_k) of every segment computed in parallel, the state
// entering segment k+1 is
//     S_in[k+1] = M_k S_in[k] + S~_k,     S_in[0] = the sequence's initial state (or zero),
// S_in[0] included in what it writes.
// This kernel walks that short chain.  Value columns are independent (column j of S only meets
// column j), so the grid splits them: one CTA per (sequence, head, block of 16 columns).
//
// The product runs on the tensor cores (mma.sync m16n8k16) with both operands split into bf16
// pairs, M = M_hi + M_lo and S = S_hi + S_lo, as M_hi S_hi + M_hi S_lo + M_lo S_hi accumulated in
// fp32: each operand keeps about 16 significant bits, so a step adds a relative error of order
// 2^-16 -- far below the bf16 rounding of everything the tensor-core prefill reads and writes.
// The summary pass stores every M_k already split and in the operand layout (seg_m_off); one bulk
// copy brings it (64 KB) into shared memory while the previous step computes.  Warp w owns output
// rows 16 w .. 16 w + 15 over the whole contraction, so no partial sums cross warps; S_in is kept in
// fp32 registers (the accumulator fragments) and as a double-buffered bf16 hi/lo B operand in
// shared memory, so one barrier per step suffices.  Every wait is bounded; a copy that does not
// arrive raises the timeout bit of the check word.
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {

namespace {

constexpr int D = 128;
constexpr int COLS = 16;          // value columns per CTA
constexpr int NTHREADS = 256;     // 8 warps x 16 output rows
constexpr uint32_t WAIT_LIMIT = 1u << 17;

// shared memory (bytes)
constexpr uint32_t M_BYTES = 2 * kSegMPlane;              // one transition: hi and lo planes
constexpr uint32_t S_PLANE = COLS * 256;                   // S^T [16 j][128 c] bf16, seg_m_off layout
constexpr uint32_t OFF_M = 0;                              // [2] transitions, double-buffered
constexpr uint32_t OFF_S = 2 * M_BYTES;                    // [2] S_in operands (hi plane, lo plane)
constexpr uint32_t OFF_BAR = OFF_S + 2 * 2 * S_PLANE;
constexpr uint32_t OFF_ABORT = OFF_BAR + 16;
constexpr uint32_t SMEM_BYTES = OFF_ABORT + 16;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// S_in[c][j] as the hi/lo B operand (element (k = c, n = j) at seg_m_off(j, c) of each plane)
__device__ __forceinline__ void put_s(unsigned char* splane, int c, int j, float x)
{
    const __nv_bfloat16 hi = __float2bfloat16_rn(x);
    const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
    *reinterpret_cast<__nv_bfloat16*>(splane + seg_m_off(j, c)) = hi;
    *reinterpret_cast<__nv_bfloat16*>(splane + S_PLANE + seg_m_off(j, c)) = lo;
}

}  // namespace

__global__ void __launch_bounds__(NTHREADS, 1) kda_segment_scan_kernel(PrefillArgs a)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw + OFF_BAR);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem_raw + OFF_ABORT);

    const int n = blockIdx.x;
    const int h = blockIdx.y;
    const int j0 = blockIdx.z * COLS;
    const int tid = threadIdx.x;
    const int w = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    griddep_launch_dependents();

    int64_t q0, q1;
    if (!seq_range(a, n, q0, q1)) return;
    const int64_t seq_chunks = (q1 - q0 + kChunk - 1) / kChunk;
    if (seq_chunks <= 0 || a.seg_chunks <= 0) return;
    const int64_t nseg = (seq_chunks + a.seg_chunks - 1) / a.seg_chunks;
    if (nseg < 2) return;

    const int H = a.H;
    const int64_t sbase = ((int64_t)n * H + h) * D * D;
    const int64_t seg0 = ((int64_t)n * H + h) * a.max_seg * D * D;
    if (tid == 0) {
        tc::mbar_init(&bar[0], 1);
        tc::mbar_init(&bar[1], 1);
        *abort_flag = 0u;
    }
    // the caller's initial state is an input of the call (no kernel of this call writes it before
    // the output pass): stage it while the summaries finish, and copy it to the first segment's
    // incoming state, which the output pass reads instead of the caller's buffer (that buffer may
    // receive the final state while the first segment is still starting)
    for (int e = tid; e < D * COLS; e += NTHREADS) {
        const int c = e / COLS, jj = e % COLS;
        const float x = a.s0 ? a.s0[sbase + (int64_t)c * D + j0 + jj] : 0.f;
        put_s(smem_raw + OFF_S, c, jj, x);
        a.seg_in[seg0 + (int64_t)c * D + j0 + jj] = x;
    }
    tc::fence_async_smem();
    __syncthreads();
    griddep_wait();  // the segment summaries come from the previous kernel

    uint32_t pend = 0, ph = 0;  // thread 0: copies issued and not seen complete; every thread: parities
    auto issue = [&](int64_t k) {
        const int b = (int)(k & 1);
        tc::mbar_arrive_expect_tx(&bar[b], M_BYTES);
        tc::bulk_load(smem_raw + OFF_M + b * M_BYTES, a.seg_mt + seg0 + k * D * D, M_BYTES, &bar[b]);
        pend |= 1u << b;
    };
    if (tid == 0) issue(0);

    // this thread's accumulator positions: rows c0, c0 + 8; columns jj, jj + 1 of n-tiles 0 and 1
    const int c0 = 16 * w + g;
    // ldmatrix row addresses: A (rows of M, k = input row) and B (k = input row c, n = column j)
    const int arow = 16 * w + (lane & 7) + 8 * ((lane >> 3) & 1), akh = 8 * (lane >> 4);
    const int bj = (lane & 7) + 8 * (lane >> 4), bkh = 8 * ((lane >> 3) & 1);
    const uint32_t m_u32 = tc::smem_u32(smem_raw + OFF_M);
    const uint32_t s_u32 = tc::smem_u32(smem_raw + OFF_S);

    for (int64_t k = 0; k + 1 < nseg; ++k) {
        const int b = (int)(k & 1);
        const int64_t segk = seg0 + k * D * D;
        float2 st[2][2];  // S~_k at the accumulator positions
        {
            const float* St = a.seg_st + segk + j0;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                st[nt][0] = *reinterpret_cast<const float2*>(St + (int64_t)c0 * D + 8 * nt + 2 * t);
                st[nt][1] = *reinterpret_cast<const float2*>(St + (int64_t)(c0 + 8) * D + 8 * nt + 2 * t);
            }
        }
        if (tc::mbar_wait(&bar[b], (ph >> b) & 1u, WAIT_LIMIT)) {
            ph ^= 1u << b;
            if (tid == 0) pend &= ~(1u << b);
        } else {
            *abort_flag = 1u;
        }
        __syncthreads();  // M_k has landed; S_in[k] is in operand buffer k & 1; step k - 1's buffers are free
        if (*abort_flag != 0u) break;
        if (tid == 0 && k + 2 < nseg) issue(k + 1);

        const uint32_t mb = m_u32 + b * M_BYTES;
        const uint32_t sb = s_u32 + b * (2 * S_PLANE);
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t oa = seg_m_off(arow, 16 * ks + akh);
            const uint32_t ob = seg_m_off(bj, 16 * ks + bkh);
            uint32_t ah[4], al[4], bh[4], bl[4];
            ldsm_x4(mb + oa, ah[0], ah[1], ah[2], ah[3]);
            ldsm_x4(mb + kSegMPlane + oa, al[0], al[1], al[2], al[3]);
            ldsm_x4(sb + ob, bh[0], bh[1], bh[2], bh[3]);
            ldsm_x4(sb + S_PLANE + ob, bl[0], bl[1], bl[2], bl[3]);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                tc::mma16816(acc[nt], ah, bh[2 * nt], bh[2 * nt + 1]);
                tc::mma16816(acc[nt], ah, bl[2 * nt], bl[2 * nt + 1]);
                tc::mma16816(acc[nt], al, bh[2 * nt], bh[2 * nt + 1]);
            }
        }
        // S_in[k+1] = M_k S_in[k] + S~_k: fp32 to the workspace, hi/lo into the other operand buffer
        float* out = a.seg_in + segk + D * D + j0;
        unsigned char* sn = smem_raw + OFF_S + (b ^ 1) * (2 * S_PLANE);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int jj = 8 * nt + 2 * t;
            const float2 u0 = make_float2(acc[nt][0] + st[nt][0].x, acc[nt][1] + st[nt][0].y);
            const float2 u1 = make_float2(acc[nt][2] + st[nt][1].x, acc[nt][3] + st[nt][1].y);
            *reinterpret_cast<float2*>(out + (int64_t)c0 * D + jj) = u0;
            *reinterpret_cast<float2*>(out + (int64_t)(c0 + 8) * D + jj) = u1;
            put_s(sn, c0, jj, u0.x);
            put_s(sn, c0, jj + 1, u0.y);
            put_s(sn, c0 + 8, jj, u1.x);
            put_s(sn, c0 + 8, jj + 1, u1.y);
        }
    }
    if (tid == 0 && *abort_flag != 0u) {
        atomicOr(a.check, kCheckTimeout);
        // a copy still in flight must land before the shared memory is released
        for (int b = 0; b < 2; ++b)
            if (pend & (1u << b)) (void)tc::mbar_wait(&bar[b], (ph >> b) & 1u, WAIT_LIMIT);
    }
}

cudaError_t launch_segment_scan(const PrefillArgs& a, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(kda_segment_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return launch_dependent(kda_segment_scan_kernel, dim3((unsigned)a.N, (unsigned)a.H, D / COLS), dim3(NTHREADS),
                            SMEM_BYTES, s, a);
}

}  // namespace kda
