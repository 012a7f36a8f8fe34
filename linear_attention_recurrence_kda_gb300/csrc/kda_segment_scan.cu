// kda_segment_scan.cu -- incoming state of every segment of a segmented prefill (fp32).
//
// A segment's tokens act on the state as one affine map S -> M S + S~ (the composition of the
// tokens' maps; "Kimi K3: architecture, derivations and a pinned-source audit", section 4.5, and
// the KDA context-parallel decomposition of the "Kimi K3" reading notes, section 7:
// S_t = S~_t + M_{t<-1} S_in).  With (M_k, S~_k) of every segment computed in parallel, the state
// entering segment k+1 is
//     S_in[k+1] = M_k S_in[k] + S~_k,     S_in[0] = the sequence's initial state (or zero).
// This kernel walks that short chain.  Value columns are independent (column j of S only meets
// column j), so the grid splits them: one CTA per (sequence, head, block of 16 columns).  M_k is
// staged through shared memory with asynchronous copies, the next one while the current step
// computes (double buffer, padded rows); each thread produces a 4 x 2 tile of the 128 x 16 result
// with fp32 FMAs.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int D = 128;
constexpr int COLS = 16;         // value columns per CTA
constexpr int NTHREADS = 256;    // 32 row groups of 4 x 8 column pairs
constexpr int MROW = D + 4;      // padded row of the staged M (floats; keeps 16-byte alignment)

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all_but_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Asynchronously stage M (row-major [128][128] fp32) into padded shared rows.
__device__ __forceinline__ void stage_m(float* dst, const float* M, int tid)
{
#pragma unroll 4
    for (int e4 = tid; e4 < D * D / 4; e4 += NTHREADS) {
        const int r = (4 * e4) / D, c = (4 * e4) % D;
        cp_async16(dst + r * MROW + c, M + 4 * e4);
    }
}

}  // namespace

__global__ void __launch_bounds__(NTHREADS) kda_segment_scan_kernel(PrefillArgs a)
{
    extern __shared__ __align__(16) float smem_f[];
    float* sM = smem_f;                       // [2][D][MROW] double-buffered transition
    float* sS = smem_f + 2 * D * MROW;        // [D][COLS] incoming state slice

    const int n = blockIdx.x;
    const int h = blockIdx.y;
    const int j0 = blockIdx.z * COLS;
    const int tid = threadIdx.x;
    const int rg = tid >> 3;            // rows 4 rg .. 4 rg + 3
    const int cp = tid & 7;             // columns j0 + 2 cp, j0 + 2 cp + 1

    int64_t q0, q1;
    if (!seq_range(a, n, q0, q1)) return;
    const int64_t seq_chunks = (q1 - q0 + kChunk - 1) / kChunk;
    if (seq_chunks <= 0 || a.seg_chunks <= 0) return;
    const int64_t nseg = (seq_chunks + a.seg_chunks - 1) / a.seg_chunks;
    if (nseg < 2) return;

    const int H = a.H;
    const int64_t sbase = ((int64_t)n * H + h) * D * D;
    const int64_t seg0 = ((int64_t)n * H + h) * a.max_seg * D * D;
    stage_m(sM, a.seg_mt + seg0, tid);
    cp_async_commit();
    for (int e = tid; e < D * COLS; e += NTHREADS) {
        const int c = e / COLS, jj = e % COLS;
        sS[e] = a.s0 ? a.s0[sbase + (int64_t)c * D + j0 + jj] : 0.f;
    }

    for (int64_t k = 0; k + 1 < nseg; ++k) {
        const int64_t segk = seg0 + k * D * D;
        float* Mk = sM + (k & 1) * D * MROW;
        // prefetch the next transition into the other buffer (an empty group on the last step)
        if (k + 2 < nseg) stage_m(sM + ((k + 1) & 1) * D * MROW, a.seg_mt + segk + D * D, tid);
        cp_async_commit();
        const float* St = a.seg_st + segk;
        float acc[4][2];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 st = *reinterpret_cast<const float2*>(St + (int64_t)(4 * rg + i) * D + j0 + 2 * cp);
            acc[i][0] = st.x;
            acc[i][1] = st.y;
        }
        cp_async_wait_all_but_one();   // M_k has landed (this thread's part)
        __syncthreads();               // ... and every thread's part; sS of the previous step is written
#pragma unroll 4
        for (int c = 0; c < D; ++c) {
            const float2 sv = *reinterpret_cast<const float2*>(sS + c * COLS + 2 * cp);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float m = Mk[(4 * rg + i) * MROW + c];
                acc[i][0] = fmaf(m, sv.x, acc[i][0]);
                acc[i][1] = fmaf(m, sv.y, acc[i][1]);
            }
        }
        __syncthreads();               // every read of sS and Mk is done
        float* out = a.seg_in + segk + D * D;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 4 * rg + i;
            *reinterpret_cast<float2*>(sS + r * COLS + 2 * cp) = make_float2(acc[i][0], acc[i][1]);
            *reinterpret_cast<float2*>(out + (int64_t)r * D + j0 + 2 * cp) = make_float2(acc[i][0], acc[i][1]);
        }
    }
}

cudaError_t launch_segment_scan(const PrefillArgs& a, cudaStream_t s)
{
    const size_t smem = (size_t)(2 * D * MROW + D * COLS) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(kda_segment_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kda_segment_scan_kernel<<<dim3((unsigned)a.N, (unsigned)a.H, D / COLS), NTHREADS, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
