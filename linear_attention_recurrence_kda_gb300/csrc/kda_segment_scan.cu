// kda_segment_scan.cu -- incoming state of every segment of a segmented prefill (fp32).
//
// A segment's tokens act on the state as one affine map S -> M S + S~ (the composition of the
// tokens' maps; "Kimi K3: architecture, derivations and a pinned-source audit", section 4.5, and
// the KDA context-parallel decomposition of the "Kimi K3" reading notes, section 7:
// S_t = S~_t + M_{t<-1} S_in).  With (M_k, S~_k) of every segment computed in parallel, the state
// entering segment k+1 is
//     S_in[k+1] = M_k S_in[k] + S~_k,     S_in[0] = the sequence's initial state (or zero).
// This kernel walks that short chain.  Value columns are independent (column j of S only meets
// column j), so the grid splits them: one CTA per (sequence, head, block of 16 columns).
//
// The summary pass stores every M_k transposed (M_k^T[c'][c], so that column c' of M_k -- the
// coefficients of input row c' -- is contiguous).  M_k^T is staged through shared memory with
// asynchronous copies, the next one while the current step computes.  Each of the 512 threads owns
// a 4 x 4 tile of the 128 x 16 result over one quarter of the contraction (32 of the 128 input rows):
// per input row one 16-byte load of M^T, one (broadcast) 16-byte load of S_in and 16 fp32 FMAs; the
// four quarters are added through shared memory.  512 threads keep enough warps in flight to hide
// the shared-memory latency of the short inner loop.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int D = 128;
constexpr int COLS = 16;         // value columns per CTA
constexpr int KSPLIT = 4;        // contraction quarters
constexpr int NTHREADS = 128 * KSPLIT;  // quarters x 4 column groups x 32 row groups

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all_but_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Asynchronously stage M^T ([128][128] fp32, rows contiguous) into shared memory.
__device__ __forceinline__ void stage_mt(float* dst, const float* Mt, int tid)
{
#pragma unroll 4
    for (int e4 = tid; e4 < D * D / 4; e4 += NTHREADS) cp_async16(dst + 4 * e4, Mt + 4 * e4);
}

}  // namespace

__global__ void __launch_bounds__(NTHREADS, 1) kda_segment_scan_kernel(PrefillArgs a)
{
    extern __shared__ __align__(16) float smem_f[];
    float* sM = smem_f;                       // [2][D][D] double-buffered M^T
    float* sS = smem_f + 2 * D * D;           // [D][COLS] incoming state slice
    float* sP = sS + D * COLS;                // [3][128 threads][16] partial tiles of quarters 1..3

    const int n = blockIdx.x;
    const int h = blockIdx.y;
    const int j0 = blockIdx.z * COLS;
    const int tid = threadIdx.x;
    const int kh = tid >> 7;             // contraction quarter: input rows [32 kh, 32 kh + 32)
    const int cg = (tid >> 5) & 3;       // columns j0 + 4 cg .. + 3
    const int rg = tid & 31;             // rows 4 rg .. 4 rg + 3
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
    griddep_wait();  // the segment summaries come from the previous kernel
    stage_mt(sM, a.seg_mt + seg0, tid);
    cp_async_commit();
    for (int e = tid; e < D * COLS; e += NTHREADS) {
        const int c = e / COLS, jj = e % COLS;
        sS[e] = a.s0 ? a.s0[sbase + (int64_t)c * D + j0 + jj] : 0.f;
    }

    for (int64_t k = 0; k + 1 < nseg; ++k) {
        const int64_t segk = seg0 + k * D * D;
        const float* Mt = sM + (k & 1) * D * D;
        // prefetch the next transition into the other buffer (an empty group on the last step)
        if (k + 2 < nseg) stage_mt(sM + ((k + 1) & 1) * D * D, a.seg_mt + segk + D * D, tid);
        cp_async_commit();
        float4 st[4];
        if (kh == 0) {
            const float* St = a.seg_st + segk;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                st[i] = *reinterpret_cast<const float4*>(St + (int64_t)(4 * rg + i) * D + j0 + 4 * cg);
        }
        cp_async_wait_all_but_one();   // M_k^T has landed (this thread's part)
        __syncthreads();               // ... and every thread's part; sS of the previous step is written
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) acc[i][jj] = 0.f;
#pragma unroll 8
        for (int cc = 0; cc < D / KSPLIT; ++cc) {
            const int c = (D / KSPLIT) * kh + cc;
            const float4 m = *reinterpret_cast<const float4*>(Mt + c * D + 4 * rg);      // M_k[4 rg + i][c]
            const float4 sv = *reinterpret_cast<const float4*>(sS + c * COLS + 4 * cg);  // S_in[c][j]
            const float mi[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[i][0] = fmaf(mi[i], sv.x, acc[i][0]);
                acc[i][1] = fmaf(mi[i], sv.y, acc[i][1]);
                acc[i][2] = fmaf(mi[i], sv.z, acc[i][2]);
                acc[i][3] = fmaf(mi[i], sv.w, acc[i][3]);
            }
        }
        if (kh > 0) {
            // partials laid out [quarter][i][thread] so that a warp's float4 stores are contiguous
            float4* pp = reinterpret_cast<float4*>(sP) + (kh - 1) * 4 * 128;
#pragma unroll
            for (int i = 0; i < 4; ++i) pp[i * 128 + (tid & 127)] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
        __syncthreads();               // every read of sS and Mt is done; the other quarters' partials are in
        if (kh == 0) {
            const float4* pp = reinterpret_cast<const float4*>(sP);
            float* out = a.seg_in + segk + D * D;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int q = 0; q < KSPLIT - 1; ++q) {
                    const float4 p4 = pp[(q * 4 + i) * 128 + tid];
                    u.x += p4.x;
                    u.y += p4.y;
                    u.z += p4.z;
                    u.w += p4.w;
                }
                const float4 r = make_float4(acc[i][0] + u.x + st[i].x, acc[i][1] + u.y + st[i].y,
                                             acc[i][2] + u.z + st[i].z, acc[i][3] + u.w + st[i].w);
                const int row = 4 * rg + i;
                *reinterpret_cast<float4*>(sS + row * COLS + 4 * cg) = r;
                *reinterpret_cast<float4*>(out + (int64_t)row * D + j0 + 4 * cg) = r;
            }
        }
    }
}

cudaError_t launch_segment_scan(const PrefillArgs& a, cudaStream_t s)
{
    const size_t smem = (size_t)(2 * D * D + D * COLS + (KSPLIT - 1) * 128 * 16) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(kda_segment_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_dependent(kda_segment_scan_kernel, dim3((unsigned)a.N, (unsigned)a.H, D / COLS), dim3(NTHREADS), smem,
                            s, a);
}

}  // namespace kda
