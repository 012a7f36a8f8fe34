// kda_segment_scan.cu -- incoming state of every segment of a segmented prefill (fp32).
//
// A segment's tokens act on the state as one affine map S -> M S + S~ (the composition of the
// tokens' maps; "Kimi K3: architecture, derivations and a pinned-source audit", section 4.5, and
// the KDA context-parallel decomposition of the "Kimi K3" reading notes, section 7:
// S_t = S~_t + M_{t<-1} S_in).  With (M_k, S~_k) of every segment computed in parallel, the state
// entering segment k+1 is
//     S_in[k+1] = M_k S_in[k] + S~_k,     S_in[0] = the sequence's initial state (or zero).
// This kernel walks that short chain.  Value columns are independent (column j of S only meets
// column j), so the grid splits them: one CTA per (sequence, head, block of 8 columns), M_k staged
// through shared memory (rows padded to avoid bank conflicts), each thread producing a 4 x 2 tile
// of the 128 x 8 result with fp32 FMAs.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int D = 128;
constexpr int COLS = 8;          // value columns per CTA
constexpr int NTHREADS = 128;    // 32 row groups of 4 x 4 column pairs
constexpr int MROW = D + 1;      // padded row of the staged M (floats)

}  // namespace

__global__ void __launch_bounds__(NTHREADS) kda_segment_scan_kernel(PrefillArgs a)
{
    extern __shared__ float smem_f[];
    float* sM = smem_f;                 // [D][MROW]
    float* sS = smem_f + D * MROW;      // [D][COLS] incoming state slice

    const int n = blockIdx.x;
    const int h = blockIdx.y;
    const int j0 = blockIdx.z * COLS;
    const int tid = threadIdx.x;
    const int rg = tid >> 2;            // rows 4 rg .. 4 rg + 3
    const int cp = tid & 3;             // columns j0 + 2 cp, j0 + 2 cp + 1

    int64_t q0, q1;
    if (!seq_range(a, n, q0, q1)) return;
    const int64_t seq_chunks = (q1 - q0 + kChunk - 1) / kChunk;
    if (seq_chunks <= 0 || a.seg_chunks <= 0) return;
    const int64_t nseg = (seq_chunks + a.seg_chunks - 1) / a.seg_chunks;
    if (nseg < 2) return;

    const int H = a.H;
    const int64_t sbase = ((int64_t)n * H + h) * D * D;
    for (int e = tid; e < D * COLS; e += NTHREADS) {
        const int c = e / COLS, jj = e % COLS;
        sS[e] = a.s0 ? a.s0[sbase + (int64_t)c * D + j0 + jj] : 0.f;
    }

    for (int64_t k = 0; k + 1 < nseg; ++k) {
        const int64_t segk = (((int64_t)n * H + h) * a.max_seg + k) * D * D;
        const float* M = a.seg_mt + segk;
        for (int e4 = tid; e4 < D * D / 4; e4 += NTHREADS) {
            const float4 m = reinterpret_cast<const float4*>(M)[e4];
            const int r = (4 * e4) / D, c = (4 * e4) % D;
            float* dst = sM + r * MROW + c;
            dst[0] = m.x;
            dst[1] = m.y;
            dst[2] = m.z;
            dst[3] = m.w;
        }
        const float* St = a.seg_st + segk;
        float acc[4][2];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 st = *reinterpret_cast<const float2*>(St + (int64_t)(4 * rg + i) * D + j0 + 2 * cp);
            acc[i][0] = st.x;
            acc[i][1] = st.y;
        }
        __syncthreads();
#pragma unroll 4
        for (int c = 0; c < D; ++c) {
            const float2 sv = *reinterpret_cast<const float2*>(sS + c * COLS + 2 * cp);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float m = sM[(4 * rg + i) * MROW + c];
                acc[i][0] = fmaf(m, sv.x, acc[i][0]);
                acc[i][1] = fmaf(m, sv.y, acc[i][1]);
            }
        }
        __syncthreads();
        float* out = a.seg_in + (((int64_t)n * H + h) * a.max_seg + k + 1) * D * D;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 4 * rg + i;
            *reinterpret_cast<float2*>(sS + r * COLS + 2 * cp) = make_float2(acc[i][0], acc[i][1]);
            *reinterpret_cast<float2*>(out + (int64_t)r * D + j0 + 2 * cp) = make_float2(acc[i][0], acc[i][1]);
        }
        __syncthreads();
    }
}

cudaError_t launch_segment_scan(const PrefillArgs& a, cudaStream_t s)
{
    const size_t smem = (size_t)(D * MROW + D * COLS) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(kda_segment_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kda_segment_scan_kernel<<<dim3((unsigned)a.N, (unsigned)a.H, D / COLS), NTHREADS, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
