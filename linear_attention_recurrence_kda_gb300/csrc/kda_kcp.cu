// kda_kcp.cu -- the pieces of context-parallel prefill (KCP) that are not a prefill themselves.
//
// A stretch of tokens acts on the recurrent state as an affine map S -> M S + S~ ("Kimi K3"
// reading notes, section 7, "Scaling to 1M Tokens: NoPE and KDA Context Parallelism": each rank
// turns its token range into such a summary, the summaries are exchanged once, and a prefix scan
// gives every rank its incoming state; "Kimi K3: architecture, derivations and a pinned-source
// audit", section 4.5: the maps compose associatively).  M (d_k x d_k) is the range's end state
// from the identity with v = 0 and S~ (d_k x d_v) its end state from zero; both come from
// kda_forward runs (see kda_forward_summary).  This file holds:
//   kda_identity_states_kernel  identity initial states [N][H][d_k][d_k]
//   kda_state_scan_kernel       S <- M_i S + S~_i for i = 0 .. count - 1, from the initial state
// The scan is fp32 SIMT: it runs once per exchange on count <= a few dozen summaries.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int NT = 256;
constexpr int JS = 32;  // value columns per CTA of the scan

}  // namespace

__global__ void __launch_bounds__(NT) kda_identity_states_kernel(float* S, int64_t units, int dk)
{
    const int64_t e = (int64_t)blockIdx.x * NT + threadIdx.x;
    const int64_t per = (int64_t)dk * dk;
    if (e >= units * per) return;
    const int64_t r = e % per;
    S[e] = (r / dk == r % dk) ? 1.f : 0.f;
}

template <int DK, int DV>
__global__ void __launch_bounds__(NT) kda_state_scan_kernel(const float* __restrict__ M, const float* __restrict__ St,
                                                            const float* __restrict__ S0, float* __restrict__ out,
                                                            int N, int H, int count)
{
    constexpr int W = DV < JS ? DV : JS;
    extern __shared__ __align__(16) float smem[];
    float* Ms = smem;                // [DK][DK + 1]
    float* Ss = Ms + DK * (DK + 1);  // [DK][W]
    const int n = blockIdx.x, h = blockIdx.y, j0 = blockIdx.z * W;
    const int tid = threadIdx.x;
    const int64_t unit = (int64_t)n * H + h;
    const int64_t sbase = unit * DK * DV;
    for (int e = tid; e < DK * W; e += NT) {
        const int c = e / W, j = e % W;
        Ss[e] = S0 ? S0[sbase + (int64_t)c * DV + j0 + j] : 0.f;
    }
    constexpr int PER = (DK * W + NT - 1) / NT;
    const int64_t mstride = (int64_t)N * H * DK * DK;
    const int64_t sstride = (int64_t)N * H * DK * DV;
    for (int i = 0; i < count; ++i) {
        __syncthreads();  // the previous step's state is complete
        const float* Mi = M + i * mstride + unit * DK * DK;
        for (int e = tid; e < DK * DK; e += NT) Ms[(e / DK) * (DK + 1) + e % DK] = Mi[e];
        __syncthreads();
        float acc[PER];
        const float* Si = St + i * sstride + sbase;
#pragma unroll
        for (int p = 0; p < PER; ++p) {
            const int e = tid + p * NT;
            acc[p] = 0.f;
            if (e < DK * W) {
                const int c = e / W, j = e % W;
                float a = Si[(int64_t)c * DV + j0 + j];
#pragma unroll 8
                for (int x = 0; x < DK; ++x) a += Ms[c * (DK + 1) + x] * Ss[x * W + j];
                acc[p] = a;
            }
        }
        __syncthreads();  // every thread has read the old state
#pragma unroll
        for (int p = 0; p < PER; ++p) {
            const int e = tid + p * NT;
            if (e < DK * W) Ss[e] = acc[p];
        }
    }
    __syncthreads();
    for (int e = tid; e < DK * W; e += NT) {
        const int c = e / W, j = e % W;
        out[sbase + (int64_t)c * DV + j0 + j] = Ss[e];
    }
}

cudaError_t launch_identity_states(float* S, int64_t units, int dk, cudaStream_t s)
{
    const int64_t n = units * dk * dk;
    if (n == 0) return cudaSuccess;
    kda_identity_states_kernel<<<(unsigned)((n + NT - 1) / NT), NT, 0, s>>>(S, units, dk);
    return cudaGetLastError();
}

template <int DK, int DV>
static cudaError_t launch_scan_t(const float* M, const float* St, const float* S0, float* out, int N, int H, int count,
                                 cudaStream_t s)
{
    constexpr int W = DV < JS ? DV : JS;
    const size_t smem = (size_t)(DK * (DK + 1) + DK * W) * sizeof(float);
    auto kern = kda_state_scan_kernel<DK, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)N, (unsigned)H, (unsigned)(DV / W)), NT, smem, s>>>(M, St, S0, out, N, H, count);
    return cudaGetLastError();
}

cudaError_t launch_state_scan(const float* M, const float* St, const float* S0, float* out, int N, int H, int dk, int dv,
                              int count, cudaStream_t s)
{
#define KDA_SCAN_CASE(DKv, DVv) \
    if (dk == DKv && dv == DVv) return launch_scan_t<DKv, DVv>(M, St, S0, out, N, H, count, s);
    KDA_SCAN_CASE(32, 32) KDA_SCAN_CASE(32, 64) KDA_SCAN_CASE(32, 128)
    KDA_SCAN_CASE(64, 32) KDA_SCAN_CASE(64, 64) KDA_SCAN_CASE(64, 128)
    KDA_SCAN_CASE(128, 32) KDA_SCAN_CASE(128, 64) KDA_SCAN_CASE(128, 128)
#undef KDA_SCAN_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda
