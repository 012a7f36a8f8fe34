// kda_gate.cu -- bounded channel-wise decay and its in-chunk cumulative sum.
//
// "Kimi K3: the paper and proofs side by side", section 2.1.1, Equation 5:
//   g = g_min * sigmoid(exp(A_h) * z)  in (g_min, 0)  per key channel,
// and (same section, and "Kimi K3" reading notes, section 2) the accumulated log-decay over a
// 16-token chunk stays in (16 g_min, 0) = (-80, 0) for g_min = -5.
//
// Output G[t, h, c] = sum of g over the tokens of t's chunk up to and including t (the chunk
// restarts at every sequence start).  One CTA per (chunk, head), one thread per key channel:
// every load and store is a contiguous d_k-wide row, so the kernel is a plain coalesced stream.
#include "kda_internal.cuh"

namespace kda {

template <typename TIO>
__global__ void __launch_bounds__(128) kda_gate_kernel(PrefillArgs a)
{
    const int slot = blockIdx.x;
    const int h = blockIdx.y;
    const int n = slot / a.chunks_per_seq;
    const int j = slot - n * a.chunks_per_seq;
    const int c = threadIdx.x;
    int64_t s0, s1;
    if (!seq_range(a, n, s0, s1)) return;
    const int64_t t0 = s0 + (int64_t)j * kChunk;
    if (t0 >= s1) return;
    const int64_t t1 = min(t0 + (int64_t)kChunk, s1);
    const float expA = expf(a.A[h]);
    const TIO* z = static_cast<const TIO*>(a.z);
    float G = 0.f;
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t idx = (t * a.H + h) * a.dk + c;
        G += log_decay(ld_io(z, idx), expA, a.g_min);
        a.G[idx] = G;
    }
}

cudaError_t launch_gate(const PrefillArgs& a, kda_dtype_t dt, cudaStream_t s)
{
    dim3 grid((unsigned)((int64_t)a.N * a.chunks_per_seq), (unsigned)a.H);
    dim3 block((unsigned)a.dk);
    if (dt == KDA_BF16) {
        kda_gate_kernel<__nv_bfloat16><<<grid, block, 0, s>>>(a);
    } else {
        kda_gate_kernel<float><<<grid, block, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace kda
