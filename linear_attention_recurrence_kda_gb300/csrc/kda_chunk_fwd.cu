// kda_chunk_fwd.cu -- inter-chunk state pass and chunk outputs, fp32 SIMT.
//
// Chunk form of Equation 1 ("Kimi K3: the paper and proofs side by side", section 2.1.1), with
// the chunk's in-chunk cumulative log-decay G (Gamma = exp(G)) and W, U~ from kda_ut_wy:
//     U     = U~ - W S_in                                       (delta-rule corrections)
//     O     = (Q*Gamma) S_in + tril_incl((Q*Gamma)(K/Gamma)^T) U (read after each update)
//     S_out = Diag(Gamma_C) S_in + (K * Gamma_C/Gamma)^T U
// The state is carried from chunk to chunk ("Kimi K3: architecture, derivations and a
// pinned-source audit", section 4.5: the state map of a chunk is the composition of its tokens'
// affine maps), restarting from the sequence's initial state at every sequence start.
//
// Value columns evolve independently (column j of S only meets column j of V and U), so the
// grid splits d_v into slices: one CTA per (sequence, head, 32-column slice) walks its
// sequence's chunks in order, keeping its d_k x 32 slice of the state in shared memory in fp32.
// Every product is an fp32 FMA and every pairwise decay exp(G_r - G_i) is formed directly, so
// this kernel carries the fp32-input path's accuracy; bf16 inputs are widened on load.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kThreads = 256;

template <int DK, int JS>
struct ChunkSmem {
    float S[DK][JS];
    float Q[kChunk][DK];
    float K[kChunk][DK];
    float G[kChunk][DK];
    float W[kChunk][DK];
    float U[kChunk][JS];
    float P[kChunk][kChunk];
    float GL[DK];
};

}  // namespace

template <typename TIO, int DK, int DV, int JS>
__global__ void __launch_bounds__(kThreads) kda_chunk_fwd_kernel(PrefillArgs a)
{
    constexpr int C = kChunk;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ChunkSmem<DK, JS>& sm = *reinterpret_cast<ChunkSmem<DK, JS>*>(smem_raw);

    const int n = blockIdx.x;
    const int h = blockIdx.y;
    const int j0 = blockIdx.z * JS;
    const int tid = threadIdx.x;
    int64_t s0, s1;
    if (!seq_range(a, n, s0, s1)) return;

    const TIO* qp = static_cast<const TIO*>(a.q);
    const TIO* kp = static_cast<const TIO*>(a.k);
    TIO* op = static_cast<TIO*>(a.out);
    const int64_t sbase = ((int64_t)n * a.H + h) * DK * DV;

    for (int e = tid; e < DK * JS; e += kThreads) {
        const int c = e / JS, j = e % JS;
        sm.S[c][j] = a.s0 ? a.s0[sbase + (int64_t)c * DV + j0 + j] : 0.f;
    }

    for (int64_t t0 = s0; t0 < s1; t0 += C) {
        const int len = (int)min((int64_t)C, s1 - t0);
        __syncthreads();  // previous chunk's state update is complete
        for (int e = tid; e < C * DK; e += kThreads) {
            const int r = e / DK, c = e % DK;
            const int64_t idx = ((t0 + r) * a.H + h) * (int64_t)DK + c;
            const bool ok = r < len;
            sm.Q[r][c] = ok ? ld_io(qp, idx) : 0.f;
            sm.K[r][c] = ok ? ld_io(kp, idx) : 0.f;
            sm.G[r][c] = ok ? a.G[idx] : 0.f;
            sm.W[r][c] = ok ? a.W[idx] : 0.f;
        }
        for (int e = tid; e < C * JS; e += kThreads) {
            const int r = e / JS, j = e % JS;
            sm.U[r][j] = (r < len) ? a.Ut[((t0 + r) * a.H + h) * (int64_t)DV + j0 + j] : 0.f;
        }
        __syncthreads();

        // P = tril_incl((Q*Gamma)(K/Gamma)^T) with the pairwise decay exp(G_r - G_i);
        // U = U~ - W S_in; GL = G at the chunk's last token.
        for (int e = tid; e < C * C; e += kThreads) {
            const int r = e / C, i = e % C;
            float acc = 0.f;
            if (i <= r) {
#pragma unroll 8
                for (int c = 0; c < DK; ++c) acc += sm.Q[r][c] * sm.K[i][c] * expf(sm.G[r][c] - sm.G[i][c]);
            }
            sm.P[r][i] = acc;
        }
        float uacc[(C * JS + kThreads - 1) / kThreads];
#pragma unroll
        for (int q = 0; q < (C * JS + kThreads - 1) / kThreads; ++q) {
            const int e = tid + q * kThreads;
            uacc[q] = 0.f;
            if (e < C * JS) {
                const int r = e / JS, j = e % JS;
                float acc = sm.U[r][j];
#pragma unroll 8
                for (int c = 0; c < DK; ++c) acc -= sm.W[r][c] * sm.S[c][j];
                uacc[q] = acc;
            }
        }
        for (int c = tid; c < DK; c += kThreads) sm.GL[c] = sm.G[len - 1][c];
        __syncthreads();
#pragma unroll
        for (int q = 0; q < (C * JS + kThreads - 1) / kThreads; ++q) {
            const int e = tid + q * kThreads;
            if (e < C * JS) sm.U[e / JS][e % JS] = uacc[q];
        }
        // Q*Gamma and K*Gamma_C/Gamma (both factors <= 1)
        for (int e = tid; e < C * DK; e += kThreads) {
            const int r = e / DK, c = e % DK;
            const float g = sm.G[r][c];
            sm.Q[r][c] *= expf(g);
            sm.K[r][c] *= expf(sm.GL[c] - g);
        }
        __syncthreads();

        // O = (Q*Gamma) S_in + P U
        for (int e = tid; e < C * JS; e += kThreads) {
            const int r = e / JS, j = e % JS;
            if (r >= len) continue;
            float acc = 0.f;
#pragma unroll 8
            for (int c = 0; c < DK; ++c) acc += sm.Q[r][c] * sm.S[c][j];
            for (int i = 0; i <= r; ++i) acc += sm.P[r][i] * sm.U[i][j];
            st_io(op, ((t0 + r) * a.H + h) * (int64_t)DV + j0 + j, acc);
        }
        __syncthreads();

        // S_out = Diag(Gamma_C) S_in + (K*Gamma_C/Gamma)^T U
        for (int e = tid; e < DK * JS; e += kThreads) {
            const int c = e / JS, j = e % JS;
            float acc = expf(sm.GL[c]) * sm.S[c][j];
            for (int i = 0; i < len; ++i) acc += sm.K[i][c] * sm.U[i][j];
            sm.S[c][j] = acc;
        }
    }
    __syncthreads();
    if (a.s_final) {
        for (int e = tid; e < DK * JS; e += kThreads) {
            const int c = e / JS, j = e % JS;
            a.s_final[sbase + (int64_t)c * DV + j0 + j] = sm.S[c][j];
        }
    }
}

template <typename TIO, int DK, int DV>
static cudaError_t launch_chunk_t(const PrefillArgs& a, cudaStream_t s)
{
    constexpr int JS = DV < 32 ? DV : 32;
    const size_t smem = sizeof(ChunkSmem<DK, JS>);
    auto kern = kda_chunk_fwd_kernel<TIO, DK, DV, JS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)a.N, (unsigned)a.H, (unsigned)(DV / JS));
    kern<<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename TIO>
static cudaError_t launch_chunk_io(const PrefillArgs& a, cudaStream_t s)
{
#define KDA_CHUNK_CASE(DKv, DVv) \
    if (a.dk == DKv && a.dv == DVv) return launch_chunk_t<TIO, DKv, DVv>(a, s);
    KDA_CHUNK_CASE(32, 32) KDA_CHUNK_CASE(32, 64) KDA_CHUNK_CASE(32, 128)
    KDA_CHUNK_CASE(64, 32) KDA_CHUNK_CASE(64, 64) KDA_CHUNK_CASE(64, 128)
    KDA_CHUNK_CASE(128, 32) KDA_CHUNK_CASE(128, 64) KDA_CHUNK_CASE(128, 128)
#undef KDA_CHUNK_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_chunk_fwd(const PrefillArgs& a, kda_dtype_t dt, cudaStream_t s)
{
    return dt == KDA_BF16 ? launch_chunk_io<__nv_bfloat16>(a, s) : launch_chunk_io<float>(a, s);
}

}  // namespace kda
