// kda_ut_wy.cu -- per-chunk UT transform of the keys and values (fp32 SIMT).
//
// Chunk form of Equation 1 ("Kimi K3: the paper and proofs side by side", section 2.1.1;
// regrouping justified by the associativity of the affine state maps, "Kimi K3: architecture,
// derivations and a pinned-source audit", section 4.5).  Within a chunk of C <= 16 tokens with
// in-chunk cumulative log-decay G_r (Gamma_r = exp(G_r), per key channel), the delta-rule
// corrections u_r solve the unit lower-triangular system
//     (I + A) U = diag(beta) (V - (K*Gamma) S_in),   A[r][i] = beta_r <k_r*Gamma_r, k_i/Gamma_i>, i < r,
// so with T = (I + A)^-1:  U = U~ - W S_in,  W = T diag(beta)(K*Gamma),  U~ = T diag(beta) V.
// This kernel produces W and U~ for every chunk; they do not depend on the state, so all chunks
// run in parallel.  The pairwise decay Gamma_r/Gamma_i is formed as exp(G_r - G_i) <= 1.
//
// One CTA per (chunk, head), 128 threads.  T is obtained by forward substitution on the 16x16
// unit lower-triangular matrix (one lane per column).
#include "kda_internal.cuh"

namespace kda {

template <typename TIO, int DK, int DV>
__global__ void __launch_bounds__(128) kda_ut_wy_kernel(PrefillArgs a)
{
    constexpr int C = kChunk;
    __shared__ float Ks[C][DK];   // raw keys, then beta_i k_i Gamma_i
    __shared__ float Gs[C][DK];
    __shared__ float Vs[C][DV];
    __shared__ float bs[C];
    __shared__ float Am[C][C];
    __shared__ float Tm[C][C];

    const int slot = blockIdx.x;
    const int h = blockIdx.y;
    const int n = slot / a.chunks_per_seq;
    const int jc = slot - n * a.chunks_per_seq;
    const int tid = threadIdx.x;
    int64_t s0, s1;
    if (!seq_range(a, n, s0, s1)) return;
    const int64_t t0 = s0 + (int64_t)jc * C;
    if (t0 >= s1) return;
    const int len = (int)min((int64_t)C, s1 - t0);

    const TIO* kp = static_cast<const TIO*>(a.k);
    const TIO* vp = static_cast<const TIO*>(a.v);
    for (int e = tid; e < C * DK; e += blockDim.x) {
        const int r = e / DK, c = e % DK;
        const int64_t idx = ((t0 + r) * a.H + h) * (int64_t)DK + c;
        const bool ok = r < len;
        Ks[r][c] = ok ? ld_io(kp, idx) : 0.f;
        Gs[r][c] = ok ? a.G[idx] : 0.f;
    }
    for (int e = tid; e < C * DV; e += blockDim.x) {
        const int r = e / DV, c = e % DV;
        Vs[r][c] = (r < len) ? ld_io(vp, ((t0 + r) * a.H + h) * (int64_t)DV + c) : 0.f;
    }
    if (tid < C) bs[tid] = (tid < len) ? a.beta[(t0 + tid) * a.H + h] : 0.f;
    __syncthreads();

    // A[r][i] = beta_r sum_c k_rc k_ic exp(G_rc - G_ic), i < r (zero elsewhere)
    for (int e = tid; e < C * C; e += blockDim.x) {
        const int r = e / C, i = e % C;
        float acc = 0.f;
        if (i < r) {
#pragma unroll 8
            for (int c = 0; c < DK; ++c) acc += Ks[r][c] * Ks[i][c] * expf(Gs[r][c] - Gs[i][c]);
            acc *= bs[r];
        }
        Am[r][i] = acc;
    }
    __syncthreads();

    // T = (I + A)^-1 by forward substitution: row r of T is e_r - sum_{i<r} A[r][i] T[i][:].
    if (tid < C) {
        const int j = tid;
        for (int r = 0; r < C; ++r) {
            float x = (r == j) ? 1.f : 0.f;
            for (int i = j; i < r; ++i) x -= Am[r][i] * Tm[i][j];
            Tm[r][j] = (j <= r) ? x : 0.f;
        }
    }
    // keys scaled for W: beta_i k_i Gamma_i (the raw keys are no longer needed)
    for (int e = tid; e < C * DK; e += blockDim.x) {
        const int r = e / DK, c = e % DK;
        Ks[r][c] = bs[r] * Ks[r][c] * expf(Gs[r][c]);
    }
    __syncthreads();

    for (int e = tid; e < C * DK; e += blockDim.x) {
        const int r = e / DK, c = e % DK;
        if (r >= len) continue;
        float acc = 0.f;
        for (int i = 0; i <= r; ++i) acc += Tm[r][i] * Ks[i][c];
        a.W[((t0 + r) * a.H + h) * (int64_t)DK + c] = acc;
    }
    for (int e = tid; e < C * DV; e += blockDim.x) {
        const int r = e / DV, c = e % DV;
        if (r >= len) continue;
        float acc = 0.f;
        for (int i = 0; i <= r; ++i) acc += Tm[r][i] * bs[i] * Vs[i][c];
        a.Ut[((t0 + r) * a.H + h) * (int64_t)DV + c] = acc;
    }
}

template <typename TIO>
static cudaError_t launch_ut_wy_t(const PrefillArgs& a, cudaStream_t s)
{
    dim3 grid((unsigned)((int64_t)a.N * a.chunks_per_seq), (unsigned)a.H);
    dim3 block(128);
#define KDA_UTWY_CASE(DKv, DVv)                                           \
    if (a.dk == DKv && a.dv == DVv) {                                      \
        kda_ut_wy_kernel<TIO, DKv, DVv><<<grid, block, 0, s>>>(a);         \
        return cudaGetLastError();                                         \
    }
    KDA_UTWY_CASE(32, 32) KDA_UTWY_CASE(32, 64) KDA_UTWY_CASE(32, 128)
    KDA_UTWY_CASE(64, 32) KDA_UTWY_CASE(64, 64) KDA_UTWY_CASE(64, 128)
    KDA_UTWY_CASE(128, 32) KDA_UTWY_CASE(128, 64) KDA_UTWY_CASE(128, 128)
#undef KDA_UTWY_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_ut_wy(const PrefillArgs& a, kda_dtype_t dt, cudaStream_t s)
{
    return dt == KDA_BF16 ? launch_ut_wy_t<__nv_bfloat16>(a, s) : launch_ut_wy_t<float>(a, s);
}

}  // namespace kda
