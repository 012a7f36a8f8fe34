// kda_backward.cu -- gradients of the KDA prefill (fp32 SIMT, every supported width and io dtype).
//
// For L = <dO, out> + <dS_final, S_final> the chunk form of Equation 1 ("Kimi K3: the paper and
// proofs side by side", section 2.1.1, gate of Equation 5) is differentiated chunk by chunk; the
// analytic derivative is the one the audit's CPU laboratory checks against finite differences
// ("Kimi K3: architecture, derivations and a pinned-source audit", "CPU laboratory").  Per chunk
// entering with state S (G the in-chunk inclusive cumulative log-decay, KG = K e^G, QG = Q e^G,
// KI = K e^-G, Kt = K e^(G_C - G), A = tril_strict(diag(b) KG KI^T), T = (I + A)^-1,
// W = T diag(b) KG, U = T diag(b) V - W S, P = tril(QG KI^T), O = QG S + P U,
// S' = e^G_C S + Kt^T U), going back from dO and dS' (the gradient reaching S'):
//     dU = Kt dS' + P^T dO,   dS = e^G_C dS' + QG^T dO - W^T dU                  (state pass)
//     dKt = U dS'^T,  dP = tril(dO U^T),  dQG = dO S^T + dP KI,  dW = -dU S^T
//     dT = dU (diag(b) V)^T + dW (diag(b) KG)^T,  dA = -tril_strict(T^T dT T^T)
//     dV = diag(b) T^T dU,  dKG = diag(b) T^T dW + diag(b) dA KI,  dKI = (diag(b) dA)^T KG + dP^T QG
//     db = rowsum(T^T dU * V) + rowsum(T^T dW * KG) + rowsum(dA * KG KI^T)
//     dG = dKG KG + dQG QG - dKI KI - dKt Kt,  dG_C += colsum(dKt Kt) + e^G_C rowsum(dS' * S)
//     dg = reversed in-chunk cumulative sum of dG;  x = e^A z, dz = dg g_min s'(x) e^A,
//     dA_h = sum dg g_min s'(x) x   (s' = s(1 - s) the slope of the sigmoid s)
// The gradients reach G through the scaled rows themselves, so no 1/Gamma^2 appears; with
// g_min >= -5.4 every factor of one chunk is a finite fp32 number (e^-G <= e^86.4).
//
// Kernels, in order (after kda_gate and kda_ut_wy, which fill G, W and U~):
//   kda_bwd_gram    per (chunk, head): P = tril(QG KI^T)
//   kda_bwd_states  per (sequence, head, value-column slice), chunks in order: the state entering
//                   every chunk and U = U~ - W S
//   kda_bwd_dstates per (sequence, head, value-column slice), chunks in reverse: the gradient
//                   reaching every chunk's end state, dU, and dS0
//   kda_bwd_chunk   per (chunk, head): every input gradient and the chunk's share of dA
//   kda_bwd_da      per head: dA from the chunks' shares (fixed order, deterministic)
// Value columns are independent in both state passes (column j of S and dS only meets column j of
// V, U, dO and dU), which is what the slices use.
#include <type_traits>

#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int C = kChunk;
constexpr int NT = 256;

// Slot of chunk ci of sequence n (s0 = cu[n]).
__device__ __forceinline__ int64_t chunk_slot(int n, int64_t s0, int64_t ci) { return s0 / C + n + ci; }

// Slope of the logistic function, s(x)(1 - s(x)) = e / (1 + e)^2 with e = exp(-|x|): no
// cancellation where the sigmoid saturates (1 - s(x) is not formed).
__device__ __forceinline__ float sigmoid_slope(float x)
{
    const float e = expf(-fabsf(x));
    return e / ((1.f + e) * (1.f + e));
}

// (sequence, chunk) of a CTA of a chunk-parallel grid; false if the chunk is past its sequence.
__device__ __forceinline__ bool chunk_of(const PrefillArgs& a, int& n, int64_t& s0, int64_t& t0, int& len, int64_t& ci)
{
    const int64_t x = blockIdx.x;
    n = (int)(x / a.chunks_per_seq);
    ci = x - (int64_t)n * a.chunks_per_seq;
    int64_t s1;
    if (!seq_range(a, n, s0, s1)) return false;
    t0 = s0 + ci * C;
    if (t0 >= s1) return false;
    len = (int)min((int64_t)C, s1 - t0);
    return true;
}

}  // namespace

// ---------------------------------------------------------------- P = tril(QG KI^T) per chunk

template <typename TIO, int DK>
__global__ void __launch_bounds__(NT) kda_bwd_gram_kernel(BackwardArgs b)
{
    const PrefillArgs& a = b.f;
    __shared__ float QG[C][DK];
    __shared__ float KI[C][DK];
    int n, len;
    int64_t s0, t0, ci;
    if (!chunk_of(a, n, s0, t0, len, ci)) return;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const TIO* qp = static_cast<const TIO*>(a.q);
    const TIO* kp = static_cast<const TIO*>(a.k);
    for (int e = tid; e < C * DK; e += NT) {
        const int r = e / DK, c = e % DK;
        float q = 0.f, k = 0.f, g = 0.f;
        if (r < len) {
            const int64_t idx = ((t0 + r) * a.H + h) * (int64_t)DK + c;
            q = ld_io(qp, idx);
            k = ld_io(kp, idx);
            g = a.G[idx];
        }
        QG[r][c] = q * expf(g);
        KI[r][c] = k * expf(-g);
    }
    __syncthreads();
    const int r = tid / C, i = tid % C;
    if (r < len) {
        float acc = 0.f;
        if (i <= r) {
#pragma unroll 8
            for (int c = 0; c < DK; ++c) acc += QG[r][c] * KI[i][c];
        }
        b.P[((t0 + r) * a.H + h) * (int64_t)C + i] = acc;
    }
}

// ---------------------------------------------------------------- forward state pass (states kept)

template <int DK, int JS>
struct StatesSmem {
    float S[DK][JS];
    float K[C][DK];  // keys, then K e^(G_C - G)
    float G[C][DK];
    float W[C][DK];
    float U[C][JS];
    float GL[DK];
};

template <typename TIO, int DK, int DV, int JS>
__global__ void __launch_bounds__(NT) kda_bwd_states_kernel(BackwardArgs b)
{
    const PrefillArgs& a = b.f;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    StatesSmem<DK, JS>& sm = *reinterpret_cast<StatesSmem<DK, JS>*>(smem_raw);
    const int n = blockIdx.x;
    const int h = blockIdx.y;
    const int j0 = blockIdx.z * JS;
    const int tid = threadIdx.x;
    int64_t s0, s1;
    if (!seq_range(a, n, s0, s1)) return;
    const TIO* kp = static_cast<const TIO*>(a.k);
    const int64_t sbase = ((int64_t)n * a.H + h) * DK * DV;
    for (int e = tid; e < DK * JS; e += NT) {
        const int c = e / JS, j = e % JS;
        sm.S[c][j] = a.s0 ? a.s0[sbase + (int64_t)c * DV + j0 + j] : 0.f;
    }
    constexpr int NU = (C * JS + NT - 1) / NT;
    for (int64_t ci = 0; s0 + ci * C < s1; ++ci) {
        const int64_t t0 = s0 + ci * C;
        const int len = (int)min((int64_t)C, s1 - t0);
        __syncthreads();  // the previous chunk's state update is complete
        float* dst = b.S_chunk + (chunk_slot(n, s0, ci) * a.H + h) * (int64_t)DK * DV + j0;
        for (int e = tid; e < DK * JS; e += NT) {
            const int c = e / JS, j = e % JS;
            dst[(int64_t)c * DV + j] = sm.S[c][j];
        }
        for (int e = tid; e < C * DK; e += NT) {
            const int r = e / DK, c = e % DK;
            const bool ok = r < len;
            const int64_t idx = ((t0 + r) * a.H + h) * (int64_t)DK + c;
            sm.K[r][c] = ok ? ld_io(kp, idx) : 0.f;
            sm.G[r][c] = ok ? a.G[idx] : 0.f;
            sm.W[r][c] = ok ? a.W[idx] : 0.f;
        }
        for (int e = tid; e < C * JS; e += NT) {
            const int r = e / JS, j = e % JS;
            sm.U[r][j] = (r < len) ? a.Ut[((t0 + r) * a.H + h) * (int64_t)DV + j0 + j] : 0.f;
        }
        __syncthreads();
        float uacc[NU];
#pragma unroll
        for (int q = 0; q < NU; ++q) {
            const int e = tid + q * NT;
            uacc[q] = 0.f;
            if (e < C * JS) {
                const int r = e / JS, j = e % JS;
                float acc = sm.U[r][j];
#pragma unroll 8
                for (int c = 0; c < DK; ++c) acc -= sm.W[r][c] * sm.S[c][j];
                uacc[q] = (r < len) ? acc : 0.f;
            }
        }
        for (int c = tid; c < DK; c += NT) sm.GL[c] = sm.G[len - 1][c];
        __syncthreads();
#pragma unroll
        for (int q = 0; q < NU; ++q) {
            const int e = tid + q * NT;
            if (e < C * JS) {
                const int r = e / JS, j = e % JS;
                sm.U[r][j] = uacc[q];
                if (r < len) b.U[((t0 + r) * a.H + h) * (int64_t)DV + j0 + j] = uacc[q];
            }
        }
        for (int e = tid; e < C * DK; e += NT) {
            const int r = e / DK, c = e % DK;
            sm.K[r][c] *= expf(sm.GL[c] - sm.G[r][c]);
        }
        __syncthreads();
        for (int e = tid; e < DK * JS; e += NT) {
            const int c = e / JS, j = e % JS;
            float acc = expf(sm.GL[c]) * sm.S[c][j];
            for (int i = 0; i < len; ++i) acc += sm.K[i][c] * sm.U[i][j];
            sm.S[c][j] = acc;
        }
    }
}

// ---------------------------------------------------------------- reverse state pass

template <int DK, int JS>
struct DStatesSmem {
    float dS[DK][JS];
    float Q[C][DK];  // queries, then Q e^G
    float K[C][DK];  // keys, then K e^(G_C - G)
    float G[C][DK];
    float W[C][DK];
    float P[C][C];
    float dO[C][JS];
    float dU[C][JS];
    float GL[DK];
};

template <typename TIO, int DK, int DV, int JS>
__global__ void __launch_bounds__(NT) kda_bwd_dstates_kernel(BackwardArgs b)
{
    const PrefillArgs& a = b.f;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    DStatesSmem<DK, JS>& sm = *reinterpret_cast<DStatesSmem<DK, JS>*>(smem_raw);
    const int n = blockIdx.x;
    const int h = blockIdx.y;
    const int j0 = blockIdx.z * JS;
    const int tid = threadIdx.x;
    int64_t s0, s1;
    if (!seq_range(a, n, s0, s1)) return;
    const TIO* qp = static_cast<const TIO*>(a.q);
    const TIO* kp = static_cast<const TIO*>(a.k);
    const TIO* dop = static_cast<const TIO*>(b.dout);
    const int64_t sbase = ((int64_t)n * a.H + h) * DK * DV;
    for (int e = tid; e < DK * JS; e += NT) {
        const int c = e / JS, j = e % JS;
        sm.dS[c][j] = b.dS_final ? b.dS_final[sbase + (int64_t)c * DV + j0 + j] : 0.f;
    }
    constexpr int NU = (C * JS + NT - 1) / NT;
    const int64_t nch = (s1 - s0 + C - 1) / C;
    for (int64_t ci = nch - 1; ci >= 0; --ci) {
        const int64_t t0 = s0 + ci * C;
        const int len = (int)min((int64_t)C, s1 - t0);
        __syncthreads();  // the previous (later) chunk's update is complete
        float* dst = b.dS_chunk + (chunk_slot(n, s0, ci) * a.H + h) * (int64_t)DK * DV + j0;
        for (int e = tid; e < DK * JS; e += NT) {
            const int c = e / JS, j = e % JS;
            dst[(int64_t)c * DV + j] = sm.dS[c][j];
        }
        for (int e = tid; e < C * DK; e += NT) {
            const int r = e / DK, c = e % DK;
            const bool ok = r < len;
            const int64_t idx = ((t0 + r) * a.H + h) * (int64_t)DK + c;
            sm.Q[r][c] = ok ? ld_io(qp, idx) : 0.f;
            sm.K[r][c] = ok ? ld_io(kp, idx) : 0.f;
            sm.G[r][c] = ok ? a.G[idx] : 0.f;
            sm.W[r][c] = ok ? a.W[idx] : 0.f;
        }
        for (int e = tid; e < C * C; e += NT) {
            const int r = e / C, i = e % C;
            sm.P[r][i] = (r < len) ? b.P[((t0 + r) * a.H + h) * (int64_t)C + i] : 0.f;
        }
        for (int e = tid; e < C * JS; e += NT) {
            const int r = e / JS, j = e % JS;
            sm.dO[r][j] = (r < len) ? ld_io(dop, ((t0 + r) * a.H + h) * (int64_t)DV + j0 + j) : 0.f;
        }
        __syncthreads();
        for (int c = tid; c < DK; c += NT) sm.GL[c] = sm.G[len - 1][c];
        __syncthreads();
        for (int e = tid; e < C * DK; e += NT) {
            const int r = e / DK, c = e % DK;
            const float g = sm.G[r][c];
            sm.Q[r][c] *= expf(g);
            sm.K[r][c] *= expf(sm.GL[c] - g);
        }
        __syncthreads();
        // dU = Kt dS' + P^T dO
        float uacc[NU];
#pragma unroll
        for (int q = 0; q < NU; ++q) {
            const int e = tid + q * NT;
            uacc[q] = 0.f;
            if (e < C * JS) {
                const int r = e / JS, j = e % JS;
                float acc = 0.f;
                if (r < len) {
#pragma unroll 8
                    for (int c = 0; c < DK; ++c) acc += sm.K[r][c] * sm.dS[c][j];
                    for (int i = r; i < len; ++i) acc += sm.P[i][r] * sm.dO[i][j];
                }
                uacc[q] = acc;
            }
        }
#pragma unroll
        for (int q = 0; q < NU; ++q) {
            const int e = tid + q * NT;
            if (e < C * JS) {
                const int r = e / JS, j = e % JS;
                sm.dU[r][j] = uacc[q];
                if (r < len) b.dU[((t0 + r) * a.H + h) * (int64_t)DV + j0 + j] = uacc[q];
            }
        }
        __syncthreads();
        // dS = e^G_C dS' + QG^T dO - W^T dU
        for (int e = tid; e < DK * JS; e += NT) {
            const int c = e / JS, j = e % JS;
            float acc = expf(sm.GL[c]) * sm.dS[c][j];
            for (int r = 0; r < len; ++r) acc += sm.Q[r][c] * sm.dO[r][j] - sm.W[r][c] * sm.dU[r][j];
            sm.dS[c][j] = acc;
        }
    }
    __syncthreads();
    if (b.dS0) {
        for (int e = tid; e < DK * JS; e += NT) {
            const int c = e / JS, j = e % JS;
            b.dS0[sbase + (int64_t)c * DV + j0 + j] = sm.dS[c][j];
        }
    }
}

// ---------------------------------------------------------------- per-chunk gradients

template <int DK, int DV>
struct ChunkGradSmem {
    static constexpr int JB = DV < 32 ? DV : 32;  // value columns per staged state tile
    float EG[C][DK];   // e^G
    float K[C][DK];
    float G[C][DK];
    float KG[C][DK];
    float KI[C][DK];
    float QG[C][DK];
    float dKt[C][DK];
    float dQa[C][DK];  // dO S^T
    float dW[C][DK];   // -dU S^T, later dG
    float TdW[C][DK];
    float V[C][DV];
    float dO[C][DV];
    float U[C][DV];
    float dU[C][DV];
    float TdU[C][DV];
    float Sin[DK][JB + 1];
    float dSo[DK][JB + 1];
    float M[C][C], P[C][C], T[C][C], dP[C][C], dTn[C][C], X[C][C], dA[C][C];
    float rs[DK], GL[DK], ktsum[DK];
    float beta[C];
    float red[NT / 32];
};

template <typename TIO, int DK, int DV>
__global__ void __launch_bounds__(NT) kda_bwd_chunk_kernel(BackwardArgs b)
{
    using Sm = ChunkGradSmem<DK, DV>;
    constexpr int JB = Sm::JB;
    const PrefillArgs& a = b.f;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Sm& sm = *reinterpret_cast<Sm*>(smem_raw);
    int n, len;
    int64_t s0, t0, ci;
    if (!chunk_of(a, n, s0, t0, len, ci)) return;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int H = a.H;
    const TIO* qp = static_cast<const TIO*>(a.q);
    const TIO* kp = static_cast<const TIO*>(a.k);
    const TIO* vp = static_cast<const TIO*>(a.v);
    const TIO* zp = static_cast<const TIO*>(a.z);
    const TIO* dop = static_cast<const TIO*>(b.dout);
    const int64_t slot = chunk_slot(n, s0, ci);
    const float* Sg = b.S_chunk + (slot * H + h) * (int64_t)DK * DV;
    const float* dSg = b.dS_chunk + (slot * H + h) * (int64_t)DK * DV;

    // 1. the chunk's rows (absent tokens as zeros)
    for (int e = tid; e < C * DK; e += NT) {
        const int r = e / DK, c = e % DK;
        float q = 0.f, k = 0.f, g = 0.f;
        if (r < len) {
            const int64_t idx = ((t0 + r) * H + h) * (int64_t)DK + c;
            q = ld_io(qp, idx);
            k = ld_io(kp, idx);
            g = a.G[idx];
        }
        const float eg = expf(g);
        sm.EG[r][c] = eg;
        sm.K[r][c] = k;
        sm.G[r][c] = g;
        sm.KG[r][c] = k * eg;
        sm.KI[r][c] = k * expf(-g);
        sm.QG[r][c] = q * eg;
    }
    for (int e = tid; e < C * DV; e += NT) {
        const int r = e / DV, j = e % DV;
        const bool ok = r < len;
        const int64_t idx = ((t0 + r) * H + h) * (int64_t)DV + j;
        sm.V[r][j] = ok ? ld_io(vp, idx) : 0.f;
        sm.dO[r][j] = ok ? ld_io(dop, idx) : 0.f;
        sm.U[r][j] = ok ? b.U[idx] : 0.f;
        sm.dU[r][j] = ok ? b.dU[idx] : 0.f;
    }
    for (int e = tid; e < C * C; e += NT) {
        const int r = e / C, i = e % C;
        sm.P[r][i] = (r < len) ? b.P[((t0 + r) * H + h) * (int64_t)C + i] : 0.f;
    }
    if (tid < C) sm.beta[tid] = tid < len ? a.beta[(t0 + tid) * H + h] : 0.f;

    // 2. the products with the states, over value-column tiles:
    //    dKt = U dS'^T, dQa = dO S^T, dW = -dU S^T, rs = rowsum(dS' * S)
    {
        constexpr int CG = NT / DK;   // thread groups per key channel
        constexpr int RPT = C / CG;   // rows per thread
        const int c = tid % DK, grp = tid / DK;
        float akt[RPT], aqa[RPT], aw[RPT];
#pragma unroll
        for (int rr = 0; rr < RPT; ++rr) akt[rr] = aqa[rr] = aw[rr] = 0.f;
        float rsum = 0.f;
        for (int jb = 0; jb < DV; jb += JB) {
            __syncthreads();  // the previous tile is consumed (and step 1 is complete)
            for (int e = tid; e < DK * JB; e += NT) {
                const int c2 = e / JB, j = e % JB;
                sm.Sin[c2][j] = Sg[(int64_t)c2 * DV + jb + j];
                sm.dSo[c2][j] = dSg[(int64_t)c2 * DV + jb + j];
            }
            __syncthreads();
#pragma unroll 4
            for (int j = 0; j < JB; ++j) {
                const float s = sm.Sin[c][j], d = sm.dSo[c][j];
                rsum += s * d;
#pragma unroll
                for (int rr = 0; rr < RPT; ++rr) {
                    const int r = grp * RPT + rr;
                    akt[rr] += sm.U[r][jb + j] * d;
                    aqa[rr] += sm.dO[r][jb + j] * s;
                    aw[rr] -= sm.dU[r][jb + j] * s;
                }
            }
        }
#pragma unroll
        for (int rr = 0; rr < RPT; ++rr) {
            const int r = grp * RPT + rr;
            sm.dKt[r][c] = akt[rr];
            sm.dQa[r][c] = aqa[rr];
            sm.dW[r][c] = aw[rr];
        }
        if (grp == 0) {
            sm.rs[c] = rsum;
            sm.GL[c] = sm.G[len - 1][c];
        }
    }
    __syncthreads();

    // 3. 16 x 16 products: M = KG KI^T, dP = tril(dO U^T), A = tril_strict(diag(b) M) (in X);
    //    colsum(dKt Kt) per key channel
    {
        const int r = tid / C, i = tid % C;
        float m = 0.f;
#pragma unroll 8
        for (int c = 0; c < DK; ++c) m += sm.KG[r][c] * sm.KI[i][c];
        float dp = 0.f;
        if (i <= r) {
#pragma unroll 8
            for (int j = 0; j < DV; ++j) dp += sm.dO[r][j] * sm.U[i][j];
        }
        sm.M[r][i] = m;
        sm.dP[r][i] = dp;
        sm.X[r][i] = (i < r) ? sm.beta[r] * m : 0.f;
    }
    for (int c = tid; c < DK; c += NT) {
        float acc = 0.f;
        for (int i = 0; i < len; ++i) acc += sm.dKt[i][c] * sm.K[i][c] * expf(sm.GL[c] - sm.G[i][c]);
        sm.ktsum[c] = acc;
    }
    __syncthreads();

    // 4. T = (I + A)^-1 by forward substitution, one thread per column
    if (tid < C) {
        const int j = tid;
        float col[C];
#pragma unroll
        for (int r = 0; r < C; ++r) {
            float t = (r == j) ? 1.f : 0.f;
            if (r > j) {
                for (int i = j; i < r; ++i) t -= sm.X[r][i] * col[i];
            }
            col[r] = t;
        }
#pragma unroll
        for (int r = 0; r < C; ++r) sm.T[r][j] = col[r];
    }
    __syncthreads();

    // 5. dT = dU (diag(b) V)^T + dW (diag(b) KG)^T
    {
        const int r = tid / C, i = tid % C;
        float acc = 0.f;
#pragma unroll 8
        for (int j = 0; j < DV; ++j) acc += sm.dU[r][j] * sm.V[i][j];
#pragma unroll 8
        for (int c = 0; c < DK; ++c) acc += sm.dW[r][c] * sm.KG[i][c];
        sm.dTn[r][i] = sm.beta[i] * acc;
    }
    __syncthreads();
    // 6. dA = -tril_strict(T^T dT T^T)
    {
        const int r = tid / C, i = tid % C;
        float acc = 0.f;
#pragma unroll
        for (int s = 0; s < C; ++s) acc += sm.T[s][r] * sm.dTn[s][i];
        sm.X[r][i] = acc;
    }
    __syncthreads();
    {
        const int r = tid / C, i = tid % C;
        float acc = 0.f;
#pragma unroll
        for (int s = 0; s < C; ++s) acc += sm.X[r][s] * sm.T[i][s];
        sm.dA[r][i] = (i < r) ? -acc : 0.f;
    }
    // 7. T^T dU and T^T dW
    for (int e = tid; e < C * DV; e += NT) {
        const int r = e / DV, j = e % DV;
        float acc = 0.f;
#pragma unroll
        for (int s = 0; s < C; ++s) acc += sm.T[s][r] * sm.dU[s][j];
        sm.TdU[r][j] = acc;
    }
    for (int e = tid; e < C * DK; e += NT) {
        const int r = e / DK, c = e % DK;
        float acc = 0.f;
#pragma unroll
        for (int s = 0; s < C; ++s) acc += sm.T[s][r] * sm.dW[s][c];
        sm.TdW[r][c] = acc;
    }
    __syncthreads();

    // 8. dq, dk and dG per element
    TIO* dqp = static_cast<TIO*>(b.dq);
    TIO* dkp = static_cast<TIO*>(b.dk);
    for (int e = tid; e < C * DK; e += NT) {
        const int r = e / DK, c = e % DK;
        if (r >= len) continue;
        const float br = sm.beta[r];
        float t = 0.f;
        for (int i = 0; i < r; ++i) t += sm.dA[r][i] * sm.KI[i][c];
        const float dKG = br * (sm.TdW[r][c] + t);
        float dKI = 0.f;
        for (int s = r + 1; s < len; ++s) dKI += sm.beta[s] * sm.dA[s][r] * sm.KG[s][c];
        for (int s = r; s < len; ++s) dKI += sm.dP[s][r] * sm.QG[s][c];
        float dQG = sm.dQa[r][c];
        for (int i = 0; i <= r; ++i) dQG += sm.dP[r][i] * sm.KI[i][c];
        const float dKt = sm.dKt[r][c];
        const float g = sm.G[r][c];
        const float ekt = expf(sm.GL[c] - g);
        const float k = sm.K[r][c];
        const int64_t idx = ((t0 + r) * H + h) * (int64_t)DK + c;
        st_io(dkp, idx, dKG * sm.EG[r][c] + dKI * expf(-g) + dKt * ekt);
        st_io(dqp, idx, dQG * sm.EG[r][c]);
        float dG = dKG * sm.KG[r][c] + dQG * sm.QG[r][c] - dKI * sm.KI[r][c] - dKt * k * ekt;
        if (r == len - 1) dG += sm.ktsum[c] + expf(sm.GL[c]) * sm.rs[c];
        sm.dW[r][c] = dG;  // dW is no longer read (steps 5 and 7 are done)
    }
    // 9. dv and dbeta
    TIO* dvp = static_cast<TIO*>(b.dv);
    for (int e = tid; e < C * DV; e += NT) {
        const int r = e / DV, j = e % DV;
        if (r < len) st_io(dvp, ((t0 + r) * H + h) * (int64_t)DV + j, sm.beta[r] * sm.TdU[r][j]);
    }
    {
        const int w = tid >> 5, lane = tid & 31;
        for (int r = w; r < len; r += NT / 32) {
            float acc = 0.f;
            for (int j = lane; j < DV; j += 32) acc += sm.TdU[r][j] * sm.V[r][j];
            for (int c = lane; c < DK; c += 32) acc += sm.TdW[r][c] * sm.KG[r][c];
            if (lane < C) acc += sm.dA[r][lane] * sm.M[r][lane];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) b.dbeta[(t0 + r) * H + h] = acc;
        }
    }
    __syncthreads();

    // 10. dg (reversed in-chunk cumulative sum of dG), the gate's chain rule, dz and dA's share
    TIO* dzp = static_cast<TIO*>(b.dz);
    const float expA = expf(a.A[h]);
    float da = 0.f;
    for (int c = tid; c < DK; c += NT) {
        float dg = 0.f;
        for (int r = len - 1; r >= 0; --r) {
            dg += sm.dW[r][c];
            const int64_t idx = ((t0 + r) * H + h) * (int64_t)DK + c;
            const float x = expA * ld_io(zp, idx);
            const float dx = dg * a.g_min * sigmoid_slope(x);
            st_io(dzp, idx, dx * expA);
            da += dx * x;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) da += __shfl_xor_sync(0xffffffffu, da, o);
    if ((tid & 31) == 0) sm.red[tid >> 5] = da;
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) s += sm.red[w];
        b.dA_part[slot * H + h] = s;
    }
}

// ---------------------------------------------------------------- dA from the chunks' shares

__global__ void __launch_bounds__(NT) kda_bwd_da_kernel(BackwardArgs b)
{
    __shared__ float red[NT / 32];
    const int h = blockIdx.x;
    const int tid = threadIdx.x;
    float s = 0.f;
    for (int64_t i = tid; i < b.slots; i += NT) s += b.dA_part[i * b.f.H + h];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((tid & 31) == 0) red[tid >> 5] = s;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) t += red[w];
        b.dA[h] = t;
    }
}

// ---------------------------------------------------------------- launch

namespace {

template <typename K>
cudaError_t set_smem(K kern, size_t bytes)
{
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename TIO, int DK, int DV>
cudaError_t launch_backward_t(const BackwardArgs& b, cudaStream_t s)
{
    const PrefillArgs& a = b.f;
    const dim3 chunk_grid((unsigned)((int64_t)a.N * a.chunks_per_seq), (unsigned)a.H);
    cudaError_t e = cudaSuccess;
    if (a.chunks_per_seq > 0) {
        prof_start("kda_gate", s);
        e = launch_gate(a, std::is_same<TIO, float>::value ? KDA_F32 : KDA_BF16, s);
        prof_stop(s);
        if (e != cudaSuccess) return e;
        prof_start("kda_ut_wy", s);
        e = launch_ut_wy(a, std::is_same<TIO, float>::value ? KDA_F32 : KDA_BF16, s);
        prof_stop(s);
        if (e != cudaSuccess) return e;
        prof_start("kda_bwd_gram", s);
        kda_bwd_gram_kernel<TIO, DK><<<chunk_grid, NT, 0, s>>>(b);
        prof_stop(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // value-column slices of the state passes: 32 columns, or 16 when that is needed to give every
    // SM a chain
    const int64_t chains32 = (int64_t)a.N * a.H * (DV >= 32 ? DV / 32 : 1);
    const bool narrow = DV >= 32 && chains32 < sm_count_of_current_device();
    if (a.chunks_per_seq > 0) {
        if (narrow) {
            constexpr int JS = 16;
            const size_t smem = sizeof(StatesSmem<DK, JS>);
            auto kern = kda_bwd_states_kernel<TIO, DK, DV, JS>;
            if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
            prof_start("kda_bwd_states", s);
            kern<<<dim3((unsigned)a.N, (unsigned)a.H, DV / JS), NT, smem, s>>>(b);
            prof_stop(s);
        } else {
            constexpr int JS = DV < 32 ? DV : 32;
            const size_t smem = sizeof(StatesSmem<DK, JS>);
            auto kern = kda_bwd_states_kernel<TIO, DK, DV, JS>;
            if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
            prof_start("kda_bwd_states", s);
            kern<<<dim3((unsigned)a.N, (unsigned)a.H, DV / JS), NT, smem, s>>>(b);
            prof_stop(s);
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // the reverse pass also runs for empty sequences (dS0 = dS_final)
    if (narrow) {
        constexpr int JS = 16;
        const size_t smem = sizeof(DStatesSmem<DK, JS>);
        auto kern = kda_bwd_dstates_kernel<TIO, DK, DV, JS>;
        if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
        prof_start("kda_bwd_dstates", s);
        kern<<<dim3((unsigned)a.N, (unsigned)a.H, DV / JS), NT, smem, s>>>(b);
        prof_stop(s);
    } else {
        constexpr int JS = DV < 32 ? DV : 32;
        const size_t smem = sizeof(DStatesSmem<DK, JS>);
        auto kern = kda_bwd_dstates_kernel<TIO, DK, DV, JS>;
        if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
        prof_start("kda_bwd_dstates", s);
        kern<<<dim3((unsigned)a.N, (unsigned)a.H, DV / JS), NT, smem, s>>>(b);
        prof_stop(s);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (a.chunks_per_seq > 0) {
        const size_t smem = sizeof(ChunkGradSmem<DK, DV>);
        auto kern = kda_bwd_chunk_kernel<TIO, DK, DV>;
        if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
        prof_start("kda_bwd_chunk", s);
        kern<<<chunk_grid, NT, smem, s>>>(b);
        prof_stop(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    prof_start("kda_bwd_da", s);
    kda_bwd_da_kernel<<<(unsigned)a.H, NT, 0, s>>>(b);
    prof_stop(s);
    return cudaGetLastError();
}

template <typename TIO>
cudaError_t launch_backward_io(const BackwardArgs& b, cudaStream_t s)
{
#define KDA_BWD_CASE(DKv, DVv) \
    if (b.f.dk == DKv && b.f.dv == DVv) return launch_backward_t<TIO, DKv, DVv>(b, s);
    KDA_BWD_CASE(32, 32) KDA_BWD_CASE(32, 64) KDA_BWD_CASE(32, 128)
    KDA_BWD_CASE(64, 32) KDA_BWD_CASE(64, 64) KDA_BWD_CASE(64, 128)
    KDA_BWD_CASE(128, 32) KDA_BWD_CASE(128, 64) KDA_BWD_CASE(128, 128)
#undef KDA_BWD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_backward(const BackwardArgs& b, kda_dtype_t dt, cudaStream_t s)
{
    return dt == KDA_BF16 ? launch_backward_io<__nv_bfloat16>(b, s) : launch_backward_io<float>(b, s);
}

}  // namespace kda
