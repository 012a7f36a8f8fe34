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
//   kda_bwd_gram    per (chunk, head): P = tril(QG KI^T), and QG, Kt for the walks
//   kda_bwd_states  per (sequence, head, value-column slice), one launch, two independent walks:
//                   chunks in order for the state entering every chunk and U = U~ - W S; chunks
//                   in reverse for the gradient reaching every chunk's end state, dU, and dS0
//   kda_bwd_chunk   per (chunk, head): every input gradient and the chunk's share of dA
//   kda_bwd_da      per head: dA from the chunks' shares (fixed order, deterministic)
// Value columns are independent in both state passes (column j of S and dS only meets column j of
// V, U, dO and dU), which is what the slices use.
#include <algorithm>
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
        const int64_t idx = ((t0 + r) * a.H + h) * (int64_t)DK + c;
        if (r < len) {
            q = ld_io(qp, idx);
            k = ld_io(kp, idx);
            g = a.G[idx];
        }
        const float qg = q * expf(g);
        QG[r][c] = qg;
        KI[r][c] = k * expf(-g);
        if (r < len) {
            // Q Gamma and K Gamma_C / Gamma for the sequential state walks
            const float gl = a.G[((t0 + len - 1) * a.H + h) * (int64_t)DK + c];
            b.QG[idx] = qg;
            b.Kt[idx] = k * expf(gl - g);
        }
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

// ---------------------------------------------------------------- state passes (shared pieces)
//
// Both walks visit one (sequence, head, value-column slice) chunk by chunk.  The slice of the state
// lives in shared memory transposed, St[j][c] (rows padded to keep 16-byte alignment), so that both
// products of a chunk read their operands as float4 along the key channels.  The rows of the next
// two chunks travel into a three-slot ring by asynchronous 16-byte copies while the current chunk
// computes (rows past the sequence end are zero-filled by the copies themselves; every iteration
// commits one copy group, empty near the end, so that "all but the newest group" is always the
// current chunk).

__device__ __forceinline__ void cp_async16_zfill(void* smem_dst, const void* gmem_src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gmem_src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gmem_src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// every copy group but the most recent one has landed
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

constexpr int kBufs = 3;  // chunks in shared memory: the current one and two in flight

// Copy `rows` rows of `bytes_per_row` bytes (a multiple of 16) of a chunk into dst (row pitch
// `pitch` bytes); row r of the chunk starts at src + r * src_stride bytes; rows r >= len are zeroed.
__device__ __forceinline__ void copy_rows(unsigned char* dst, int pitch, const unsigned char* src, int64_t src_stride,
                                          int rows, int bytes_per_row, int len, int tid)
{
    const int per = bytes_per_row / 16;
    for (int e = tid; e < rows * per; e += NT) {
        const int r = e / per, c = e - r * per;
        const bool ok = r < len;
        cp_async16_zfill(dst + r * pitch + c * 16, ok ? src + r * src_stride + c * 16 : src, ok);
    }
}

template <typename T>
__device__ __forceinline__ float to_f(T x) { return static_cast<float>(x); }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// ---------------------------------------------------------------- forward state pass (states kept)

template <int DK, int JS>
struct StatesSmem {
    static constexpr int SP = DK + 4;  // padded row of the transposed state
    float St[JS][SP];                  // state slice, transposed: St[j][c] = S[c][j0 + j]
    float K[kBufs][C][DK];             // K e^(G_C - G), ring of chunks
    float W[kBufs][C][DK];
    float Ut[kBufs][C][JS];            // U~ slice
    float GL[kBufs][DK];               // G of the chunk's last token
    float U[C][JS];
    float eGL[DK];                     // e^(G_C)
};

template <typename TIO, int DK, int DV, int JS>
__device__ __forceinline__ void bwd_states(const BackwardArgs& b, unsigned char* smem_raw, int slice)
{
    using Sm = StatesSmem<DK, JS>;
    const PrefillArgs& a = b.f;
    Sm& sm = *reinterpret_cast<Sm*>(smem_raw);
    const int n = blockIdx.x;
    const int h = blockIdx.y;
    const int j0 = slice * JS;
    const int tid = threadIdx.x;
    const int H = a.H;
    int64_t s0, s1;
    if (!seq_range(a, n, s0, s1)) return;
    const int64_t sbase = ((int64_t)n * H + h) * DK * DV;
    for (int e = tid; e < DK * JS; e += NT) {
        const int c = e / JS, j = e % JS;
        sm.St[j][c] = a.s0 ? a.s0[sbase + (int64_t)c * DV + j0 + j] : 0.f;
    }
    constexpr int NU = (C * JS + NT - 1) / NT;       // U entries per thread
    constexpr int NS = (JS * DK / 4 + NT - 1) / NT;  // (j, 4 channels) state items per thread
    const int64_t rowk = (int64_t)H * DK * 4, rowv = (int64_t)H * DV * 4;  // bytes between token rows
    auto fetch = [&](int buf, int64_t t0, int len) {
        const int64_t base = (t0 * H + h);
        copy_rows(reinterpret_cast<unsigned char*>(sm.K[buf]), DK * 4,
                  reinterpret_cast<const unsigned char*>(b.Kt + base * DK), rowk, C, DK * 4, len, tid);
        copy_rows(reinterpret_cast<unsigned char*>(sm.W[buf]), DK * 4,
                  reinterpret_cast<const unsigned char*>(a.W + base * DK), rowk, C, DK * 4, len, tid);
        copy_rows(reinterpret_cast<unsigned char*>(sm.Ut[buf]), JS * 4,
                  reinterpret_cast<const unsigned char*>(a.Ut + base * DV + j0), rowv, C, JS * 4, len, tid);
        copy_rows(reinterpret_cast<unsigned char*>(sm.GL[buf]), DK * 4,
                  reinterpret_cast<const unsigned char*>(a.G + ((t0 + len - 1) * H + h) * DK), 0, 1, DK * 4, 1, tid);
        cp_async_commit();
    };
    auto fetch_chunk = [&](int64_t c) {  // chunk c into its ring slot (an empty group past the end)
        const int64_t t = s0 + c * C;
        if (t < s1) fetch((int)(c % kBufs), t, (int)min((int64_t)C, s1 - t));
        else cp_async_commit();
    };
    fetch_chunk(0);
    fetch_chunk(1);
    for (int64_t ci = 0; s0 + ci * C < s1; ++ci) {
        const int64_t t0 = s0 + ci * C;
        const int len = (int)min((int64_t)C, s1 - t0);
        const int buf = (int)(ci % kBufs);
        cp_async_wait_prev();
        __syncthreads();  // this chunk's rows have landed; the previous chunk's update is complete
        fetch_chunk(ci + 2);
        if (tid < DK) sm.eGL[tid] = expf(sm.GL[buf][tid]);
        float* dst = b.S_chunk + (chunk_slot(n, s0, ci) * H + h) * (int64_t)DK * DV + j0;
        for (int e = tid; e < DK * JS; e += NT) {
            const int c = e / JS, j = e % JS;
            dst[(int64_t)c * DV + j] = sm.St[j][c];
        }
        // U = U~ - W S (four accumulators along the key channels)
        float uacc[NU];
#pragma unroll
        for (int q = 0; q < NU; ++q) {
            const int e = tid + q * NT;
            uacc[q] = 0.f;
            if (e < C * JS) {
                const int r = e / JS, j = e % JS;
                float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll 8
                for (int c = 0; c < DK; c += 4) {
                    const float4 w = *reinterpret_cast<const float4*>(&sm.W[buf][r][c]);
                    const float4 x = *reinterpret_cast<const float4*>(&sm.St[j][c]);
                    a01 = __ffma2_rn(make_float2(w.x, w.y), make_float2(x.x, x.y), a01);
                    a23 = __ffma2_rn(make_float2(w.z, w.w), make_float2(x.z, x.w), a23);
                }
                uacc[q] = r < len ? sm.Ut[buf][r][j] - ((a01.x + a01.y) + (a23.x + a23.y)) : 0.f;
            }
        }
#pragma unroll
        for (int q = 0; q < NU; ++q) {
            const int e = tid + q * NT;
            if (e < C * JS) {
                const int r = e / JS, j = e % JS;
                sm.U[r][j] = uacc[q];
                if (r < len) b.U[((t0 + r) * H + h) * (int64_t)DV + j0 + j] = uacc[q];
            }
        }
        __syncthreads();  // U and e^G_C complete; every thread has read the old state
        // S = e^G_C S + Kt^T U, four key channels of one column per item
#pragma unroll
        for (int q = 0; q < NS; ++q) {
            const int e = tid + q * NT;
            if (e < JS * DK / 4) {
                const int j = e / (DK / 4), c = 4 * (e % (DK / 4));
                const float4 g = *reinterpret_cast<const float4*>(&sm.eGL[c]);
                const float4 x = *reinterpret_cast<const float4*>(&sm.St[j][c]);
                float2 x01 = __fmul2_rn(make_float2(g.x, g.y), make_float2(x.x, x.y));
                float2 x23 = __fmul2_rn(make_float2(g.z, g.w), make_float2(x.z, x.w));
#pragma unroll
                for (int i = 0; i < C; ++i) {  // rows past the chunk's end are zero
                    const float u = sm.U[i][j];
                    const float4 kt = *reinterpret_cast<const float4*>(&sm.K[buf][i][c]);
                    x01 = __ffma2_rn(make_float2(kt.x, kt.y), make_float2(u, u), x01);
                    x23 = __ffma2_rn(make_float2(kt.z, kt.w), make_float2(u, u), x23);
                }
                *reinterpret_cast<float4*>(&sm.St[j][c]) = make_float4(x01.x, x01.y, x23.x, x23.y);
            }
        }
    }
}

// ---------------------------------------------------------------- reverse state pass

template <typename TIO, int DK, int JS>
struct DStatesSmem {
    static constexpr int SP = DK + 4;
    float dSt[JS][SP];      // gradient slice, transposed: dSt[j][c] = dS[c][j0 + j]
    float Q[kBufs][C][DK];      // Q e^G, double buffered
    float K[kBufs][C][DK];      // K e^(G_C - G)
    float W[kBufs][C][DK];
    float P[kBufs][C][C];
    TIO dO[kBufs][C][JS];   // raw dO slice
    float GL[kBufs][DK];
    float dU[C][JS];
    float eGL[DK];
};

template <typename TIO, int DK, int DV, int JS>
__device__ __forceinline__ void bwd_dstates(const BackwardArgs& b, unsigned char* smem_raw, int slice)
{
    using Sm = DStatesSmem<TIO, DK, JS>;
    const PrefillArgs& a = b.f;
    Sm& sm = *reinterpret_cast<Sm*>(smem_raw);
    const int n = blockIdx.x;
    const int h = blockIdx.y;
    const int j0 = slice * JS;
    const int tid = threadIdx.x;
    const int H = a.H;
    int64_t s0, s1;
    if (!seq_range(a, n, s0, s1)) return;
    const TIO* dop = static_cast<const TIO*>(b.dout);
    const int64_t sbase = ((int64_t)n * H + h) * DK * DV;
    for (int e = tid; e < DK * JS; e += NT) {
        const int c = e / JS, j = e % JS;
        sm.dSt[j][c] = b.dS_final ? b.dS_final[sbase + (int64_t)c * DV + j0 + j] : 0.f;
    }
    constexpr int NU = (C * JS + NT - 1) / NT;
    constexpr int NS = (JS * DK / 4 + NT - 1) / NT;
    const int64_t rowk = (int64_t)H * DK * 4, rowp = (int64_t)H * C * 4, rowo = (int64_t)H * DV * sizeof(TIO);
    auto fetch = [&](int buf, int64_t t0, int len) {
        const int64_t base = (t0 * H + h);
        copy_rows(reinterpret_cast<unsigned char*>(sm.Q[buf]), DK * 4,
                  reinterpret_cast<const unsigned char*>(b.QG + base * DK), rowk, C, DK * 4, len, tid);
        copy_rows(reinterpret_cast<unsigned char*>(sm.K[buf]), DK * 4,
                  reinterpret_cast<const unsigned char*>(b.Kt + base * DK), rowk, C, DK * 4, len, tid);
        copy_rows(reinterpret_cast<unsigned char*>(sm.W[buf]), DK * 4,
                  reinterpret_cast<const unsigned char*>(a.W + base * DK), rowk, C, DK * 4, len, tid);
        copy_rows(reinterpret_cast<unsigned char*>(sm.P[buf]), C * 4,
                  reinterpret_cast<const unsigned char*>(b.P + base * C), rowp, C, C * 4, len, tid);
        copy_rows(reinterpret_cast<unsigned char*>(sm.dO[buf]), JS * (int)sizeof(TIO),
                  reinterpret_cast<const unsigned char*>(dop + base * DV + j0), rowo, C, JS * (int)sizeof(TIO), len, tid);
        copy_rows(reinterpret_cast<unsigned char*>(sm.GL[buf]), DK * 4,
                  reinterpret_cast<const unsigned char*>(a.G + ((t0 + len - 1) * H + h) * DK), 0, 1, DK * 4, 1, tid);
        cp_async_commit();
    };
    const int64_t nch = (s1 - s0 + C - 1) / C;
    auto chunk_len = [&](int64_t ci) { return (int)min((int64_t)C, s1 - (s0 + ci * C)); };
    // the chunks are visited last first: visit v is chunk nch - 1 - v, in ring slot v mod kBufs
    auto fetch_visit = [&](int64_t vis) {
        const int64_t c = nch - 1 - vis;
        if (c >= 0) fetch((int)(vis % kBufs), s0 + c * C, chunk_len(c));
        else cp_async_commit();
    };
    fetch_visit(0);
    fetch_visit(1);
    for (int64_t vis = 0; vis < nch; ++vis) {
        const int64_t ci = nch - 1 - vis;
        const int64_t t0 = s0 + ci * C;
        const int len = chunk_len(ci);
        const int buf = (int)(vis % kBufs);
        cp_async_wait_prev();
        __syncthreads();  // this chunk's rows have landed; the previous (later) chunk's update is complete
        fetch_visit(vis + 2);
        if (tid < DK) sm.eGL[tid] = expf(sm.GL[buf][tid]);
        float* dst = b.dS_chunk + (chunk_slot(n, s0, ci) * H + h) * (int64_t)DK * DV + j0;
        for (int e = tid; e < DK * JS; e += NT) {
            const int c = e / JS, j = e % JS;
            dst[(int64_t)c * DV + j] = sm.dSt[j][c];
        }
        // dU = Kt dS' + P^T dO
        float uacc[NU];
#pragma unroll
        for (int q = 0; q < NU; ++q) {
            const int e = tid + q * NT;
            uacc[q] = 0.f;
            if (e < C * JS) {
                const int r = e / JS, j = e % JS;
                if (r < len) {
                    float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll 8
                    for (int c = 0; c < DK; c += 4) {
                        const float4 kt = *reinterpret_cast<const float4*>(&sm.K[buf][r][c]);
                        const float4 x = *reinterpret_cast<const float4*>(&sm.dSt[j][c]);
                        a01 = __ffma2_rn(make_float2(kt.x, kt.y), make_float2(x.x, x.y), a01);
                        a23 = __ffma2_rn(make_float2(kt.z, kt.w), make_float2(x.z, x.w), a23);
                    }
                    // P^T dO over the rows i >= r (P is lower triangular and zero past the chunk's end)
                    float pd = 0.f;
#pragma unroll
                    for (int i = 0; i < C; ++i) pd = fmaf(sm.P[buf][i][r], to_f(sm.dO[buf][i][j]), pd);
                    uacc[q] = ((a01.x + a01.y) + (a23.x + a23.y)) + pd;
                }
            }
        }
#pragma unroll
        for (int q = 0; q < NU; ++q) {
            const int e = tid + q * NT;
            if (e < C * JS) {
                const int r = e / JS, j = e % JS;
                sm.dU[r][j] = uacc[q];
                if (r < len) b.dU[((t0 + r) * H + h) * (int64_t)DV + j0 + j] = uacc[q];
            }
        }
        __syncthreads();  // dU and e^G_C complete; every thread has read the old gradient
        // dS = e^G_C dS' + QG^T dO - W^T dU, four key channels of one column per item
#pragma unroll
        for (int q = 0; q < NS; ++q) {
            const int e = tid + q * NT;
            if (e < JS * DK / 4) {
                const int j = e / (DK / 4), c = 4 * (e % (DK / 4));
                const float4 g = *reinterpret_cast<const float4*>(&sm.eGL[c]);
                const float4 x = *reinterpret_cast<const float4*>(&sm.dSt[j][c]);
                float2 x01 = __fmul2_rn(make_float2(g.x, g.y), make_float2(x.x, x.y));
                float2 x23 = __fmul2_rn(make_float2(g.z, g.w), make_float2(x.z, x.w));
#pragma unroll
                for (int r = 0; r < C; ++r) {  // rows past the chunk's end are zero
                    const float o = to_f(sm.dO[buf][r][j]), mdu = -sm.dU[r][j];
                    const float4 qg = *reinterpret_cast<const float4*>(&sm.Q[buf][r][c]);
                    const float4 w = *reinterpret_cast<const float4*>(&sm.W[buf][r][c]);
                    x01 = __ffma2_rn(make_float2(qg.x, qg.y), make_float2(o, o),
                                     __ffma2_rn(make_float2(w.x, w.y), make_float2(mdu, mdu), x01));
                    x23 = __ffma2_rn(make_float2(qg.z, qg.w), make_float2(o, o),
                                     __ffma2_rn(make_float2(w.z, w.w), make_float2(mdu, mdu), x23));
                }
                *reinterpret_cast<float4*>(&sm.dSt[j][c]) = make_float4(x01.x, x01.y, x23.x, x23.y);
            }
        }
    }
    __syncthreads();
    if (b.dS0) {
        for (int e = tid; e < DK * JS; e += NT) {
            const int c = e / JS, j = e % JS;
            b.dS0[sbase + (int64_t)c * DV + j0 + j] = sm.dSt[j][c];
        }
    }
}

// The two state passes do not depend on each other (the reverse pass needs no forward state), so
// one launch runs both: CTAs with blockIdx.z < DV / JS walk forward, the others backward.  States
// from the forward pass are needed only by the per-chunk kernel that follows.
template <typename TIO, int DK, int DV, int JS>
__global__ void __launch_bounds__(NT) kda_bwd_states_kernel(BackwardArgs b, int with_forward)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int NSL = DV / JS;
    const int z = (int)blockIdx.z;
    if (with_forward && z < NSL) {
        bwd_states<TIO, DK, DV, JS>(b, smem_raw, z);
    } else {
        bwd_dstates<TIO, DK, DV, JS>(b, smem_raw, with_forward ? z - NSL : z);
    }
}

// ---------------------------------------------------------------- per-chunk gradients

// Rows of the [16][d] tiles are padded by four floats: rows stay 16-byte aligned for float4 reads
// along a row, and the 16 rows of one column fall on 8 distinct banks (the 16 x 16 products read
// columns of 16 rows at once).
template <int DK, int DV>
struct ChunkGradSmem {
    static constexpr int JB = DV < 32 ? DV : 32;  // value columns per staged state tile
    static constexpr int PK = DK + 4, PV = DV + 4;
    float K[C][PK];
    float G[C][PK];
    float KG[C][PK];
    float KI[C][PK];
    float QG[C][PK];
    float dKt[C][PK];  // U dS'^T, later dG
    float dQa[C][PK];  // dO S^T
    float dW[C][PK];   // -dU S^T, later T^T dW
    float V[C][PV];
    float dO[C][PV];
    float U[C][PV];
    float dU[C][PV];   // later T^T dU
    float Sin[2][DK][JB + 1];  // double-buffered state tiles (odd pitch: no bank conflicts)
    float dSo[2][DK][JB + 1];
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
    constexpr int NTILE = DV / JB;
    // state tile t (value columns t JB .. t JB + JB - 1) into slot t & 1 by asynchronous 4-byte copies
    auto issue_tile = [&](int t) {
        if (t < NTILE) {
            const int jb = t * JB;
            for (int e = tid; e < DK * JB; e += NT) {
                const int c2 = e / JB, j = e % JB;
                cp_async4(&sm.Sin[t & 1][c2][j], Sg + (int64_t)c2 * DV + jb + j);
                cp_async4(&sm.dSo[t & 1][c2][j], dSg + (int64_t)c2 * DV + jb + j);
            }
        }
        cp_async_commit();
    };
    issue_tile(0);  // in flight while the chunk's rows are read

    // 1. the chunk's rows (absent tokens as zeros); the loops are unrolled so that every load of a
    //    thread is in flight at once
    static_assert((C * DK) % NT == 0 && (C * DV) % NT == 0, "whole rows per pass");
#pragma unroll
    for (int pass = 0; pass < C * DK / NT; ++pass) {
        const int e = tid + pass * NT;
        const int r = e / DK, c = e % DK;
        float q = 0.f, k = 0.f, g = 0.f;
        if (r < len) {
            const int64_t idx = ((t0 + r) * H + h) * (int64_t)DK + c;
            q = ld_io(qp, idx);
            k = ld_io(kp, idx);
            g = a.G[idx];
        }
        const float eg = expf(g);
        sm.K[r][c] = k;
        sm.G[r][c] = g;
        sm.KG[r][c] = k * eg;
        sm.KI[r][c] = k * expf(-g);
        sm.QG[r][c] = q * eg;
    }
#pragma unroll
    for (int pass = 0; pass < C * DV / NT; ++pass) {
        const int e = tid + pass * NT;
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
        constexpr int RP = RPT / 2;   // row pairs per thread (packed fp32 arithmetic on a pair)
        const int c = tid % DK, grp = tid / DK;
        float2 akt[RP], aqa[RP], aw[RP];
#pragma unroll
        for (int rp = 0; rp < RP; ++rp) akt[rp] = aqa[rp] = aw[rp] = make_float2(0.f, 0.f);
        float rsum = 0.f;
        for (int t = 0; t < NTILE; ++t) {
            const int jb = t * JB, sl = t & 1;
            issue_tile(t + 1);  // its slot was consumed before the previous iteration's last barrier
            cp_async_wait_prev();
            __syncthreads();    // tile t has landed (and step 1 is complete)
#pragma unroll 2
            for (int j = 0; j < JB; j += 4) {
                float sv[4], dv[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    sv[q] = sm.Sin[sl][c][j + q];
                    dv[q] = sm.dSo[sl][c][j + q];
                    rsum = fmaf(sv[q], dv[q], rsum);
                }
#pragma unroll
                for (int rp = 0; rp < RP; ++rp) {
                    const int r = grp * RPT + 2 * rp;
                    const float4 u0 = *reinterpret_cast<const float4*>(&sm.U[r][jb + j]);
                    const float4 u1 = *reinterpret_cast<const float4*>(&sm.U[r + 1][jb + j]);
                    const float4 o0 = *reinterpret_cast<const float4*>(&sm.dO[r][jb + j]);
                    const float4 o1 = *reinterpret_cast<const float4*>(&sm.dO[r + 1][jb + j]);
                    const float4 d0 = *reinterpret_cast<const float4*>(&sm.dU[r][jb + j]);
                    const float4 d1 = *reinterpret_cast<const float4*>(&sm.dU[r + 1][jb + j]);
                    akt[rp] = __ffma2_rn(make_float2(u0.x, u1.x), make_float2(dv[0], dv[0]), akt[rp]);
                    akt[rp] = __ffma2_rn(make_float2(u0.y, u1.y), make_float2(dv[1], dv[1]), akt[rp]);
                    akt[rp] = __ffma2_rn(make_float2(u0.z, u1.z), make_float2(dv[2], dv[2]), akt[rp]);
                    akt[rp] = __ffma2_rn(make_float2(u0.w, u1.w), make_float2(dv[3], dv[3]), akt[rp]);
                    aqa[rp] = __ffma2_rn(make_float2(o0.x, o1.x), make_float2(sv[0], sv[0]), aqa[rp]);
                    aqa[rp] = __ffma2_rn(make_float2(o0.y, o1.y), make_float2(sv[1], sv[1]), aqa[rp]);
                    aqa[rp] = __ffma2_rn(make_float2(o0.z, o1.z), make_float2(sv[2], sv[2]), aqa[rp]);
                    aqa[rp] = __ffma2_rn(make_float2(o0.w, o1.w), make_float2(sv[3], sv[3]), aqa[rp]);
                    aw[rp] = __ffma2_rn(make_float2(-d0.x, -d1.x), make_float2(sv[0], sv[0]), aw[rp]);
                    aw[rp] = __ffma2_rn(make_float2(-d0.y, -d1.y), make_float2(sv[1], sv[1]), aw[rp]);
                    aw[rp] = __ffma2_rn(make_float2(-d0.z, -d1.z), make_float2(sv[2], sv[2]), aw[rp]);
                    aw[rp] = __ffma2_rn(make_float2(-d0.w, -d1.w), make_float2(sv[3], sv[3]), aw[rp]);
                }
            }
            __syncthreads();  // tile t is consumed: its slot can take tile t + 2
        }
#pragma unroll
        for (int rp = 0; rp < RP; ++rp) {
            const int r = grp * RPT + 2 * rp;
            sm.dKt[r][c] = akt[rp].x;
            sm.dKt[r + 1][c] = akt[rp].y;
            sm.dQa[r][c] = aqa[rp].x;
            sm.dQa[r + 1][c] = aqa[rp].y;
            sm.dW[r][c] = aw[rp].x;
            sm.dW[r + 1][c] = aw[rp].y;
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
        float2 m2 = make_float2(0.f, 0.f);
#pragma unroll 8
        for (int c = 0; c < DK; c += 2)
            m2 = __ffma2_rn(*reinterpret_cast<const float2*>(&sm.KG[r][c]), *reinterpret_cast<const float2*>(&sm.KI[i][c]),
                            m2);
        float2 dp2 = make_float2(0.f, 0.f);
        if (i <= r) {
#pragma unroll 8
            for (int j = 0; j < DV; j += 2)
                dp2 = __ffma2_rn(*reinterpret_cast<const float2*>(&sm.dO[r][j]), *reinterpret_cast<const float2*>(&sm.U[i][j]),
                                 dp2);
        }
        const float m = m2.x + m2.y;
        sm.M[r][i] = m;
        sm.dP[r][i] = dp2.x + dp2.y;
        sm.X[r][i] = (i < r) ? sm.beta[r] * m : 0.f;
    }
    for (int c = tid; c < DK; c += NT) {
        float acc = 0.f;
        for (int i = 0; i < len; ++i) acc += sm.dKt[i][c] * sm.K[i][c] * expf(sm.GL[c] - sm.G[i][c]);
        sm.ktsum[c] = acc;
    }
    __syncthreads();

    // 4. T = (I + A)^-1 by column-oriented forward substitution, one lane per column
    if (tid < C) {
        const int j = tid;
        float col[C];
#pragma unroll
        for (int r = 0; r < C; ++r) col[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
        for (int i = 0; i < C; ++i) {
            const float ti = col[i];
#pragma unroll
            for (int r = i + 1; r < C; ++r) col[r] = fmaf(-sm.X[r][i], ti, col[r]);
        }
#pragma unroll
        for (int r = 0; r < C; ++r) sm.T[r][j] = col[r];
    }
    __syncthreads();

    // 5. dT = dU (diag(b) V)^T + dW (diag(b) KG)^T
    {
        const int r = tid / C, i = tid % C;
        float2 a2 = make_float2(0.f, 0.f);
#pragma unroll 8
        for (int j = 0; j < DV; j += 2)
            a2 = __ffma2_rn(*reinterpret_cast<const float2*>(&sm.dU[r][j]), *reinterpret_cast<const float2*>(&sm.V[i][j]), a2);
#pragma unroll 8
        for (int c = 0; c < DK; c += 2)
            a2 = __ffma2_rn(*reinterpret_cast<const float2*>(&sm.dW[r][c]), *reinterpret_cast<const float2*>(&sm.KG[i][c]), a2);
        sm.dTn[r][i] = sm.beta[i] * (a2.x + a2.y);
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
    // 7. T^T dU and T^T dW, in place of dU and dW once every thread has its values
    constexpr int NTU = (C * DV + NT - 1) / NT, NTW = (C * DK + NT - 1) / NT;
    float tdu[NTU], tdw[NTW];
#pragma unroll
    for (int q = 0; q < NTU; ++q) {
        const int e = tid + q * NT;
        const int r = e / DV, j = e % DV;
        float acc = 0.f;
#pragma unroll
        for (int s = 0; s < C; ++s) acc = fmaf(sm.T[s][r], sm.dU[s][j], acc);
        tdu[q] = acc;
    }
#pragma unroll
    for (int q = 0; q < NTW; ++q) {
        const int e = tid + q * NT;
        const int r = e / DK, c = e % DK;
        float acc = 0.f;
#pragma unroll
        for (int s = 0; s < C; ++s) acc = fmaf(sm.T[s][r], sm.dW[s][c], acc);
        tdw[q] = acc;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < NTU; ++q) {
        const int e = tid + q * NT;
        sm.dU[e / DV][e % DV] = tdu[q];
    }
#pragma unroll
    for (int q = 0; q < NTW; ++q) {
        const int e = tid + q * NT;
        sm.dW[e / DK][e % DK] = tdw[q];
    }
    __syncthreads();

    // 8. dq, dk and dG per element (dG into dKt's place: each entry is read only by its own thread)
    TIO* dqp = static_cast<TIO*>(b.dq);
    TIO* dkp = static_cast<TIO*>(b.dk);
    for (int e = tid; e < C * DK; e += NT) {
        const int r = e / DK, c = e % DK;
        if (r >= len) continue;
        const float br = sm.beta[r];
        float t = 0.f;
        for (int i = 0; i < r; ++i) t = fmaf(sm.dA[r][i], sm.KI[i][c], t);
        const float dKG = br * (sm.dW[r][c] + t);
        float dKI = 0.f;
        for (int s = r + 1; s < len; ++s) dKI = fmaf(sm.beta[s] * sm.dA[s][r], sm.KG[s][c], dKI);
        for (int s = r; s < len; ++s) dKI = fmaf(sm.dP[s][r], sm.QG[s][c], dKI);
        float dQG = sm.dQa[r][c];
        for (int i = 0; i <= r; ++i) dQG = fmaf(sm.dP[r][i], sm.KI[i][c], dQG);
        const float dKt = sm.dKt[r][c];
        const float g = sm.G[r][c];
        const float eg = expf(g);
        const float ekt = expf(sm.GL[c] - g);
        const float k = sm.K[r][c];
        const int64_t idx = ((t0 + r) * H + h) * (int64_t)DK + c;
        st_io(dkp, idx, dKG * eg + dKI * expf(-g) + dKt * ekt);
        st_io(dqp, idx, dQG * eg);
        float dG = dKG * sm.KG[r][c] + dQG * sm.QG[r][c] - dKI * sm.KI[r][c] - dKt * k * ekt;
        if (r == len - 1) dG += sm.ktsum[c] + expf(sm.GL[c]) * sm.rs[c];
        sm.dKt[r][c] = dG;
    }
    // 9. dv and dbeta (T^T dU now in dU, T^T dW in dW)
    TIO* dvp = static_cast<TIO*>(b.dv);
    for (int e = tid; e < C * DV; e += NT) {
        const int r = e / DV, j = e % DV;
        if (r < len) st_io(dvp, ((t0 + r) * H + h) * (int64_t)DV + j, sm.beta[r] * sm.dU[r][j]);
    }
    {
        const int w = tid >> 5, lane = tid & 31;
        for (int r = w; r < len; r += NT / 32) {
            float acc = 0.f;
            for (int j = lane; j < DV; j += 32) acc = fmaf(sm.dU[r][j], sm.V[r][j], acc);
            for (int c = lane; c < DK; c += 32) acc = fmaf(sm.dW[r][c], sm.KG[r][c], acc);
            if (lane < C) acc = fmaf(sm.dA[r][lane], sm.M[r][lane], acc);
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
        float zr[C];  // the channel's z over the chunk, every load in flight at once
#pragma unroll
        for (int r = 0; r < C; ++r) zr[r] = r < len ? ld_io(zp, ((t0 + r) * H + h) * (int64_t)DK + c) : 0.f;
        float dg = 0.f;
#pragma unroll
        for (int r = C - 1; r >= 0; --r) {
            if (r >= len) continue;
            dg += sm.dKt[r][c];
            const int64_t idx = ((t0 + r) * H + h) * (int64_t)DK + c;
            const float x = expA * zr[r];
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
    // SM a chain; the forward pass is skipped when no sequence has a token (the reverse pass still
    // writes dS0 = dS_final)
    const int64_t chains32 = 2 * (int64_t)a.N * a.H * (DV >= 32 ? DV / 32 : 1);
    const bool narrow = DV >= 32 && chains32 < sm_count_of_current_device();
    const int with_forward = a.chunks_per_seq > 0 ? 1 : 0;
    auto launch_states = [&](auto kern, size_t smem, int nsl) -> cudaError_t {
        cudaError_t err = set_smem(kern, smem);
        if (err != cudaSuccess) return err;
        prof_start("kda_bwd_states", s);
        kern<<<dim3((unsigned)a.N, (unsigned)a.H, (unsigned)(nsl * (1 + with_forward))), NT, smem, s>>>(b, with_forward);
        prof_stop(s);
        return cudaGetLastError();
    };
    if (narrow) {
        constexpr int JS = 16;
        const size_t smem = std::max(sizeof(StatesSmem<DK, JS>), sizeof(DStatesSmem<TIO, DK, JS>));
        e = launch_states(kda_bwd_states_kernel<TIO, DK, DV, JS>, smem, DV / JS);
    } else {
        constexpr int JS = DV < 32 ? DV : 32;
        const size_t smem = std::max(sizeof(StatesSmem<DK, JS>), sizeof(DStatesSmem<TIO, DK, JS>));
        e = launch_states(kda_bwd_states_kernel<TIO, DK, DV, JS>, smem, DV / JS);
    }
    if (e != cudaSuccess) return e;
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
