// kda_decode.cu -- one recurrent decode step: the state read-modify-write.
//
// KDA.step ("Kimi K3: the paper and proofs side by side", section "A recurrent step and its
// return type", with the update of section 2.1.1, Equation 1, and the gate of Equation 5):
//     alpha = exp(g_min sigmoid(exp(A_h) z))
//     r = (Diag(alpha) S)^T k,  y = (Diag(alpha) S)^T q,  u = beta (v - r)
//     S' = Diag(alpha) S + k u^T,   o = S'^T q = y + (q.k) u
// The step is bound by moving the fp32 state: d_k x d_v x 4 bytes in and out once per
// (sequence, head).  One CTA of 256 threads owns one (sequence, head): each warp streams whole
// rows of S with 128-bit loads (lane l holds columns 4l..4l+3 for d_v = 128), keeps its rows in
// registers, reduces r and y over its rows, combines the eight warps' partial sums through shared
// memory (q.k is a warp-shuffle reduction), and writes S' back from the same registers.  Loads
// and stores use the streaming cache policy: every state byte is touched once per step.  For
// d_k = d_v = 128 the state goes through shared memory instead (kda_decode_step_smem_kernel).
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;

template <int VEC> struct VecT;
template <> struct VecT<4> { using T = float4; };
template <> struct VecT<2> { using T = float2; };
template <> struct VecT<1> { using T = float; };

__device__ __forceinline__ void vset(float4& v, int i, float x) { (&v.x)[i] = x; }
__device__ __forceinline__ void vset(float2& v, int i, float x) { (&v.x)[i] = x; }
__device__ __forceinline__ void vset(float& v, int, float x) { v = x; }
__device__ __forceinline__ float vget(const float4& v, int i) { return (&v.x)[i]; }
__device__ __forceinline__ float vget(const float2& v, int i) { return (&v.x)[i]; }
__device__ __forceinline__ float vget(const float& v, int) { return v; }

}  // namespace

template <typename TIO, int DK, int DV>
__global__ void __launch_bounds__(kDecThreads, 2) kda_decode_step_kernel(DecodeArgs a)
{
    constexpr int VEC = DV / 32;
    constexpr int RPW = DK / kDecWarps;  // rows per warp
    using V = typename VecT<VEC>::T;
    __shared__ float s_alpha[DK];
    __shared__ float s_k[DK];
    __shared__ float s_q[DK];
    __shared__ float s_u[DV];
    __shared__ float s_red[2][kDecWarps][DV];
    __shared__ float s_qk;

    const int nh = blockIdx.x;            // sequence * H + head
    const int h = nh % a.H;
    const int tid = threadIdx.x;
    const int w = tid >> 5;
    const int l = tid & 31;
    float* S = a.state + (int64_t)nh * DK * DV;

    // issue every state load of this thread before anything else
    V s[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int c = w + kDecWarps * i;
        s[i] = __ldcs(reinterpret_cast<const V*>(S + (int64_t)c * DV) + l);
    }

    const TIO* qp = static_cast<const TIO*>(a.q);
    const TIO* kp = static_cast<const TIO*>(a.k);
    const TIO* zp = static_cast<const TIO*>(a.z);
    if (tid < DK) {
        const int64_t idx = (int64_t)nh * DK + tid;
        s_alpha[tid] = expf(log_decay(ld_io(zp, idx), expf(a.A[h]), a.g_min));
        s_k[tid] = ld_io(kp, idx);
        s_q[tid] = ld_io(qp, idx);
    }
    __syncthreads();
    if (w == 0) {
        float p = 0.f;
        for (int c = l; c < DK; c += 32) p += s_q[c] * s_k[c];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
        if (l == 0) s_qk = p;
    }

    float r[VEC], y[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) r[e] = y[e] = 0.f;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int c = w + kDecWarps * i;
        const float al = s_alpha[c], kc = s_k[c], qc = s_q[c];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const float d = al * vget(s[i], e);  // decayed state, kept for the write-back
            vset(s[i], e, d);
            r[e] += kc * d;
            y[e] += qc * d;
        }
    }
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        s_red[0][w][l * VEC + e] = r[e];
        s_red[1][w][l * VEC + e] = y[e];
    }
    __syncthreads();
    if (tid < DV) {
        float rr = 0.f, yy = 0.f;
#pragma unroll
        for (int ww = 0; ww < kDecWarps; ++ww) {
            rr += s_red[0][ww][tid];
            yy += s_red[1][ww][tid];
        }
        const int64_t vidx = (int64_t)nh * DV + tid;
        const float u = a.beta[nh] * (ld_io(static_cast<const TIO*>(a.v), vidx) - rr);
        s_u[tid] = u;
        st_io(static_cast<TIO*>(a.out), vidx, yy + s_qk * u);
    }
    __syncthreads();
    float u[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) u[e] = s_u[l * VEC + e];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int c = w + kDecWarps * i;
        const float kc = s_k[c];
#pragma unroll
        for (int e = 0; e < VEC; ++e) vset(s[i], e, vget(s[i], e) + kc * u[e]);
        __stcs(reinterpret_cast<V*>(S + (int64_t)c * DV) + l, s[i]);
    }
}

// d_k = d_v = 128: the same step with the state staged through shared memory instead of registers
// (64 KB per (sequence, head), brought in by 16-byte asynchronous copies), so that a thread holds
// no state between the phases and three CTAs -- 192 KB of state in flight -- share an SM.
constexpr int kSmemD = 128;
constexpr size_t kDecSmemBytes = (size_t)kSmemD * kSmemD * 4;

template <typename TIO>
__global__ void __launch_bounds__(kDecThreads, 3) kda_decode_step_smem_kernel(DecodeArgs a)
{
    constexpr int D = kSmemD;
    constexpr int RPW = D / kDecWarps;  // rows per warp
    extern __shared__ __align__(16) float s_state[];  // [D][D]
    __shared__ float s_alpha[D];
    __shared__ float s_k[D];
    __shared__ float s_q[D];
    __shared__ float s_u[D];
    __shared__ float s_red[2][kDecWarps][D];
    __shared__ float s_qk;

    const int nh = blockIdx.x;  // sequence * H + head
    const int h = nh % a.H;
    const int tid = threadIdx.x;
    const int w = tid >> 5;
    const int l = tid & 31;
    float* S = a.state + (int64_t)nh * D * D;

    // the whole state in flight first: 4096 16-byte pieces, 16 per thread, coalesced
#pragma unroll
    for (int i = 0; i < D * D / 4 / kDecThreads; ++i) {
        const int e4 = tid + kDecThreads * i;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(s_state + 4 * e4)),
                     "l"(S + 4 * e4)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");

    const TIO* qp = static_cast<const TIO*>(a.q);
    const TIO* kp = static_cast<const TIO*>(a.k);
    const TIO* zp = static_cast<const TIO*>(a.z);
    if (tid < D) {
        const int64_t idx = (int64_t)nh * D + tid;
        s_alpha[tid] = expf(log_decay(ld_io(zp, idx), expf(a.A[h]), a.g_min));
        s_k[tid] = ld_io(kp, idx);
        s_q[tid] = ld_io(qp, idx);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    if (w == 0) {
        float p = 0.f;
        for (int c = l; c < D; c += 32) p += s_q[c] * s_k[c];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
        if (l == 0) s_qk = p;
    }

    // decay the rows this warp owns (lane l: columns 4l .. 4l + 3), keep them in shared memory, and
    // reduce r = (Diag alpha S)^T k and y = (Diag alpha S)^T q over them
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f), y = r;
#pragma unroll 4
    for (int i = 0; i < RPW; ++i) {
        const int c = w + kDecWarps * i;
        float4* row = reinterpret_cast<float4*>(s_state + c * D) + l;
        const float al = s_alpha[c], kc = s_k[c], qc = s_q[c];
        float4 d = *row;
        d.x *= al;
        d.y *= al;
        d.z *= al;
        d.w *= al;
        *row = d;
        r.x += kc * d.x;
        r.y += kc * d.y;
        r.z += kc * d.z;
        r.w += kc * d.w;
        y.x += qc * d.x;
        y.y += qc * d.y;
        y.z += qc * d.z;
        y.w += qc * d.w;
    }
    *reinterpret_cast<float4*>(&s_red[0][w][4 * l]) = r;
    *reinterpret_cast<float4*>(&s_red[1][w][4 * l]) = y;
    __syncthreads();
    if (tid < D) {
        float rr = 0.f, yy = 0.f;
#pragma unroll
        for (int ww = 0; ww < kDecWarps; ++ww) {
            rr += s_red[0][ww][tid];
            yy += s_red[1][ww][tid];
        }
        const int64_t vidx = (int64_t)nh * D + tid;
        const float u = a.beta[nh] * (ld_io(static_cast<const TIO*>(a.v), vidx) - rr);
        s_u[tid] = u;
        st_io(static_cast<TIO*>(a.out), vidx, yy + s_qk * u);
    }
    __syncthreads();
    // S' = Diag(alpha) S + k u^T, streamed back in the load's coalesced order
    const float4 u4 = *reinterpret_cast<const float4*>(&s_u[4 * (tid & 31)]);
#pragma unroll 4
    for (int i = 0; i < D * D / 4 / kDecThreads; ++i) {
        const int e4 = tid + kDecThreads * i;
        const int c = e4 / (D / 4);  // row; the column group is e4 mod 32 = tid mod 32
        const float kc = s_k[c];
        float4 d = reinterpret_cast<const float4*>(s_state)[e4];
        d.x += kc * u4.x;
        d.y += kc * u4.y;
        d.z += kc * u4.z;
        d.w += kc * u4.w;
        __stcs(reinterpret_cast<float4*>(S) + e4, d);
    }
}

template <typename TIO>
static cudaError_t launch_decode_io(const DecodeArgs& a, int dk, int dv, cudaStream_t s)
{
    const unsigned grid = (unsigned)((int64_t)a.N * a.H);
    if (dk == kSmemD && dv == kSmemD) {
        cudaError_t e = cudaFuncSetAttribute(kda_decode_step_smem_kernel<TIO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kDecSmemBytes);
        if (e != cudaSuccess) return e;
        kda_decode_step_smem_kernel<TIO><<<grid, kDecThreads, kDecSmemBytes, s>>>(a);
        return cudaGetLastError();
    }
#define KDA_DEC_CASE(DKv, DVv)                                                 \
    if (dk == DKv && dv == DVv) {                                               \
        kda_decode_step_kernel<TIO, DKv, DVv><<<grid, kDecThreads, 0, s>>>(a);  \
        return cudaGetLastError();                                              \
    }
    KDA_DEC_CASE(32, 32) KDA_DEC_CASE(32, 64) KDA_DEC_CASE(32, 128)
    KDA_DEC_CASE(64, 32) KDA_DEC_CASE(64, 64) KDA_DEC_CASE(64, 128)
    KDA_DEC_CASE(128, 32) KDA_DEC_CASE(128, 64) KDA_DEC_CASE(128, 128)
#undef KDA_DEC_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const DecodeArgs& a, int dk, int dv, kda_dtype_t dt, cudaStream_t s)
{
    return dt == KDA_BF16 ? launch_decode_io<__nv_bfloat16>(a, dk, dv, s) : launch_decode_io<float>(a, dk, dv, s);
}

}  // namespace kda
