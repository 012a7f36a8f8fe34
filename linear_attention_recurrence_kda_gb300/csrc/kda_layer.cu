// kda_layer.cu -- the per-head work around the recurrence in a KDA layer: the prologue that turns
// the q, k, v projections into the recurrence's inputs, and the epilogue applied to its output.
//
// "Kimi K3: the paper and proofs side by side", section 2.1.1 ("Preparing the queries, keys,
// values, and decay", Equations 2-6) and "Kimi K3: architecture, derivations and a pinned-source
// audit", section 4.3:
//   prologue  y_t = sum_{i<K} w[h,c,i] x_{t-i}     causal depthwise short convolution (zero before
//                                                  each sequence start)
//             y_t = y_t sigmoid(y_t)               Swish
//             y_t = y_t / sqrt(|y_t|^2 + 1e-6)     regularised L2 normalisation (q and k only)
//   epilogue  y = o / sqrt(mean_c o^2 + eps) * weight * sigmoid(gate)
//                                                  head-wise RMSNorm and sigmoid output gate
// The projections themselves (x W) are plain GEMMs outside this library.
//
// Both are streaming kernels: every element is read and written once.  A prologue CTA takes 64
// consecutive tokens of one head and one tensor: its threads first copy the 64 rows (and the K-1
// rows before them) into shared memory with asynchronous 16-byte copies, so that a whole tile is in
// flight at once, then every warp walks 8 of the tokens (lane l owns channels l*VEC ..
// l*VEC + VEC - 1), convolving from the staged rows (zero before each sequence start); the L2 norm is
// a warp reduction.  An epilogue warp normalises whole token-head rows with one warp reduction each.  Swish and the gate use the hardware exponential
// and reciprocal approximations, the norms rsqrt.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kLayerThreads = 256;
constexpr int kLayerWarps = kLayerThreads / 32;
constexpr int kProTokens = 8;  // tokens per prologue warp
constexpr int kProTile = kLayerWarps * kProTokens;  // tokens per prologue CTA

template <typename TIO, int VEC>
__device__ __forceinline__ void ld_vec(const TIO* p, float (&x)[VEC])
{
    if constexpr (sizeof(TIO) == 2 && VEC == 4) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
        x[0] = __low2float(a); x[1] = __high2float(a); x[2] = __low2float(b); x[3] = __high2float(b);
    } else if constexpr (sizeof(TIO) == 4 && VEC == 4) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(p));
        x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) x[e] = ld_io(p, e);
    }
}

template <typename TIO, int VEC>
__device__ __forceinline__ void st_vec(TIO* p, const float (&x)[VEC])
{
    if constexpr (sizeof(TIO) == 2 && VEC == 4) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
        const __nv_bfloat162 b = __floats2bfloat162_rn(x[2], x[3]);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t*>(&a);
        u.y = *reinterpret_cast<const uint32_t*>(&b);
        *reinterpret_cast<uint2*>(p) = u;
    } else if constexpr (sizeof(TIO) == 4 && VEC == 4) {
        *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) st_io(p, e, x[e]);
    }
}

template <typename TIO, int VEC>
__device__ __forceinline__ void lds_vec(const TIO* p, float (&x)[VEC])
{
    if constexpr (sizeof(TIO) == 2 && VEC == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
        x[0] = __low2float(a); x[1] = __high2float(a); x[2] = __low2float(b); x[3] = __high2float(b);
    } else if constexpr (sizeof(TIO) == 4 && VEC == 4) {
        const float4 f = *reinterpret_cast<const float4*>(p);
        x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) x[e] = ld_io(p, e);
    }
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gmem_src)
                 : "memory");
}

// logistic function from the hardware base-2 exponential and reciprocal approximations (relative
// error near 2^-22): 1 / (1 + 2^(-x log2 e)); the exponential saturates to +inf for very negative x
// and the reciprocal of +inf is 0, so no input gives a NaN
__device__ __forceinline__ float sigmoid_f(float x)
{
    float e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-1.4426950408889634f * x));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
    return r;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// sequence containing token t: the largest n with cu[n] <= t (so an empty sequence is skipped),
// clamped so that garbage offsets never index outside [0, N]
__device__ __forceinline__ int find_seq(const int32_t* cu, int N, int64_t t)
{
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)cu[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

}  // namespace

template <typename TIO, int VEC>
__global__ void __launch_bounds__(kLayerThreads) kda_prologue_kernel(PrologueArgs a, int first)
{
    constexpr int D = 32 * VEC;
    constexpr int HALO = kMaxConv - 1;
    constexpr int CH = D * (int)sizeof(TIO) / 16;  // 16-byte pieces per row
    extern __shared__ __align__(16) unsigned char smem_raw[];
    TIO* rows = reinterpret_cast<TIO*>(smem_raw);  // [HALO + kProTile][D]: row HALO + r is token t0 + r
    const int which = first + blockIdx.z;  // 0: q, 1: k, 2: v
    const int h = blockIdx.y;
    const int w = threadIdx.x >> 5;
    const int l = threadIdx.x & 31;
    const int64_t t0 = (int64_t)blockIdx.x * kProTile;
    if (t0 >= a.T) return;
    // selected without indexing the parameter arrays (which would copy them to local memory)
    const TIO* x = static_cast<const TIO*>(which == 0 ? a.x[0] : which == 1 ? a.x[1] : a.x[2]);
    TIO* y = static_cast<TIO*>(which == 0 ? a.y[0] : which == 1 ? a.y[1] : a.y[2]);
    const float* wt = which == 0 ? a.w[0] : which == 1 ? a.w[1] : a.w[2];
    const int K = a.K;

    // the tile's rows and the K-1 rows before it (tokens outside [0, T) are not copied and never read)
    const int64_t r_lo = t0 - HALO;
    const int nrows = HALO + kProTile;
    for (int e = threadIdx.x; e < nrows * CH; e += kLayerThreads) {
        const int r = e / CH, ch = e - r * CH;
        const int64_t t = r_lo + r;
        if (t >= 0 && t < a.T) {
            cp_async16(reinterpret_cast<unsigned char*>(rows + r * D) + ch * 16,
                       reinterpret_cast<const unsigned char*>(x + (t * a.H + h) * D) + ch * 16);
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");

    float wk[VEC][kMaxConv];
#pragma unroll
    for (int e = 0; e < VEC; ++e)
#pragma unroll
        for (int i = 0; i < kMaxConv; ++i) wk[e][i] = (i < K) ? wt[((int64_t)h * D + l * VEC + e) * K + i] : 0.f;

    // this warp's tokens [tw, tw1) and the start of the sequence holding tw
    const int64_t tw = t0 + (int64_t)w * kProTokens;
    const int64_t tw1 = min(tw + (int64_t)kProTokens, a.T);
    int64_t start = 0, end = 0;
    int n = 0;
    if (tw < a.T) {
        if (a.cu != nullptr) {
            n = find_seq(a.cu, a.N, tw);
            start = min((int64_t)max(a.cu[n], 0), tw);
            end = max((int64_t)a.cu[n + 1], tw + 1);
        } else {
            const int64_t len = a.T / a.N;
            start = (tw / len) * len;
            end = start + len;
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();

    for (int64_t t = tw; t < tw1; ++t) {
        if (t >= end) {  // a new sequence starts here
            if (a.cu != nullptr) {
                while (n + 1 < a.N && (int64_t)a.cu[n + 1] <= t) ++n;
                start = t;
                end = max((int64_t)a.cu[n + 1], t + 1);
            } else {
                start = t;
                end = t + a.T / a.N;
            }
        }
        const int r = (int)(t - r_lo);
        float s[VEC];
        {
            float xt[VEC];
            lds_vec<TIO, VEC>(rows + r * D + l * VEC, xt);
#pragma unroll
            for (int e = 0; e < VEC; ++e) s[e] = wk[e][0] * xt[e];
        }
#pragma unroll
        for (int i = 1; i < kMaxConv; ++i) {
            if (i < K && t - i >= start) {
                float xp[VEC];
                lds_vec<TIO, VEC>(rows + (r - i) * D + l * VEC, xp);
#pragma unroll
                for (int e = 0; e < VEC; ++e) s[e] = fmaf(wk[e][i], xp[e], s[e]);
            }
        }
        float yv[VEC];
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const float sw = s[e] * sigmoid_f(s[e]);
            yv[e] = sw;
            ss = fmaf(sw, sw, ss);
        }
        if (which < 2) {
            const float inv = rsqrtf(warp_sum(ss) + 1e-6f);
#pragma unroll
            for (int e = 0; e < VEC; ++e) yv[e] *= inv;
        }
        st_vec<TIO, VEC>(y + (t * a.H + h) * D + l * VEC, yv);
    }
}

template <typename TIO, int VEC>
__global__ void __launch_bounds__(kLayerThreads) kda_epilogue_kernel(EpilogueArgs a)
{
    constexpr int D = 32 * VEC;
    const int l = threadIdx.x & 31;
    const TIO* o = static_cast<const TIO*>(a.o);
    const TIO* g = static_cast<const TIO*>(a.gate);
    TIO* y = static_cast<TIO*>(a.y);
    float wt[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) wt[e] = a.weight[l * VEC + e];
    const int64_t stride = (int64_t)gridDim.x * kLayerWarps;
    for (int64_t row = (int64_t)blockIdx.x * kLayerWarps + (threadIdx.x >> 5); row < a.rows; row += stride) {
        float ov[VEC], gv[VEC];
        ld_vec<TIO, VEC>(o + row * D + l * VEC, ov);
        ld_vec<TIO, VEC>(g + row * D + l * VEC, gv);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) ss += ov[e] * ov[e];
        const float inv = rsqrtf(warp_sum(ss) * (1.f / D) + a.eps);
#pragma unroll
        for (int e = 0; e < VEC; ++e) ov[e] = ov[e] * inv * wt[e] * sigmoid_f(gv[e]);
        st_vec<TIO, VEC>(y + row * D + l * VEC, ov);
    }
}

template <typename TIO>
static cudaError_t launch_prologue_io(const PrologueArgs& a, cudaStream_t s)
{
    const unsigned gx = (unsigned)((a.T + kProTile - 1) / kProTile);
    if (gx == 0) return cudaSuccess;
    auto go = [&](int d, int first, int count) -> cudaError_t {
        const dim3 grid(gx, (unsigned)a.H, (unsigned)count);
        const size_t smem = (size_t)(kMaxConv - 1 + kProTile) * d * sizeof(TIO);
        if (d == 32) kda_prologue_kernel<TIO, 1><<<grid, kLayerThreads, smem, s>>>(a, first);
        else if (d == 64) kda_prologue_kernel<TIO, 2><<<grid, kLayerThreads, smem, s>>>(a, first);
        else if (d == 128) kda_prologue_kernel<TIO, 4><<<grid, kLayerThreads, smem, s>>>(a, first);
        else return cudaErrorInvalidValue;
        return cudaGetLastError();
    };
    if (a.dk == a.dv) return go(a.dk, 0, 3);
    const cudaError_t e = go(a.dk, 0, 2);
    return e != cudaSuccess ? e : go(a.dv, 2, 1);
}

cudaError_t launch_prologue(const PrologueArgs& a, kda_dtype_t dt, cudaStream_t s)
{
    return dt == KDA_BF16 ? launch_prologue_io<__nv_bfloat16>(a, s) : launch_prologue_io<float>(a, s);
}

template <typename TIO>
static cudaError_t launch_epilogue_io(const EpilogueArgs& a, int dv, cudaStream_t s)
{
    if (a.rows == 0) return cudaSuccess;
    const int64_t ctas = (a.rows + kLayerWarps - 1) / kLayerWarps;
    const int64_t cap = (int64_t)sm_count_of_current_device() * 8 * 4;  // a few waves of 8 CTAs per SM
    const unsigned grid = (unsigned)(ctas < cap ? ctas : cap);
    if (dv == 32) kda_epilogue_kernel<TIO, 1><<<grid, kLayerThreads, 0, s>>>(a);
    else if (dv == 64) kda_epilogue_kernel<TIO, 2><<<grid, kLayerThreads, 0, s>>>(a);
    else if (dv == 128) kda_epilogue_kernel<TIO, 4><<<grid, kLayerThreads, 0, s>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_epilogue(const EpilogueArgs& a, int dv, kda_dtype_t dt, cudaStream_t s)
{
    return dt == KDA_BF16 ? launch_epilogue_io<__nv_bfloat16>(a, dv, s) : launch_epilogue_io<float>(a, dv, s);
}

}  // namespace kda
