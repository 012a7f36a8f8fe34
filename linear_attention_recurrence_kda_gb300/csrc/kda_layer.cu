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
// Both are streaming kernels (every element is read and written once), written to spend few
// instructions per element so that HBM, not instruction issue, bounds them:
//   * a lane owns one 16-byte vector of a row (8 bf16 or 4 fp32 channels), so a row of d channels
//     is a group of G = d / 8 (or d / 4) lanes, a warp covers 32 / G consecutive rows (heads) of a
//     token at once, and the row reductions are log2(G) shuffles within the group;
//   * arithmetic runs on packed fp32 pairs; the logistic function of a channel pair is one packed
//     half-precision tanh where the result is rounded to bf16, and otherwise two exponentials
//     sharing one hardware reciprocal (1/a = b / (ab), 1/b = a / (ab));
//   * the prologue is a persistent grid: a CTA walks consecutive tiles of 64 tokens (and the K-1
//     before them) of its heads, staged with asynchronous 16-byte copies into two alternating
//     buffers; each warp walks 8 consecutive tokens of a tile with the convolution's window of
//     earlier inputs held in registers, so every input vector is read from shared memory once.
#include <cuda_fp16.h>

#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kLayerThreads = 256;
constexpr int kLayerWarps = kLayerThreads / 32;
constexpr int kProTokens = 8;                       // tokens per prologue warp
constexpr int kProTile = kLayerWarps * kProTokens;  // tokens per prologue CTA
constexpr int kVecBytes = 16;                       // bytes a lane owns in a row
constexpr int kWarpRowBytes = 32 * kVecBytes;       // bytes a warp covers per token (512)
constexpr int kEpiRows = 2;                         // row groups a warp has in flight in the epilogue
constexpr float kLog2e = 1.4426950408889634f;

// 16 bytes of TIO as packed fp32 pairs
template <typename TIO> struct Vec16;
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void unpack(const uint4& u, float2 (&x)[4])
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) x[p] = make_float2(__uint_as_float(w[p] << 16), __uint_as_float(w[p] & 0xffff0000u));
    }
    __device__ __forceinline__ static uint4 pack(const float2 (&x)[4])
    {
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const __nv_bfloat162 b = __float22bfloat162_rn(x[p]);
            w[p] = *reinterpret_cast<const uint32_t*>(&b);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct Vec16<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void unpack(const uint4& u, float2 (&x)[2])
    {
        x[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
        x[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
    }
    __device__ __forceinline__ static uint4 pack(const float2 (&x)[2])
    {
        return make_uint4(__float_as_uint(x[0].x), __float_as_uint(x[0].y), __float_as_uint(x[1].x),
                          __float_as_uint(x[1].y));
    }
};

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gmem_src)
                 : "memory");
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// logistic function of a pair, 1 / (1 + 2^(-x log2 e)), from the hardware base-2 exponential and
// one reciprocal approximation for both (relative error a few 2^-23).  The exponent is capped at
// 2^60 so that the product of the two denominators stays finite (below 2^121): inputs under -41.6
// give 2^-60 instead of a smaller number, and no input gives a NaN.
__device__ __forceinline__ float2 sigmoid2(float2 x)
{
    const float2 y = __fmul2_rn(x, make_float2(-kLog2e, -kLog2e));
    const float a0 = 1.f + ex2_approx(fminf(y.x, 60.f));
    const float a1 = 1.f + ex2_approx(fminf(y.y, 60.f));
    const float r = rcp_approx(a0 * a1);
    return make_float2(a1 * r, a0 * r);
}

// tanh of a pair by one packed half-precision hardware instruction (absolute error about 2^-11;
// halves beyond the f16 range round to +-inf, where tanh is +-1)
__device__ __forceinline__ float2 tanh2_h(float2 x)
{
    const __half2 hx = __floats2half2_rn(x.x, x.y);
    uint32_t t = *reinterpret_cast<const uint32_t*>(&hx);
    asm("tanh.approx.f16x2 %0, %0;" : "+r"(t));
    return __half22float2(*reinterpret_cast<const __half2*>(&t));
}

// Where the result is rounded to bf16 (relative precision 2^-9) the logistic function is taken as
// sigmoid(x) = (1 + tanh(x / 2)) / 2, one packed tanh for a channel pair; fp32 results use the
// exponential-and-reciprocal form (sigmoid2).  kHalf<TIO> is the factor 1/2 the bf16 form needs,
// folded by the callers into the convolution taps and into the gate's scale.
template <typename TIO>
constexpr float kHalf = sizeof(TIO) == 2 ? 0.5f : 1.f;

// Swish x sigmoid(x) of a pair from s = kHalf x: s (1 + tanh s) in bf16, x sigmoid(x) in fp32
template <typename TIO>
__device__ __forceinline__ float2 swish_io(float2 s)
{
    if constexpr (sizeof(TIO) == 2) return __ffma2_rn(s, tanh2_h(s), s);
    else return __fmul2_rn(s, sigmoid2(s));
}

// h sigmoid(g) of a pair from h = kHalf u: h (1 + tanh(g / 2)) in bf16, u sigmoid(g) in fp32
template <typename TIO>
__device__ __forceinline__ float2 gate_io(float2 h, float2 g)
{
    if constexpr (sizeof(TIO) == 2) return __ffma2_rn(h, tanh2_h(__fmul2_rn(g, make_float2(0.5f, 0.5f))), h);
    else return __fmul2_rn(h, sigmoid2(g));
}

// sum over the G lanes of a row group (G a power of two; the groups are aligned runs of lanes;
// every lane of the warp takes part)
template <int G>
__device__ __forceinline__ float group_sum(float x)
{
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
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

// One warp's run of `run` (<= kProTokens) tokens for a convolution of width KT; every lane takes
// part (the row reductions are warp-wide shuffles) and lanes with `store` false write nothing.
//   st     this lane's vector in the staged row of the run's first token (rows kWarpRowBytes apart)
//   y      this lane's vector of the first token's output (tokens ystride elements apart)
//   wk     the lane's taps times kHalf (pairs of channels), zero beyond the width
//   win0   valid inputs before the first token (those of its own sequence, at most KT - 1)
//   fresh  bit j: token j starts a sequence (nothing before it enters the window)
template <typename TIO, int D, int KT>
__device__ __forceinline__ void prologue_tokens(const unsigned char* st, TIO* y, int64_t ystride,
                                                const float2 (&wk)[kMaxConv][Vec16<TIO>::N / 2], bool norm,
                                                bool store, int run, int win0, uint32_t fresh)
{
    using V = Vec16<TIO>;
    constexpr int P = V::N / 2;
    constexpr int G = D / V::N;
    // window of earlier inputs: xw[i - 1] = x_{t - i}
    float2 xw[KT > 1 ? KT - 1 : 1][P];
#pragma unroll
    for (int i = 1; i < KT; ++i) {
        if (i <= win0) {
            V::unpack(*reinterpret_cast<const uint4*>(st - i * kWarpRowBytes), xw[i - 1]);
        } else {
#pragma unroll
            for (int p = 0; p < P; ++p) xw[i - 1][p] = make_float2(0.f, 0.f);
        }
    }
    // one token: convolution over the window, Swish, the optional norm, the store; then the
    // window moves on by one token
    auto step = [&](int j) {
        float2 x[P];
        V::unpack(*reinterpret_cast<const uint4*>(st + j * kWarpRowBytes), x);
        float2 s[P];
        float2 ss = make_float2(0.f, 0.f);
#pragma unroll
        for (int p = 0; p < P; ++p) {
            s[p] = __fmul2_rn(wk[0][p], x[p]);
#pragma unroll
            for (int i = 1; i < KT; ++i) s[p] = __ffma2_rn(wk[i][p], xw[i - 1][p], s[p]);
            s[p] = swish_io<TIO>(s[p]);
            ss = __ffma2_rn(s[p], s[p], ss);
        }
        if (norm) {
            const float inv = rsqrtf(group_sum<G>(ss.x + ss.y) + 1e-6f);
#pragma unroll
            for (int p = 0; p < P; ++p) s[p] = __fmul2_rn(s[p], make_float2(inv, inv));
        }
        if (store) *reinterpret_cast<uint4*>(y + j * ystride) = V::pack(s);
#pragma unroll
        for (int i = KT - 2; i > 0; --i)
#pragma unroll
            for (int p = 0; p < P; ++p) xw[i][p] = xw[i - 1][p];
        if (KT > 1) {
#pragma unroll
            for (int p = 0; p < P; ++p) xw[0][p] = x[p];
        }
    };
    // two tokens at once (the common case): one butterfly reduces both rows' sums of squares, the
    // two halves of a lane group holding one token's total each after log2(G) levels, and one more
    // exchange hands each half the other's
    auto step2 = [&](int j) {
        float2 x0[P], x1[P];
        V::unpack(*reinterpret_cast<const uint4*>(st + j * kWarpRowBytes), x0);
        V::unpack(*reinterpret_cast<const uint4*>(st + (j + 1) * kWarpRowBytes), x1);
        float2 s0[P], s1[P];
        float2 q0 = make_float2(0.f, 0.f), q1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int p = 0; p < P; ++p) {
            s0[p] = __fmul2_rn(wk[0][p], x0[p]);
            s1[p] = __fmul2_rn(wk[0][p], x1[p]);
            if (KT > 1) s1[p] = __ffma2_rn(wk[1][p], x0[p], s1[p]);
#pragma unroll
            for (int i = 1; i < KT; ++i) s0[p] = __ffma2_rn(wk[i][p], xw[i - 1][p], s0[p]);
#pragma unroll
            for (int i = 2; i < KT; ++i) s1[p] = __ffma2_rn(wk[i][p], xw[i - 2][p], s1[p]);
            s0[p] = swish_io<TIO>(s0[p]);
            s1[p] = swish_io<TIO>(s1[p]);
            q0 = __ffma2_rn(s0[p], s0[p], q0);
            q1 = __ffma2_rn(s1[p], s1[p], q1);
        }
        if (norm) {
            const bool upper = (threadIdx.x & (G / 2)) != 0;
            const float a0 = q0.x + q0.y, a1 = q1.x + q1.y;
            float keep = upper ? a1 : a0;
            keep += __shfl_xor_sync(0xffffffffu, upper ? a0 : a1, G / 2);
#pragma unroll
            for (int off = G / 4; off > 0; off >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, off);
            const float other = __shfl_xor_sync(0xffffffffu, keep, G / 2);
            const float inv0 = rsqrtf((upper ? other : keep) + 1e-6f);
            const float inv1 = rsqrtf((upper ? keep : other) + 1e-6f);
#pragma unroll
            for (int p = 0; p < P; ++p) {
                s0[p] = __fmul2_rn(s0[p], make_float2(inv0, inv0));
                s1[p] = __fmul2_rn(s1[p], make_float2(inv1, inv1));
            }
        }
        if (store) {
            *reinterpret_cast<uint4*>(y + j * ystride) = V::pack(s0);
            *reinterpret_cast<uint4*>(y + (j + 1) * ystride) = V::pack(s1);
        }
        // the window moves on by two tokens
#pragma unroll
        for (int i = KT - 2; i > 1; --i)
#pragma unroll
            for (int p = 0; p < P; ++p) xw[i][p] = xw[i - 2][p];
        if (KT > 2) {
#pragma unroll
            for (int p = 0; p < P; ++p) xw[1][p] = x0[p];
        }
        if (KT > 1) {
#pragma unroll
            for (int p = 0; p < P; ++p) xw[0][p] = x1[p];
        }
    };
    if (run == kProTokens && fresh == 0u) {
        // the common case: straight-line code over the run, so the tokens' work interleaves
        static_assert(kProTokens % 2 == 0, "token pairs");
#pragma unroll
        for (int j = 0; j < kProTokens; j += 2) step2(j);
        return;
    }
    for (int j = 0; j < run; ++j) {
        if ((fresh >> j) & 1u) {
#pragma unroll
            for (int i = 0; i < KT - 1; ++i)
#pragma unroll
                for (int p = 0; p < P; ++p) xw[i][p] = make_float2(0.f, 0.f);
        }
        step(j);
    }
}

}  // namespace

// A persistent grid: CTA b takes the tiles [b ntiles / grid, (b + 1) ntiles / grid) in order, a
// tile being kProTile tokens of one group of 32 / G heads of one tensor, ordered tokens fastest,
// so that a CTA's consecutive tiles are consecutive token ranges with the same weights.  Tiles are
// staged into two alternating buffers: the copy of the next tile is in flight while the warps
// work on the current one.  tiles_t = ceil(T / kProTile), groups = ceil(H / (32 / G)); seq_len
// is T / N when there are no offsets.
template <typename TIO, int D>
__global__ void __launch_bounds__(kLayerThreads, 2)
    kda_prologue_kernel(PrologueArgs a, int first, int count, int tiles_t, int groups, int64_t seq_len)
{
    using V = Vec16<TIO>;
    constexpr int P = V::N / 2;
    constexpr int G = D / V::N;      // lanes per row
    constexpr int RPW = 32 / G;      // heads per warp (and per tile)
    constexpr int HALO = kMaxConv - 1;
    constexpr int ROWS = HALO + kProTile;
    constexpr int TILE_BYTES = ROWS * kWarpRowBytes;
    extern __shared__ __align__(16) unsigned char stage[];  // [2][ROWS][kWarpRowBytes]
    const int w = threadIdx.x >> 5;
    const int l = threadIdx.x & 31;
    const int ntiles = tiles_t * groups * count;
    const int b0 = (int)((int64_t)ntiles * blockIdx.x / gridDim.x);
    const int b1 = (int)((int64_t)ntiles * (blockIdx.x + 1) / gridDim.x);
    if (b0 >= b1) return;
    const int64_t tok_stride = (int64_t)a.H * D;  // elements from one token's row to the next

    struct Tile {
        int64_t t0;
        int h0, which, key;
    };
    auto decode = [&](int ti) {
        Tile t;
        const int gz = ti / tiles_t;
        t.t0 = (int64_t)(ti - gz * tiles_t) * kProTile;
        t.key = gz;
        t.which = first + gz / groups;
        t.h0 = (gz % groups) * RPW;
        return t;
    };
    // the tile's rows and the K-1 rows before it, 16 bytes a copy: piece l of a token is lane l's
    // vector (heads h0 .. h0 + RPW - 1 are contiguous), so thread (w, l) copies piece l of rows
    // w, w + 8, ...; tokens outside [0, T) and heads >= H are not copied (their lanes compute on
    // whatever the buffer holds and store nothing)
    auto stage_tile = [&](const Tile& t, unsigned char* buf) {
        if (l < min(RPW, a.H - t.h0) * G) {
            const unsigned char* x = static_cast<const unsigned char*>(t.which == 0 ? a.x[0]
                                                                       : t.which == 1 ? a.x[1]
                                                                                      : a.x[2]);
            int64_t tt = t.t0 - HALO + w;
            int64_t off = (tt * a.H + t.h0) * D * (int64_t)sizeof(TIO) + l * kVecBytes;
            const int64_t step = kLayerWarps * tok_stride * (int64_t)sizeof(TIO);
            for (int r = w; r < ROWS; r += kLayerWarps, tt += kLayerWarps, off += step) {
                if (tt >= 0 && tt < a.T) cp_async16(buf + r * kWarpRowBytes + l * kVecBytes, x + off);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    Tile cur = decode(b0);
    stage_tile(cur, stage);
    float2 wk[kMaxConv][P];
    int wkey = -1;
    int n = 0;                    // this warp's sequence and its bounds, carried from tile to tile
    int64_t start = 0, end = 0, prev_tw = -1;
    for (int ti = b0; ti < b1; ++ti) {
        const int k = ti - b0;
        const unsigned char* buf = stage + (k & 1) * TILE_BYTES;
        Tile next{};
        if (ti + 1 < b1) {
            next = decode(ti + 1);
            stage_tile(next, stage + ((k + 1) & 1) * TILE_BYTES);
        }
        const int hl = cur.h0 + l / G;
        const int c0 = (l % G) * V::N;
        const bool lane_ok = hl < a.H;
        if (cur.key != wkey) {  // this lane's taps times kHalf, zero beyond K (and for absent heads)
            const float* wt = cur.which == 0 ? a.w[0] : cur.which == 1 ? a.w[1] : a.w[2];
            const float* wrow = wt + ((int64_t)(lane_ok ? hl : 0) * D + c0) * a.K;
#pragma unroll
            for (int i = 0; i < kMaxConv; ++i)
#pragma unroll
                for (int p = 0; p < P; ++p)
                    wk[i][p] = (i < a.K && lane_ok) ? make_float2(kHalf<TIO> * wrow[(2 * p) * a.K + i],
                                                                  kHalf<TIO> * wrow[(2 * p + 1) * a.K + i])
                                                    : make_float2(0.f, 0.f);
            wkey = cur.key;
        }
        // this warp's tokens [tw, tw1): the sequence holding tw (advanced from the previous
        // tile's, searched afresh when the tokens start over), how many inputs before tw belong to
        // it, and which tokens of the run start a sequence
        const int64_t tw = cur.t0 + (int64_t)w * kProTokens;
        const int64_t tw1 = min(tw + (int64_t)kProTokens, a.T);
        int win0 = 0;
        uint32_t fresh = 0u;
        if (tw < a.T) {
            if (a.cu != nullptr) {
                if (tw < prev_tw || prev_tw < 0) n = find_seq(a.cu, a.N, tw);
                while (n + 1 < a.N && (int64_t)a.cu[n + 1] <= tw) ++n;
                start = min((int64_t)max(a.cu[n], 0), tw);
                end = max((int64_t)a.cu[n + 1], tw + 1);
                int nn = n;
                for (int64_t e = end; e < tw1;) {
                    fresh |= 1u << (int)(e - tw);
                    while (nn + 1 < a.N && (int64_t)a.cu[nn + 1] <= e) ++nn;
                    e = max((int64_t)a.cu[nn + 1], e + 1);
                }
            } else {
                if (tw < start || tw >= end) {
                    start = (tw / seq_len) * seq_len;
                    end = start + seq_len;
                }
                for (int64_t e = end; e < tw1; e += seq_len) fresh |= 1u << (int)(e - tw);
            }
            win0 = (int)min(tw - start, (int64_t)(kMaxConv - 1));
            prev_tw = tw;
        }
        if (ti + 1 < b1) asm volatile("cp.async.wait_group 1;" ::: "memory");
        else asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        if (tw < a.T) {  // warp-uniform: every lane of the warp takes part
            TIO* y = static_cast<TIO*>(cur.which == 0 ? a.y[0] : cur.which == 1 ? a.y[1] : a.y[2]);
            const unsigned char* st = buf + (int)(tw - (cur.t0 - HALO)) * kWarpRowBytes + l * kVecBytes;
            TIO* yl = y + (tw * a.H + (lane_ok ? hl : 0)) * D + c0;
            const bool norm = cur.which < 2;
            const int run = (int)(tw1 - tw);
            switch (a.K) {
                case 1: prologue_tokens<TIO, D, 1>(st, yl, tok_stride, wk, norm, lane_ok, run, win0, fresh); break;
                case 2: prologue_tokens<TIO, D, 2>(st, yl, tok_stride, wk, norm, lane_ok, run, win0, fresh); break;
                case 3: prologue_tokens<TIO, D, 3>(st, yl, tok_stride, wk, norm, lane_ok, run, win0, fresh); break;
                default: prologue_tokens<TIO, D, 4>(st, yl, tok_stride, wk, norm, lane_ok, run, win0, fresh); break;
            }
        }
        __syncthreads();  // the buffer is free for the tile after next
        cur = next;
    }
}

// Rows of d_v channels, 32 / G rows a warp at once and kEpiRows such groups in flight.
template <typename TIO, int D>
__global__ void __launch_bounds__(kLayerThreads) kda_epilogue_kernel(EpilogueArgs a)
{
    using V = Vec16<TIO>;
    constexpr int P = V::N / 2;
    constexpr int G = D / V::N;
    constexpr int RPW = 32 / G;
    const int l = threadIdx.x & 31;
    const int c0 = (l % G) * V::N;
    const TIO* o = static_cast<const TIO*>(a.o);
    const TIO* g = static_cast<const TIO*>(a.gate);
    TIO* y = static_cast<TIO*>(a.y);
    float2 wt[P];
#pragma unroll
    for (int p = 0; p < P; ++p) wt[p] = make_float2(a.weight[c0 + 2 * p], a.weight[c0 + 2 * p + 1]);
    const int64_t warp = (int64_t)blockIdx.x * kLayerWarps + (threadIdx.x >> 5);
    const int64_t stride = (int64_t)gridDim.x * kLayerWarps * kEpiRows * RPW;
    for (int64_t base = warp * kEpiRows * RPW; base < a.rows; base += stride) {
        uint4 ou[kEpiRows], gu[kEpiRows];
#pragma unroll
        for (int u = 0; u < kEpiRows; ++u) {
            const int64_t row = base + u * RPW + l / G;
            if (row < a.rows) {
                ou[u] = *reinterpret_cast<const uint4*>(o + row * D + c0);
                gu[u] = *reinterpret_cast<const uint4*>(g + row * D + c0);
            } else {
                ou[u] = gu[u] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < kEpiRows; ++u) {
            const int64_t row = base + u * RPW + l / G;
            float2 ov[P], gv[P];
            V::unpack(ou[u], ov);
            V::unpack(gu[u], gv);
            float2 ss = make_float2(0.f, 0.f);
#pragma unroll
            for (int p = 0; p < P; ++p) ss = __ffma2_rn(ov[p], ov[p], ss);
            const float inv = rsqrtf(group_sum<G>(ss.x + ss.y) * (1.f / D) + a.eps);
            const float hinv = kHalf<TIO> * inv;
#pragma unroll
            for (int p = 0; p < P; ++p)
                ov[p] = gate_io<TIO>(__fmul2_rn(ov[p], __fmul2_rn(wt[p], make_float2(hinv, hinv))), gv[p]);
            if (row < a.rows) *reinterpret_cast<uint4*>(y + row * D + c0) = V::pack(ov);
        }
    }
}

template <typename TIO>
static cudaError_t launch_prologue_io(const PrologueArgs& a, cudaStream_t s)
{
    const int64_t tiles_t = (a.T + kProTile - 1) / kProTile;
    if (tiles_t == 0) return cudaSuccess;
    constexpr int smem = 2 * (kMaxConv - 1 + kProTile) * kWarpRowBytes;
    static_assert(2 * (smem + 1024) <= 232448, "two CTAs' staging buffers fit an SM");
    const int64_t seq_len = a.cu != nullptr ? 0 : a.T / a.N;
    auto go = [&](int d, int first, int count) -> cudaError_t {
        const int rpw = 32 / (d / Vec16<TIO>::N);  // heads per tile
        const int64_t groups = (a.H + rpw - 1) / rpw;
        const int64_t ntiles = tiles_t * groups * count;
        if (ntiles >= (int64_t)1 << 31) return cudaErrorInvalidValue;
        void (*kern)(PrologueArgs, int, int, int, int, int64_t) = d == 32   ? kda_prologue_kernel<TIO, 32>
                                                                 : d == 64  ? kda_prologue_kernel<TIO, 64>
                                                                 : d == 128 ? kda_prologue_kernel<TIO, 128>
                                                                            : nullptr;
        if (kern == nullptr) return cudaErrorInvalidValue;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        int per_sm = 0;  // resident CTAs per SM: the persistent grid is one wave of them
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kLayerThreads, smem);
        if (e != cudaSuccess) return e;
        const int64_t slots = (int64_t)sm_count_of_current_device() * (per_sm > 0 ? per_sm : 1);
        const unsigned grid = (unsigned)(ntiles < slots ? ntiles : slots);
        kern<<<grid, kLayerThreads, smem, s>>>(a, first, count, (int)tiles_t, (int)groups, seq_len);
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
    if (dv != 32 && dv != 64 && dv != 128) return cudaErrorInvalidValue;
    const int64_t rows_per_cta = (int64_t)kLayerWarps * kEpiRows * (32 / (dv / Vec16<TIO>::N));
    const int64_t ctas = (a.rows + rows_per_cta - 1) / rows_per_cta;
    const int64_t cap = (int64_t)sm_count_of_current_device() * 8 * 16;  // the loop takes the rest
    const unsigned grid = (unsigned)(ctas < cap ? ctas : cap);
    if (dv == 32) kda_epilogue_kernel<TIO, 32><<<grid, kLayerThreads, 0, s>>>(a);
    else if (dv == 64) kda_epilogue_kernel<TIO, 64><<<grid, kLayerThreads, 0, s>>>(a);
    else kda_epilogue_kernel<TIO, 128><<<grid, kLayerThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_epilogue(const EpilogueArgs& a, int dv, kda_dtype_t dt, cudaStream_t s)
{
    return dt == KDA_BF16 ? launch_epilogue_io<__nv_bfloat16>(a, dv, s) : launch_epilogue_io<float>(a, dv, s);
}

}  // namespace kda
