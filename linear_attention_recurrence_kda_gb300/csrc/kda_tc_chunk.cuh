// kda_tc_chunk.cuh -- per-chunk preparation of the bf16, d = 128 prefill, shared by the fused
// tensor-core kernel (kda_chunk_tc.cu) and the parallel chunk-preparation kernel (kda_prep_tc.cu).
//
// For one 16-token chunk of one head these functions compute, from the q, k, v, z tiles and beta
// (the chunk form of Equation 1, "Kimi K3: the paper and proofs side by side", section 2.1.1, with
// the gate of Equation 5):
//   g = g_min sigmoid(e^{A_h} z), G_r = in-chunk inclusive cumsum, Gamma_r = e^{G_r}, Gamma_C = Gamma_16
//   K Gamma, Q Gamma (hi/lo), K / Gamma (hi/lo), (K Gamma_C / Gamma) (hi/lo), V^T
//   A[r][i] = beta_r <k_r Gamma_r, k_i / Gamma_i> (i < r),  P = tril_incl((Q Gamma)(K / Gamma)^T)
//   T = (I + A)^-1 by forward substitution, T' = T diag(beta) (hi/lo)
// With g_min = -5 a 16-token chunk keeps G in [-80, 0] ("Kimi K3" reading notes, section 2), so
// Gamma and 1/Gamma are normal fp32/bf16 numbers with one reference point per chunk.
//
// The shared-memory placement of every tile is a template parameter (a struct of byte offsets), so
// the two kernels can lay out their buffers differently.  All functions are called by the 256
// threads of one warp group; `p` is the thread's index in the group.
#pragma once

#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {

// 3-D views [T_tot][H][128] of the bf16 q, k, v, z inputs with a [16 tokens][1 head][128] box.
struct TileMaps {
    CUtensorMap q, k, v, z;
};
bool encode_tile_maps(TileMaps& m, const PrefillArgs& a);

namespace tcc {

constexpr int D = 128;            // d_k = d_v
constexpr int C = kChunk;         // 16
constexpr int NGROUP = 256;       // threads of one warp group
constexpr int LROW = 136;         // padded row (elements) of the row-major mma.sync operand tiles
constexpr uint32_t STAGE_TILE = C * D * 2;  // 4096 bytes per input tensor and chunk
constexpr uint32_t NONE_TILE = 4096;        // [128][16] bf16 NONE tile
constexpr uint32_t SMALL_TILE = 512;        // [16][16] bf16 NONE tile
constexpr uint32_t ROW_TILE = C * LROW * 2; // [16][LROW] bf16 row-major tile: 4352 bytes

// Per-chunk operand block: everything the state pass needs for one chunk of one head, laid out
// exactly as the state pass stages it in shared memory (one contiguous bulk copy).  P and
// (K Gamma_C / Gamma)^T are stored as one NONE-layout operand [P ; (K Gamma_C / Gamma)^T]
// (16 + 128 rows of 16 tokens), so that the output and state-update products of a chunk share one
// tensor-core instruction (N = 144); hi and lo parts are two such operands.
constexpr uint32_t BLK_WQ = 0;        // [W ; Q Gamma (hi)] [32][128 c] bf16 SW128           8192
constexpr uint32_t BLK_PK = 8192;     // [P ; (K Gamma_C / Gamma)^T] hi [144][16] NONE         4608
constexpr uint32_t BLK_PK_LO = 4608;  //   ... and its lo part at BLK_PK + BLK_PK_LO          4608
constexpr uint32_t BLK_KT = BLK_PK + SMALL_TILE;  // (K Gamma_C / Gamma)^T hi (lo: + BLK_PK_LO)
constexpr uint32_t BLK_UT = 17408;    // U~ = T' V fp32 [16 r][128 j]                         8192
constexpr uint32_t BLK_GC = 25600;    // Gamma_C fp32 [128]                                    512
constexpr uint32_t BLK_BYTES = 26112;

__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_arrive(uint32_t id, uint32_t count)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// NONE-style tile [rows][16] with an 8-row-group stride of RG bytes (256: the tensor-core operand
// layout; 272: padded, so that the transposed per-channel stores of prep_factors spread over the
// shared-memory banks).
template <uint32_t RG>
__host__ __device__ __forceinline__ uint32_t none_off_rg(int r, int k)
{
    return (uint32_t)((r >> 3) * RG + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// Equation 5 with the fast exponential and division (relative error ~1e-6, far below bf16).
__device__ __forceinline__ float log_decay_fast(float z, float expA, float g_min)
{
    const float x = expA * z;
    const float e = __expf(-fabsf(x));
    const float sig = (x >= 0.f) ? __fdividef(1.f, 1.f + e) : __fdividef(e, 1.f + e);
    return g_min * sig;
}

__device__ __forceinline__ void st_bf16(unsigned char* base, uint32_t off, __nv_bfloat16 x)
{
    *reinterpret_cast<__nv_bfloat16*>(base + off) = x;
}

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi)
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo)
{
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

// (x0, x1) = hi + lo as bf16 pairs: one packed conversion each.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<uint32_t*>(&h);
    lo = *reinterpret_cast<uint32_t*>(&l);
}

__device__ __forceinline__ uint32_t pack_f2(float x0, float x1)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    return *reinterpret_cast<uint32_t*>(&h);
}

// 16x16 partial product over one k-step (16 channels): acc += L[:, k0:k0+16] R[:, k0:k0+16]^T,
// L and R row-major [16][LROW] bf16.
__device__ __forceinline__ void mma_kstep(float (&acc)[2][4], const __nv_bfloat16* L, const __nv_bfloat16* R, int k0,
                                          int lane)
{
    const int g = lane >> 2, t = lane & 3;
    uint32_t af[4];
    af[0] = *reinterpret_cast<const uint32_t*>(L + g * LROW + k0 + 2 * t);
    af[1] = *reinterpret_cast<const uint32_t*>(L + (g + 8) * LROW + k0 + 2 * t);
    af[2] = *reinterpret_cast<const uint32_t*>(L + g * LROW + k0 + 8 + 2 * t);
    af[3] = *reinterpret_cast<const uint32_t*>(L + (g + 8) * LROW + k0 + 8 + 2 * t);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int n0 = 8 * nt;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(R + (n0 + g) * LROW + k0 + 2 * t);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(R + (n0 + g) * LROW + k0 + 8 + 2 * t);
        tc::mma16816(acc[nt], af, b0, b1);
    }
}

// Gate, in-chunk cumulative log-decay and every per-element factor of one chunk.
// Thread p owns the channel pair (2 cp, 2 cp + 1), cp = p % 64, and tokens [4 tq, 4 tq + 4),
// tq = p / 64; pairs make every row-tile store a 32-bit word.  Input tiles (q, k, v, z [16][128]
// bf16, row-major) are at Map::OFF_STAGE; tokens r >= len are treated as absent (zero).
// Writes: row-major K Gamma (OFF_LL), Q Gamma hi/lo (OFF_QL), K/Gamma hi/lo (OFF_KD); rows 16..31
// of the SW128 [W ; Q Gamma] tile at `wq` (Q Gamma hi); (K Gamma)^T and V^T (NONE, OFF_XT / OFF_VT);
// (K Gamma_C / Gamma)^T hi/lo at `kt` and `kt + kt_lo` (NONE); Gamma_C at `gc`.  One barrier
// (Map::NB) inside.
template <class Map>
__device__ __forceinline__ void prep_factors(unsigned char* sm, int p, int len, unsigned char* wq, unsigned char* kt,
                                             float* gc, float expA, float g_min, bool zero_v,
                                             uint32_t kt_lo = NONE_TILE)
{
    const int cp = p & 63;
    const int tq = p >> 6;
    const int c0 = 2 * cp;
    const int r0 = 4 * tq;
    const uint32_t* tq32 = reinterpret_cast<const uint32_t*>(sm + Map::OFF_STAGE);
    const uint32_t* tk32 = reinterpret_cast<const uint32_t*>(sm + Map::OFF_STAGE + STAGE_TILE);
    const uint32_t* tv32 = reinterpret_cast<const uint32_t*>(sm + Map::OFF_STAGE + 2 * STAGE_TILE);
    const uint32_t* tz32 = reinterpret_cast<const uint32_t*>(sm + Map::OFF_STAGE + 3 * STAGE_TILE);
    float* hs = reinterpret_cast<float*>(sm + Map::OFF_HS);  // [4 quarters][128 channels]

    float G0[4], G1[4];
    float2 kv[4], qv[4];
    uint32_t vv[4];
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int r = r0 + e;
        const bool ok = r < len;
        const uint32_t zw = tz32[(r * D + c0) >> 1];
        const float2 z2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&zw));
        a0 += ok ? log_decay_fast(z2.x, expA, g_min) : 0.f;
        a1 += ok ? log_decay_fast(z2.y, expA, g_min) : 0.f;
        G0[e] = a0;
        G1[e] = a1;
        const uint32_t kw = ok ? tk32[(r * D + c0) >> 1] : 0u;
        const uint32_t qw = ok ? tq32[(r * D + c0) >> 1] : 0u;
        kv[e] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kw));
        qv[e] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qw));
        vv[e] = (ok && !zero_v) ? tv32[(r * D + c0) >> 1] : 0u;
    }
    *reinterpret_cast<float2*>(hs + tq * D + c0) = make_float2(a0, a1);
    named_sync(Map::NB, NGROUP);
    float off0 = 0.f, off1 = 0.f, tot0 = 0.f, tot1 = 0.f;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
        const float2 hq = *reinterpret_cast<const float2*>(hs + qq * D + c0);
        if (qq < tq) {
            off0 += hq.x;
            off1 += hq.y;
        }
        tot0 += hq.x;
        tot1 += hq.y;
    }
    const float eGC0 = __expf(tot0), eGC1 = __expf(tot1);
    if (tq == 3) *reinterpret_cast<float2*>(gc + c0) = make_float2(eGC0, eGC1);

    uint32_t* sLl = reinterpret_cast<uint32_t*>(sm + Map::OFF_LL);
    uint32_t* sQl = reinterpret_cast<uint32_t*>(sm + Map::OFF_QL);
    uint32_t* sQll = sQl + C * LROW / 2;
    uint32_t* sKd = reinterpret_cast<uint32_t*>(sm + Map::OFF_KD);
    uint32_t* sKdl = sKd + C * LROW / 2;
    // transposed tiles: 4 tokens of one channel = 8 bytes at none_off(c, 4 tq)
    uint32_t xt0[2], xt1[2], kh0[2], kh1[2], kl0[2], kl1[2];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int r = r0 + e;
        const float eG0 = __expf(G0[e] + off0), eG1 = __expf(G1[e] + off1);  // Gamma in [e^-80, 1]
        const float iG0 = __fdividef(1.f, eG0), iG1 = __fdividef(1.f, eG1);  // 1/Gamma in [1, e^80]
        const float ll0 = kv[e].x * eG0, ll1 = kv[e].y * eG1;
        const uint32_t llw = pack_f2(ll0, ll1);
        const int ri = (r * LROW + c0) >> 1;
        sLl[ri] = llw;
        uint32_t hi, lo;
        split2(qv[e].x * eG0, qv[e].y * eG1, hi, lo);
        sQl[ri] = hi;
        sQll[ri] = lo;
        *reinterpret_cast<uint32_t*>(wq + tc::sw128_off(C + r, c0, 2 * C)) = hi;
        split2(kv[e].x * iG0, kv[e].y * iG1, hi, lo);
        sKd[ri] = hi;
        sKdl[ri] = lo;
        uint32_t th, tl;
        split2(kv[e].x * (eGC0 * iG0), kv[e].y * (eGC1 * iG1), th, tl);  // k Gamma_C / Gamma <= 1
        // de-interleave the pairs into per-channel token runs
        const int slot = e >> 1, sh = (e & 1) * 16;
        if ((e & 1) == 0) {
            xt0[slot] = llw & 0xffffu;
            xt1[slot] = llw >> 16;
            kh0[slot] = th & 0xffffu;
            kh1[slot] = th >> 16;
            kl0[slot] = tl & 0xffffu;
            kl1[slot] = tl >> 16;
        } else {
            xt0[slot] |= (llw & 0xffffu) << sh;
            xt1[slot] |= (llw >> 16) << sh;
            kh0[slot] |= (th & 0xffffu) << sh;
            kh1[slot] |= (th >> 16) << sh;
            kl0[slot] |= (tl & 0xffffu) << sh;
            kl1[slot] |= (tl >> 16) << sh;
        }
    }
    const uint32_t v00 = (vv[0] & 0xffffu) | (vv[1] << 16), v01 = (vv[2] & 0xffffu) | (vv[3] << 16);
    const uint32_t v10 = (vv[0] >> 16) | (vv[1] & 0xffff0000u), v11 = (vv[2] >> 16) | (vv[3] & 0xffff0000u);
    const uint32_t p0 = none_off_rg<Map::XT_RG>(c0, r0), p1 = none_off_rg<Map::XT_RG>(c0 + 1, r0);
    *reinterpret_cast<uint2*>(sm + Map::OFF_XT + p0) = make_uint2(xt0[0], xt0[1]);
    *reinterpret_cast<uint2*>(sm + Map::OFF_XT + p1) = make_uint2(xt1[0], xt1[1]);
    *reinterpret_cast<uint2*>(sm + Map::OFF_VT + p0) = make_uint2(v00, v01);
    *reinterpret_cast<uint2*>(sm + Map::OFF_VT + p1) = make_uint2(v10, v11);
    const uint32_t o0 = tc::none_off(c0, r0), o1 = tc::none_off(c0 + 1, r0);
    *reinterpret_cast<uint2*>(kt + o0) = make_uint2(kh0[0], kh0[1]);
    *reinterpret_cast<uint2*>(kt + o1) = make_uint2(kh1[0], kh1[1]);
    *reinterpret_cast<uint2*>(kt + kt_lo + o0) = make_uint2(kl0[0], kl0[1]);
    *reinterpret_cast<uint2*>(kt + kt_lo + o1) = make_uint2(kl1[0], kl1[1]);
}

// A and P over K = 128 with mma.sync, two k-steps per warp (warps 0..3: A, warps 4..7: P as
// hi*hi + hi*lo + lo*hi), partial sums reduced in shared memory (OFF_PART, 8 KB); then
// T = (I + A)^-1 by forward substitution and T' = T diag(beta) (hi/lo, OFF_T), P finalised into
// `pb` and `pb + p_lo` (hi/lo NONE).  beta of the chunk is read from OFF_BETA.  Two barriers (Map::NB) inside.
template <class Map>
__device__ __forceinline__ void prep_solve(unsigned char* sm, int p, unsigned char* pb, uint32_t p_lo = SMALL_TILE)
{
    const int pw = p >> 5, lane = p & 31;
    float* sA = reinterpret_cast<float*>(sm + Map::OFF_A);
    float* part = reinterpret_cast<float*>(sm + Map::OFF_PART);
    const float* beta = reinterpret_cast<const float*>(sm + Map::OFF_BETA);
    const __nv_bfloat16* sLl = reinterpret_cast<const __nv_bfloat16*>(sm + Map::OFF_LL);
    const __nv_bfloat16* sQl = reinterpret_cast<const __nv_bfloat16*>(sm + Map::OFF_QL);
    const __nv_bfloat16* sQll = sQl + C * LROW;
    const __nv_bfloat16* sKd = reinterpret_cast<const __nv_bfloat16*>(sm + Map::OFF_KD);
    const __nv_bfloat16* sKdl = sKd + C * LROW;
    {
        const int g = lane >> 2, t = lane & 3;
        const int k0 = 32 * (pw & 3);
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if (pw < 4) {
            mma_kstep(acc, sLl, sKd, k0, lane);
            mma_kstep(acc, sLl, sKd, k0 + 16, lane);
        } else {
#pragma unroll
            for (int kk = 0; kk < 32; kk += 16) {
                mma_kstep(acc, sQl, sKd, k0 + kk, lane);
                mma_kstep(acc, sQl, sKdl, k0 + kk, lane);
                mma_kstep(acc, sQll, sKd, k0 + kk, lane);
            }
        }
        float* pp = part + pw * C * C;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            *reinterpret_cast<float2*>(pp + g * C + 8 * nt + 2 * t) = make_float2(acc[nt][0], acc[nt][1]);
            *reinterpret_cast<float2*>(pp + (g + 8) * C + 8 * nt + 2 * t) = make_float2(acc[nt][2], acc[nt][3]);
        }
    }
    named_sync(Map::NB, NGROUP);
    {
        const int idx = p;  // one entry of A and one of P per thread
        const int r = idx >> 4, i = idx & 15;
        float sa = 0.f, sp = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            sa += part[k * C * C + idx];
            sp += part[(4 + k) * C * C + idx];
        }
        sA[idx] = (i < r) ? beta[r] * sa : 0.f;
        __nv_bfloat16 hi, lo;
        split_bf16((i <= r) ? sp : 0.f, hi, lo);
        st_bf16(pb, tc::none_off(r, i), hi);
        st_bf16(pb, p_lo + tc::none_off(r, i), lo);
    }
    named_sync(Map::NB, NGROUP);
    if (pw == 0 && lane < C) {
        // forward substitution, one lane per column j, column-oriented: once T[i][j] is final it is
        // eliminated from every later row, p_r -= A[r][i] T[i][j] (r > i), so each step adds one
        // dependent multiply-add instead of a length-r dot product
        const int j = lane;
        float p[C];
#pragma unroll
        for (int r = 0; r < C; ++r) p[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
        for (int i = 0; i < C; ++i) {
            const float ti = p[i];
#pragma unroll
            for (int r = i + 1; r < C; ++r) p[r] = fmaf(-sA[r * C + i], ti, p[r]);
        }
        const float bj = beta[j];
#pragma unroll
        for (int r = 0; r < C; ++r) {
            __nv_bfloat16 hi, lo;
            split_bf16(p[r] * bj, hi, lo);
            st_bf16(sm, Map::OFF_T + tc::none_off(r, j), hi);
            st_bf16(sm, Map::OFF_T + SMALL_TILE + tc::none_off(r, j), lo);
        }
    }
}

}  // namespace tcc
}  // namespace kda
