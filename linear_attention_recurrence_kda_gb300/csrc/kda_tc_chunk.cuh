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

// Per-pair operand block: everything the state pass needs for one 32-token step (two consecutive
// 16-token chunks a, b of one head), laid out exactly as the state pass stages it in shared memory
// (one contiguous bulk copy).  With X = W_b K~_a^T and Z = (Q Gamma)_b K~_a^T (K~ = K Gamma_C /
// Gamma), the pair acts on the state like one chunk of 32 tokens:
//   W = [W_a ; W_b Gamma_Ca - X W_a],  U~ = [U~_a ; U~_b - X U~_a],  Q = [(Q Gamma)_a ; (Q Gamma)_b Gamma_Ca],
//   K~ = [K~_a Gamma_Cb ; K~_b],       P = [[P_a, 0] ; [Z, P_b]],     Gamma_C = Gamma_Ca Gamma_Cb
// (substitute chunk a's end state into chunk b's equations), and every factor stays bounded by one
// in magnitude as in the 16-token form.  P and K~^T are stored as one no-swizzle operand
// [P ; K~^T] (32 + 128 rows of 32 tokens), so that the output and state-update products of a step
// share one tensor-core instruction (N = 160); hi and lo parts are two such operands.
constexpr int PAIR = 2 * C;                          // tokens per state step
constexpr uint32_t PK_RG = 512;                      // 8-row-group stride of the [P ; K~^T] operand
constexpr uint32_t BLK_WQ = 0;        // [W ; Q Gamma (hi)] [64][128 c] bf16 SW128               16384
constexpr uint32_t BLK_PK = 16384;    // [P ; K~^T] hi [160][32] no-swizzle (LBO 128, SBO 512)    10240
constexpr uint32_t BLK_PK_LO = 10240; //   ... and its lo part at BLK_PK + BLK_PK_LO              10240
constexpr uint32_t BLK_KT = BLK_PK + 4 * PK_RG;  // the K~^T rows (from row 32)
constexpr uint32_t BLK_UT = 36864;    // U~ fp32 [32 r][128 j]                                    16384
constexpr uint32_t BLK_GC = 53248;    // Gamma_C fp32 [128]                                         512
constexpr uint32_t BLK_BYTES = 53760;

// Byte offset of element (row, k) of the [P ; K~^T] operand (k < 32 tokens).
__host__ __device__ __forceinline__ uint32_t pk_off(int row, int k)
{
    return (uint32_t)((row >> 3) * PK_RG + (k >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

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

// Placement of a no-swizzle K-major tile inside a larger operand: element (r, k) of the tile is
// element (r + row0, k + k0) of an operand whose 8-row groups are `rg` bytes apart.
struct NonePlace {
    uint32_t rg, row0, k0;
    __device__ __forceinline__ uint32_t off(int r, int k) const
    {
        const int rr = r + (int)row0, kk = k + (int)k0;
        return (uint32_t)((rr >> 3) * (int)rg + (kk >> 3) * 128 + (rr & 7) * 16 + (kk & 7) * 2);
    }
};
constexpr NonePlace kNoneTile{256u, 0u, 0u};  // a standalone [rows][16] tile

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
// Optional outputs: `wq` (Q Gamma hi into rows wq_row0 + r of an SW128 tile of wq_rows rows,
// multiplied per channel by `wq_scale` if that is not null) and `kt` may be null; `kt_place` /
// `kt_lo` place the transposed (K Gamma_C / Gamma) hi/lo tiles inside a larger operand; `kr`, if
// not null, receives (K Gamma_C / Gamma) row-major hi/lo ([16][LROW] each).
template <class Map>
__device__ __forceinline__ void prep_factors(unsigned char* sm, int p, int len, unsigned char* wq, unsigned char* kt,
                                             float* gc, float expA, float g_min, bool zero_v,
                                             uint32_t kt_lo = NONE_TILE, NonePlace kt_place = kNoneTile,
                                             int wq_row0 = C, int wq_rows = 2 * C, unsigned char* kr = nullptr,
                                             const float* wq_scale = nullptr)
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
    const float2 wsc = wq_scale ? *reinterpret_cast<const float2*>(wq_scale + c0) : make_float2(1.f, 1.f);
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
        if (wq) {
            const uint32_t wv = wq_scale ? pack_f2(qv[e].x * eG0 * wsc.x, qv[e].y * eG1 * wsc.y) : hi;
            *reinterpret_cast<uint32_t*>(wq + tc::sw128_off(wq_row0 + r, c0, wq_rows)) = wv;
        }
        split2(kv[e].x * iG0, kv[e].y * iG1, hi, lo);
        sKd[ri] = hi;
        sKdl[ri] = lo;
        uint32_t th, tl;
        split2(kv[e].x * (eGC0 * iG0), kv[e].y * (eGC1 * iG1), th, tl);  // k Gamma_C / Gamma <= 1
        if (kr) {
            reinterpret_cast<uint32_t*>(kr)[ri] = th;
            reinterpret_cast<uint32_t*>(kr)[C * LROW / 2 + ri] = tl;
        }
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
    if (kt) {
        const uint32_t o0 = kt_place.off(c0, r0), o1 = kt_place.off(c0 + 1, r0);
        *reinterpret_cast<uint2*>(kt + o0) = make_uint2(kh0[0], kh0[1]);
        *reinterpret_cast<uint2*>(kt + o1) = make_uint2(kh1[0], kh1[1]);
        *reinterpret_cast<uint2*>(kt + kt_lo + o0) = make_uint2(kl0[0], kl0[1]);
        *reinterpret_cast<uint2*>(kt + kt_lo + o1) = make_uint2(kl1[0], kl1[1]);
    }
}

// Variants of the per-chunk solve (template argument of prep_solve).
enum SolveVariant : int {
    SOLVE_ONE = 0,    // a chunk on its own
    SOLVE_FIRST = 1,  // chunk a of a pair: also zeroes the upper-right block of the pair's P
    SOLVE_SECOND = 2  // chunk b of a pair: also the cross products with chunk a's K~ (below)
};

// A and P over K = 128 with mma.sync, partial sums reduced in shared memory (OFF_PART, 8 KB);
// then T = (I + A)^-1 by forward substitution and T' = T diag(beta) (hi/lo, OFF_T), P finalised
// into `pb` and `pb + p_lo` (hi/lo, placed by p_place).  beta of the chunk is read from OFF_BETA.
// SOLVE_ONE / SOLVE_FIRST: warps 0..3 A, warps 4..7 P as hi*hi + hi*lo + lo*hi, two k-steps each.
// SOLVE_SECOND: chunk a's K~ = K Gamma_C / Gamma (row-major hi/lo at Map::OFF_KRA) also enters
//   Y = (K Gamma) K~_a^T  (so that X = W K~_a^T = T' Y)   -> bf16 hi/lo B operand at Map::OFF_YT
//   Z = (Q Gamma) K~_a^T  (the pair's lower-left output block) -> `pb` rows 16..31, tokens 0..15
// with warp 0: A, warps 1, 2: Y (K~ hi, lo), warps 3..5: P, warps 6, 7: Z (k-steps 0..3, 4..7).
// Two barriers (Map::NB) inside.
template <class Map, int VAR = SOLVE_ONE>
__device__ __forceinline__ void prep_solve(unsigned char* sm, int p, unsigned char* pb, uint32_t p_lo = SMALL_TILE,
                                           NonePlace p_place = kNoneTile)
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
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if constexpr (VAR != SOLVE_SECOND) {
            const int k0 = 32 * (pw & 3);
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
        } else {
            const __nv_bfloat16* sKa = reinterpret_cast<const __nv_bfloat16*>(sm + Map::OFF_KRA);
            const __nv_bfloat16* sKal = sKa + C * LROW;
            // one product over all eight k-steps per warp (two half-ranges of three for Z)
            const __nv_bfloat16* L = (pw < 3) ? sLl : (pw == 4 ? sQl : (pw == 5 ? sQll : sQl));
            const __nv_bfloat16* R = (pw == 0)   ? sKd
                                     : (pw == 1) ? sKa
                                     : (pw == 2) ? sKal
                                     : (pw == 3) ? sKd
                                     : (pw == 4) ? sKdl
                                     : (pw == 5) ? sKd
                                                 : sKa;
            if (pw < 6) {
#pragma unroll 4
                for (int k0 = 0; k0 < D; k0 += 16) mma_kstep(acc, L, R, k0, lane);
            } else {
                const int kb = 64 * (pw - 6);
#pragma unroll 2
                for (int k0 = kb; k0 < kb + 64; k0 += 16) {
                    mma_kstep(acc, sQl, sKa, k0, lane);
                    mma_kstep(acc, sQl, sKal, k0, lane);
                    mma_kstep(acc, sQll, sKa, k0, lane);
                }
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
        const int idx = p;  // one entry of each 16 x 16 result per thread
        const int r = idx >> 4, i = idx & 15;
        float sa, sp;
        if constexpr (VAR != SOLVE_SECOND) {
            sa = 0.f;
            sp = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                sa += part[k * C * C + idx];
                sp += part[(4 + k) * C * C + idx];
            }
        } else {
            sa = part[idx];
            sp = part[3 * C * C + idx] + part[4 * C * C + idx] + part[5 * C * C + idx];
            const float sy = part[1 * C * C + idx] + part[2 * C * C + idx];
            const float sz = part[6 * C * C + idx] + part[7 * C * C + idx];
            __nv_bfloat16 hi, lo;
            // Y[r][i] as the B operand of T' Y: element (k = r, n = i) of a no-swizzle [16 n][16 k] tile
            split_bf16(sy, hi, lo);
            st_bf16(sm, Map::OFF_YT + tc::none_off(i, r), hi);
            st_bf16(sm, Map::OFF_YT + SMALL_TILE + tc::none_off(i, r), lo);
            split_bf16(sz, hi, lo);
            const NonePlace zp{p_place.rg, p_place.row0, p_place.k0 - C};
            st_bf16(pb, zp.off(r, i), hi);
            st_bf16(pb, p_lo + zp.off(r, i), lo);
        }
        sA[idx] = (i < r) ? beta[r] * sa : 0.f;
        __nv_bfloat16 hi, lo;
        split_bf16((i <= r) ? sp : 0.f, hi, lo);
        st_bf16(pb, p_place.off(r, i), hi);
        st_bf16(pb, p_lo + p_place.off(r, i), lo);
        if constexpr (VAR == SOLVE_FIRST) {
            const NonePlace up{p_place.rg, p_place.row0, p_place.k0 + C};
            st_bf16(pb, up.off(r, i), __float2bfloat16_rn(0.f));
            st_bf16(pb, p_lo + up.off(r, i), __float2bfloat16_rn(0.f));
        }
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
