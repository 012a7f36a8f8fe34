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
// layout; 264: padded, so that the transposed per-channel stores of prep_factors spread over the
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

constexpr float kLog2e = 1.4426950408889634f;

// 2^x and 1/x by the hardware approximations (relative errors ~2^-22, far below bf16)
__device__ __forceinline__ float ex2_fast(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_fast(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// a packed pair of bf16 as two floats (low half first)
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
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
__device__ __forceinline__ uint32_t pack_f2(float2 x) { return pack_f2(x.x, x.y); }

// x = hi + lo as bf16 pairs, the residual by one packed subtraction
__device__ __forceinline__ void split2v(float2 x, uint32_t& hi, uint32_t& lo)
{
    hi = pack_f2(x);
    lo = pack_f2(__fadd2_rn(x, make_float2(-__uint_as_float(hi << 16), -__uint_as_float(hi & 0xffff0000u))));
}

// mma.sync operands of row-major [16][LROW] bf16 tiles by ldmatrix (rows 272 bytes apart, so the
// eight rows of each 8 x 8 matrix fall on distinct banks)
__device__ __forceinline__ void ldsm4(const void* p, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(tc::smem_u32(p)));
}
// A fragment: rows 0..15 of L, columns k0 .. k0 + 15
__device__ __forceinline__ void frag_a(const __nv_bfloat16* L, int k0, int lane, uint32_t (&a)[4])
{
    ldsm4(L + ((lane & 7) + 8 * ((lane >> 3) & 1)) * LROW + k0 + 8 * (lane >> 4), a);
}
// B fragments of the two n-tiles (rows 0..7 and 8..15 of R: b[0..1] and b[2..3]), columns k0 .. k0 + 15
__device__ __forceinline__ void frag_b(const __nv_bfloat16* R, int k0, int lane, uint32_t (&b)[4])
{
    ldsm4(R + ((lane & 7) + 8 * (lane >> 4)) * LROW + k0 + 8 * ((lane >> 3) & 1), b);
}
// acc += A B^T over one k-step for both n-tiles
__device__ __forceinline__ void mma2(float (&acc)[2][4], const uint32_t (&a)[4], const uint32_t (&b)[4])
{
    tc::mma16816(acc[0], a, b[0], b[1]);
    tc::mma16816(acc[1], a, b[2], b[3]);
}
// acc += (Lh + Ll)(Rh + Rl)^T without the lo*lo term, over k-steps [k0, k1)
__device__ __forceinline__ void mma_hilo(float (&acc)[2][4], const __nv_bfloat16* Lh, const __nv_bfloat16* Ll,
                                         const __nv_bfloat16* Rh, const __nv_bfloat16* Rl, int k0, int k1, int lane)
{
    for (int k = k0; k < k1; k += 16) {
        uint32_t ah[4], al[4], bh[4], bl[4];
        frag_a(Lh, k, lane, ah);
        frag_a(Ll, k, lane, al);
        frag_b(Rh, k, lane, bh);
        frag_b(Rl, k, lane, bl);
        mma2(acc, ah, bh);
        mma2(acc, ah, bl);
        mma2(acc, al, bh);
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

    // Both channels of the pair go through packed fp32 arithmetic.  Decays are kept in base 2:
    // the gate g log2(e) = g_min log2(e) / (1 + 2^(-log2(e) e^{A_h} z)) (Equation 5), G its in-chunk
    // cumulative sum, Gamma = 2^G and 1/Gamma = 2^-G.
    const float2 zs = make_float2(-kLog2e * expA, -kLog2e * expA);
    const float2 gm = make_float2(kLog2e * g_min, kLog2e * g_min);
    const float2 one = make_float2(1.f, 1.f);
    float2 G[4], kv[4], qv[4];
    uint32_t vv[4];
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int r = r0 + e;
        const bool ok = r < len;
        const uint32_t zw = tz32[(r * D + c0) >> 1];
        const float2 y = __fmul2_rn(zs, bf2_to_f2(zw));
        const float2 den = __fadd2_rn(one, make_float2(ex2_fast(y.x), ex2_fast(y.y)));
        const float2 g = __fmul2_rn(gm, make_float2(rcp_fast(den.x), rcp_fast(den.y)));
        acc = ok ? __fadd2_rn(acc, g) : acc;
        G[e] = acc;
        kv[e] = bf2_to_f2(ok ? tk32[(r * D + c0) >> 1] : 0u);
        qv[e] = bf2_to_f2(ok ? tq32[(r * D + c0) >> 1] : 0u);
        vv[e] = (ok && !zero_v) ? tv32[(r * D + c0) >> 1] : 0u;
    }
    *reinterpret_cast<float2*>(hs + tq * D + c0) = acc;
    named_sync(Map::NB, NGROUP);
    float2 off = make_float2(0.f, 0.f), tot = make_float2(0.f, 0.f);
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
        const float2 hq = *reinterpret_cast<const float2*>(hs + qq * D + c0);
        if (qq < tq) off = __fadd2_rn(off, hq);
        tot = __fadd2_rn(tot, hq);
    }
    const float2 eGC = make_float2(ex2_fast(tot.x), ex2_fast(tot.y));
    if (tq == 3) *reinterpret_cast<float2*>(gc + c0) = eGC;
    const float2 wsc = wq_scale ? *reinterpret_cast<const float2*>(wq_scale + c0) : one;

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
        const float2 Gs = __fadd2_rn(G[e], off);
        const float2 eG = make_float2(ex2_fast(Gs.x), ex2_fast(Gs.y));     // Gamma in [e^-80, 1]
        const float2 iG = make_float2(ex2_fast(-Gs.x), ex2_fast(-Gs.y));   // 1/Gamma in [1, e^80]
        const uint32_t llw = pack_f2(__fmul2_rn(kv[e], eG));
        const int ri = (r * LROW + c0) >> 1;
        sLl[ri] = llw;
        const float2 qg = __fmul2_rn(qv[e], eG);
        uint32_t hi, lo;
        split2v(qg, hi, lo);
        sQl[ri] = hi;
        sQll[ri] = lo;
        if (wq) {
            const uint32_t wv = wq_scale ? pack_f2(__fmul2_rn(qg, wsc)) : hi;
            *reinterpret_cast<uint32_t*>(wq + tc::sw128_off(wq_row0 + r, c0, wq_rows)) = wv;
        }
        split2v(__fmul2_rn(kv[e], iG), hi, lo);
        sKd[ri] = hi;
        sKdl[ri] = lo;
        uint32_t th, tl;
        split2v(__fmul2_rn(kv[e], __fmul2_rn(eGC, iG)), th, tl);  // k Gamma_C / Gamma <= 1
        if (kr) {
            reinterpret_cast<uint32_t*>(kr)[ri] = th;
            reinterpret_cast<uint32_t*>(kr)[C * LROW / 2 + ri] = tl;
        }
        // de-interleave the pairs into per-channel token runs
        const int slot = e >> 1;
        if ((e & 1) == 0) {
            xt0[slot] = llw & 0xffffu;
            xt1[slot] = llw >> 16;
            kh0[slot] = th & 0xffffu;
            kh1[slot] = th >> 16;
            kl0[slot] = tl & 0xffffu;
            kl1[slot] = tl >> 16;
        } else {
            xt0[slot] = __byte_perm(xt0[slot], llw, 0x5410);
            xt1[slot] = __byte_perm(xt1[slot], llw, 0x7610);
            kh0[slot] = __byte_perm(kh0[slot], th, 0x5410);
            kh1[slot] = __byte_perm(kh1[slot], th, 0x7610);
            kl0[slot] = __byte_perm(kl0[slot], tl, 0x5410);
            kl1[slot] = __byte_perm(kl1[slot], tl, 0x7610);
        }
    }
    const uint32_t v00 = __byte_perm(vv[0], vv[1], 0x5410), v01 = __byte_perm(vv[2], vv[3], 0x5410);
    const uint32_t v10 = __byte_perm(vv[0], vv[1], 0x7632), v11 = __byte_perm(vv[2], vv[3], 0x7632);
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

// Index of element (r, c) of a 16 x 16 fp32 partial tile: rows with bit 1 set hold their two
// column halves swapped.
__device__ __forceinline__ int part_idx(int r, int c) { return r * C + (c ^ (((r >> 1) & 1) << 3)); }

// A and P over K = 128 with mma.sync, partial sums reduced in shared memory (OFF_PART, 8 KB);
// then T = (I + A)^-1 by forward substitution and T' = T diag(beta) (hi/lo, OFF_T), P finalised
// into `pb` and `pb + p_lo` (hi/lo, placed by p_place).  beta of the chunk is read from OFF_BETA.
// SOLVE_ONE / SOLVE_FIRST: warps 0..3 A, warps 4..7 P as hi*hi + hi*lo + lo*hi, two k-steps each.
// SOLVE_SECOND: chunk a's K~ = K Gamma_C / Gamma (row-major hi/lo at Map::OFF_KRA) also enters
//   Y = (K Gamma) K~_a^T  (so that X = W K~_a^T = T' Y)   -> bf16 hi/lo B operand at Map::OFF_YT
//   Z = (Q Gamma) K~_a^T  (the pair's lower-left output block) -> `pb` rows 16..31, tokens 0..15
// with warp 0: A, warps 1, 2: Y (k-steps 0..3, 4..7), warps 3..5: P (k-steps 0..2, 3..5, 6..7),
// warps 6, 7: Z (k-steps 0..3, 4..7).
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
#pragma unroll
                for (int k = k0; k < k0 + 32; k += 16) {
                    uint32_t a[4], b[4];
                    frag_a(sLl, k, lane, a);
                    frag_b(sKd, k, lane, b);
                    mma2(acc, a, b);
                }
            } else {
                mma_hilo(acc, sQl, sQll, sKd, sKdl, k0, k0 + 32, lane);
            }
        } else {
            const __nv_bfloat16* sKa = reinterpret_cast<const __nv_bfloat16*>(sm + Map::OFF_KRA);
            const __nv_bfloat16* sKal = sKa + C * LROW;
            if (pw == 0) {  // A over all k-steps
#pragma unroll 4
                for (int k = 0; k < D; k += 16) {
                    uint32_t a[4], b[4];
                    frag_a(sLl, k, lane, a);
                    frag_b(sKd, k, lane, b);
                    mma2(acc, a, b);
                }
            } else if (pw < 3) {  // Y = (K Gamma) (K~hi + K~lo)^T over one half of the k-steps
#pragma unroll 2
                for (int k = 64 * (pw - 1); k < 64 * pw; k += 16) {
                    uint32_t a[4], bh[4], bl[4];
                    frag_a(sLl, k, lane, a);
                    frag_b(sKa, k, lane, bh);
                    frag_b(sKal, k, lane, bl);
                    mma2(acc, a, bh);
                    mma2(acc, a, bl);
                }
            } else if (pw < 6) {  // P over k-steps [0, 3), [3, 6), [6, 8)
                const int kb = 48 * (pw - 3);
                mma_hilo(acc, sQl, sQll, sKd, sKdl, kb, min(kb + 48, D), lane);
            } else {  // Z over one half of the k-steps
                mma_hilo(acc, sQl, sQll, sKa, sKal, 64 * (pw - 6), 64 * (pw - 5), lane);
            }
        }
        // partial tiles [16][16] with the column halves of rows 2, 3 (mod 4) swapped, so that each
        // half-warp's 8-byte stores cover all 32 banks (part_idx)
        float* pp = part + pw * C * C;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            *reinterpret_cast<float2*>(pp + part_idx(g, 8 * nt + 2 * t)) = make_float2(acc[nt][0], acc[nt][1]);
            *reinterpret_cast<float2*>(pp + part_idx(g + 8, 8 * nt + 2 * t)) = make_float2(acc[nt][2], acc[nt][3]);
        }
    }
    named_sync(Map::NB, NGROUP);
    {
        const int r = p >> 4, i = p & 15;  // one entry of each 16 x 16 result per thread
        const int idx = part_idx(r, i);
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
        sA[p] = (i < r) ? beta[r] * sa : 0.f;
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
