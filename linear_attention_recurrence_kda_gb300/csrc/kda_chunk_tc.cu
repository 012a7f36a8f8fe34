// kda_chunk_tc.cu -- fused KDA prefill on the sm_103a tensor cores (bf16 inputs, d_k = d_v = 128).
//
// One CTA walks one sequence of one head in 16-token chunks and does, per chunk, every stage of
// the chunk form of Equation 1 ("Kimi K3: the paper and proofs side by side", section 2.1.1):
//
//   gate      g = g_min sigmoid(e^{A_h} z)  (Equation 5), G_r = in-chunk inclusive cumsum,
//             Gamma_r = e^{G_r}.  With g_min = -5 a 16-token chunk keeps G in [-80, 0] ("Kimi K3"
//             reading notes, section 2), so both Gamma_r and 1/Gamma_r are normal fp32/bf16
//             numbers and one reference point per chunk (its start) suffices.
//   UT / WY   A[r][i] = beta_r <k_r Gamma_r, k_i / Gamma_i> (i < r), T = (I + A)^-1,
//             W = T diag(beta) (K Gamma),  U~ = T diag(beta) V
//   chain     U = U~ - W S,   O = (Q Gamma) S + tril_incl((Q Gamma)(K / Gamma)^T) U,
//             S <- Diag(Gamma_C) S + (K Gamma_C / Gamma)^T U
// (derivation: substitute the token recurrence into itself across the chunk; the regrouping is
// exact -- "Kimi K3: architecture, derivations and a pinned-source audit", section 4.5).
//
// Mapping onto the hardware (value channels j and key channels c are the 128 TMEM lanes):
//   * 16x16 products A = (K Gamma)(K/Gamma)^T and P = (Q Gamma)(K/Gamma)^T: warp-level mma.sync
//     (their M is 16, below the tensor-core instruction's minimum of 64);
//   * T by fp32 forward substitution (one lane per column); beta is folded into its columns,
//     T' = T diag(beta), so that V enters the tensor core exactly as given;
//   * W^T = (K Gamma)^T T'^T and U~^T = V^T T'^T: tcgen05, M = 128 channels, N = K = 16;
//   * D1 = S^T [W ; Q Gamma]^T (M = 128, N = 32, K = 128), then U^T = U~^T - D1[:, :16] and
//     D1[:, 16:] += U^T P^T (N = K = 16) gives O^T, and dS^T = U^T (K Gamma_C/Gamma) (N = 128,
//     K = 16): tcgen05 with fp32 accumulators in tensor memory;
//   * the fp32 state S^T lives in registers (thread = one value channel x 64 key channels) and is
//     re-staged as a bf16 SW128 operand after every chunk.
// Precision: outputs are compared with the exact result as max|error| / RMS(output), and the
// outputs of long sequences are heavy-tailed (max/RMS ~ 14), so a single bf16 rounding of an
// operand on the output path already costs ~2e-2 of that budget.  The operands whose rounding
// reaches the outputs directly are therefore carried as bf16 pairs x = hi + lo (hi = bf16(x),
// lo = bf16(x - hi), ~16 significant bits) and multiplied as hi*hi + hi*lo + lo*hi: Q Gamma and
// K/Gamma inside P, P and U in U P^T, U and K Gamma_C/Gamma in the state update, and T'.  The
// remaining bf16 roundings (the state as the read operand, W, K Gamma) reach the outputs only
// through products that the decay keeps small.
// The loop is software-pipelined across chunks: while the tensor core runs chunk n's state-read,
// output and state-update products, all 256 threads prepare chunk n+1 (gate, factors, A, P, T')
// into the other half of double-buffered operand tiles, and TMA fetches chunk n+2's inputs.
// Every mbarrier wait is bounded; a wait that gives up raises the timeout bit of the check word
// and the CTA stops cleanly.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {

namespace {

constexpr int D = 128;            // d_k = d_v
constexpr int C = kChunk;         // 16
constexpr int NTHREADS = 256;
constexpr int LROW = 136;         // padded row (elements) of the mma.sync operand tiles
constexpr uint32_t WAIT_LIMIT = 1u << 24;

// shared-memory map (bytes from a 1024-aligned base); "[2]" = double-buffered by chunk parity
constexpr uint32_t OFF_S = 0;          // S^T [128 j][128 c] SW128                      32768
constexpr uint32_t OFF_WQ = 32768;     // [2] [W ; Q Gamma] [32][128 c] SW128            2 x 8192
constexpr uint32_t OFF_STAGE = 49152;  // q, k, v, z tiles [16][128] bf16 (TMA)         16384
constexpr uint32_t OFF_KT = 65536;     // [2] (K Gamma_C/Gamma)^T hi, lo [128 c][16 i]   2 x 8192
constexpr uint32_t OFF_XT = 81920;     // (K Gamma)^T [128 c][16 i] NONE                4096
constexpr uint32_t OFF_VT = 86016;     // V^T [128 j][16 i] NONE                        4096
constexpr uint32_t OFF_UT = 90112;     // U^T hi, lo [128 j][16 i] NONE                 8192
constexpr uint32_t OFF_P = 98304;      // [2] P hi, lo [16 r][16 i] NONE                 2 x 1024
constexpr uint32_t OFF_T = 100352;     // T' hi, lo [16 r][16 i] NONE                   1024
constexpr uint32_t OFF_LL = 101376;    // K Gamma [16][LROW] bf16                       4352
constexpr uint32_t OFF_QL = 105728;    // Q Gamma hi, lo                                2 x 4352
constexpr uint32_t OFF_KD = 114432;    // K / Gamma hi, lo                              2 x 4352
constexpr uint32_t OFF_A = 123136;     // A fp32 [16][16]                               1024
constexpr uint32_t OFF_PF = 124160;    // P partial sums fp32 [2][16][16]               2048
constexpr uint32_t OFF_GC = 126208;    // [2] Gamma_C fp32 [128]                         2 x 512
constexpr uint32_t OFF_HS = 127232;    // per-channel half-chunk log-decay sums [2][128] 1024
constexpr uint32_t OFF_BETA = 128256;  // [2] beta [16]                                  2 x 64
constexpr uint32_t OFF_BAR = 128384;   // mbarrier of the tensor-core commits           8
constexpr uint32_t OFF_BARLD = 128392; // mbarrier of the TMA tile loads                8
constexpr uint32_t OFF_TSLOT = 128400; // TMEM base address                             4
constexpr uint32_t OFF_ABORT = 128404; // stop flag                                     4
constexpr uint32_t SMEM_USED = 128408;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
constexpr uint32_t STAGE_TILE = C * D * 2;  // 4096 bytes per tensor and chunk
constexpr uint32_t NONE_TILE = 4096;        // [128][16] bf16 NONE tile
constexpr uint32_t SMALL_TILE = 512;        // [16][16] bf16 NONE tile

// tensor-memory columns
constexpr uint32_t TM_D1 = 0;    // [0,16): (W S)^T, [16,32): O^T
constexpr uint32_t TM_W = 32;    // W^T  (lanes = c)
constexpr uint32_t TM_U = 48;    // U~^T (lanes = j)
constexpr uint32_t TM_D3 = 128;  // dS^T (lanes = j, columns = c)
constexpr uint32_t TM_COLS = 256;

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

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

__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 a, __nv_bfloat16 b)
{
    return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

// acc[16 x 16] += L R^T over K = 128 (L, R: 16 rows of LROW bf16) with mma.sync m16n8k16.
__device__ __forceinline__ void mma_rows16(float (&acc)[2][4], const __nv_bfloat16* L, const __nv_bfloat16* R, int lane)
{
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const int k0 = 16 * ks;
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
}

// Commit the issued tensor-core work, bounded wait by thread 0, CTA barrier.  False: stop.
__device__ __forceinline__ bool tc_join(uint64_t* bar, uint32_t& phase, volatile uint32_t* abort_flag)
{
    if (threadIdx.x == 0) {
        tc::umma_commit(bar);
        if (!tc::mbar_wait(bar, phase, WAIT_LIMIT)) *abort_flag = 1u;
    }
    phase ^= 1u;
    __syncthreads();
    tc::fence_after_sync();
    return *abort_flag == 0u;
}

// Generic-proxy writes to operand tiles -> visible to the tensor core; CTA barrier.
__device__ __forceinline__ void tc_publish()
{
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
}

struct Ctx {
    unsigned char* sm;
    int tid, w, lane;
    int h, H;
    float expA, g_min;
};

// Gate, in-chunk cumulative log-decay and every per-element factor of one chunk (all threads).
// Thread (c, half) owns key/value channel c and tokens [8 half, 8 half + 8).
// Writes: row-major K Gamma, Q Gamma (hi/lo), K/Gamma (hi/lo); WQ[b] rows 16..31 (Q Gamma hi);
// (K Gamma)^T, V^T; KT[b] (K Gamma_C/Gamma hi/lo); GC[b] = Gamma_C.  Contains one CTA barrier.
__device__ __forceinline__ void prep_factors(const Ctx& x, int len, int b)
{
    unsigned char* sm = x.sm;
    const int c = x.tid & (D - 1);
    const int half = x.tid >> 7;
    const int r0 = 8 * half;
    const __nv_bfloat16* tq = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_STAGE);
    const __nv_bfloat16* tk = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_STAGE + STAGE_TILE);
    const __nv_bfloat16* tv = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_STAGE + 2 * STAGE_TILE);
    const __nv_bfloat16* tz = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_STAGE + 3 * STAGE_TILE);
    float* hs = reinterpret_cast<float*>(sm + OFF_HS);

    float Gl[8], kv[8], qv[8];
    uint32_t vpk[4];
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int r = r0 + e;
        const bool ok = r < len;
        const float g = ok ? log_decay(__bfloat162float(tz[r * D + c]), x.expA, x.g_min) : 0.f;
        acc += g;
        Gl[e] = acc;
        kv[e] = ok ? __bfloat162float(tk[r * D + c]) : 0.f;
        qv[e] = ok ? __bfloat162float(tq[r * D + c]) : 0.f;
    }
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const __nv_bfloat16 z0 = __float2bfloat16_rn(0.f);
        vpk[e / 2] = pack2((r0 + e < len) ? tv[(r0 + e) * D + c] : z0, (r0 + e + 1 < len) ? tv[(r0 + e + 1) * D + c] : z0);
    }
    hs[half * D + c] = acc;
    __syncthreads();
    const float off = half ? hs[c] : 0.f;
    const float GC = hs[c] + hs[D + c];
    const float eGC = expf(GC);
    if (half) reinterpret_cast<float*>(sm + OFF_GC + b * 512)[c] = eGC;

    __nv_bfloat16* sLl = reinterpret_cast<__nv_bfloat16*>(sm + OFF_LL);
    __nv_bfloat16* sQl = reinterpret_cast<__nv_bfloat16*>(sm + OFF_QL);
    __nv_bfloat16* sQll = sQl + C * LROW;
    __nv_bfloat16* sKd = reinterpret_cast<__nv_bfloat16*>(sm + OFF_KD);
    __nv_bfloat16* sKdl = sKd + C * LROW;
    unsigned char* wq = sm + OFF_WQ + b * 8192;
    __nv_bfloat16 xt[8], kth[8], ktl[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int r = r0 + e;
        const float eG = expf(Gl[e] + off);      // Gamma_r in [e^-80, 1]
        const float ieG = __frcp_rn(eG);          // 1 / Gamma_r in [1, e^80]
        const float ll = kv[e] * eG;
        __nv_bfloat16 hi, lo;
        xt[e] = __float2bfloat16_rn(ll);
        sLl[r * LROW + c] = xt[e];
        split_bf16(qv[e] * eG, hi, lo);
        sQl[r * LROW + c] = hi;
        sQll[r * LROW + c] = lo;
        st_bf16(wq, tc::sw128_off(C + r, c, 2 * C), hi);
        split_bf16(kv[e] * ieG, hi, lo);
        sKd[r * LROW + c] = hi;
        sKdl[r * LROW + c] = lo;
        split_bf16(kv[e] * (eGC * ieG), kth[e], ktl[e]);   // k Gamma_C / Gamma_r <= 1
    }
    *reinterpret_cast<uint4*>(sm + OFF_XT + tc::none_off(c, r0)) =
        make_uint4(pack2(xt[0], xt[1]), pack2(xt[2], xt[3]), pack2(xt[4], xt[5]), pack2(xt[6], xt[7]));
    *reinterpret_cast<uint4*>(sm + OFF_VT + tc::none_off(c, r0)) = make_uint4(vpk[0], vpk[1], vpk[2], vpk[3]);
    unsigned char* kt = sm + OFF_KT + b * 8192;
    *reinterpret_cast<uint4*>(kt + tc::none_off(c, r0)) =
        make_uint4(pack2(kth[0], kth[1]), pack2(kth[2], kth[3]), pack2(kth[4], kth[5]), pack2(kth[6], kth[7]));
    *reinterpret_cast<uint4*>(kt + NONE_TILE + tc::none_off(c, r0)) =
        make_uint4(pack2(ktl[0], ktl[1]), pack2(ktl[2], ktl[3]), pack2(ktl[4], ktl[5]), pack2(ktl[6], ktl[7]));
}

// A, P (mma.sync), T = (I + A)^-1 and T' = T diag(beta) (hi/lo), P finalised into P[b] (hi/lo).
// Contains one CTA barrier; the caller publishes afterwards.
__device__ __forceinline__ void prep_solve(const Ctx& x, int b)
{
    unsigned char* sm = x.sm;
    const int w = x.w, lane = x.lane, tid = x.tid;
    float* sA = reinterpret_cast<float*>(sm + OFF_A);
    float* sPf = reinterpret_cast<float*>(sm + OFF_PF);
    const float* beta = reinterpret_cast<const float*>(sm + OFF_BETA + b * 64);
    const __nv_bfloat16* sLl = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_LL);
    const __nv_bfloat16* sQl = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_QL);
    const __nv_bfloat16* sQll = sQl + C * LROW;
    const __nv_bfloat16* sKd = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_KD);
    const __nv_bfloat16* sKdl = sKd + C * LROW;
    if (w < 3) {
        const int g = lane >> 2, t = lane & 3;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if (w == 0) {
            mma_rows16(acc, sLl, sKd, lane);
        } else if (w == 1) {
            mma_rows16(acc, sQl, sKd, lane);
            mma_rows16(acc, sQl, sKdl, lane);
        } else {
            mma_rows16(acc, sQll, sKd, lane);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = g + ((e >> 1) << 3);
                const int i = 8 * nt + 2 * t + (e & 1);
                if (w == 0) {
                    sA[r * C + i] = (i < r) ? beta[r] * acc[nt][e] : 0.f;
                } else {
                    sPf[(w - 1) * C * C + r * C + i] = acc[nt][e];
                }
            }
        }
    }
    __syncthreads();
    if (w == 0 && lane < C) {
        // forward substitution, one lane per column j: T[r][j] = delta_rj - sum_{i<r} A[r][i] T[i][j]
        const int j = lane;
        float tcol[C];
#pragma unroll
        for (int r = 0; r < C; ++r) {
            float p0 = (r == j) ? 1.f : 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
            for (int i = 0; i < r; i += 4) {
                p0 -= sA[r * C + i] * tcol[i];
                if (i + 1 < r) p1 -= sA[r * C + i + 1] * tcol[i + 1];
                if (i + 2 < r) p2 -= sA[r * C + i + 2] * tcol[i + 2];
                if (i + 3 < r) p3 -= sA[r * C + i + 3] * tcol[i + 3];
            }
            tcol[r] = (p0 + p1) + (p2 + p3);
        }
        const float bj = beta[j];
#pragma unroll
        for (int r = 0; r < C; ++r) {
            __nv_bfloat16 hi, lo;
            split_bf16(tcol[r] * bj, hi, lo);
            st_bf16(sm, OFF_T + tc::none_off(r, j), hi);
            st_bf16(sm, OFF_T + SMALL_TILE + tc::none_off(r, j), lo);
        }
    } else if (tid >= 128) {
        unsigned char* pb = sm + OFF_P + b * 1024;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int idx = 2 * (tid - 128) + e;
            const int r = idx >> 4, i = idx & 15;
            const float pv = (i <= r) ? sPf[idx] + sPf[C * C + idx] : 0.f;
            __nv_bfloat16 hi, lo;
            split_bf16(pv, hi, lo);
            st_bf16(pb, tc::none_off(r, i), hi);
            st_bf16(pb, SMALL_TILE + tc::none_off(r, i), lo);
        }
    }
}

}  // namespace

struct TileMaps {
    CUtensorMap q, k, v, z;  // 3-D views [T_tot][H][128] of the bf16 inputs, box [16][1][128]
};

__global__ void __launch_bounds__(NTHREADS, 1) kda_chunk_fwd_tc_kernel(PrefillArgs a, const __grid_constant__ TileMaps maps)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint64_t* bar_ld = reinterpret_cast<uint64_t*>(sm + OFF_BARLD);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_TSLOT);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sm + OFF_ABORT);

    const int n = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int w = tid >> 5;
    const int lane = tid & 31;
    const int q4 = w & 3;    // TMEM lane quarter
    const int h2 = w >> 2;   // which half of the columns this warp handles
    const int jrow = 32 * q4 + lane;

    int64_t s0, s1;
    if (!seq_range(a, n, s0, s1)) return;
    const int H = a.H;
    const Ctx x{sm, tid, w, lane, h, H, expf(a.A[h]), a.g_min};
    __nv_bfloat16* op = static_cast<__nv_bfloat16*>(a.out);
    const int nchunks = (int)((s1 - s0 + C - 1) / C);

    auto issue_tiles = [&](int chunk) {  // thread 0
        const int tn = (int)(s0 + (int64_t)chunk * C);
        tc::fence_async_smem();
        tc::mbar_arrive_expect_tx(bar_ld, 4 * STAGE_TILE);
        tc::tma_load_3d(sm + OFF_STAGE, &maps.q, 0, h, tn, bar_ld);
        tc::tma_load_3d(sm + OFF_STAGE + STAGE_TILE, &maps.k, 0, h, tn, bar_ld);
        tc::tma_load_3d(sm + OFF_STAGE + 2 * STAGE_TILE, &maps.v, 0, h, tn, bar_ld);
        tc::tma_load_3d(sm + OFF_STAGE + 3 * STAGE_TILE, &maps.z, 0, h, tn, bar_ld);
    };
    auto load_beta = [&](int chunk) -> float {  // threads 0..15
        const int64_t t = s0 + (int64_t)chunk * C + tid;
        return (chunk < nchunks && t < s1) ? a.beta[t * H + h] : 0.f;
    };
    auto chunk_len = [&](int chunk) -> int { return (int)min((int64_t)C, s1 - (s0 + (int64_t)chunk * C)); };

    if (w == 0) tc::tmem_alloc(tslot, TM_COLS);
    float beta_next = 0.f;
    if (tid == 0) {
        tc::mbar_init(bar, 1);
        tc::mbar_init(bar_ld, 1);
        *abort_flag = 0u;
        if (nchunks > 0) issue_tiles(0);
    }
    if (tid < C) beta_next = load_beta(0);

    // state slice: S[c][jrow] for c in [64*h2, 64*h2 + 64)
    float S[64];
    const int64_t sbase = ((int64_t)n * H + h) * D * D;
#pragma unroll
    for (int cc = 0; cc < 64; ++cc) {
        S[cc] = a.s0 ? a.s0[sbase + (int64_t)(64 * h2 + cc) * D + jrow] : 0.f;
    }
    auto stage_state = [&]() {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
            uint4 pk;
            pk.x = tc::pack_bf16(S[8 * ch + 0], S[8 * ch + 1]);
            pk.y = tc::pack_bf16(S[8 * ch + 2], S[8 * ch + 3]);
            pk.z = tc::pack_bf16(S[8 * ch + 4], S[8 * ch + 5]);
            pk.w = tc::pack_bf16(S[8 * ch + 6], S[8 * ch + 7]);
            *reinterpret_cast<uint4*>(sm + OFF_S + tc::sw128_chunk_off(jrow, 8 * h2 + ch, D)) = pk;
        }
    };
    stage_state();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tslot;
    const uint32_t lane_base = tbase + ((uint32_t)(32 * q4) << 16);
    uint32_t phase = 0, ld_phase = 0;

    // prepare chunk c into buffer (c & 1): wait for its tiles, factors, then prefetch chunk c+1
    auto prepare_factors = [&](int chunk) -> bool {
        const int b = chunk & 1;
        if (tid < C) reinterpret_cast<float*>(sm + OFF_BETA + b * 64)[tid] = beta_next;
        if (tid == 0 && !tc::mbar_wait(bar_ld, ld_phase, WAIT_LIMIT)) *abort_flag = 1u;
        ld_phase ^= 1u;
        __syncthreads();
        if (*abort_flag) return false;
        prep_factors(x, chunk_len(chunk), b);
        __syncthreads();  // stage consumed
        if (chunk + 1 < nchunks) {
            if (tid == 0) issue_tiles(chunk + 1);
            if (tid < C) beta_next = load_beta(chunk + 1);
        }
        return true;
    };
    auto issue_mw_mu = [&](int b) {  // thread 0: W^T = (K Gamma)^T T'^T, U~^T = V^T T'^T
        (void)b;
        const uint32_t id16 = tc::idesc_bf16(128, 16);
        const uint64_t dT = tc::desc_none(tc::smem_u32(sm + OFF_T));
        const uint64_t dTl = tc::desc_none(tc::smem_u32(sm + OFF_T + SMALL_TILE));
        const uint64_t dX = tc::desc_none(tc::smem_u32(sm + OFF_XT));
        const uint64_t dV = tc::desc_none(tc::smem_u32(sm + OFF_VT));
        tc::umma(tbase + TM_W, dX, dT, id16, 0u);
        tc::umma(tbase + TM_W, dX, dTl, id16, 1u);
        tc::umma(tbase + TM_U, dV, dT, id16, 0u);
        tc::umma(tbase + TM_U, dV, dTl, id16, 1u);
    };
    auto issue_m1 = [&](int b) {  // thread 0: D1 = S^T [W ; Q Gamma]^T (M = 128, N = 32, K = 128)
        const uint32_t id32 = tc::idesc_bf16(128, 2 * C);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
            tc::umma(tbase + TM_D1, tc::desc_sw128(tc::smem_u32(sm + OFF_S + kb * 16384 + off)),
                     tc::desc_sw128(tc::smem_u32(sm + OFF_WQ + b * 8192 + kb * (2 * C * 128) + off)), id32,
                     ks > 0 ? 1u : 0u);
        }
    };
    auto transpose_w = [&](int b) {  // warps 0..3: W^T (TMEM, lanes = c) -> rows 0..15 of WQ[b]
        if (w < 4) {
            uint32_t v[16];
            KDA_TMEM_LD16(lane_base + TM_W, v);
            tc::tmem_wait_ld();
            unsigned char* wq = sm + OFF_WQ + b * 8192;
#pragma unroll
            for (int r = 0; r < C; ++r) st_bf16(wq, tc::sw128_off(r, jrow, 2 * C), __float2bfloat16_rn(u2f(v[r])));
        }
    };

    bool ok = true;
    if (nchunks > 0) {
        // prologue: chunk 0 prepared and its state-read issued
        ok = prepare_factors(0);
        if (ok) {
            prep_solve(x, 0);
            tc_publish();
            if (tid == 0) issue_mw_mu(0);
            ok = tc_join(bar, phase, abort_flag);
        }
        if (ok) {
            transpose_w(0);
            tc_publish();
            if (tid == 0) issue_m1(0);
        }
    }

    for (int ch = 0; ok && ch < nchunks; ++ch) {
        const int b = ch & 1, nb = b ^ 1;
        const bool has_next = ch + 1 < nchunks;
        const int64_t t0 = s0 + (int64_t)ch * C;
        const int len = chunk_len(ch);

        // (1) while the state-read of chunk ch runs: factors of chunk ch+1
        if (has_next && !(ok = prepare_factors(ch + 1))) break;

        // (2) U^T = U~^T - (W S)^T as a hi/lo pair
        if (!(ok = tc_join(bar, phase, abort_flag))) break;
        {
            uint32_t dv[8], uv[8];
            KDA_TMEM_LD8(lane_base + TM_D1 + 8 * h2, dv);
            KDA_TMEM_LD8(lane_base + TM_U + 8 * h2, uv);
            tc::tmem_wait_ld();
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float u0 = u2f(uv[2 * e]) - u2f(dv[2 * e]);
                const float u1 = u2f(uv[2 * e + 1]) - u2f(dv[2 * e + 1]);
                __nv_bfloat162 h2v = __floats2bfloat162_rn(u0, u1);
                const float2 hf = __bfloat1622float2(h2v);
                __nv_bfloat162 l2v = __floats2bfloat162_rn(u0 - hf.x, u1 - hf.y);
                hi[e] = *reinterpret_cast<uint32_t*>(&h2v);
                lo[e] = *reinterpret_cast<uint32_t*>(&l2v);
            }
            *reinterpret_cast<uint4*>(sm + OFF_UT + tc::none_off(jrow, 8 * h2)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(sm + OFF_UT + NONE_TILE + tc::none_off(jrow, 8 * h2)) =
                make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        tc_publish();

        // (3) O^T += U^T P^T and dS^T = U^T (K Gamma_C / Gamma), each as hi*hi + hi*lo + lo*hi
        if (tid == 0) {
            const uint32_t id16 = tc::idesc_bf16(128, 16);
            const uint32_t id128 = tc::idesc_bf16(128, 128);
            const uint64_t dU = tc::desc_none(tc::smem_u32(sm + OFF_UT));
            const uint64_t dUl = tc::desc_none(tc::smem_u32(sm + OFF_UT + NONE_TILE));
            const uint64_t dP = tc::desc_none(tc::smem_u32(sm + OFF_P + b * 1024));
            const uint64_t dPl = tc::desc_none(tc::smem_u32(sm + OFF_P + b * 1024 + SMALL_TILE));
            const uint64_t dK = tc::desc_none(tc::smem_u32(sm + OFF_KT + b * 8192));
            const uint64_t dKl = tc::desc_none(tc::smem_u32(sm + OFF_KT + b * 8192 + NONE_TILE));
            tc::umma(tbase + TM_D1 + C, dU, dP, id16, 1u);
            tc::umma(tbase + TM_D1 + C, dU, dPl, id16, 1u);
            tc::umma(tbase + TM_D1 + C, dUl, dP, id16, 1u);
            tc::umma(tbase + TM_D3, dU, dK, id128, 0u);
            tc::umma(tbase + TM_D3, dU, dKl, id128, 1u);
            tc::umma(tbase + TM_D3, dUl, dK, id128, 1u);
        }

        // (4) while those run: A, P, T' of chunk ch+1, then its W / U~ products
        if (has_next) {
            prep_solve(x, nb);
            tc_publish();
            if (tid == 0) issue_mw_mu(nb);
        }
        if (!(ok = tc_join(bar, phase, abort_flag))) break;

        // (5) S <- Diag(Gamma_C) S + dS ; outputs of chunk ch ; W of chunk ch+1
        {
            const float* gc = reinterpret_cast<const float*>(sm + OFF_GC + b * 512) + 64 * h2;
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                uint32_t v[16];
                KDA_TMEM_LD16(lane_base + TM_D3 + 64 * h2 + 16 * blk, v);
                tc::tmem_wait_ld();
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    const float4 g4 = *reinterpret_cast<const float4*>(gc + 16 * blk + 4 * e4);
                    const int cc = 16 * blk + 4 * e4;
                    S[cc + 0] = g4.x * S[cc + 0] + u2f(v[4 * e4 + 0]);
                    S[cc + 1] = g4.y * S[cc + 1] + u2f(v[4 * e4 + 1]);
                    S[cc + 2] = g4.z * S[cc + 2] + u2f(v[4 * e4 + 2]);
                    S[cc + 3] = g4.w * S[cc + 3] + u2f(v[4 * e4 + 3]);
                }
            }
            stage_state();
            uint32_t ov[8];
            KDA_TMEM_LD8(lane_base + TM_D1 + C + 8 * h2, ov);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int r = 8 * h2 + e;
                if (r < len) op[((t0 + r) * H + h) * D + jrow] = __float2bfloat16_rn(u2f(ov[e]));
            }
        }
        if (has_next) {
            transpose_w(nb);
            tc_publish();
            if (tid == 0) issue_m1(nb);
        }
    }

    if (!ok || *abort_flag) {
        if (tid == 0) atomicOr(a.check, kCheckTimeout);
    } else if (a.s_final) {
#pragma unroll
        for (int cc = 0; cc < 64; ++cc) a.s_final[sbase + (int64_t)(64 * h2 + cc) * D + jrow] = S[cc];
    }
    tc::fence_before_sync();
    __syncthreads();
    if (w == 0) tc::tmem_dealloc(tbase, TM_COLS);
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        }
    });
    return fn;
}

// [T_tot][H][128] bf16 -> 3-D tensor map with a [16 tokens][1 head][128 channels] box.
bool encode_tile_map(CUtensorMap* m, const void* base, int64_t T_tot, int H)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T_tot};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    const cuuint32_t box[3] = {(cuuint32_t)D, 1u, (cuuint32_t)C};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_chunk_fwd_tc(const PrefillArgs& a, cudaStream_t s)
{
    TileMaps maps;
    if (!encode_tile_map(&maps.q, a.q, a.T_tot, a.H) || !encode_tile_map(&maps.k, a.k, a.T_tot, a.H) ||
        !encode_tile_map(&maps.v, a.v, a.T_tot, a.H) || !encode_tile_map(&maps.z, a.z, a.T_tot, a.H)) {
        return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(kda_chunk_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)a.N, (unsigned)a.H);
    kda_chunk_fwd_tc_kernel<<<grid, NTHREADS, SMEM_BYTES, s>>>(a, maps);
    return cudaGetLastError();
}

static_assert(SMEM_USED + 1024 <= SMEM_BYTES, "shared-memory map exceeds the request");

}  // namespace kda
