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
// Two CTAs share an SM (256 TMEM columns and ~100 KB of shared memory each), so one CTA's SIMT
// stages overlap the other's tensor-core work.  Every mbarrier wait is bounded; a wait that gives
// up raises the timeout bit of the check word and the CTA stops cleanly.
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

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_S = 0;         // S^T  [128 j][128 c] SW128          32768
constexpr uint32_t OFF_WQ = 32768;    // [W ; Q Gamma] [32][128 c] SW128     8192
constexpr uint32_t OFF_XT = 40960;    // (K Gamma)^T [128 c][16 i] NONE      4096
constexpr uint32_t OFF_VT = 45056;    // V^T  [128 j][16 i] NONE             4096
constexpr uint32_t OFF_UT = 49152;    // U^T hi [128 j][16 i] NONE           4096
constexpr uint32_t OFF_UL = 53248;    // U^T lo                              4096
constexpr uint32_t OFF_KT = 57344;    // (K Gamma_C/Gamma)^T hi [128 c][16 i] 4096
constexpr uint32_t OFF_KTL = 61440;   // (K Gamma_C/Gamma)^T lo              4096
constexpr uint32_t OFF_P = 65536;     // P hi [16 r][16 i] NONE              512
constexpr uint32_t OFF_PL = 66048;    // P lo                                512
constexpr uint32_t OFF_T = 66560;     // T' hi [16 r][16 i] NONE             512
constexpr uint32_t OFF_TL = 67072;    // T' lo                               512
constexpr uint32_t OFF_LL = 67584;    // K Gamma   [16][LROW] bf16           4352
constexpr uint32_t OFF_QL = 71936;    // Q Gamma hi                          4352
constexpr uint32_t OFF_QLL = 76288;   // Q Gamma lo                          4352
constexpr uint32_t OFF_KD = 80640;    // K / Gamma hi                        4352
constexpr uint32_t OFF_KDL = 84992;   // K / Gamma lo                        4352
constexpr uint32_t OFF_A = 89344;     // A fp32 [16][16]                     1024
constexpr uint32_t OFF_PF = 90368;    // P partial sums fp32 [2][16][16]     2048
constexpr uint32_t OFF_GC = 92416;    // Gamma_C fp32 [128]                  512
constexpr uint32_t OFF_BAR = 92928;   // mbarrier                            8
constexpr uint32_t OFF_TSLOT = 92936; // TMEM base address                   4
constexpr uint32_t OFF_ABORT = 92940; // stop flag                           4
constexpr uint32_t OFF_STAGE = 93184; // q, k, v, z tiles [16][128] bf16 (TMA)  16384
constexpr uint32_t OFF_BETA = 109568; // beta of the chunk                   64
constexpr uint32_t OFF_BARLD = 109632;// mbarrier of the tile loads          8
constexpr uint32_t SMEM_USED = 109640;
constexpr uint32_t STAGE_TILE = C * D * 2;  // 4096 bytes per tensor and chunk
// Two CTAs per SM fit (the number whose 256 TMEM columns fit in the SM's 512).
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;

// tensor-memory columns (256 allocated)
constexpr uint32_t TM_D1 = 0;    // [0,16): (W S)^T, [16,32): O^T
constexpr uint32_t TM_W = 32;    // W^T  (lanes = c)
constexpr uint32_t TM_U = 48;    // U~^T (lanes = j)
constexpr uint32_t TM_D3 = 128;  // dS^T (lanes = j, columns = c)
constexpr uint32_t TM_COLS = 256;

__device__ __forceinline__ void st_bf16(unsigned char* base, uint32_t off, float x)
{
    *reinterpret_cast<__nv_bfloat16*>(base + off) = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi)
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo)
{
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
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

// Issue + commit + bounded wait by thread 0, then a CTA barrier.  Returns false if the CTA must stop.
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

}  // namespace

struct TileMaps {
    CUtensorMap q, k, v, z;  // 3-D views [T_tot][H][128] of the bf16 inputs, box [16][1][128]
};

__global__ void __launch_bounds__(NTHREADS, 2) kda_chunk_fwd_tc_kernel(PrefillArgs a, const __grid_constant__ TileMaps maps)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_TSLOT);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sm + OFF_ABORT);
    __nv_bfloat16* sLl = reinterpret_cast<__nv_bfloat16*>(sm + OFF_LL);
    __nv_bfloat16* sQl = reinterpret_cast<__nv_bfloat16*>(sm + OFF_QL);
    __nv_bfloat16* sQll = reinterpret_cast<__nv_bfloat16*>(sm + OFF_QLL);
    __nv_bfloat16* sKd = reinterpret_cast<__nv_bfloat16*>(sm + OFF_KD);
    __nv_bfloat16* sKdl = reinterpret_cast<__nv_bfloat16*>(sm + OFF_KDL);
    float* sA = reinterpret_cast<float*>(sm + OFF_A);
    float* sPf = reinterpret_cast<float*>(sm + OFF_PF);
    float* sBeta = reinterpret_cast<float*>(sm + OFF_BETA);
    uint64_t* bar_ld = reinterpret_cast<uint64_t*>(sm + OFF_BARLD);
    const __nv_bfloat16* tq = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_STAGE);
    const __nv_bfloat16* tk = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_STAGE + STAGE_TILE);
    const __nv_bfloat16* tv = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_STAGE + 2 * STAGE_TILE);
    const __nv_bfloat16* tz = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_STAGE + 3 * STAGE_TILE);
    float* sGC = reinterpret_cast<float*>(sm + OFF_GC);

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

    __nv_bfloat16* op = static_cast<__nv_bfloat16*>(a.out);
    const int H = a.H;
    const float expA = expf(a.A[h]);
    const float g_min = a.g_min;

    if (w == 0) tc::tmem_alloc(tslot, TM_COLS);
    if (tid == 0) {
        tc::mbar_init(bar, 1);
        tc::mbar_init(bar_ld, 1);
        *abort_flag = 0u;
        tc::fence_async_smem();
        // first chunk's tiles
        if (s0 < s1) {
            tc::mbar_arrive_expect_tx(bar_ld, 4 * STAGE_TILE);
            tc::tma_load_3d(sm + OFF_STAGE, &maps.q, 0, h, (int)s0, bar_ld);
            tc::tma_load_3d(sm + OFF_STAGE + STAGE_TILE, &maps.k, 0, h, (int)s0, bar_ld);
            tc::tma_load_3d(sm + OFF_STAGE + 2 * STAGE_TILE, &maps.v, 0, h, (int)s0, bar_ld);
            tc::tma_load_3d(sm + OFF_STAGE + 3 * STAGE_TILE, &maps.z, 0, h, (int)s0, bar_ld);
        }
    }
    float beta_next = (tid < C && s0 + tid < s1) ? a.beta[(s0 + tid) * H + h] : 0.f;
    uint32_t ld_phase = 0;

    // state slice: S[c][jrow] for c in [64*h2, 64*h2 + 64)
    float S[64];
    const int64_t sbase = ((int64_t)n * H + h) * D * D;
#pragma unroll
    for (int cc = 0; cc < 64; ++cc) {
        S[cc] = a.s0 ? a.s0[sbase + (int64_t)(64 * h2 + cc) * D + jrow] : 0.f;
    }
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        uint4 pk;
        pk.x = tc::pack_bf16(S[8 * ch + 0], S[8 * ch + 1]);
        pk.y = tc::pack_bf16(S[8 * ch + 2], S[8 * ch + 3]);
        pk.z = tc::pack_bf16(S[8 * ch + 4], S[8 * ch + 5]);
        pk.w = tc::pack_bf16(S[8 * ch + 6], S[8 * ch + 7]);
        *reinterpret_cast<uint4*>(sm + OFF_S + tc::sw128_chunk_off(jrow, 8 * h2 + ch, D)) = pk;
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tslot;
    const uint32_t lane_base = tbase + ((uint32_t)(32 * q4) << 16);
    uint32_t phase = 0;

    for (int64_t t0 = s0; t0 < s1; t0 += C) {
        const int len = (int)min((int64_t)C, s1 - t0);
        if (tid < C) sBeta[tid] = beta_next;
        if (tid == 0 && !tc::mbar_wait(bar_ld, ld_phase, WAIT_LIMIT)) *abort_flag = 1u;
        ld_phase ^= 1u;
        __syncthreads();
        if (*abort_flag) break;

        // ---------------- gate + per-token factors (kda_gate / kda_ut_wy prologue)
        if (tid < D) {
            const int c = tid;
            float Gr[C];
            float G = 0.f;
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float g = 0.f;
                if (r < len) g = log_decay(__bfloat162float(tz[r * D + c]), expA, g_min);
                G += g;
                Gr[r] = G;
            }
            const float eGC = expf(G);
            sGC[c] = eGC;
            uint32_t xpk[C / 2], kpk[C / 2], kpl[C / 2];
#pragma unroll
            for (int r = 0; r < C; r += 2) {
                float xv[2], kt[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int rr = r + e;
                    float kv = 0.f, qv = 0.f;
                    if (rr < len) {
                        kv = __bfloat162float(tk[rr * D + c]);
                        qv = __bfloat162float(tq[rr * D + c]);
                    }
                    const float eG = expf(Gr[rr]);       // Gamma_r in [e^-80, 1]
                    const float ieG = __frcp_rn(eG);      // 1 / Gamma_r in [1, e^80]
                    const float ll = kv * eG;
                    __nv_bfloat16 hi, lo;
                    sLl[rr * LROW + c] = __float2bfloat16_rn(ll);
                    split_bf16(qv * eG, hi, lo);
                    sQl[rr * LROW + c] = hi;
                    sQll[rr * LROW + c] = lo;
                    *reinterpret_cast<__nv_bfloat16*>(sm + OFF_WQ + tc::sw128_off(C + rr, c, 2 * C)) = hi;
                    split_bf16(kv * ieG, hi, lo);
                    sKd[rr * LROW + c] = hi;
                    sKdl[rr * LROW + c] = lo;
                    xv[e] = ll;
                    kt[e] = kv * (eGC * ieG);            // k Gamma_C / Gamma_r <= 1
                }
                xpk[r / 2] = tc::pack_bf16(xv[0], xv[1]);
                __nv_bfloat162 kh = __floats2bfloat162_rn(kt[0], kt[1]);
                const float2 khf = __bfloat1622float2(kh);
                __nv_bfloat162 kl = __floats2bfloat162_rn(kt[0] - khf.x, kt[1] - khf.y);
                kpk[r / 2] = *reinterpret_cast<uint32_t*>(&kh);
                kpl[r / 2] = *reinterpret_cast<uint32_t*>(&kl);
            }
            *reinterpret_cast<uint4*>(sm + OFF_XT + tc::none_off(c, 0)) = make_uint4(xpk[0], xpk[1], xpk[2], xpk[3]);
            *reinterpret_cast<uint4*>(sm + OFF_XT + tc::none_off(c, 8)) = make_uint4(xpk[4], xpk[5], xpk[6], xpk[7]);
            *reinterpret_cast<uint4*>(sm + OFF_KT + tc::none_off(c, 0)) = make_uint4(kpk[0], kpk[1], kpk[2], kpk[3]);
            *reinterpret_cast<uint4*>(sm + OFF_KT + tc::none_off(c, 8)) = make_uint4(kpk[4], kpk[5], kpk[6], kpk[7]);
            *reinterpret_cast<uint4*>(sm + OFF_KTL + tc::none_off(c, 0)) = make_uint4(kpl[0], kpl[1], kpl[2], kpl[3]);
            *reinterpret_cast<uint4*>(sm + OFF_KTL + tc::none_off(c, 8)) = make_uint4(kpl[4], kpl[5], kpl[6], kpl[7]);
        } else {
            // V^T rows as given (beta is applied through T')
            const int j = tid - D;
            uint32_t vpk[C / 2];
#pragma unroll
            for (int r = 0; r < C; r += 2) {
                const __nv_bfloat16 zero = __float2bfloat16_rn(0.f);
                __nv_bfloat162 pr;
                pr.x = (r < len) ? tv[r * D + j] : zero;
                pr.y = (r + 1 < len) ? tv[(r + 1) * D + j] : zero;
                vpk[r / 2] = *reinterpret_cast<uint32_t*>(&pr);
            }
            *reinterpret_cast<uint4*>(sm + OFF_VT + tc::none_off(j, 0)) = make_uint4(vpk[0], vpk[1], vpk[2], vpk[3]);
            *reinterpret_cast<uint4*>(sm + OFF_VT + tc::none_off(j, 8)) = make_uint4(vpk[4], vpk[5], vpk[6], vpk[7]);
        }
        __syncthreads();

        // the staged tiles are consumed: fetch the next chunk's while this one computes
        if (t0 + C < s1) {
            if (tid == 0) {
                tc::fence_async_smem();
                tc::mbar_arrive_expect_tx(bar_ld, 4 * STAGE_TILE);
                const int tn = (int)(t0 + C);
                tc::tma_load_3d(sm + OFF_STAGE, &maps.q, 0, h, tn, bar_ld);
                tc::tma_load_3d(sm + OFF_STAGE + STAGE_TILE, &maps.k, 0, h, tn, bar_ld);
                tc::tma_load_3d(sm + OFF_STAGE + 2 * STAGE_TILE, &maps.v, 0, h, tn, bar_ld);
                tc::tma_load_3d(sm + OFF_STAGE + 3 * STAGE_TILE, &maps.z, 0, h, tn, bar_ld);
            }
            if (tid < C) beta_next = (t0 + C + tid < s1) ? a.beta[(t0 + C + tid) * H + h] : 0.f;
        }

        // ---------------- A (warp 0) and the two halves of P (warps 1, 2): 16x16, K = 128, mma.sync
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
                        sA[r * C + i] = (i < r) ? sBeta[r] * acc[nt][e] : 0.f;
                    } else {
                        sPf[(w - 1) * C * C + r * C + i] = acc[nt][e];
                    }
                }
            }
        }
        __syncthreads();

        // ---------------- T = (I + A)^-1 by forward substitution (lane = column); T' = T diag(beta)
        if (w == 0 && lane < C) {
            const int j = lane;
            const float bj = sBeta[j];
            float tcol[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float x = (r == j) ? 1.f : 0.f;
#pragma unroll
                for (int i = 0; i < r; ++i) x -= sA[r * C + i] * tcol[i];
                tcol[r] = x;
            }
#pragma unroll
            for (int r = 0; r < C; ++r) {
                __nv_bfloat16 hi, lo;
                split_bf16(tcol[r] * bj, hi, lo);
                *reinterpret_cast<__nv_bfloat16*>(sm + OFF_T + tc::none_off(r, j)) = hi;
                *reinterpret_cast<__nv_bfloat16*>(sm + OFF_TL + tc::none_off(r, j)) = lo;
            }
        } else if (tid >= 128) {
            // P = tril_incl(sum of the partial products), as a hi/lo pair
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int idx = 2 * (tid - 128) + e;
                const int r = idx >> 4, i = idx & 15;
                const float pv = (i <= r) ? sPf[idx] + sPf[C * C + idx] : 0.f;
                __nv_bfloat16 hi, lo;
                split_bf16(pv, hi, lo);
                *reinterpret_cast<__nv_bfloat16*>(sm + OFF_P + tc::none_off(r, i)) = hi;
                *reinterpret_cast<__nv_bfloat16*>(sm + OFF_PL + tc::none_off(r, i)) = lo;
            }
        }
        tc_publish();

        // ---------------- W^T = (K Gamma)^T T'^T, U~^T = V^T T'^T  (T' = hi + lo)
        if (tid == 0) {
            const uint32_t id16 = tc::idesc_bf16(128, 16);
            const uint64_t dT = tc::desc_none(tc::smem_u32(sm + OFF_T));
            const uint64_t dTl = tc::desc_none(tc::smem_u32(sm + OFF_TL));
            const uint64_t dX = tc::desc_none(tc::smem_u32(sm + OFF_XT));
            const uint64_t dV = tc::desc_none(tc::smem_u32(sm + OFF_VT));
            tc::umma(tbase + TM_W, dX, dT, id16, 0u);
            tc::umma(tbase + TM_W, dX, dTl, id16, 1u);
            tc::umma(tbase + TM_U, dV, dT, id16, 0u);
            tc::umma(tbase + TM_U, dV, dTl, id16, 1u);
        }
        if (!tc_join(bar, phase, abort_flag)) break;

        // ---------------- W -> rows 0..15 of the [W ; Q Gamma] operand
        if (w < 4) {
            const int c = jrow;
            uint32_t v[16];
            KDA_TMEM_LD16(lane_base + TM_W, v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int r = 0; r < C; ++r) st_bf16(sm, OFF_WQ + tc::sw128_off(r, c, 2 * C), u2f(v[r]));
        }
        tc_publish();

        // ---------------- D1 = S^T [W ; Q Gamma]^T  (M = 128, N = 32, K = 128)
        if (tid == 0) {
            const uint32_t id32 = tc::idesc_bf16(128, 2 * C);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
                tc::umma(tbase + TM_D1, tc::desc_sw128(tc::smem_u32(sm + OFF_S + kb * 16384 + off)),
                         tc::desc_sw128(tc::smem_u32(sm + OFF_WQ + kb * (2 * C * 128) + off)), id32, ks > 0 ? 1u : 0u);
            }
        }
        if (!tc_join(bar, phase, abort_flag)) break;

        // ---------------- U^T = U~^T - (W S)^T  -> bf16 operand
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
            *reinterpret_cast<uint4*>(sm + OFF_UL + tc::none_off(jrow, 8 * h2)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        tc_publish();

        // ---------------- O^T += U^T P^T ;  dS^T = U^T (K Gamma_C / Gamma)  (hi/lo pairs)
        if (tid == 0) {
            const uint32_t id16 = tc::idesc_bf16(128, 16);
            const uint64_t dU = tc::desc_none(tc::smem_u32(sm + OFF_UT));
            const uint64_t dUl = tc::desc_none(tc::smem_u32(sm + OFF_UL));
            const uint64_t dP = tc::desc_none(tc::smem_u32(sm + OFF_P));
            const uint64_t dPl = tc::desc_none(tc::smem_u32(sm + OFF_PL));
            tc::umma(tbase + TM_D1 + C, dU, dP, id16, 1u);
            tc::umma(tbase + TM_D1 + C, dU, dPl, id16, 1u);
            tc::umma(tbase + TM_D1 + C, dUl, dP, id16, 1u);
            const uint32_t id128 = tc::idesc_bf16(128, 128);
            const uint64_t dK = tc::desc_none(tc::smem_u32(sm + OFF_KT));
            const uint64_t dKl = tc::desc_none(tc::smem_u32(sm + OFF_KTL));
            tc::umma(tbase + TM_D3, dU, dK, id128, 0u);
            tc::umma(tbase + TM_D3, dU, dKl, id128, 1u);
            tc::umma(tbase + TM_D3, dUl, dK, id128, 1u);
        }
        if (!tc_join(bar, phase, abort_flag)) break;

        // ---------------- S <- Diag(Gamma_C) S + dS ; outputs
        {
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                uint32_t v[16];
                KDA_TMEM_LD16(lane_base + TM_D3 + 64 * h2 + 16 * blk, v);
                tc::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int cc = 16 * blk + e;
                    S[cc] = sGC[64 * h2 + cc] * S[cc] + u2f(v[e]);
                }
            }
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint4 pk;
                pk.x = tc::pack_bf16(S[8 * ch + 0], S[8 * ch + 1]);
                pk.y = tc::pack_bf16(S[8 * ch + 2], S[8 * ch + 3]);
                pk.z = tc::pack_bf16(S[8 * ch + 4], S[8 * ch + 5]);
                pk.w = tc::pack_bf16(S[8 * ch + 6], S[8 * ch + 7]);
                *reinterpret_cast<uint4*>(sm + OFF_S + tc::sw128_chunk_off(jrow, 8 * h2 + ch, D)) = pk;
            }
            uint32_t ov[8];
            KDA_TMEM_LD8(lane_base + TM_D1 + C + 8 * h2, ov);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int r = 8 * h2 + e;
                if (r < len) op[((t0 + r) * H + h) * D + jrow] = __float2bfloat16_rn(u2f(ov[e]));
            }
        }
        tc_publish();
    }

    if (*abort_flag) {
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
