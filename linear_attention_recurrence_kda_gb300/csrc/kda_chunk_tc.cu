// kda_chunk_tc.cu -- fused KDA prefill on the sm_103a tensor cores (bf16 inputs, d_k = d_v = 128).
//
// One CTA walks one sequence of one head in 16-token chunks and computes, per chunk, every stage of
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
//
// Warp specialisation.  Warps 8..15 (producer) prepare chunk n+1 -- TMA tile loads, gate and
// factors, A, P and T', the W / U~ products and W's transposition into the read operand -- while
// warps 0..7 (consumer) run chunk n's state pass: the state read, U, the output and state-update
// products, the state update and the outputs.  The per-chunk operands the consumer reads are
// double-buffered by chunk parity; the two groups hand them over with named barriers (FULL[b]:
// producer -> consumer, EMPTY[b]: consumer -> producer).  Every mbarrier wait is bounded; a wait
// that gives up raises the timeout bit of the check word, and from then on both groups skip all
// work but still walk the whole barrier protocol, so neither can be left waiting on the other.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_tc_chunk.cuh"

namespace kda {

namespace {

using tcc::C;
using tcc::D;
using tcc::NGROUP;
using tcc::NONE_TILE;
using tcc::SMALL_TILE;
using tcc::STAGE_TILE;
using tcc::named_arrive;
using tcc::named_sync;
using tcc::st_bf16;
using tcc::u2f;
constexpr int NTHREADS = 512;     // 8 consumer + 8 producer warps
constexpr uint32_t WAIT_LIMIT = 1u << 17;  // tries of up to 20 us each: ~2.6 s at most

// named barriers (0 is __syncthreads)
constexpr uint32_t NB_CONS = 1;   // consumer group only
constexpr uint32_t NB_PROD = 2;   // producer group only
constexpr uint32_t NB_FULL = 3;   // + b: chunk parity b's operands are ready (512 threads)
constexpr uint32_t NB_EMPTY = 5;  // + b: chunk parity b's operands may be overwritten (512 threads)

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
constexpr uint32_t OFF_PART = 124160;  // k-step partial products fp32 [8 warps][16][16] 8192
constexpr uint32_t OFF_GC = 132352;    // [2] Gamma_C fp32 [128]                         2 x 512
constexpr uint32_t OFF_HS = 133376;    // per-channel quarter-chunk log-decay sums [4][128] 2048
constexpr uint32_t OFF_BETA = 135424;  // beta [16]                                      64
constexpr uint32_t OFF_BARC = 135488;  // mbarrier: consumer tensor-core commits        8
constexpr uint32_t OFF_BARP = 135496;  // mbarrier: producer tensor-core commits        8
constexpr uint32_t OFF_BARLD = 135504; // mbarrier: TMA tile loads                      8
constexpr uint32_t OFF_TSLOT = 135512; // TMEM base address                             4
constexpr uint32_t OFF_ABORT = 135516; // stop flag                                     4
constexpr uint32_t SMEM_USED = 135520;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;

// tensor-memory columns
constexpr uint32_t TM_D1 = 0;    // consumer: [0,16) (W S)^T, [16,32) O^T
constexpr uint32_t TM_W = 32;    // producer: W^T  (lanes = c)
constexpr uint32_t TM_U = 48;    // producer -> consumer: [2] U~^T (lanes = j), 16 columns each
constexpr uint32_t TM_D3 = 128;  // consumer: dS^T (lanes = j, columns = c)
constexpr uint32_t TM_COLS = 256;

// Placement of the per-chunk preparation tiles in this kernel's shared memory.
struct FusedMap {
    static constexpr uint32_t OFF_STAGE = ::kda::OFF_STAGE;
    static constexpr uint32_t OFF_HS = ::kda::OFF_HS;
    static constexpr uint32_t OFF_LL = ::kda::OFF_LL;
    static constexpr uint32_t OFF_QL = ::kda::OFF_QL;
    static constexpr uint32_t OFF_KD = ::kda::OFF_KD;
    static constexpr uint32_t OFF_XT = ::kda::OFF_XT;
    static constexpr uint32_t OFF_VT = ::kda::OFF_VT;
    static constexpr uint32_t OFF_A = ::kda::OFF_A;
    static constexpr uint32_t OFF_PART = ::kda::OFF_PART;
    static constexpr uint32_t OFF_BETA = ::kda::OFF_BETA;
    static constexpr uint32_t OFF_T = ::kda::OFF_T;
    static constexpr uint32_t NB = 2;       // producer-group barrier
    static constexpr uint32_t XT_RG = 256;  // (K Gamma)^T and V^T are tensor-core operands here
};

// Abort flag, read identically by every lane of the warp (it guards warp-collective instructions).
__device__ __forceinline__ bool read_dead(const volatile uint32_t* abort_flag)
{
    return __any_sync(0xffffffffu, *abort_flag != 0u);
}

// Thread 0 of a group: commit its issued tensor-core work and wait (bounded) for it.
__device__ __forceinline__ void commit_wait(uint64_t* bar, uint32_t phase, volatile uint32_t* abort_flag)
{
    tc::umma_commit(bar);
    if (!tc::mbar_wait(bar, phase, WAIT_LIMIT)) *abort_flag = 1u;
}

}  // namespace

__global__ void __launch_bounds__(NTHREADS, 1) kda_chunk_fwd_tc_kernel(PrefillArgs a, const __grid_constant__ TileMaps maps)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned base (SW128 atoms), derived from the __shared__ array so that every access
    // stays a shared-memory access
    unsigned char* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bar_c = reinterpret_cast<uint64_t*>(sm + OFF_BARC);
    uint64_t* bar_p = reinterpret_cast<uint64_t*>(sm + OFF_BARP);
    uint64_t* bar_ld = reinterpret_cast<uint64_t*>(sm + OFF_BARLD);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_TSLOT);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sm + OFF_ABORT);

    const int n = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int w = tid >> 5;
    const int lane = tid & 31;

    int64_t q0, q1;
    if (!seq_range(a, n, q0, q1)) return;
    // segment k of the sequence, and what this CTA computes for it (mode 0: outputs and, for the
    // last segment, the final state; 1: S~, the end state from a zero start; 2: M, the transition,
    // as the end state from the identity with V = 0)
    const int mode = a.seg_mode == 0 ? 0 : 1 + (int)(blockIdx.z & 1);
    const int k = a.seg_mode == 0 ? (int)blockIdx.z : (int)(blockIdx.z >> 1);
    const int64_t seq_chunks = (q1 - q0 + C - 1) / C;
    const int64_t seg_c = a.seg_chunks > 0 ? (int64_t)a.seg_chunks : (seq_chunks > 0 ? seq_chunks : 1);
    const int64_t nseg = seq_chunks > 0 ? (seq_chunks + seg_c - 1) / seg_c : 1;
    if (mode == 0 ? (int64_t)k >= nseg : (int64_t)k >= nseg - 1) return;
    const int64_t s0 = q0 + (int64_t)k * seg_c * C;
    const int64_t s1 = min(q1, s0 + seg_c * C);
    const int H = a.H;
    const int nchunks = (int)((s1 - s0 + C - 1) / C);
    auto chunk_len = [&](int chunk) -> int { return (int)min((int64_t)C, s1 - (s0 + (int64_t)chunk * C)); };

    if (w == 0) tc::tmem_alloc(tslot, TM_COLS);
    if (tid == 0) {
        tc::mbar_init(bar_c, 1);
        tc::mbar_init(bar_p, 1);
        tc::mbar_init(bar_ld, 1);
        *abort_flag = 0u;
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tslot;

    if (w >= 8) {
        // ======================================================================== producer
        const int p = tid - NGROUP;
        const int pw = w - 8;
        const float expA = expf(a.A[h]);
        const float g_min = a.g_min;
        const uint32_t lane_base = tbase + ((uint32_t)(32 * (pw & 3)) << 16);
        uint32_t ph_p = 0, ph_ld = 0;
        auto issue_tiles = [&](int chunk) {  // producer thread 0
            const int tn = (int)(s0 + (int64_t)chunk * C);
            tc::fence_async_smem();
            tc::mbar_arrive_expect_tx(bar_ld, 4 * STAGE_TILE);
            tc::tma_load_3d(sm + OFF_STAGE, &maps.q, 0, h, tn, bar_ld);
            tc::tma_load_3d(sm + OFF_STAGE + STAGE_TILE, &maps.k, 0, h, tn, bar_ld);
            tc::tma_load_3d(sm + OFF_STAGE + 2 * STAGE_TILE, &maps.v, 0, h, tn, bar_ld);
            tc::tma_load_3d(sm + OFF_STAGE + 3 * STAGE_TILE, &maps.z, 0, h, tn, bar_ld);
        };
        auto load_beta = [&](int chunk) -> float {  // producer threads 0..15
            const int64_t t = s0 + (int64_t)chunk * C + p;
            return (chunk < nchunks && t < s1) ? a.beta[t * H + h] : 0.f;
        };
        float beta_next = (p < C) ? load_beta(0) : 0.f;
        if (p == 0 && nchunks > 0) issue_tiles(0);

        for (int ch = 0; ch < nchunks; ++ch) {
            const int b = ch & 1;
            if (ch >= 2) {
                named_sync(NB_EMPTY + b, NTHREADS);  // the consumer is done with chunk ch-2
                tc::fence_after_sync();
            }
            bool dead = read_dead(abort_flag);
            // tiles of chunk ch
            if (p < C) reinterpret_cast<float*>(sm + OFF_BETA)[p] = beta_next;
            if (p == 0 && !dead && !tc::mbar_wait(bar_ld, ph_ld, WAIT_LIMIT)) *abort_flag = 1u;
            ph_ld ^= 1u;
            named_sync(NB_PROD, NGROUP);
            dead = read_dead(abort_flag);
            if (!dead) tcc::prep_factors<FusedMap>(sm, p, chunk_len(ch), sm + OFF_WQ + b * 8192, sm + OFF_KT + b * 8192,
                                                 reinterpret_cast<float*>(sm + OFF_GC + b * 512), expA, g_min, mode == 2);
            else named_sync(NB_PROD, NGROUP);  // the barrier inside prep_factors
            named_sync(NB_PROD, NGROUP);       // stage consumed
            if (ch + 1 < nchunks) {
                if (p == 0 && !dead) issue_tiles(ch + 1);
                if (p < C) beta_next = load_beta(ch + 1);
            }
            if (!dead) {
                tcc::prep_solve<FusedMap>(sm, p, sm + OFF_P + b * 1024);
            } else {
                named_sync(NB_PROD, NGROUP);
                named_sync(NB_PROD, NGROUP);
            }
            tc::fence_async_smem();
            tc::fence_before_sync();
            named_sync(NB_PROD, NGROUP);
            tc::fence_after_sync();
            if (p == 0 && !dead) {
                // W^T = (K Gamma)^T T'^T, U~^T = V^T T'^T (T' = hi + lo)
                const uint32_t id16 = tc::idesc_bf16(128, 16);
                const uint64_t dT = tc::desc_none(tc::smem_u32(sm + OFF_T));
                const uint64_t dTl = tc::desc_none(tc::smem_u32(sm + OFF_T + SMALL_TILE));
                const uint64_t dX = tc::desc_none(tc::smem_u32(sm + OFF_XT));
                const uint64_t dV = tc::desc_none(tc::smem_u32(sm + OFF_VT));
                const uint32_t du = tbase + TM_U + 16 * b;
                tc::umma(tbase + TM_W, dX, dT, id16, 0u);
                tc::umma(tbase + TM_W, dX, dTl, id16, 1u);
                tc::umma(du, dV, dT, id16, 0u);
                tc::umma(du, dV, dTl, id16, 1u);
                commit_wait(bar_p, ph_p, abort_flag);
            }
            ph_p ^= 1u;
            named_sync(NB_PROD, NGROUP);
            tc::fence_after_sync();
            dead = read_dead(abort_flag);
            if (!dead) {
                // W^T (lanes = c) -> rows 0..15 of WQ[b]; producer warp pw handles rows 8 (pw / 4) .. +8
                uint32_t v[8];
                KDA_TMEM_LD8(lane_base + TM_W + 8 * (pw >> 2), v);
                tc::tmem_wait_ld();
                unsigned char* wq = sm + OFF_WQ + b * 8192;
                const int c = 32 * (pw & 3) + lane;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    st_bf16(wq, tc::sw128_off(8 * (pw >> 2) + e, c, 2 * C), __float2bfloat16_rn(u2f(v[e])));
                }
            }
            tc::fence_async_smem();
            tc::fence_before_sync();
            named_arrive(NB_FULL + b, NTHREADS);
        }
    } else {
        // ======================================================================== consumer
        const int q4 = w & 3;    // TMEM lane quarter
        const int h2 = w >> 2;   // which half of the key channels this warp's state slice covers
        const int jrow = 32 * q4 + lane;
        const uint32_t lane_base = tbase + ((uint32_t)(32 * q4) << 16);
        __nv_bfloat16* op = static_cast<__nv_bfloat16*>(a.out);
        uint32_t ph_c = 0;

        // state slice: S[c][jrow] for c in [64*h2, 64*h2 + 64)
        float S[64];
        const int64_t sbase = ((int64_t)n * H + h) * D * D;
        const int64_t segbase = (((int64_t)n * H + h) * a.max_seg + k) * D * D;
        const float* init = nullptr;
        // with several segments every segment, the first included, starts from the scan's copy: the
        // final state may overwrite the caller's initial state (in-place carry) while the first
        // segment's CTA has not read it yet
        if (mode == 0) init = (nseg == 1) ? (a.s0 ? a.s0 + sbase : nullptr) : a.seg_in + segbase;
#pragma unroll
        for (int cc = 0; cc < 64; ++cc) {
            const int c = 64 * h2 + cc;
            S[cc] = init ? init[(int64_t)c * D + jrow] : ((mode == 2 && c == jrow) ? 1.f : 0.f);
        }
        auto stage_state = [&]() {
#pragma unroll
            for (int chn = 0; chn < 8; ++chn) {
                uint4 pk;
                pk.x = tc::pack_bf16(S[8 * chn + 0], S[8 * chn + 1]);
                pk.y = tc::pack_bf16(S[8 * chn + 2], S[8 * chn + 3]);
                pk.z = tc::pack_bf16(S[8 * chn + 4], S[8 * chn + 5]);
                pk.w = tc::pack_bf16(S[8 * chn + 6], S[8 * chn + 7]);
                *reinterpret_cast<uint4*>(sm + OFF_S + tc::sw128_chunk_off(jrow, 8 * h2 + chn, D)) = pk;
            }
        };
        stage_state();
        tc::fence_async_smem();

        for (int ch = 0; ch < nchunks; ++ch) {
            const int b = ch & 1;
            const int64_t t0 = s0 + (int64_t)ch * C;
            const int len = chunk_len(ch);
            named_sync(NB_FULL + b, NTHREADS);  // chunk ch's operands are ready; the state is staged
            tc::fence_after_sync();
            bool dead = read_dead(abort_flag);

            // D1 = S^T [W ; Q Gamma]^T  (M = 128, N = 32, K = 128)
            if (tid == 0 && !dead) {
                const uint32_t id32 = tc::idesc_bf16(128, 2 * C);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
                    tc::umma(tbase + TM_D1, tc::desc_sw128(tc::smem_u32(sm + OFF_S + kb * 16384 + off)),
                             tc::desc_sw128(tc::smem_u32(sm + OFF_WQ + b * 8192 + kb * (2 * C * 128) + off)), id32,
                             ks > 0 ? 1u : 0u);
                }
                commit_wait(bar_c, ph_c, abort_flag);
            }
            ph_c ^= 1u;
            named_sync(NB_CONS, NGROUP);
            tc::fence_after_sync();
            dead = read_dead(abort_flag);

            // U^T = U~^T - (W S)^T as a hi/lo pair; warp half h2 takes columns 8 h2 .. 8 h2 + 7
            if (!dead) {
                uint32_t dv[8], uv[8];
                KDA_TMEM_LD8(lane_base + TM_D1 + 8 * h2, dv);
                KDA_TMEM_LD8(lane_base + TM_U + 16 * b + 8 * h2, uv);
                tc::tmem_wait_ld();
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float u0 = u2f(uv[2 * e]) - u2f(dv[2 * e]);
                    const float u1 = u2f(uv[2 * e + 1]) - u2f(dv[2 * e + 1]);
                    __nv_bfloat162 hv = __floats2bfloat162_rn(u0, u1);
                    const float2 hf = __bfloat1622float2(hv);
                    __nv_bfloat162 lv = __floats2bfloat162_rn(u0 - hf.x, u1 - hf.y);
                    hi[e] = *reinterpret_cast<uint32_t*>(&hv);
                    lo[e] = *reinterpret_cast<uint32_t*>(&lv);
                }
                *reinterpret_cast<uint4*>(sm + OFF_UT + tc::none_off(jrow, 8 * h2)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(sm + OFF_UT + NONE_TILE + tc::none_off(jrow, 8 * h2)) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            tc::fence_async_smem();
            tc::fence_before_sync();
            named_sync(NB_CONS, NGROUP);
            tc::fence_after_sync();

            // O^T += U^T P^T and dS^T = U^T (K Gamma_C / Gamma), each as hi*hi + hi*lo + lo*hi
            if (tid == 0 && !dead) {
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
                commit_wait(bar_c, ph_c, abort_flag);
            }
            ph_c ^= 1u;
            named_sync(NB_CONS, NGROUP);
            tc::fence_after_sync();
            dead = read_dead(abort_flag);

            // S <- Diag(Gamma_C) S + dS (staged for the next read), outputs of chunk ch
            if (!dead) {
                const float* gc = reinterpret_cast<const float*>(sm + OFF_GC + b * 512) + 64 * h2;
#pragma unroll
                for (int blk = 0; blk < 4; blk += 2) {
                    uint32_t v0[16], v1[16];
                    KDA_TMEM_LD16(lane_base + TM_D3 + 64 * h2 + 16 * blk, v0);
                    KDA_TMEM_LD16(lane_base + TM_D3 + 64 * h2 + 16 * blk + 16, v1);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        const float4 g4 = *reinterpret_cast<const float4*>(gc + 16 * blk + 4 * e4);
                        const int cc = 16 * blk + 4 * e4;
                        const uint32_t* vv = (e4 < 4) ? v0 : v1;
                        const int o = (e4 & 3) * 4;
                        S[cc + 0] = g4.x * S[cc + 0] + u2f(vv[o + 0]);
                        S[cc + 1] = g4.y * S[cc + 1] + u2f(vv[o + 1]);
                        S[cc + 2] = g4.z * S[cc + 2] + u2f(vv[o + 2]);
                        S[cc + 3] = g4.w * S[cc + 3] + u2f(vv[o + 3]);
                    }
                }
                stage_state();
                uint32_t ov[8];
                KDA_TMEM_LD8(lane_base + TM_D1 + C + 8 * h2, ov);
                tc::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int r = 8 * h2 + e;
                    if (mode == 0 && r < len) op[((t0 + r) * H + h) * D + jrow] = __float2bfloat16_rn(u2f(ov[e]));
                }
            }
            tc::fence_async_smem();
            tc::fence_before_sync();
            if (ch + 2 < nchunks) named_arrive(NB_EMPTY + b, NTHREADS);
        }
        float* dst = nullptr;
        if (mode == 0) dst = ((int64_t)k == nseg - 1 && a.s_final) ? a.s_final + sbase : nullptr;
        else dst = (mode == 1 ? a.seg_st : a.seg_mt) + segbase;
        if (*abort_flag) {
            if (tid == 0) atomicOr(a.check, kCheckTimeout);
        } else if (dst && mode == 2) {
            // the transition M[c][j] (this lane holds column j = jrow) in the scan's operand format
#pragma unroll
            for (int cc = 0; cc < 64; ++cc) store_seg_m(dst, 64 * h2 + cc, jrow, S[cc]);
        } else if (dst) {
#pragma unroll
            for (int cc = 0; cc < 64; ++cc) dst[(int64_t)(64 * h2 + cc) * D + jrow] = S[cc];
        }
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

bool encode_tile_maps(TileMaps& m, const PrefillArgs& a)
{
    return encode_tile_map(&m.q, a.q, a.T_tot, a.H) && encode_tile_map(&m.k, a.k, a.T_tot, a.H) &&
           encode_tile_map(&m.v, a.v, a.T_tot, a.H) && encode_tile_map(&m.z, a.z, a.T_tot, a.H);
}

cudaError_t launch_chunk_fwd_tc(const PrefillArgs& a, cudaStream_t s)
{
    TileMaps maps;
    if (!encode_tile_maps(maps, a)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kda_chunk_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (a.seg_chunks > 0 && a.max_seg > 1) {
        // pass 1: (S~, M) of every segment but the last; pass 2: scan; pass 3: outputs
        PrefillArgs a1 = a;
        a1.seg_mode = 1;
        prof_start("kda_seg_summary_tc", s);
        kda_chunk_fwd_tc_kernel<<<dim3((unsigned)a.N, (unsigned)a.H, (unsigned)(2 * (a.max_seg - 1))), NTHREADS,
                                  SMEM_BYTES, s>>>(a1, maps);
        e = cudaGetLastError();
        prof_stop(s);
        if (e != cudaSuccess) return e;
        prof_start("kda_seg_scan", s);
        e = launch_segment_scan(a, s);
        prof_stop(s);
        if (e != cudaSuccess) return e;
    }
    PrefillArgs a3 = a;
    a3.seg_mode = 0;
    prof_start("kda_chunk_fwd_tc", s);
    kda_chunk_fwd_tc_kernel<<<dim3((unsigned)a.N, (unsigned)a.H, (unsigned)(a.max_seg > 1 ? a.max_seg : 1)), NTHREADS,
                              SMEM_BYTES, s>>>(a3, maps);
    e = cudaGetLastError();
    prof_stop(s);
    return e;
}

static_assert(SMEM_USED + 1024 <= SMEM_BYTES, "shared-memory map exceeds the request");

}  // namespace kda
