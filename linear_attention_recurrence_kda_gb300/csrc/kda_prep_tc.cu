// kda_prep_tc.cu -- parallel preparation of the bf16, d = 128 prefill in pairs of chunks.
//
// Everything of a 32-token step that does not depend on the recurrent state -- the gate
// (Equation 5), the in-chunk decays, the WY/UT transform and the in-step output product -- is
// computed here for every step of every (sequence, head) at once, and written as one contiguous
// operand block per step (layout: tcc::BLK_*; the chunk form of Equation 1, "Kimi K3: the paper and
// proofs side by side", section 2.1.1; "Kimi K3: architecture, derivations and a pinned-source
// audit", section 4.5).  A step is two 16-token chunks a, b, each prepared with its own decay
// reference point (so that Gamma and 1/Gamma stay normal numbers); the pair is then assembled by
// substituting chunk a's end state into chunk b's equations:
//   X = W_b K~_a^T = T'_b Y,  Y = (K Gamma)_b K~_a^T,  Z = (Q Gamma)_b K~_a^T   (K~ = K Gamma_C / Gamma)
//   W = [W_a ; W_b Gamma_Ca - X W_a],  U~ = [U~_a ; U~_b - X U~_a],  Q = [(Q Gamma)_a ; (Q Gamma)_b Gamma_Ca]
//   [P ; K~^T] = [[P_a, 0] ; [Z, P_b] ; (K~_a Gamma_Cb)^T, K~_b^T],   Gamma_C = Gamma_Ca Gamma_Cb
// The sequential state pass (kda_state_tc.cu) then only streams these blocks.
//
// One CTA of 256 threads (three per SM) walks a run of 2 (small grids) or 8 (grids of many waves)
// pairs of one (sequence, head): the q, k, v, z tiles arrive by TMA one chunk ahead; the factors, A, P, T and the cross
// products Y, Z come from the shared preparation functions, W and U~ from warp-level mma.sync, and
// every part is stored straight into the block in global memory.  Block slot of step s of sequence
// n: cu[n] / 32 + n + s, so the slots of consecutive sequences never overlap
// (ceil(len / 32) <= floor((cu[n] mod 32 + len) / 32) + 1).
#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_tc_chunk.cuh"

namespace kda {

namespace {

using tcc::C;
using tcc::D;
using tcc::NGROUP;
using tcc::PAIR;

constexpr int kRunShort = 2;                 // 32-token steps per CTA: small grids (short tail)
constexpr int kRunLong = 8;                  // ... grids of many waves (CTA start-up amortised)
constexpr uint32_t WAIT_LIMIT = 1u << 17;    // tries of up to 20 us each

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t XT_RG = 264;          // padded 8-row-group stride of the transposed tiles (the
                                         // 8-byte per-channel stores of a half-warp cover all banks)
constexpr uint32_t OFF_STAGE = 0;        // q, k, v, z tiles [16][128] bf16 (TMA)     16384
constexpr uint32_t OFF_LL = 16384;       // K Gamma [16][LROW] bf16                     4352
constexpr uint32_t OFF_QL = 20736;       // Q Gamma hi, lo                          2 x 4352
constexpr uint32_t OFF_KD = 29440;       // K / Gamma hi, lo                        2 x 4352
constexpr uint32_t OFF_XT = 38144;       // (K Gamma)^T [128 c][16 i], padded           4352
constexpr uint32_t OFF_VT = 42496;       // V^T [128 j][16 i], padded                   4352
constexpr uint32_t OFF_A = 46848;        // A fp32 [16][16]                             1024
constexpr uint32_t OFF_PART = 47872;     // partial products fp32 [8][16][16]           8192
constexpr uint32_t OFF_T = 56064;        // T' hi, lo [16][16] NONE                     1024
constexpr uint32_t OFF_HS = 57088;       // quarter-chunk log-decay sums [4][128]       2048
constexpr uint32_t OFF_YT = OFF_HS;      //   chunk b, after the factors: Y^T hi, lo NONE  1024
constexpr uint32_t OFF_KRA = 59136;      // chunk a's K~ hi, lo [16][LROW]          2 x 4352
constexpr uint32_t OFF_FRAGW = 67840;    // chunk a's W as mma.sync B fragments [4][256]  4096
constexpr uint32_t OFF_GCA = 71936;      // Gamma_C of chunk a [128]                     512
constexpr uint32_t OFF_GCB = 72448;      // Gamma_C of chunk b [128]                     512
constexpr uint32_t OFF_BETA = 72960;     // beta [16]                                     64
constexpr uint32_t OFF_BAR = 73024;      // mbarrier: TMA tile loads                       8
constexpr uint32_t OFF_ABORT = 73032;    // stop flag                                      4
constexpr uint32_t SMEM_USED = 73036;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;

struct PrepMap {
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
    static constexpr uint32_t OFF_KRA = ::kda::OFF_KRA;
    static constexpr uint32_t OFF_YT = ::kda::OFF_YT;
    static constexpr uint32_t NB = 1;
    static constexpr uint32_t XT_RG = ::kda::XT_RG;
};

static_assert(OFF_XT + 16 * XT_RG <= OFF_VT && OFF_VT + 16 * XT_RG <= OFF_A, "shared-memory map overlaps");
static_assert(OFF_HS + 4 * 128 * 4 <= OFF_KRA && OFF_KRA + 2 * tcc::ROW_TILE <= OFF_FRAGW &&
                  OFF_FRAGW + 4 * NGROUP * 4 <= OFF_GCA,
              "shared-memory map overlaps");
static_assert(3 * (SMEM_BYTES + 1024) <= 232448, "three CTAs must fit on an SM");

__device__ __forceinline__ void sync_all() { tcc::named_sync(1, NGROUP); }

// 8 x 8 bf16 block held one row per four lanes, transposed across the warp
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// T' hi/lo as mma.sync A fragments (M = 16 tokens, K = 16 tokens): the four 8 x 8 core matrices
// of the no-swizzle tile, rows 0..7 / 8..15 at +0 / +256 bytes, tokens 8..15 at +128
__device__ __forceinline__ void load_tprime(const unsigned char* sm, int lane, uint32_t (&th)[4], uint32_t (&tl)[4])
{
    const int mi = lane >> 3;
    const unsigned char* row = sm + OFF_T + (mi & 1) * 256 + (mi >> 1) * 128 + (lane & 7) * 16;
    tcc::ldsm4(row, th);
    tcc::ldsm4(row + tcc::SMALL_TILE, tl);
}

// W = T' (K Gamma) and U~ = T' V of the current chunk for the 8 channels [n0, n0 + 8) (N = 8 per
// tile, K = 16 tokens; T' = hi + lo, two products each).
__device__ __forceinline__ void wu_tile(const unsigned char* sm, const uint32_t (&th)[4], const uint32_t (&tl)[4], int n0,
                                        int g, int t, float (&wa)[4], float (&ua)[4])
{
    const uint32_t o0 = tcc::none_off_rg<XT_RG>(n0 + g, 2 * t), o1 = tcc::none_off_rg<XT_RG>(n0 + g, 2 * t + 8);
    const uint32_t xb0 = *reinterpret_cast<const uint32_t*>(sm + OFF_XT + o0);
    const uint32_t xb1 = *reinterpret_cast<const uint32_t*>(sm + OFF_XT + o1);
    const uint32_t vb0 = *reinterpret_cast<const uint32_t*>(sm + OFF_VT + o0);
    const uint32_t vb1 = *reinterpret_cast<const uint32_t*>(sm + OFF_VT + o1);
#pragma unroll
    for (int e = 0; e < 4; ++e) wa[e] = ua[e] = 0.f;
    tc::mma16816(wa, th, xb0, xb1);
    tc::mma16816(wa, tl, xb0, xb1);
    tc::mma16816(ua, th, vb0, vb1);
    tc::mma16816(ua, tl, vb0, vb1);
}

// Chunk a: W_a (rows 0..15 of the block's SW128 [W ; Q] tile, bf16) and U~_a (rows 0..15 of its
// fp32 tile) for the 16 channels [16 w, 16 w + 16) of warp w; W_a is also kept as the B operand of
// X W_a (k = token, n = channel), which is the transpose of the 8 x 8 blocks just computed.
__device__ __forceinline__ void wy_first(unsigned char* sm, unsigned char* blk, int w, int lane, int tid)
{
    const int g = lane >> 2, t = lane & 3;
    uint32_t th[4], tl[4];
    load_tprime(sm, lane, th, tl);
    float* ut = reinterpret_cast<float*>(blk + tcc::BLK_UT);
    uint32_t* fragw = reinterpret_cast<uint32_t*>(sm + OFF_FRAGW);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int n0 = 16 * w + 8 * nt;
        float wa[4], ua[4];
        wu_tile(sm, th, tl, n0, g, t, wa, ua);
        const int c = n0 + 2 * t;
        const uint32_t w01 = tcc::pack_f2(wa[0], wa[1]), w23 = tcc::pack_f2(wa[2], wa[3]);
        *reinterpret_cast<uint32_t*>(blk + tcc::BLK_WQ + tc::sw128_off(g, c, 2 * PAIR)) = w01;
        *reinterpret_cast<uint32_t*>(blk + tcc::BLK_WQ + tc::sw128_off(g + 8, c, 2 * PAIR)) = w23;
        *reinterpret_cast<float2*>(ut + g * D + c) = make_float2(ua[0], ua[1]);
        *reinterpret_cast<float2*>(ut + (g + 8) * D + c) = make_float2(ua[2], ua[3]);
        fragw[(2 * nt) * NGROUP + tid] = transpose8x8(w01);
        fragw[(2 * nt + 1) * NGROUP + tid] = transpose8x8(w23);
    }
}

// Chunk b and the pair assembly: rows 16..31 of W and U~ (see the file comment), the pair's K~ rows
// of chunk a's tokens and the pair's Gamma_C.  U~_a is read back from the block (rows 0..15,
// written by this CTA in wy_first).
__device__ __forceinline__ void wy_second(unsigned char* sm, unsigned char* blk, int w, int lane, int tid)
{
    const int g = lane >> 2, t = lane & 3;
    float* ut = reinterpret_cast<float*>(blk + tcc::BLK_UT);
    float ur[2][4];  // U~_a as B operands: (k = token 2t, 2t + 1, 2t + 8, 2t + 9; n = channel)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int j = 16 * w + 8 * nt + g;
        ur[nt][0] = ut[(2 * t) * D + j];
        ur[nt][1] = ut[(2 * t + 1) * D + j];
        ur[nt][2] = ut[(2 * t + 8) * D + j];
        ur[nt][3] = ut[(2 * t + 9) * D + j];
    }
    uint32_t th[4], tl[4];
    load_tprime(sm, lane, th, tl);
    // X = T' Y, every warp the whole 16 x 16 (its accumulator fragments are the A fragments of X W_a)
    float xa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const unsigned char* yt = sm + OFF_YT;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const uint32_t o0 = tc::none_off(8 * nt + g, 2 * t), o1 = tc::none_off(8 * nt + g, 2 * t + 8);
        const uint32_t yh0 = *reinterpret_cast<const uint32_t*>(yt + o0);
        const uint32_t yh1 = *reinterpret_cast<const uint32_t*>(yt + o1);
        const uint32_t yl0 = *reinterpret_cast<const uint32_t*>(yt + tcc::SMALL_TILE + o0);
        const uint32_t yl1 = *reinterpret_cast<const uint32_t*>(yt + tcc::SMALL_TILE + o1);
        tc::mma16816(xa[nt], th, yh0, yh1);
        tc::mma16816(xa[nt], th, yl0, yl1);
        tc::mma16816(xa[nt], tl, yh0, yh1);
    }
    uint32_t xh[4], xl[4];
    tcc::split2(xa[0][0], xa[0][1], xh[0], xl[0]);  // (g, 2t)
    tcc::split2(xa[0][2], xa[0][3], xh[1], xl[1]);  // (g + 8, 2t)
    tcc::split2(xa[1][0], xa[1][1], xh[2], xl[2]);  // (g, 2t + 8)
    tcc::split2(xa[1][2], xa[1][3], xh[3], xl[3]);  // (g + 8, 2t + 8)
    const float* gca = reinterpret_cast<const float*>(sm + OFF_GCA);
    const float* gcb = reinterpret_cast<const float*>(sm + OFF_GCB);
    const uint32_t* fragw = reinterpret_cast<const uint32_t*>(sm + OFF_FRAGW);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int n0 = 16 * w + 8 * nt;
        float wa[4], ua[4];
        wu_tile(sm, th, tl, n0, g, t, wa, ua);
        const uint32_t bw0 = fragw[(2 * nt) * NGROUP + tid], bw1 = fragw[(2 * nt + 1) * NGROUP + tid];
        float xw[4] = {0.f, 0.f, 0.f, 0.f};
        tc::mma16816(xw, xh, bw0, bw1);
        tc::mma16816(xw, xl, bw0, bw1);
        uint32_t bu0h, bu0l, bu1h, bu1l;
        tcc::split2(ur[nt][0], ur[nt][1], bu0h, bu0l);
        tcc::split2(ur[nt][2], ur[nt][3], bu1h, bu1l);
        float xu[4] = {0.f, 0.f, 0.f, 0.f};
        tc::mma16816(xu, xh, bu0h, bu1h);
        tc::mma16816(xu, xh, bu0l, bu1l);
        tc::mma16816(xu, xl, bu0h, bu1h);
        const int c = n0 + 2 * t;
        const float2 ga = *reinterpret_cast<const float2*>(gca + c);
        *reinterpret_cast<uint32_t*>(blk + tcc::BLK_WQ + tc::sw128_off(C + g, c, 2 * PAIR)) =
            tcc::pack_f2(wa[0] * ga.x - xw[0], wa[1] * ga.y - xw[1]);
        *reinterpret_cast<uint32_t*>(blk + tcc::BLK_WQ + tc::sw128_off(C + 8 + g, c, 2 * PAIR)) =
            tcc::pack_f2(wa[2] * ga.x - xw[2], wa[3] * ga.y - xw[3]);
        *reinterpret_cast<float2*>(ut + (C + g) * D + c) = make_float2(ua[0] - xu[0], ua[1] - xu[1]);
        *reinterpret_cast<float2*>(ut + (C + 8 + g) * D + c) = make_float2(ua[2] - xu[2], ua[3] - xu[3]);
    }
    {
        // (K~_a Gamma_Cb)^T: channel c = tid / 2, tokens 8 (tid & 1) .. + 7, one 16-byte store each
        const int c = tid >> 1, i0 = 8 * (tid & 1);
        const float gb = gcb[c];
        const __nv_bfloat16* ka = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_KRA);
        const __nv_bfloat16* kal = ka + C * tcc::LROW;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = i0 + 2 * e;
            const float x0 = (__bfloat162float(ka[i * tcc::LROW + c]) + __bfloat162float(kal[i * tcc::LROW + c])) * gb;
            const float x1 =
                (__bfloat162float(ka[(i + 1) * tcc::LROW + c]) + __bfloat162float(kal[(i + 1) * tcc::LROW + c])) * gb;
            tcc::split2(x0, x1, hi[e], lo[e]);
        }
        const uint32_t o = tcc::pk_off(2 * C + c, i0);
        *reinterpret_cast<uint4*>(blk + tcc::BLK_PK + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(blk + tcc::BLK_PK + tcc::BLK_PK_LO + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        if (tid < D) reinterpret_cast<float*>(blk + tcc::BLK_GC)[tid] = gca[tid] * gcb[tid];
    }
}

}  // namespace

__global__ void __launch_bounds__(NGROUP, 3) kda_chunk_prep_tc_kernel(PrefillArgs a, const __grid_constant__ TileMaps maps)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sm + OFF_ABORT);
    float* sbeta = reinterpret_cast<float*>(sm + OFF_BETA);
    float* gca = reinterpret_cast<float*>(sm + OFF_GCA);
    float* gcb = reinterpret_cast<float*>(sm + OFF_GCB);

    const int run_pairs = a.prep_run;
    const int64_t pairs_max = ((int64_t)a.chunks_per_seq + 1) / 2;
    const int runs = (int)((pairs_max + run_pairs - 1) / run_pairs);
    const int n = (int)(blockIdx.x / (unsigned)runs);
    const int run = (int)(blockIdx.x % (unsigned)runs);
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int w = tid >> 5, lane = tid & 31;
    griddep_launch_dependents();

    int64_t q0, q1;
    if (!seq_range(a, n, q0, q1)) return;
    const int64_t seq_chunks = (q1 - q0 + C - 1) / C;
    const int64_t seq_pairs = (seq_chunks + 1) / 2;
    const int64_t pb = (int64_t)run * run_pairs;
    const int64_t pe = min(pb + run_pairs, seq_pairs);
    if (pb >= pe) return;
    const int H = a.H;
    const int64_t slot0 = q0 / PAIR + n;  // block slot of the sequence's first step
    const float expA = expf(a.A[h]);
    const float g_min = a.g_min;

    if (tid == 0) {
        tc::mbar_init(bar, 1);
        *abort_flag = 0u;
    }
    tc::fence_async_smem();
    __syncthreads();

    // chunk c of the sequence; the second chunk of the last pair may hold no tokens (then nothing
    // is loaded and every token of it counts as absent)
    auto has_tokens = [&](int64_t c) { return q0 + c * C < q1; };
    auto issue_tiles = [&](int64_t c) {
        const int tn = (int)(q0 + c * C);
        tc::mbar_arrive_expect_tx(bar, 4 * tcc::STAGE_TILE);
        tc::tma_load_3d(sm + OFF_STAGE, &maps.q, 0, h, tn, bar);
        tc::tma_load_3d(sm + OFF_STAGE + tcc::STAGE_TILE, &maps.k, 0, h, tn, bar);
        tc::tma_load_3d(sm + OFF_STAGE + 2 * tcc::STAGE_TILE, &maps.v, 0, h, tn, bar);
        tc::tma_load_3d(sm + OFF_STAGE + 3 * tcc::STAGE_TILE, &maps.z, 0, h, tn, bar);
    };
    auto load_beta = [&](int64_t c) -> float {  // threads 0..15
        const int64_t t = q0 + c * C + tid;
        return (t < q1) ? a.beta[t * H + h] : 0.f;
    };
    const int64_t cb = 2 * pb, ce = 2 * pe;
    bool pend_ld = false;  // thread 0: a tile load whose completion was not observed
    if (tid == 0) {
        issue_tiles(cb);
        pend_ld = true;
    }
    float beta_next = (tid < C) ? load_beta(cb) : 0.f;
    uint32_t ph = 0;

    for (int64_t c = cb; c < ce; ++c) {
        const bool second = (c & 1) != 0;
        const int len = (int)max((int64_t)0, min((int64_t)C, q1 - (q0 + c * C)));
        if (tid < C) sbeta[tid] = beta_next;
        if (tid == 0 && pend_ld) {
            if (tc::mbar_wait(bar, ph, WAIT_LIMIT)) pend_ld = false, ph ^= 1u;
            else *abort_flag = 1u;
        }
        sync_all();
        const bool dead = *abort_flag != 0u;
        unsigned char* blk = a.blocks + ((slot0 + (c >> 1)) * H + h) * (int64_t)tcc::BLK_BYTES;  // global
        if (!dead) {
            if (!second) {
                // Q Gamma hi into rows 32..47 of [W ; Q]; K~ row-major to shared memory for the pair
                tcc::prep_factors<PrepMap>(sm, tid, len, blk + tcc::BLK_WQ, nullptr, gca, expA, g_min, false,
                                           tcc::BLK_PK_LO, tcc::kNoneTile, 2 * C, 2 * PAIR, sm + OFF_KRA);
            } else {
                // (Q Gamma)_b Gamma_Ca into rows 48..63; K~_b^T into the [P ; K~^T] rows 32.., tokens 16..31
                tcc::prep_factors<PrepMap>(sm, tid, len, blk + tcc::BLK_WQ, blk + tcc::BLK_PK, gcb, expA, g_min,
                                           false, tcc::BLK_PK_LO, tcc::NonePlace{tcc::PK_RG, 2 * C, C}, 3 * C,
                                           2 * PAIR, nullptr, gca);
            }
        } else {
            sync_all();  // the barrier inside prep_factors
        }
        tc::fence_async_smem();
        sync_all();  // the stage has been consumed
        if (c + 1 < ce) {
            if (tid == 0 && !dead && has_tokens(c + 1)) {
                issue_tiles(c + 1);
                pend_ld = true;
            }
            if (tid < C) beta_next = load_beta(c + 1);
        }
        if (!dead) {
            if (!second) {
                tcc::prep_solve<PrepMap, tcc::SOLVE_FIRST>(sm, tid, blk + tcc::BLK_PK, tcc::BLK_PK_LO,
                                                           tcc::NonePlace{tcc::PK_RG, 0, 0});
            } else {
                tcc::prep_solve<PrepMap, tcc::SOLVE_SECOND>(sm, tid, blk + tcc::BLK_PK, tcc::BLK_PK_LO,
                                                            tcc::NonePlace{tcc::PK_RG, C, C});
            }
        } else {
            sync_all();
            sync_all();
        }
        sync_all();  // T' (and for chunk b: Y^T, Z) complete
        if (!dead) {
            if (!second) wy_first(sm, blk, w, lane, tid);
            else wy_second(sm, blk, w, lane, tid);
        }
    }
    if (tid == 0) {
        if (*abort_flag) {
            atomicOr(a.check, kCheckTimeout);
            if (pend_ld) (void)tc::mbar_wait(bar, ph, WAIT_LIMIT);  // a load in flight must land first
        }
    }
}

cudaError_t launch_chunk_prep_tc(const PrefillArgs& a, cudaStream_t s)
{
    TileMaps maps;
    if (!encode_tile_maps(maps, a)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kda_chunk_prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // runs of kRunLong steps once the short-run grid would take more than ~8 waves of resident CTAs
    const int64_t pairs = ((int64_t)a.chunks_per_seq + 1) / 2;
    const int64_t short_ctas = (pairs + kRunShort - 1) / kRunShort * a.N * a.H;
    PrefillArgs b = a;
    b.prep_run = short_ctas > 8LL * 3 * sm_count_of_current_device() ? kRunLong : kRunShort;
    const int64_t runs = (pairs + b.prep_run - 1) / b.prep_run;
    const int64_t gx = runs * a.N;  // at most N x chunks_per_seq < 2^31 (checked by the caller)
    if (gx == 0) return cudaSuccess;
    kda_chunk_prep_tc_kernel<<<dim3((unsigned)gx, (unsigned)a.H, 1), NGROUP, SMEM_BYTES, s>>>(b, maps);
    return cudaGetLastError();
}

}  // namespace kda
