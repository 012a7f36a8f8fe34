// kda_prep_tc.cu -- parallel per-chunk preparation of the bf16, d = 128 prefill.
//
// Everything of a 16-token chunk that does not depend on the recurrent state -- the gate
// (Equation 5), the in-chunk decays, the WY/UT transform and the in-chunk output product -- is
// computed here for every chunk of every (sequence, head) at once, and written as one contiguous
// operand block per chunk (layout: tcc::BLK_*):
//   [W ; Q Gamma] SW128, [P ; (K Gamma_C / Gamma)^T] hi/lo, U~ = T' V (fp32), Gamma_C
// with W = T diag(beta) (K Gamma), U~ = T diag(beta) V, T = (I + A)^-1 (the chunk form of Equation 1,
// "Kimi K3: the paper and proofs side by side", section 2.1.1; "Kimi K3: architecture, derivations
// and a pinned-source audit", section 4.5).  The sequential state pass (kda_state_tc.cu) then
// only streams these blocks.
//
// One CTA of 256 threads (three per SM) walks a run of up to kRun chunks of one (sequence, head):
// the q, k, v, z tiles arrive by TMA one chunk ahead, the factors, A, P and T come from the shared preparation
// functions, W and U~ from warp-level mma.sync (T' hi/lo against (K Gamma)^T and V^T), and the
// assembled block leaves shared memory as one bulk copy.  Block slot of chunk c of sequence n:
// cu[n] / 16 + n + c, so the slots of consecutive sequences never overlap
// (ceil(len / 16) <= floor((cu[n] mod 16 + len) / 16) + 1).
#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_tc_chunk.cuh"

namespace kda {

namespace {

using tcc::C;
using tcc::D;
using tcc::NGROUP;

constexpr int kRun = 4;                      // chunks per CTA
constexpr uint32_t WAIT_LIMIT = 1u << 17;    // tries of up to 20 us each

// shared-memory map (bytes from a 1024-aligned base); the operand block itself is written straight
// to global memory
constexpr uint32_t XT_RG = 272;          // padded 8-row-group stride of the transposed tiles
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
constexpr uint32_t OFF_BETA = 59136;     // beta [16]                                     64
constexpr uint32_t OFF_BAR = 59200;      // mbarrier: TMA tile loads                       8
constexpr uint32_t OFF_ABORT = 59208;    // stop flag                                      4
constexpr uint32_t SMEM_USED = 59212;
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
    static constexpr uint32_t NB = 1;
    static constexpr uint32_t XT_RG = ::kda::XT_RG;
};

static_assert(OFF_XT + 16 * XT_RG <= OFF_VT && OFF_VT + 16 * XT_RG <= OFF_A, "shared-memory map overlaps");
static_assert(3 * (SMEM_BYTES + 1024) <= 232448, "three CTAs must fit on an SM");

__device__ __forceinline__ void sync_all() { tcc::named_sync(1, NGROUP); }

// W = T' (K Gamma) and U~ = T' V for the 16 channels [16 w, 16 w + 16) of warp w, by mma.sync
// (M = 16 tokens, N = 8 channels per tile, K = 16 tokens; T' = hi + lo, two products each).
// W goes to rows 0..15 of the block's SW128 [W ; Q Gamma] tile (bf16), U~ to its fp32 tile.
__device__ __forceinline__ void wy_products(const unsigned char* sm, unsigned char* blk, int w, int lane)
{
    const int g = lane >> 2, t = lane & 3;
    const unsigned char* tt = sm + OFF_T;
    uint32_t th[4], tl[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t o = tc::none_off(g + 8 * (e & 1), 2 * t + 8 * (e >> 1));
        th[e] = *reinterpret_cast<const uint32_t*>(tt + o);
        tl[e] = *reinterpret_cast<const uint32_t*>(tt + tcc::SMALL_TILE + o);
    }
    float* ut = reinterpret_cast<float*>(blk + tcc::BLK_UT);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int n0 = 16 * w + 8 * nt;
        const uint32_t o0 = tcc::none_off_rg<XT_RG>(n0 + g, 2 * t), o1 = tcc::none_off_rg<XT_RG>(n0 + g, 2 * t + 8);
        const uint32_t xb0 = *reinterpret_cast<const uint32_t*>(sm + OFF_XT + o0);
        const uint32_t xb1 = *reinterpret_cast<const uint32_t*>(sm + OFF_XT + o1);
        const uint32_t vb0 = *reinterpret_cast<const uint32_t*>(sm + OFF_VT + o0);
        const uint32_t vb1 = *reinterpret_cast<const uint32_t*>(sm + OFF_VT + o1);
        float wa[4] = {0.f, 0.f, 0.f, 0.f}, ua[4] = {0.f, 0.f, 0.f, 0.f};
        tc::mma16816(wa, th, xb0, xb1);
        tc::mma16816(wa, tl, xb0, xb1);
        tc::mma16816(ua, th, vb0, vb1);
        tc::mma16816(ua, tl, vb0, vb1);
        const int c = n0 + 2 * t;
        *reinterpret_cast<uint32_t*>(blk + tcc::BLK_WQ + tc::sw128_off(g, c, 2 * C)) = tcc::pack_f2(wa[0], wa[1]);
        *reinterpret_cast<uint32_t*>(blk + tcc::BLK_WQ + tc::sw128_off(g + 8, c, 2 * C)) = tcc::pack_f2(wa[2], wa[3]);
        *reinterpret_cast<float2*>(ut + g * D + c) = make_float2(ua[0], ua[1]);
        *reinterpret_cast<float2*>(ut + (g + 8) * D + c) = make_float2(ua[2], ua[3]);
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

    const int runs = (a.chunks_per_seq + kRun - 1) / kRun;
    const int n = (int)(blockIdx.x / (unsigned)runs);
    const int run = (int)(blockIdx.x % (unsigned)runs);
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int w = tid >> 5, lane = tid & 31;
    griddep_launch_dependents();

    int64_t q0, q1;
    if (!seq_range(a, n, q0, q1)) return;
    const int64_t seq_chunks = (q1 - q0 + C - 1) / C;
    const int64_t cb = (int64_t)run * kRun;
    const int64_t ce = min(cb + kRun, seq_chunks);
    if (cb >= ce) return;
    const int H = a.H;
    const int64_t slot0 = q0 / C + n;  // block slot of the sequence's first chunk
    const float expA = expf(a.A[h]);
    const float g_min = a.g_min;

    if (tid == 0) {
        tc::mbar_init(bar, 1);
        *abort_flag = 0u;
    }
    tc::fence_async_smem();
    __syncthreads();

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
    bool pend_ld = false;  // thread 0: a tile load whose completion was not observed
    if (tid == 0) {
        issue_tiles(cb);
        pend_ld = true;
    }
    float beta_next = (tid < C) ? load_beta(cb) : 0.f;
    uint32_t ph = 0;

    for (int64_t c = cb; c < ce; ++c) {
        const int len = (int)min((int64_t)C, q1 - (q0 + c * C));
        if (tid < C) sbeta[tid] = beta_next;
        if (tid == 0 && pend_ld) {
            if (tc::mbar_wait(bar, ph, WAIT_LIMIT)) pend_ld = false, ph ^= 1u;
            else *abort_flag = 1u;
        }
        sync_all();
        const bool dead = *abort_flag != 0u;
        unsigned char* blk = a.blocks + ((slot0 + c) * H + h) * (int64_t)tcc::BLK_BYTES;  // global
        if (!dead) {
            tcc::prep_factors<PrepMap>(sm, tid, len, blk + tcc::BLK_WQ, blk + tcc::BLK_KT,
                                       reinterpret_cast<float*>(blk + tcc::BLK_GC), expA, g_min, false,
                                       tcc::BLK_PK_LO);
        } else {
            sync_all();  // the barrier inside prep_factors
        }
        tc::fence_async_smem();
        sync_all();  // the stage has been consumed
        if (c + 1 < ce) {
            if (tid == 0 && !dead) {
                issue_tiles(c + 1);
                pend_ld = true;
            }
            if (tid < C) beta_next = load_beta(c + 1);
        }
        if (!dead) {
            tcc::prep_solve<PrepMap>(sm, tid, blk + tcc::BLK_PK, tcc::BLK_PK_LO);
        } else {
            sync_all();
            sync_all();
        }
        sync_all();  // T' is complete
        if (!dead) wy_products(sm, blk, w, lane);
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
    const int64_t runs = ((int64_t)a.chunks_per_seq + kRun - 1) / kRun;
    const int64_t gx = runs * a.N;  // at most N x chunks_per_seq < 2^31 (checked by the caller)
    if (gx == 0) return cudaSuccess;
    kda_chunk_prep_tc_kernel<<<dim3((unsigned)gx, (unsigned)a.H, 1), NGROUP, SMEM_BYTES, s>>>(a, maps);
    return cudaGetLastError();
}

}  // namespace kda
