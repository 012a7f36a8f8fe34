// kda_state_tc.cu -- the sequential state pass of the bf16, d = 128 prefill on the tensor cores.
//
// Per chunk of one (sequence, head[, segment]), with the chunk's operand block prepared by
// kda_prep_tc.cu (W, Q Gamma, (K Gamma_C / Gamma)^T, U~, P, Gamma_C):
//   U = U~ - W S,   O = (Q Gamma) S + P U,   S <- Diag(Gamma_C) S + (K Gamma_C / Gamma)^T U
// (the chunk form of Equation 1, "Kimi K3: the paper and proofs side by side", section 2.1.1;
// "Kimi K3: architecture, derivations and a pinned-source audit", section 4.5).
//
// Value channels j are the 128 TMEM lanes.  Per chunk: D1 = S^T [W ; Q Gamma]^T (M = 128, N = 32,
// K = 128) -> U^T = U~^T - D1[:, :16] as a bf16 hi/lo pair -> O^T += U^T P^T and
// dS^T = U^T (K Gamma_C / Gamma) (hi*hi + hi*lo + lo*hi) -> S <- Diag(Gamma_C) S + dS in registers
// (thread = one value channel x 64 key channels), re-staged as the bf16 SW128 operand of the next D1.
// The blocks stream through a two-slot shared-memory ring by plain bulk copies, the next but one
// issued as soon as a slot is free.  256 threads and ~93 KB of shared memory per CTA: two CTAs
// (two independent chains) share an SM, hiding each other's latency.
//
// Modes (segmented prefill, see the launcher): 0 writes outputs and (last segment) the final state;
// 1 computes S~, the segment's end state from a zero start; 2 computes M, the segment's transition,
// as the end state from the identity with V = 0 (columns of M evolve exactly like state columns).
// Every mbarrier wait is bounded; a wait that gives up raises the timeout bit of the check word,
// the CTA skips the remaining work, waits (bounded) for its copies in flight and frees its TMEM.
#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_tc_chunk.cuh"

namespace kda {

namespace {

using tcc::C;
using tcc::D;
using tcc::NONE_TILE;
using tcc::SMALL_TILE;
using tcc::u2f;

constexpr int NTHREADS = 256;
constexpr uint32_t WAIT_LIMIT = 1u << 17;  // tries of up to 20 us each: ~2.6 s at most
constexpr uint32_t SLOT = 26624;           // ring slot stride (a multiple of 1024 >= BLK_BYTES)

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_S = 0;           // S^T [128 j][128 c] bf16 SW128                 32768
constexpr uint32_t OFF_RING = 32768;    // [2] operand blocks                        2 x 26624
constexpr uint32_t OFF_UT = 86016;      // U^T hi, lo [128 j][16 i] NONE                  8192
constexpr uint32_t OFF_BARF = 94208;    // mbarriers: ring slot filled [2]                  16
constexpr uint32_t OFF_BARC = 94224;    // mbarrier: tensor-core commits                     8
constexpr uint32_t OFF_TSLOT = 94232;   // TMEM base address                                  4
constexpr uint32_t OFF_ABORT = 94236;   // stop flag                                          4
constexpr uint32_t SMEM_USED = 94240;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;

static_assert(SLOT >= tcc::BLK_BYTES && SLOT % 1024 == 0, "ring slots must hold a block at 1024-byte alignment");
static_assert(OFF_UT >= OFF_RING + 2 * SLOT, "shared-memory map overlaps");

// tensor-memory columns
constexpr uint32_t TM_D1 = 0;    // [0, 16) (W S)^T, [16, 32) O^T
constexpr uint32_t TM_D3 = 128;  // dS^T (lanes = j, columns = c)
constexpr uint32_t TM_COLS = 256;

__device__ __forceinline__ void sync_all() { tcc::named_sync(1, NTHREADS); }

// Abort flag, read identically by every lane of the warp; every lane of the warp must call it.
__device__ __forceinline__ bool read_dead(const volatile uint32_t* abort_flag)
{
    return __any_sync(0xffffffffu, *abort_flag != 0u);
}

}  // namespace

__global__ void __launch_bounds__(NTHREADS, 2) kda_chunk_state_tc_kernel(PrefillArgs a)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bar_f = reinterpret_cast<uint64_t*>(sm + OFF_BARF);
    uint64_t* bar_c = reinterpret_cast<uint64_t*>(sm + OFF_BARC);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_TSLOT);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sm + OFF_ABORT);

    const int n = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int w = tid >> 5;
    const int lane = tid & 31;

    int64_t q0, q1;
    if (!seq_range(a, n, q0, q1)) return;
    // segment k of the sequence and what this CTA computes for it (see the file comment)
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
    const int64_t cbase = q0 / C + n + (int64_t)k * seg_c;  // block slot of the segment's first chunk
    auto chunk_len = [&](int chunk) -> int { return (int)min((int64_t)C, s1 - (s0 + (int64_t)chunk * C)); };
    auto block_of = [&](int chunk) -> const unsigned char* {
        return a.blocks + ((cbase + chunk) * H + h) * (int64_t)tcc::BLK_BYTES;
    };

    if (w == 0) tc::tmem_alloc(tslot, TM_COLS);
    if (tid == 0) {
        tc::mbar_init(&bar_f[0], 1);
        tc::mbar_init(&bar_f[1], 1);
        tc::mbar_init(bar_c, 1);
        *abort_flag = 0u;
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tslot;

    // thread 0 owns the ring: pending loads per slot and the parity of each slot's next fill
    uint32_t pend = 0, ph_f0 = 0, ph_f1 = 0, ph_c = 0;
    bool pend_c = false;  // a tensor-core commit whose completion was not observed
    auto issue_load = [&](int chunk) {
        const int sl = chunk & 1;
        tc::mbar_arrive_expect_tx(&bar_f[sl], tcc::BLK_BYTES);
        tc::bulk_load(sm + OFF_RING + sl * SLOT, block_of(chunk), tcc::BLK_BYTES, &bar_f[sl]);
        pend |= 1u << sl;
    };
    auto wait_slot = [&](int sl) -> bool {
        const bool ok = tc::mbar_wait(&bar_f[sl], sl ? ph_f1 : ph_f0, WAIT_LIMIT);
        if (ok) {
            pend &= ~(1u << sl);
            if (sl) ph_f1 ^= 1u;
            else ph_f0 ^= 1u;
        }
        return ok;
    };
    if (tid == 0) {
        if (nchunks > 0) issue_load(0);
        if (nchunks > 1) issue_load(1);
    }

    const int q4 = w & 3;    // TMEM lane quarter
    const int h2 = w >> 2;   // which half of the key channels this warp's state slice covers
    const int jrow = 32 * q4 + lane;
    const uint32_t lane_base = tbase + ((uint32_t)(32 * q4) << 16);
    __nv_bfloat16* op = static_cast<__nv_bfloat16*>(a.out);

    // state slice: S[c][jrow] for c in [64*h2, 64*h2 + 64)
    float S[64];
    const int64_t sbase = ((int64_t)n * H + h) * D * D;
    const int64_t segbase = (((int64_t)n * H + h) * a.max_seg + k) * D * D;
    const float* init = nullptr;
    if (mode == 0) init = (k == 0) ? (a.s0 ? a.s0 + sbase : nullptr) : a.seg_in + segbase;
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
    tc::fence_before_sync();
    sync_all();
    tc::fence_after_sync();

    for (int ch = 0; ch < nchunks; ++ch) {
        const int sl = ch & 1;
        unsigned char* blk = sm + OFF_RING + sl * SLOT;
        const int64_t t0 = s0 + (int64_t)ch * C;
        const int len = chunk_len(ch);
        bool dead = read_dead(abort_flag);

        // D1 = S^T [W ; Q Gamma]^T (M = 128, K = 128; N = 32 with outputs, else 16: W only)
        if (tid == 0 && !dead) {
            if (!wait_slot(sl)) {
                *abort_flag = 1u;
            } else {
                const uint32_t nq = (mode == 0) ? 2 * C : C;
                const uint32_t idd = tc::idesc_bf16(128, (int)nq);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
                    tc::umma(tbase + TM_D1, tc::desc_sw128(tc::smem_u32(sm + OFF_S + kb * 16384 + off)),
                             tc::desc_sw128(tc::smem_u32(blk + tcc::BLK_WQ + kb * (2 * C * 128) + off)), idd,
                             ks > 0 ? 1u : 0u);
                }
                tc::umma_commit(bar_c);
                if (tc::mbar_wait(bar_c, ph_c, WAIT_LIMIT)) ph_c ^= 1u;
                else *abort_flag = 1u, pend_c = true;
            }
        }
        sync_all();
        tc::fence_after_sync();
        dead = read_dead(abort_flag);

        // U^T = U~^T - (W S)^T as a hi/lo pair; warp half h2 takes tokens 8 h2 .. 8 h2 + 7
        if (!dead) {
            uint32_t dv[8];
            KDA_TMEM_LD8(lane_base + TM_D1 + 8 * h2, dv);
            float uv[8];
            const float* ut = reinterpret_cast<const float*>(blk + tcc::BLK_UT);
#pragma unroll
            for (int e = 0; e < 8; ++e) uv[e] = (mode == 2) ? 0.f : ut[(8 * h2 + e) * D + jrow];
            tc::tmem_wait_ld();
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                tcc::split2(uv[2 * e] - u2f(dv[2 * e]), uv[2 * e + 1] - u2f(dv[2 * e + 1]), hi[e], lo[e]);
            }
            *reinterpret_cast<uint4*>(sm + OFF_UT + tc::none_off(jrow, 8 * h2)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(sm + OFF_UT + NONE_TILE + tc::none_off(jrow, 8 * h2)) =
                make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        sync_all();
        tc::fence_after_sync();

        // O^T += U^T P^T (outputs only) and dS^T = U^T (K Gamma_C / Gamma), each hi*hi + hi*lo + lo*hi
        if (tid == 0 && !dead) {
            const uint32_t id16 = tc::idesc_bf16(128, 16);
            const uint32_t id128 = tc::idesc_bf16(128, 128);
            const uint64_t dU = tc::desc_none(tc::smem_u32(sm + OFF_UT));
            const uint64_t dUl = tc::desc_none(tc::smem_u32(sm + OFF_UT + NONE_TILE));
            const uint64_t dK = tc::desc_none(tc::smem_u32(blk + tcc::BLK_KT));
            const uint64_t dKl = tc::desc_none(tc::smem_u32(blk + tcc::BLK_KT + NONE_TILE));
            if (mode == 0) {
                const uint64_t dP = tc::desc_none(tc::smem_u32(blk + tcc::BLK_P));
                const uint64_t dPl = tc::desc_none(tc::smem_u32(blk + tcc::BLK_P + SMALL_TILE));
                tc::umma(tbase + TM_D1 + C, dU, dP, id16, 1u);
                tc::umma(tbase + TM_D1 + C, dU, dPl, id16, 1u);
                tc::umma(tbase + TM_D1 + C, dUl, dP, id16, 1u);
            }
            tc::umma(tbase + TM_D3, dU, dK, id128, 0u);
            tc::umma(tbase + TM_D3, dU, dKl, id128, 1u);
            tc::umma(tbase + TM_D3, dUl, dK, id128, 1u);
            tc::umma_commit(bar_c);
            if (tc::mbar_wait(bar_c, ph_c, WAIT_LIMIT)) ph_c ^= 1u;
            else *abort_flag = 1u, pend_c = true;
        }
        sync_all();
        tc::fence_after_sync();
        dead = read_dead(abort_flag);

        // S <- Diag(Gamma_C) S + dS (staged for the next read), outputs of the chunk
        if (!dead) {
            const float* gc = reinterpret_cast<const float*>(blk + tcc::BLK_GC) + 64 * h2;
#pragma unroll
            for (int b4 = 0; b4 < 4; b4 += 2) {
                uint32_t v0[16], v1[16];
                KDA_TMEM_LD16(lane_base + TM_D3 + 64 * h2 + 16 * b4, v0);
                KDA_TMEM_LD16(lane_base + TM_D3 + 64 * h2 + 16 * b4 + 16, v1);
                tc::tmem_wait_ld();
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const float4 g4 = *reinterpret_cast<const float4*>(gc + 16 * b4 + 4 * e4);
                    const int cc = 16 * b4 + 4 * e4;
                    const uint32_t* vv = (e4 < 4) ? v0 : v1;
                    const int o = (e4 & 3) * 4;
                    S[cc + 0] = g4.x * S[cc + 0] + u2f(vv[o + 0]);
                    S[cc + 1] = g4.y * S[cc + 1] + u2f(vv[o + 1]);
                    S[cc + 2] = g4.z * S[cc + 2] + u2f(vv[o + 2]);
                    S[cc + 3] = g4.w * S[cc + 3] + u2f(vv[o + 3]);
                }
            }
            stage_state();
            if (mode == 0) {
                uint32_t ov[8];
                KDA_TMEM_LD8(lane_base + TM_D1 + C + 8 * h2, ov);
                tc::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int r = 8 * h2 + e;
                    if (r < len) op[((t0 + r) * H + h) * D + jrow] = __float2bfloat16_rn(u2f(ov[e]));
                }
            }
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        sync_all();  // every read of this slot is done; the next state is staged
        tc::fence_after_sync();
        if (tid == 0 && ch + 2 < nchunks && *abort_flag == 0u) issue_load(ch + 2);
    }

    float* dst = nullptr;
    if (mode == 0) dst = ((int64_t)k == nseg - 1 && a.s_final) ? a.s_final + sbase : nullptr;
    else dst = (mode == 1 ? a.seg_st : a.seg_mt) + segbase;
    if (*abort_flag) {
        if (tid == 0) {
            atomicOr(a.check, kCheckTimeout);
            // copies and tensor-core work still in flight must finish before the shared and tensor
            // memory are released
            for (int sl = 0; sl < 2; ++sl) {
                if (pend & (1u << sl)) (void)wait_slot(sl);
            }
            if (pend_c) (void)tc::mbar_wait(bar_c, ph_c, WAIT_LIMIT);
        }
    } else if (dst) {
#pragma unroll
        for (int cc = 0; cc < 64; ++cc) dst[(int64_t)(64 * h2 + cc) * D + jrow] = S[cc];
    }
    tc::fence_before_sync();
    __syncthreads();
    if (w == 0) tc::tmem_dealloc(tbase, TM_COLS);
}

namespace {

cudaError_t launch_chunk_state_tc(const PrefillArgs& a, int seg_mode, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(kda_chunk_state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    PrefillArgs b = a;
    b.seg_mode = seg_mode;
    const unsigned gz = seg_mode == 0 ? (unsigned)(a.max_seg > 1 ? a.max_seg : 1) : (unsigned)(2 * (a.max_seg - 1));
    if (gz == 0) return cudaSuccess;
    kda_chunk_state_tc_kernel<<<dim3((unsigned)a.N, (unsigned)a.H, gz), NTHREADS, SMEM_BYTES, s>>>(b);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_split_tc(const PrefillArgs& a, cudaStream_t s)
{
    prof_start("kda_chunk_prep_tc", s);
    cudaError_t e = launch_chunk_prep_tc(a, s);
    prof_stop(s);
    if (e != cudaSuccess) return e;
    if (a.seg_chunks > 0 && a.max_seg > 1) {
        // (S~, M) of every segment but the last, then the scan of the incoming states
        prof_start("kda_state_summary_tc", s);
        e = launch_chunk_state_tc(a, 1, s);
        prof_stop(s);
        if (e != cudaSuccess) return e;
        prof_start("kda_seg_scan", s);
        e = launch_segment_scan(a, s);
        prof_stop(s);
        if (e != cudaSuccess) return e;
    }
    prof_start("kda_chunk_state_tc", s);
    e = launch_chunk_state_tc(a, 0, s);
    prof_stop(s);
    return e;
}

}  // namespace kda
