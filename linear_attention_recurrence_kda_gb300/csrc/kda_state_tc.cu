// kda_state_tc.cu -- the sequential state pass of the bf16, d = 128 prefill on the tensor cores.
//
// The state advances in 32-token steps (two 16-token chunks fused by the preparation kernel,
// kda_prep_tc.cu, into one operand block: W, Q Gamma, [P ; (K Gamma_C / Gamma)^T], U~, Gamma_C):
//   U = U~ - W S,   O = (Q Gamma) S + P U,   S <- Diag(Gamma_C) S + (K Gamma_C / Gamma)^T U
// (the chunk form of Equation 1, "Kimi K3: the paper and proofs side by side", section 2.1.1;
// "Kimi K3: architecture, derivations and a pinned-source audit", section 4.5).
//
// Value channels j are the 128 TMEM lanes; the fp32 state S^T [j][c] itself lives in tensor memory.
// Per step:
//   D1 = bf16(S)^T [W ; Q Gamma]^T      (M = 128, N = 64, K = 128: (W S)^T and (Q Gamma S)^T)
//   U^T = U~^T - (W S)^T                (a bf16 hi/lo pair, written to tensor memory over (W S)^T)
//   [O^T | S^T] += U^T [P ; (K Gamma_C / Gamma)^T]^T   (N = 160, K = 32: per hi/lo term two
//                                        instructions update the outputs and the state together;
//                                        S^T already holds S^T Diag(Gamma_C))
//   bf16(S)^T and S^T Diag(Gamma_C of the next step)   (one read of the new state writes the next
//                                        D1's A operand and the next update's decayed state)
// A tcgen05.mma costs about the same whatever N is, so a step is organised around few
// instructions: 8 for D1 and 6 for the fused update, for 32 tokens.  The operand blocks stream
// through a two-slot shared-memory ring by plain bulk copies.  256 threads, ~107 KB of shared
// memory and 256 TMEM columns per CTA: two CTAs (two independent chains) share an SM.  Outputs are
// moved from tensor memory to registers after the update and stored while the next step's D1 runs.
//
// Modes (segmented prefill, see the launcher): 0 writes outputs and (last segment) the final state;
// 1 computes S~, the segment's end state from a zero start; 2 computes M, the segment's transition,
// as the end state from the identity with V = 0 (columns of M evolve exactly like state columns),
// stored as the scan's bf16 hi/lo operand (seg_m_off).  Every mbarrier wait is bounded; a wait
// that gives up raises the timeout bit of the check word, the CTA skips the remaining work, waits
// (bounded) for its copies and products in flight and frees its tensor memory.
#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_tc_chunk.cuh"

namespace kda {

namespace {

using tcc::C;
using tcc::D;
using tcc::u2f;

constexpr int NTHREADS = 256;
constexpr uint32_t WAIT_LIMIT = 1u << 17;  // tries of up to 20 us each: ~2.6 s at most
constexpr int CT = tcc::PAIR;              // tokens per step (32)
constexpr int NSLOT = 2;                   // ring depth (steps in flight)
constexpr uint32_t SLOT = 54272;           // ring slot stride (a multiple of 1024 >= BLK_BYTES)

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_RING = 0;                         // [NSLOT] operand blocks
constexpr uint32_t OFF_BARF = NSLOT * SLOT;              // mbarriers: ring slot filled [NSLOT]
constexpr uint32_t OFF_BARC = OFF_BARF + 8 * NSLOT;      // mbarrier: tensor-core commits
constexpr uint32_t OFF_TSLOT = OFF_BARC + 8;             // TMEM base address
constexpr uint32_t OFF_ABORT = OFF_TSLOT + 4;            // stop flag
constexpr uint32_t SMEM_USED = OFF_ABORT + 4;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;

static_assert(SLOT >= tcc::BLK_BYTES && SLOT % 1024 == 0, "ring slots must hold a block at 1024-byte alignment");
static_assert(2 * (SMEM_BYTES + 1024) <= 232448, "two CTAs must fit on an SM");

// tensor-memory columns
constexpr uint32_t TM_WU = 0;     // D1's (W S)^T [32 tokens], then U^T hi/lo: tokens 16 h .. 16 h + 15 hi at
                                  // columns 16 h .. 16 h + 7, lo at 16 h + 8 .. 16 h + 15 (h = 0, 1)
constexpr uint32_t TM_O = 32;     // D1's (Q Gamma S)^T, then O^T; immediately followed by the state
constexpr uint32_t TM_S = 64;     // S^T fp32 (lanes = j, columns = c), 128 columns
constexpr uint32_t TM_SA = 192;   // bf16 S^T as the A operand of D1: c pairs, 64 columns
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
    griddep_launch_dependents();

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
    const int nchunks = (int)((s1 - s0 + CT - 1) / CT);  // 32-token steps of the segment
    // block slot of the segment's first step (segments hold an even number of 16-token chunks)
    const int64_t cbase = q0 / CT + n + (int64_t)k * (seg_c / 2);
    auto chunk_len = [&](int chunk) -> int { return (int)min((int64_t)CT, s1 - (s0 + (int64_t)chunk * CT)); };
    auto block_of = [&](int chunk) -> const unsigned char* {
        return a.blocks + ((cbase + chunk) * H + h) * (int64_t)tcc::BLK_BYTES;
    };

    if (w == 0) tc::tmem_alloc(tslot, TM_COLS);
    if (tid == 0) {
        for (int sl = 0; sl < NSLOT; ++sl) tc::mbar_init(&bar_f[sl], 1);
        tc::mbar_init(bar_c, 1);
        *abort_flag = 0u;
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tslot;
    griddep_wait();  // the operand blocks and incoming states come from the previous kernels

    // ring bookkeeping: every thread tracks each slot's fill parity; thread 0 also the loads it
    // issued and has not seen complete, and an unobserved tensor-core commit
    uint32_t phb = 0, pend = 0, ph_c = 0;
    bool pend_c = false;
    auto issue_load = [&](int chunk) {
        const int sl = chunk % NSLOT;
        tc::mbar_arrive_expect_tx(&bar_f[sl], tcc::BLK_BYTES);
        tc::bulk_load(sm + OFF_RING + sl * SLOT, block_of(chunk), tcc::BLK_BYTES, &bar_f[sl]);
        pend |= 1u << sl;
    };
    if (tid == 0) {
        for (int c = 0; c < NSLOT && c < nchunks; ++c) issue_load(c);
    }

    const int q4 = w & 3;    // TMEM lane quarter
    const int h2 = w >> 2;   // which half of the key channels (and of the chunk's tokens) this warp covers
    const int jrow = 32 * q4 + lane;
    const uint32_t lane_base = tbase + ((uint32_t)(32 * q4) << 16);
    const uint32_t my_s = lane_base + TM_S + 64 * h2;    // this thread's 64 state columns
    const uint32_t my_sa = lane_base + TM_SA + 32 * h2;  // ... and their 32 bf16-pair columns
    __nv_bfloat16* op = static_cast<__nv_bfloat16*>(a.out);

    // bf16 copy of this thread's 64 state values (16 of them per call) into the A operand
    auto stage16 = [&](int q, const uint32_t (&v)[16]) {
        uint32_t pk[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) pk[m] = tc::pack_bf16(u2f(v[2 * m]), u2f(v[2 * m + 1]));
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(my_sa + 8 * q),
                     "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]), "r"(pk[6]), "r"(pk[7])
                     : "memory");
    };

    // initial state S[c][jrow], c in [64 h2, 64 h2 + 64), into tensor memory: the bf16 copy as is, the
    // fp32 state already multiplied by the first chunk's Gamma_C (the decay the first update applies)
    bool init_ok = true;
    if (nchunks > 0) {
        init_ok = tc::mbar_wait(&bar_f[0], 0u, WAIT_LIMIT);
        if (init_ok) {
            phb ^= 1u;
            if (tid == 0) pend &= ~1u;
        } else {
            *abort_flag = 1u;
        }
    }
    {
        const float* gc0 = reinterpret_cast<const float*>(sm + OFF_RING + tcc::BLK_GC) + 64 * h2;
        const int64_t sbase = ((int64_t)n * H + h) * D * D;
        const int64_t segbase = (((int64_t)n * H + h) * a.max_seg + k) * D * D;
        const float* init = nullptr;
        if (mode == 0) init = (k == 0) ? (a.s0 ? a.s0 + sbase : nullptr) : a.seg_in + segbase;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int c = 64 * h2 + 16 * q + e;
                v[e] = __float_as_uint(init ? init[(int64_t)c * D + jrow] : ((mode == 2 && c == jrow) ? 1.f : 0.f));
            }
            stage16(q, v);
            if (nchunks > 0 && init_ok) {
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(u2f(v[e]) * gc0[16 * q + e]);
            }
            KDA_TMEM_ST16(my_s + 16 * q, v);
        }
        tc::tmem_wait_st();
    }
    tc::fence_before_sync();
    sync_all();
    tc::fence_after_sync();

    // outputs of the previous chunk, held in registers until the next chunk's D1 runs
    uint32_t ovp[8];  // bf16 pairs: tokens 16 h2 .. 16 h2 + 15
    int64_t o_t0 = 0;
    int o_len = 0;
    bool o_have = false;
    auto store_outputs = [&]() {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int r = 16 * h2 + e;
            const unsigned short bits = (unsigned short)((e & 1) ? (ovp[e >> 1] >> 16) : (ovp[e >> 1] & 0xffffu));
            if (r < o_len) op[((o_t0 + r) * H + h) * D + jrow] = __ushort_as_bfloat16(bits);
        }
        o_have = false;
    };

    for (int ch = 0; ch < nchunks; ++ch) {
        const int sl = ch % NSLOT;
        unsigned char* blk = sm + OFF_RING + sl * SLOT;
        bool dead = read_dead(abort_flag);

        // step ch's block has landed: every thread waited for it in the previous step's re-staging
        // (or before the initial state was written).  Thread 0 issues D1 (N = 64 with outputs, else
        // 32: W only) while the other warps store the previous step's outputs.
        const bool got = !dead;
        bool issued = false;
        if (tid == 0 && got) {
            const uint32_t idd = tc::idesc_bf16(128, mode == 0 ? 2 * CT : CT);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
                tc::umma_ts(tbase + TM_WU, tbase + TM_SA + 8 * ks,
                            tc::desc_sw128(tc::smem_u32(blk + tcc::BLK_WQ + kb * (2 * CT * 128) + off)), idd,
                            ks > 0 ? 1u : 0u);
            }
            tc::umma_commit(bar_c);
            issued = true;
        }
        if (o_have && w != 0) store_outputs();
        if (issued) {
            if (tc::mbar_wait(bar_c, ph_c, WAIT_LIMIT)) ph_c ^= 1u;
            else *abort_flag = 1u, pend_c = true;
        }
        if (o_have) store_outputs();  // warp 0, after its thread 0 has issued and waited
        tc::fence_before_sync();
        sync_all();
        tc::fence_after_sync();
        dead = read_dead(abort_flag);

        // U^T = U~^T - (W S)^T as a hi/lo pair into tensor memory; warp half h2 takes tokens
        // 16 h2 .. 16 h2 + 15 and overwrites exactly the (W S)^T columns it has read
        if (!dead) {
            uint32_t dv[16];
            KDA_TMEM_LD16(lane_base + TM_WU + 16 * h2, dv);
            float uv[16];
            const float* ut = reinterpret_cast<const float*>(blk + tcc::BLK_UT);
#pragma unroll
            for (int e = 0; e < 16; ++e) uv[e] = (mode == 2) ? 0.f : ut[(16 * h2 + e) * D + jrow];
            tc::tmem_wait_ld();
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                tcc::split2(uv[2 * e] - u2f(dv[2 * e]), uv[2 * e + 1] - u2f(dv[2 * e + 1]), hi[e], lo[e]);
            }
            KDA_TMEM_ST8(lane_base + TM_WU + 16 * h2, hi);
            KDA_TMEM_ST8(lane_base + TM_WU + 16 * h2 + 8, lo);
            tc::tmem_wait_st();
        }
        tc::fence_before_sync();
        sync_all();
        tc::fence_after_sync();

        // [O^T | S^T] += U^T [P ; (K Gamma_C / Gamma)^T]^T as hi*hi + hi*lo + lo*hi, one K = 16 half of
        // the step's tokens at a time (without outputs: S^T += U^T (K Gamma_C / Gamma) alone)
        if (tid == 0 && !dead) {
            const uint32_t dst = mode == 0 ? TM_O : TM_S;
            const uint32_t idd = tc::idesc_bf16(128, mode == 0 ? CT + D : D);
            const uint32_t boff = mode == 0 ? tcc::BLK_PK : tcc::BLK_KT;
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const uint64_t dB = tc::desc_none_strided(tc::smem_u32(blk + boff + 256 * ks), 128, tcc::PK_RG);
                const uint64_t dBl =
                    tc::desc_none_strided(tc::smem_u32(blk + boff + tcc::BLK_PK_LO + 256 * ks), 128, tcc::PK_RG);
                const uint32_t ahi = tbase + TM_WU + 16 * ks, alo = ahi + 8;
                tc::umma_ts(tbase + dst, ahi, dB, idd, 1u);
                tc::umma_ts(tbase + dst, ahi, dBl, idd, 1u);
                tc::umma_ts(tbase + dst, alo, dB, idd, 1u);
            }
            tc::umma_commit(bar_c);
            if (tc::mbar_wait(bar_c, ph_c, WAIT_LIMIT)) ph_c ^= 1u;
            else *abort_flag = 1u, pend_c = true;
        }
        sync_all();
        tc::fence_after_sync();
        dead = read_dead(abort_flag);

        // the new state's bf16 copy for the next D1, and the state multiplied by the next chunk's
        // Gamma_C (the decay its update applies; its block is in the ring already); outputs to registers
        if (!dead) {
            bool next_ok = false;
            if (ch + 1 < nchunks) {
                const int sn = (ch + 1) % NSLOT;
                next_ok = tc::mbar_wait(&bar_f[sn], (phb >> sn) & 1u, WAIT_LIMIT);
                if (next_ok) {
                    phb ^= 1u << sn;
                    if (tid == 0) pend &= ~(1u << sn);
                } else {
                    *abort_flag = 1u;
                }
            }
            uint32_t v[4][16], ob[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) KDA_TMEM_LD16(my_s + 16 * q, v[q]);
            if (mode == 0) KDA_TMEM_LD16(lane_base + TM_O + 16 * h2, ob);
            tc::tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 4; ++q) stage16(q, v[q]);
            if (next_ok) {
                const float* gcn = reinterpret_cast<const float*>(sm + OFF_RING + ((ch + 1) % NSLOT) * SLOT + tcc::BLK_GC) + 64 * h2;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) {
                        const float4 g4 = *reinterpret_cast<const float4*>(gcn + 16 * q + 4 * e4);
                        v[q][4 * e4 + 0] = __float_as_uint(u2f(v[q][4 * e4 + 0]) * g4.x);
                        v[q][4 * e4 + 1] = __float_as_uint(u2f(v[q][4 * e4 + 1]) * g4.y);
                        v[q][4 * e4 + 2] = __float_as_uint(u2f(v[q][4 * e4 + 2]) * g4.z);
                        v[q][4 * e4 + 3] = __float_as_uint(u2f(v[q][4 * e4 + 3]) * g4.w);
                    }
                    KDA_TMEM_ST16(my_s + 16 * q, v[q]);
                }
            }
            if (mode == 0) {
#pragma unroll
                for (int e = 0; e < 8; ++e) ovp[e] = tc::pack_bf16(u2f(ob[2 * e]), u2f(ob[2 * e + 1]));
                o_t0 = s0 + (int64_t)ch * CT;
                o_len = chunk_len(ch);
                o_have = true;
            }
            tc::tmem_wait_st();
        }
        tc::fence_before_sync();
        sync_all();  // every read of this slot is done; the next state is staged
        tc::fence_after_sync();
        if (tid == 0 && *abort_flag == 0u && ch + NSLOT < nchunks) issue_load(ch + NSLOT);
    }
    if (o_have) store_outputs();

    const int64_t sbase = ((int64_t)n * H + h) * D * D;
    const int64_t segbase = (((int64_t)n * H + h) * a.max_seg + k) * D * D;
    float* dst = nullptr;
    if (mode == 0) dst = ((int64_t)k == nseg - 1 && a.s_final) ? a.s_final + sbase : nullptr;
    else dst = (mode == 1 ? a.seg_st : a.seg_mt) + segbase;
    if (read_dead(abort_flag)) {
        if (tid == 0) {
            atomicOr(a.check, kCheckTimeout);
            // copies and tensor-core work still in flight must finish before the shared and tensor
            // memory are released
            for (int sl = 0; sl < NSLOT; ++sl) {
                if (pend & (1u << sl)) (void)tc::mbar_wait(&bar_f[sl], (phb >> sl) & 1u, WAIT_LIMIT);
            }
            if (pend_c) (void)tc::mbar_wait(bar_c, ph_c, WAIT_LIMIT);
        }
    } else if (dst) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t v[16];
            KDA_TMEM_LD16(my_s + 16 * q, v);
            tc::tmem_wait_ld();
            if (mode == 2) {
                // the transition M[c][j] (this lane holds column j = jrow) in the scan's operand format
#pragma unroll
                for (int e = 0; e < 16; ++e) store_seg_m(dst, 64 * h2 + 16 * q + e, jrow, u2f(v[e]));
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) dst[(int64_t)(64 * h2 + 16 * q + e) * D + jrow] = u2f(v[e]);
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (w == 0) tc::tmem_dealloc(tbase, TM_COLS);
}

namespace {

// Shared memory requested by a grid that fits on the SMs one CTA each: more than half of an SM's,
// so that two chains never share an SM.  (A CTA launched early, next to the previous kernel's
// CTAs, is placed wherever there is room; without this it could land on an SM that already holds
// a chain and run at the shared speed.)
constexpr uint32_t SMEM_EXCLUSIVE = 120 * 1024;
static_assert(SMEM_EXCLUSIVE >= SMEM_BYTES && 2 * (SMEM_EXCLUSIVE + 1024) > 233472, "one CTA per SM");

cudaError_t launch_chunk_state_tc(const PrefillArgs& a, int seg_mode, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(kda_chunk_state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_EXCLUSIVE);
    if (e != cudaSuccess) return e;
    PrefillArgs b = a;
    b.seg_mode = seg_mode;
    const unsigned gz = seg_mode == 0 ? (unsigned)(a.max_seg > 1 ? a.max_seg : 1) : (unsigned)(2 * (a.max_seg - 1));
    if (gz == 0) return cudaSuccess;
    const int64_t ctas = (int64_t)a.N * a.H * gz;
    const uint32_t smem = ctas <= (int64_t)sm_count_of_current_device() ? SMEM_EXCLUSIVE : SMEM_BYTES;
    return launch_dependent(kda_chunk_state_tc_kernel, dim3((unsigned)a.N, (unsigned)a.H, gz), dim3(NTHREADS), smem, s, b);
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
