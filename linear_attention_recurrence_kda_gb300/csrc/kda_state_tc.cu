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
//   bf16(S)^T, then S^T Diag(Gamma_C of the next step)   (one read of the new state writes the
//                                        next D1's A operand and the next update's decayed state)
// A tcgen05.mma takes about as long to issue whatever its N, so a step is organised around few
// instructions: 8 for D1 and 6 for the fused update, for 32 tokens.
//
// Warp roles.  Warps 0..7 (the epilogue) own the tensor-memory lanes: warp w reads and writes lanes
// 32 (w mod 4) .. + 31 and half of the key channels.  Warp 8 (the control warp, one thread) issues
// every tensor-core instruction and every block copy.  The two sides meet only at mbarriers, one
// phase per step each:
//   sa   (epilogue -> control)  bf16(S) of the previous step is staged: D1 may start
//   d1   (tensor core -> epilogue)  D1 is complete: U epilogue
//   u    (epilogue -> control)  U is in tensor memory: the fused update may start
//   fu   (tensor core -> both)  the fused update is complete: re-stage the state; refill the slot
// so the decay of the state for the next step (during D1), the output stores (during the update) and
// the block copies run while the tensor core works on the chain, and the chain itself is staging -> D1 -> U epilogue
// -> update.  Operand blocks stream through a two-slot shared-memory ring by plain bulk copies.
// 288 threads, ~107 KB of shared memory and 256 TMEM columns per CTA: two CTAs (two independent
// chains) share an SM.
//
// Modes (segmented prefill, see the launcher): 0 writes outputs and (last segment) the final state;
// 1 computes S~, the segment's end state from a zero start; 2 computes M, the segment's transition,
// as the end state from the identity with V = 0 (columns of M evolve exactly like state columns),
// stored as the scan's bf16 hi/lo operand (seg_m_off).  Every mbarrier wait is bounded; a wait
// that gives up raises the abort flag and the timeout bit of the check word, every thread leaves
// its loop at its next wait, the control thread waits (bounded) for its copies and products in
// flight, and the CTA frees its tensor memory.
#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_tc_chunk.cuh"

namespace kda {

namespace {

using tcc::C;
using tcc::D;
using tcc::u2f;

constexpr int NEPI = 256;                  // epilogue threads (warps 0..7)
constexpr int NTHREADS = NEPI + 32;        // + the control warp
constexpr int CTRL = NEPI;                 // the control thread (warp 8, lane 0)
constexpr uint32_t WAIT_LIMIT = kWaitTries;  // drain waits: tries of up to 20 us each, ~2.6 s at most
constexpr int CT = tcc::PAIR;              // tokens per step (32)
constexpr int NSLOT = 2;                   // ring depth (steps in flight)
constexpr uint32_t SLOT = 54272;           // ring slot stride (a multiple of 1024 >= BLK_BYTES)

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_RING = 0;                         // [NSLOT] operand blocks
constexpr uint32_t OFF_BARF = NSLOT * SLOT;              // mbarriers: ring slot filled [NSLOT]
constexpr uint32_t OFF_BAR_SA = OFF_BARF + 8 * NSLOT;    // ... bf16 state staged (NEPI arrivals)
constexpr uint32_t OFF_BAR_D1 = OFF_BAR_SA + 8;          // ... D1 complete (tensor-core commit)
constexpr uint32_t OFF_BAR_U = OFF_BAR_D1 + 8;           // ... U written (NEPI arrivals)
constexpr uint32_t OFF_BAR_FU = OFF_BAR_U + 8;           // ... fused update complete (commit)
constexpr uint32_t OFF_BAR_T = OFF_BAR_FU + 8;           // ... teardown commit
constexpr uint32_t OFF_TSLOT = OFF_BAR_T + 8;            // TMEM base address
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

// Bounded hand-off wait (`tries` tries) that gives up at once when the CTA has been told to stop;
// on a timeout it raises the stop flag itself.  Returns true when the phase completed.  Giving up
// here is always safe: whoever stops touches no ring slot or tensor memory afterwards, and the
// control thread drains its copies and tensor-core work (with the full WAIT_LIMIT) before the CTA
// releases its shared and tensor memory.
__device__ __forceinline__ bool wait_or_stop(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                             uint32_t tries)
{
    if (*abort_flag != 0u) return false;
    if (tc::mbar_wait(bar, parity, tries)) return true;
    *abort_flag = 1u;
    return false;
}

}  // namespace

// The kernel body, compiled twice (see the kernels below).  SHARED: two CTAs share an SM, so the
// re-staging keeps fewer values live.
template <bool SHARED>
__device__ __forceinline__ void state_pass(const PrefillArgs& a)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bar_f = reinterpret_cast<uint64_t*>(sm + OFF_BARF);
    uint64_t* bar_sa = reinterpret_cast<uint64_t*>(sm + OFF_BAR_SA);
    uint64_t* bar_d1 = reinterpret_cast<uint64_t*>(sm + OFF_BAR_D1);
    uint64_t* bar_u = reinterpret_cast<uint64_t*>(sm + OFF_BAR_U);
    uint64_t* bar_fu = reinterpret_cast<uint64_t*>(sm + OFF_BAR_FU);
    uint64_t* bar_t = reinterpret_cast<uint64_t*>(sm + OFF_BAR_T);
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
    const int nsteps = (int)((s1 - s0 + CT - 1) / CT);  // 32-token steps of the segment
    // block slot of the segment's first step (segments hold an even number of 16-token chunks)
    const int64_t cbase = q0 / CT + n + (int64_t)k * (seg_c / 2);
    auto step_len = [&](int s) -> int { return (int)min((int64_t)CT, s1 - (s0 + (int64_t)s * CT)); };
    auto block_of = [&](int s) -> const unsigned char* {
        return a.blocks + ((cbase + s) * H + h) * (int64_t)tcc::BLK_BYTES;
    };
    // block s sits in slot s mod 2; it is that slot's fill number s / 2
    auto slot_ptr = [&](int s) -> unsigned char* { return sm + OFF_RING + (s % NSLOT) * SLOT; };
    auto fill_parity = [&](int s) -> uint32_t { return (uint32_t)((s / NSLOT) & 1); };

    if (w == 0) tc::tmem_alloc(tslot, TM_COLS);
    if (tid == 0) {
        for (int sl = 0; sl < NSLOT; ++sl) tc::mbar_init(&bar_f[sl], 1);
        tc::mbar_init(bar_sa, NEPI);
        tc::mbar_init(bar_d1, 1);
        tc::mbar_init(bar_u, NEPI);
        tc::mbar_init(bar_fu, 1);
        tc::mbar_init(bar_t, 1);
        *abort_flag = 0u;
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tslot;
    griddep_wait();  // the operand blocks and incoming states come from the previous kernels

    if (tid == CTRL) {
        // ------------------------------------------------------------------ control thread
        uint32_t issued = 0, seen = 0;  // blocks whose copies were issued / observed complete
        auto issue_load = [&](int s) {
            tc::mbar_arrive_expect_tx(&bar_f[s % NSLOT], tcc::BLK_BYTES);
            tc::bulk_load(slot_ptr(s), block_of(s), tcc::BLK_BYTES, &bar_f[s % NSLOT]);
            ++issued;
        };
        for (int s = 0; s < NSLOT && s < nsteps; ++s) issue_load(s);
        bool committed = false;  // tensor-core work issued whose completion this thread did not observe
        const uint32_t idd1 = tc::idesc_bf16(128, mode == 0 ? 2 * CT : CT);
        const uint32_t iddf = tc::idesc_bf16(128, mode == 0 ? CT + D : D);
        const uint32_t dstf = tbase + (mode == 0 ? TM_O : TM_S);
        const uint32_t boff = mode == 0 ? tcc::BLK_PK : tcc::BLK_KT;
        for (int s = 0; s < nsteps; ++s) {
            unsigned char* blk = slot_ptr(s);
            if (!wait_or_stop(&bar_f[s % NSLOT], fill_parity(s), abort_flag, a.handoff_tries)) break;
            seen = (uint32_t)s + 1;
            if (!wait_or_stop(bar_sa, (uint32_t)(s & 1), abort_flag, a.handoff_tries)) break;
            tc::fence_after_sync();
            const uint64_t d0 = tc::desc_sw128(tc::smem_u32(blk + tcc::BLK_WQ));
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
                tc::umma_ts(tbase + TM_WU, tbase + TM_SA + 8 * ks, d0 + ((kb * (2 * CT * 128) + off) >> 4), idd1,
                            ks > 0 ? 1u : 0u);
            }
            tc::umma_commit(bar_d1);
            committed = true;
            if (!wait_or_stop(bar_u, (uint32_t)(s & 1), abort_flag, a.handoff_tries)) break;
            tc::fence_after_sync();
            // [O^T | S^T] += U^T [P ; K~^T]^T as hi*hi + hi*lo + lo*hi, one K = 16 half of the step's
            // tokens at a time (without outputs: S^T += U^T K~ alone)
            const uint64_t dB0 = tc::desc_none_strided(tc::smem_u32(blk + boff), 128, tcc::PK_RG);
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const uint64_t dB = dB0 + ((256 * ks) >> 4);
                const uint64_t dBl = dB0 + ((tcc::BLK_PK_LO + 256 * ks) >> 4);
                const uint32_t ahi = tbase + TM_WU + 16 * ks, alo = ahi + 8;
                tc::umma_ts(dstf, ahi, dB, iddf, 1u);
                tc::umma_ts(dstf, ahi, dBl, iddf, 1u);
                tc::umma_ts(dstf, alo, dB, iddf, 1u);
            }
            tc::umma_commit(bar_fu);
            // the update is the last reader of this slot: refill it once the update is done
            if (s + NSLOT < nsteps) {
                if (!wait_or_stop(bar_fu, (uint32_t)(s & 1), abort_flag, a.handoff_tries)) break;
                committed = false;
                issue_load(s + NSLOT);
            }
        }
        // tensor-core work and copies still in flight must finish before the shared and tensor memory
        // are released
        if (committed) {
            tc::umma_commit(bar_t);
            (void)tc::mbar_wait(bar_t, 0u, WAIT_LIMIT);
        }
        if (*abort_flag != 0u) {
            atomicOr(a.check, kCheckTimeout);
            for (uint32_t s = seen; s < issued; ++s) (void)tc::mbar_wait(&bar_f[s % NSLOT], fill_parity((int)s), WAIT_LIMIT);
        }
    } else if (tid < NEPI) {
        // ------------------------------------------------------------------ epilogue warps
        // every wait is decided for the whole warp, so that the warp-collective tensor-memory
        // instructions below always run on all 32 lanes
        auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, wait_or_stop(bar, parity, abort_flag, a.handoff_tries));
        };
        const int q4 = w & 3;    // TMEM lane quarter
        const int h2 = w >> 2;   // which half of the key channels (and of the step's tokens) this warp covers
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

        // initial state S[c][jrow], c in [64 h2, 64 h2 + 64), into tensor memory: the bf16 copy as is,
        // the fp32 state already multiplied by the first step's Gamma_C (the decay its update applies)
        const bool have0 = nsteps > 0 && wait_warp(&bar_f[0], 0u);
        {
            const float* gc0 = reinterpret_cast<const float*>(sm + OFF_RING + tcc::BLK_GC) + 64 * h2;
            const int64_t sbase = ((int64_t)n * H + h) * D * D;
            const int64_t segbase = (((int64_t)n * H + h) * a.max_seg + k) * D * D;
            const float* init = nullptr;
            // with several segments every segment, the first included, starts from the scan's copy: the
            // final state may overwrite the caller's initial state (in-place carry) while the first
            // segment's CTA has not read it yet
            if (mode == 0) init = (nseg == 1) ? (a.s0 ? a.s0 + sbase : nullptr) : a.seg_in + segbase;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t v[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int c = 64 * h2 + 16 * q + e;
                    v[e] = __float_as_uint(init ? init[(int64_t)c * D + jrow] : ((mode == 2 && c == jrow) ? 1.f : 0.f));
                }
                stage16(q, v);
                if (have0) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(u2f(v[e]) * gc0[16 * q + e]);
                }
                KDA_TMEM_ST16(my_s + 16 * q, v);
            }
            tc::tmem_wait_st();
        }
        tc::fence_before_sync();
        tc::mbar_arrive(bar_sa);  // phase 0: the first D1 may start

        // outputs of the previous step, held in registers until the next step's D1 runs
        uint32_t ovp[8];  // bf16 pairs: tokens 16 h2 .. 16 h2 + 15
        int64_t o_t0 = 0;
        int o_len = 0;
        bool o_have = false;
        const int64_t o_stride = (int64_t)H * D;  // between consecutive tokens of one head
        auto store_outputs = [&]() {
            __nv_bfloat16* base = op + ((o_t0 + 16 * h2) * H + h) * D + jrow;
            const int n_valid = o_len - 16 * h2;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const unsigned short bits = (unsigned short)((e & 1) ? (ovp[e >> 1] >> 16) : (ovp[e >> 1] & 0xffffu));
                if (e < n_valid) base[e * o_stride] = __ushort_as_bfloat16(bits);
            }
            o_have = false;
        };

        for (int s = 0; s < nsteps; ++s) {
            const unsigned char* blk = slot_ptr(s);
            // this block's U~ (in the ring since D1 was issued) into registers while D1 runs
            if (!wait_warp(&bar_f[s % NSLOT], fill_parity(s))) break;
            float uv[16];
            {
                const float* ut = reinterpret_cast<const float*>(blk + tcc::BLK_UT);
#pragma unroll
                for (int e = 0; e < 16; ++e) uv[e] = (mode == 2) ? 0.f : ut[(16 * h2 + e) * D + jrow];
            }
            if (!wait_warp(bar_d1, (uint32_t)(s & 1))) break;
            tc::fence_after_sync();

            // U^T = U~^T - (W S)^T as a hi/lo pair into tensor memory; warp half h2 takes tokens
            // 16 h2 .. 16 h2 + 15 and overwrites exactly the (W S)^T columns it has read
            {
                uint32_t dv[16];
                KDA_TMEM_LD16(lane_base + TM_WU + 16 * h2, dv);
                tc::tmem_wait_ld();
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    tcc::split2(uv[2 * e] - u2f(dv[2 * e]), uv[2 * e + 1] - u2f(dv[2 * e + 1]), hi[e], lo[e]);
                KDA_TMEM_ST8(lane_base + TM_WU + 16 * h2, hi);
                KDA_TMEM_ST8(lane_base + TM_WU + 16 * h2 + 8, lo);
                tc::tmem_wait_st();  // also the decayed-state stores of the previous step
            }
            tc::fence_before_sync();
            tc::mbar_arrive(bar_u);  // the fused update may start
            if (o_have) store_outputs();  // the previous step's outputs, while the update runs

            if (!wait_warp(bar_fu, (uint32_t)(s & 1))) break;
            tc::fence_after_sync();

            // the new state's bf16 copy for the next D1 first (32 values at a time), then -- while that D1
            // runs -- the state multiplied by the next step's Gamma_C (the decay its update applies),
            // read again 16 columns at a time; outputs to registers
            {
                constexpr int NR = SHARED ? 2 : 4;  // 16-column groups per tensor-memory round trip
#pragma unroll
                for (int hq = 0; hq < 4 / NR; ++hq) {
                    uint32_t v[NR][16];
#pragma unroll
                    for (int qq = 0; qq < NR; ++qq) KDA_TMEM_LD16(my_s + 16 * (NR * hq + qq), v[qq]);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int qq = 0; qq < NR; ++qq) stage16(NR * hq + qq, v[qq]);
                }
            }
            if (mode == 0) {
                uint32_t ob[16];
                KDA_TMEM_LD16(lane_base + TM_O + 16 * h2, ob);
                tc::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 8; ++e) ovp[e] = tc::pack_bf16(u2f(ob[2 * e]), u2f(ob[2 * e + 1]));
                o_t0 = s0 + (int64_t)s * CT;
                o_len = step_len(s);
                o_have = true;
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            tc::mbar_arrive(bar_sa);  // phase s + 1: the next D1 may start
            if (s + 1 < nsteps) {
                if (!wait_warp(&bar_f[(s + 1) % NSLOT], fill_parity(s + 1))) break;
                const float* gcn = reinterpret_cast<const float*>(slot_ptr(s + 1) + tcc::BLK_GC) + 64 * h2;
                constexpr int NQ = SHARED ? 1 : 2;  // 16-column groups per tensor-memory round trip
#pragma unroll
                for (int hq = 0; hq < 4 / NQ; ++hq) {
                    uint32_t v[NQ][16];
#pragma unroll
                    for (int qq = 0; qq < NQ; ++qq) KDA_TMEM_LD16(my_s + 16 * (NQ * hq + qq), v[qq]);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int qq = 0; qq < NQ; ++qq) {
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) {
                            const float4 g4 = *reinterpret_cast<const float4*>(gcn + 16 * (NQ * hq + qq) + 4 * e4);
                            v[qq][4 * e4 + 0] = __float_as_uint(u2f(v[qq][4 * e4 + 0]) * g4.x);
                            v[qq][4 * e4 + 1] = __float_as_uint(u2f(v[qq][4 * e4 + 1]) * g4.y);
                            v[qq][4 * e4 + 2] = __float_as_uint(u2f(v[qq][4 * e4 + 2]) * g4.z);
                            v[qq][4 * e4 + 3] = __float_as_uint(u2f(v[qq][4 * e4 + 3]) * g4.w);
                        }
                        KDA_TMEM_ST16(my_s + 16 * (NQ * hq + qq), v[qq]);
                    }
                }
            }
        }
        tc::tmem_wait_st();
        if (o_have) store_outputs();

        const int64_t sbase = ((int64_t)n * H + h) * D * D;
        const int64_t segbase = (((int64_t)n * H + h) * a.max_seg + k) * D * D;
        float* dst = nullptr;
        if (mode == 0) dst = ((int64_t)k == nseg - 1 && a.s_final) ? a.s_final + sbase : nullptr;
        else dst = (mode == 1 ? a.seg_st : a.seg_mt) + segbase;
        if (__any_sync(0xffffffffu, *abort_flag != 0u)) {
            if (tid == 0) atomicOr(a.check, kCheckTimeout);
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
    }
    if (w == NEPI / 32) __syncwarp();  // the control warp reconverges before the CTA barrier
    tc::fence_before_sync();
    __syncthreads();
    if (w == 0) tc::tmem_dealloc(tbase, TM_COLS);
}

// Register budgets.  Registers come from each SM sub-partition's quarter of the file (16,384): two
// CTAs of 9 warps place 5 warps on some sub-partition, so 5 x 32 x 96 <= 16,384 allows 96 per
// thread; one CTA per SM places 3, which allows 168.
__global__ void __maxnreg__(96) kda_chunk_state_tc_kernel(PrefillArgs a) { state_pass<true>(a); }
__global__ void __maxnreg__(168) kda_chunk_state_tc_excl_kernel(PrefillArgs a) { state_pass<false>(a); }

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
    const dim3 grid((unsigned)a.N, (unsigned)a.H, gz);
    if (ctas <= (int64_t)sm_count_of_current_device()) {
        e = cudaFuncSetAttribute(kda_chunk_state_tc_excl_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SMEM_EXCLUSIVE);
        if (e != cudaSuccess) return e;
        return launch_dependent(kda_chunk_state_tc_excl_kernel, grid, dim3(NTHREADS), SMEM_EXCLUSIVE, s, b);
    }
    return launch_dependent(kda_chunk_state_tc_kernel, grid, dim3(NTHREADS), SMEM_BYTES, s, b);
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
