// kda_replay.cu -- a window of decode tokens per sequence from a state snapshot (speculative-decode
// state replay).
//
// "Kimi K3: architecture, derivations and a pinned-source audit", section 10.3 "KDA state replay for
// speculative decoding": a speculating server keeps just the per-token inputs of its drafts (far
// less memory than a copy of the state), checks the drafted window against a saved state, and then
// moves that state forward over the drafts that survived, on chip and in one launch; a draft that
// was rejected is therefore never applied and never has to be undone.  The arithmetic
// of every token is the decode step's (Equation 1 with the gate of Equation 5, o = S'^T q = y + (q.k) u):
//     alpha = exp(g_min sigmoid(exp(A_h) z)),  r = (Diag(alpha) S)^T k,  y = (Diag(alpha) S)^T q,
//     u = beta (v - r),  S' = Diag(alpha) S + k u^T.
//
// One CTA of 256 threads owns one (sequence, head) for the whole window.  The fp32 state is read
// from HBM once into registers (warp w holds rows w, w + 8, ...; lane l holds columns
// l*VEC .. l*VEC + VEC - 1 of each, so a warp reads whole rows with vector loads), advances token
// by token on chip and is written at most once, right after the last accepted token.  Token inputs
// are staged in shared memory eight tokens at a time (the gate is evaluated there).  Per token the
// eight warps' partial sums of r (and of y when outputs are wanted) meet in shared memory behind one
// barrier; every thread then adds the eight partials of its own columns itself, so u needs no second
// barrier to reach the threads that apply it.  The partial-sum buffer alternates between consecutive
// tokens: a buffer is written again two tokens later, after a barrier that every reader of its
// previous contents has passed.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kRepThreads = 256;
constexpr int kRepWarps = kRepThreads / 32;
constexpr int kRepGroup = 8;  // tokens staged in shared memory at a time

template <int VEC>
__device__ __forceinline__ void ld_cols(const float* p, float (&x)[VEC])
{
    if constexpr (VEC == 4) {
        const float4 t = __ldcs(reinterpret_cast<const float4*>(p));
        x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
    } else if constexpr (VEC == 2) {
        const float2 t = __ldcs(reinterpret_cast<const float2*>(p));
        x[0] = t.x; x[1] = t.y;
    } else {
        x[0] = __ldcs(p);
    }
}

template <int VEC>
__device__ __forceinline__ void st_cols(float* p, const float (&x)[VEC])
{
    if constexpr (VEC == 4) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(x[0], x[1], x[2], x[3]));
    } else if constexpr (VEC == 2) {
        __stcs(reinterpret_cast<float2*>(p), make_float2(x[0], x[1]));
    } else {
        __stcs(p, x[0]);
    }
}

}  // namespace

template <typename TIO, int DK, int DV, bool OUT>
__global__ void __launch_bounds__(kRepThreads, 2) kda_decode_replay_kernel(ReplayArgs a)
{
    constexpr int VEC = DV / 32;
    constexpr int RPW = DK / kRepWarps;  // rows per warp
    __shared__ __align__(16) float s_k[kRepGroup][DK];
    __shared__ __align__(16) float s_q[kRepGroup][DK];
    __shared__ __align__(16) float s_al[kRepGroup][DK];
    __shared__ __align__(16) float s_v[kRepGroup][DV];
    __shared__ float s_beta[kRepGroup];
    __shared__ float s_qk[kRepGroup];
    __shared__ __align__(16) float s_red[2][OUT ? 2 : 1][kRepWarps][DV];

    const int nh = blockIdx.x;  // sequence * H + head
    const int n = nh / a.H;
    const int h = nh - n * a.H;
    const int tid = threadIdx.x;
    const int w = tid >> 5;
    const int l = tid & 31;
    const int L = a.L;

    // the whole state in flight first
    float s[RPW][VEC];
    {
        const float* S = a.state_in + (int64_t)nh * DK * DV;
#pragma unroll
        for (int i = 0; i < RPW; ++i) ld_cols<VEC>(S + (int64_t)(w + kRepWarps * i) * DV + l * VEC, s[i]);
    }

    int acc = L;
    if (a.accepted != nullptr) acc = min(max(a.accepted[n], 0), L);
    float* Sout = a.state_out != nullptr ? a.state_out + (int64_t)nh * DK * DV : nullptr;
    auto store_state = [&]() {
#pragma unroll
        for (int i = 0; i < RPW; ++i) st_cols<VEC>(Sout + (int64_t)(w + kRepWarps * i) * DV + l * VEC, s[i]);
    };
    if (Sout != nullptr && acc == 0) store_state();

    const int steps = OUT ? L : acc;  // without outputs nothing after the accepted prefix matters
    const TIO* qp = static_cast<const TIO*>(a.q);
    const TIO* kp = static_cast<const TIO*>(a.k);
    const TIO* vp = static_cast<const TIO*>(a.v);
    const TIO* zp = static_cast<const TIO*>(a.z);
    TIO* op = static_cast<TIO*>(a.out);
    const float expA = expf(a.A[h]);
    const int64_t tok0 = (int64_t)n * L;  // first row of this sequence's window

    for (int g0 = 0; g0 < steps; g0 += kRepGroup) {
        const int ng = min(kRepGroup, steps - g0);
        __syncthreads();  // the previous group's staged tokens are no longer read
        for (int e = tid; e < ng * DK; e += kRepThreads) {
            const int j = e / DK;
            const int c = e - j * DK;
            const int64_t idx = ((tok0 + g0 + j) * a.H + h) * DK + c;
            s_k[j][c] = ld_io(kp, idx);
            s_q[j][c] = ld_io(qp, idx);
            s_al[j][c] = expf(log_decay(ld_io(zp, idx), expA, a.g_min));
        }
        for (int e = tid; e < ng * DV; e += kRepThreads) {
            const int j = e / DV;
            const int c = e - j * DV;
            s_v[j][c] = ld_io(vp, ((tok0 + g0 + j) * a.H + h) * DV + c);
        }
        if (tid < ng) s_beta[tid] = a.beta[(tok0 + g0 + tid) * a.H + h];
        __syncthreads();
        if (OUT && w < ng) {  // q.k of token w of the group (read after the first token's barrier)
            float p = 0.f;
            for (int c = l; c < DK; c += 32) p += s_q[w][c] * s_k[w][c];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
            if (l == 0) s_qk[w] = p;
        }

        for (int j = 0; j < ng; ++j) {
            const int t = g0 + j;
            const int buf = t & 1;
            // decay the rows this thread holds and reduce r (and y) over them
            float r[VEC], y[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) r[e] = y[e] = 0.f;
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const int c = w + kRepWarps * i;
                const float al = s_al[j][c], kc = s_k[j][c];
                const float qc = OUT ? s_q[j][c] : 0.f;
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float d = al * s[i][e];
                    s[i][e] = d;
                    r[e] += kc * d;
                    if (OUT) y[e] += qc * d;
                }
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                s_red[buf][0][w][l * VEC + e] = r[e];
                if (OUT) s_red[buf][OUT ? 1 : 0][w][l * VEC + e] = y[e];
            }
            __syncthreads();
            // every thread: u for its own columns from the eight warps' partial sums
            float u[VEC];
            const float b = s_beta[j];
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                float rr = 0.f;
#pragma unroll
                for (int ww = 0; ww < kRepWarps; ++ww) rr += s_red[buf][0][ww][l * VEC + e];
                u[e] = b * (s_v[j][l * VEC + e] - rr);
            }
            if (OUT && w == 0) {
                const float qk = s_qk[j];
                const int64_t orow = ((tok0 + t) * a.H + h) * DV + l * VEC;
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    float yy = 0.f;
#pragma unroll
                    for (int ww = 0; ww < kRepWarps; ++ww) yy += s_red[buf][OUT ? 1 : 0][ww][l * VEC + e];
                    st_io(op, orow + e, yy + qk * u[e]);
                }
            }
            // S' = Diag(alpha) S + k u^T (the decay is already applied)
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const float kc = s_k[j][w + kRepWarps * i];
#pragma unroll
                for (int e = 0; e < VEC; ++e) s[i][e] += kc * u[e];
            }
            if (Sout != nullptr && t + 1 == acc) store_state();
        }
    }
}

// ---------------------------------------------------------------- d_k = d_v = 128, bf16, L <= 8
//
// The production shape gets a persistent form of the same step: two CTAs per SM walk the
// (sequence, head) units with the grid as stride, and while one unit's state advances in registers
// the state (64 KB) and drafted tokens of the CTA's next unit already arrive in shared memory by
// 16-byte asynchronous copies, so that HBM keeps streaming through the arithmetic of every window.
// Per unit: wait for the copies, move the state into registers and the tokens into fp32 staging
// (gate evaluated there; alpha, k and q of a key channel side by side, so a row takes one 16-byte
// shared load), then start the next unit's copies and run the window.  Column pairs are updated
// with packed fp32 instructions, in the same order of operations as the kernel above.
constexpr int kRepD = 128;

struct RepLayout {
    static constexpr int kRawRow = kRepD * 2;                         // one bf16 token row of q, k, z or v
    static constexpr int kStage = 0;                                  // fp32 [128][128], next unit's state
    static constexpr int kRaw = kStage + kRepD * kRepD * 4;           // bf16 [token][q, k, z, v][128]
    static constexpr int kRawBeta = kRaw + kRepGroup * 4 * kRawRow;   // fp32 [token]
    static constexpr int kAkq = kRawBeta + kRepGroup * 4;             // float4 [token][row]: alpha, k, q, 0
    static constexpr int kV = kAkq + kRepGroup * kRepD * 16;          // fp32 [token][128]
    static constexpr int kRed = kV + kRepGroup * kRepD * 4;           // fp32 [2][r, y][warp][128]
    static constexpr int kBeta = kRed + 2 * 2 * kRepWarps * kRepD * 4;
    static constexpr int kQk = kBeta + kRepGroup * 4;
    static constexpr int kBytes = kQk + kRepGroup * 4;
};
static_assert(RepLayout::kAkq % 16 == 0 && RepLayout::kV % 16 == 0 && RepLayout::kRed % 16 == 0, "16-byte alignment");
static_assert(2 * (RepLayout::kBytes + 1024) <= 228 * 1024, "two CTAs per SM");

__device__ __forceinline__ void cp_async16(void* dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}

template <bool OUT>
__global__ void __launch_bounds__(kRepThreads, 2) kda_decode_replay_d128_kernel(ReplayArgs a)
{
    constexpr int D = kRepD;
    constexpr int RPW = D / kRepWarps;  // 16 rows per warp
    using TIO = __nv_bfloat16;
    extern __shared__ __align__(16) unsigned char smem[];
    float* stage = reinterpret_cast<float*>(smem + RepLayout::kStage);
    unsigned char* raw = smem + RepLayout::kRaw;
    float* raw_beta = reinterpret_cast<float*>(smem + RepLayout::kRawBeta);
    float4* s_akq = reinterpret_cast<float4*>(smem + RepLayout::kAkq);
    float* s_v = reinterpret_cast<float*>(smem + RepLayout::kV);
    float* s_red = reinterpret_cast<float*>(smem + RepLayout::kRed);
    float* s_beta = reinterpret_cast<float*>(smem + RepLayout::kBeta);
    float* s_qk = reinterpret_cast<float*>(smem + RepLayout::kQk);

    const int tid = threadIdx.x;
    const int w = tid >> 5;
    const int l = tid & 31;
    const int L = a.L;
    const int units = a.N * a.H;
    const TIO* qp = static_cast<const TIO*>(a.q);
    const TIO* kp = static_cast<const TIO*>(a.k);
    const TIO* vp = static_cast<const TIO*>(a.v);
    const TIO* zp = static_cast<const TIO*>(a.z);
    TIO* op = static_cast<TIO*>(a.out);

    auto acc_of = [&](int unit) {
        return a.accepted != nullptr ? min(max(a.accepted[unit / a.H], 0), L) : L;
    };
    // asynchronous copies of a unit's state and of the `steps` drafted tokens it will use
    auto prefetch = [&](int unit, int steps) {
        const int n = unit / a.H;
        const int h = unit - n * a.H;
        const float* S = a.state_in + (int64_t)unit * D * D;
#pragma unroll
        for (int i = 0; i < D * D / 4 / kRepThreads; ++i) {
            const int e4 = tid + kRepThreads * i;
            cp_async16(stage + 4 * e4, S + 4 * e4);
        }
        constexpr int CH = RepLayout::kRawRow / 16;  // 16-byte pieces per token row
        const int64_t tok0 = (int64_t)n * L;
        for (int e = tid; e < steps * 4 * CH; e += kRepThreads) {
            const int j = e / (4 * CH);
            const int rem = e - j * 4 * CH;
            const int which = rem / CH;
            const int ch = rem - which * CH;
            const TIO* base = which == 0 ? qp : which == 1 ? kp : which == 2 ? zp : vp;
            cp_async16(raw + (size_t)e * 16, base + ((tok0 + j) * a.H + h) * D + ch * 8);
        }
        if (tid < steps) cp_async4(raw_beta + tid, a.beta + (tok0 + tid) * a.H + h);
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    int unit = blockIdx.x;
    if (unit >= units) return;
    int acc = acc_of(unit);
    prefetch(unit, OUT ? L : acc);
    for (; unit < units; unit += gridDim.x) {
        const int next = unit + gridDim.x;
        const int acc_next = next < units ? acc_of(next) : 0;
        const int steps = OUT ? L : acc;
        const int n = unit / a.H;
        const int h = unit - n * a.H;
        const float expA = expf(a.A[h]);
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();  // this unit's state and tokens are in shared memory

        for (int e = tid; e < steps * D; e += kRepThreads) {
            const int j = e / D;
            const int c = e - j * D;
            const TIO* rq = reinterpret_cast<const TIO*>(raw + (j * 4 + 0) * RepLayout::kRawRow);
            const TIO* rk = reinterpret_cast<const TIO*>(raw + (j * 4 + 1) * RepLayout::kRawRow);
            const TIO* rz = reinterpret_cast<const TIO*>(raw + (j * 4 + 2) * RepLayout::kRawRow);
            const TIO* rv = reinterpret_cast<const TIO*>(raw + (j * 4 + 3) * RepLayout::kRawRow);
            s_akq[e] = make_float4(expf(log_decay(__bfloat162float(rz[c]), expA, a.g_min)), __bfloat162float(rk[c]),
                                   __bfloat162float(rq[c]), 0.f);
            s_v[e] = __bfloat162float(rv[c]);
        }
        if (tid < steps) s_beta[tid] = raw_beta[tid];
        if (OUT && w < steps) {  // q.k of token w
            const TIO* rq = reinterpret_cast<const TIO*>(raw + (w * 4 + 0) * RepLayout::kRawRow);
            const TIO* rk = reinterpret_cast<const TIO*>(raw + (w * 4 + 1) * RepLayout::kRawRow);
            float p = 0.f;
#pragma unroll
            for (int c = l; c < D; c += 32) p += __bfloat162float(rq[c]) * __bfloat162float(rk[c]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
            if (l == 0) s_qk[w] = p;
        }
        float2 s[RPW][2];  // rows w + 8 i, columns 4 l .. 4 l + 3 as two pairs
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            const float4 t4 = *reinterpret_cast<const float4*>(stage + (w + kRepWarps * i) * D + 4 * l);
            s[i][0] = make_float2(t4.x, t4.y);
            s[i][1] = make_float2(t4.z, t4.w);
        }
        __syncthreads();  // staging complete; the copy buffers are free for the next unit
        if (next < units) prefetch(next, OUT ? L : acc_next);

        float* Sout = a.state_out != nullptr ? a.state_out + (int64_t)unit * D * D : nullptr;
        auto store_state = [&]() {
#pragma unroll
            for (int i = 0; i < RPW; ++i)
                __stcs(reinterpret_cast<float4*>(Sout + (w + kRepWarps * i) * D + 4 * l),
                       make_float4(s[i][0].x, s[i][0].y, s[i][1].x, s[i][1].y));
        };
        if (Sout != nullptr && acc == 0) store_state();

        for (int t = 0; t < steps; ++t) {
            float* red = s_red + (t & 1) * (2 * kRepWarps * D);
            float2 r0 = make_float2(0.f, 0.f), r1 = r0, y0 = r0, y1 = r0;
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const float4 f = s_akq[t * D + w + kRepWarps * i];
                const float2 al = make_float2(f.x, f.x), k2 = make_float2(f.y, f.y);
                s[i][0] = __fmul2_rn(s[i][0], al);
                s[i][1] = __fmul2_rn(s[i][1], al);
                r0 = __ffma2_rn(k2, s[i][0], r0);
                r1 = __ffma2_rn(k2, s[i][1], r1);
                if (OUT) {
                    const float2 q2 = make_float2(f.z, f.z);
                    y0 = __ffma2_rn(q2, s[i][0], y0);
                    y1 = __ffma2_rn(q2, s[i][1], y1);
                }
            }
            *reinterpret_cast<float4*>(red + w * D + 4 * l) = make_float4(r0.x, r0.y, r1.x, r1.y);
            if (OUT) *reinterpret_cast<float4*>(red + (kRepWarps + w) * D + 4 * l) = make_float4(y0.x, y0.y, y1.x, y1.y);
            __syncthreads();
            float2 R0 = make_float2(0.f, 0.f), R1 = R0;
#pragma unroll
            for (int ww = 0; ww < kRepWarps; ++ww) {
                const float4 p4 = *reinterpret_cast<const float4*>(red + ww * D + 4 * l);
                R0 = __fadd2_rn(R0, make_float2(p4.x, p4.y));
                R1 = __fadd2_rn(R1, make_float2(p4.z, p4.w));
            }
            const float4 v4 = *reinterpret_cast<const float4*>(s_v + t * D + 4 * l);
            const float2 b2 = make_float2(s_beta[t], s_beta[t]);
            const float2 u0 = __fmul2_rn(b2, __fadd2_rn(make_float2(v4.x, v4.y), make_float2(-R0.x, -R0.y)));
            const float2 u1 = __fmul2_rn(b2, __fadd2_rn(make_float2(v4.z, v4.w), make_float2(-R1.x, -R1.y)));
            if (OUT && w == 0) {
                float2 Y0 = make_float2(0.f, 0.f), Y1 = Y0;
#pragma unroll
                for (int ww = 0; ww < kRepWarps; ++ww) {
                    const float4 p4 = *reinterpret_cast<const float4*>(red + (kRepWarps + ww) * D + 4 * l);
                    Y0 = __fadd2_rn(Y0, make_float2(p4.x, p4.y));
                    Y1 = __fadd2_rn(Y1, make_float2(p4.z, p4.w));
                }
                const float2 qk2 = make_float2(s_qk[t], s_qk[t]);
                const float2 o0 = __ffma2_rn(qk2, u0, Y0), o1 = __ffma2_rn(qk2, u1, Y1);
                __nv_bfloat162 b01 = __floats2bfloat162_rn(o0.x, o0.y), b23 = __floats2bfloat162_rn(o1.x, o1.y);
                uint2 pk;
                pk.x = *reinterpret_cast<uint32_t*>(&b01);
                pk.y = *reinterpret_cast<uint32_t*>(&b23);
                *reinterpret_cast<uint2*>(op + (((int64_t)n * L + t) * a.H + h) * D + 4 * l) = pk;
            }
            // S' = Diag(alpha) S + k u^T (the decay is already applied)
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const float kc = s_akq[t * D + w + kRepWarps * i].y;
                const float2 k2 = make_float2(kc, kc);
                s[i][0] = __ffma2_rn(k2, u0, s[i][0]);
                s[i][1] = __ffma2_rn(k2, u1, s[i][1]);
            }
            if (Sout != nullptr && t + 1 == acc) store_state();
        }
        acc = acc_next;
    }
}

// ---------------------------------------------------------------- verify only: the in-window chunk form
//
// A verify launch (outputs, no state written) needs only o_1 .. o_L from the snapshot S, so the window
// is treated as one chunk, with Gamma_t = alpha_1 ... alpha_t (inclusive, per key channel; at most 8
// tokens, so the accumulated log-decay stays >= 8 g_min and Gamma, 1/Gamma are normal fp32 numbers):
//     KG = K * Gamma, QG = Q * Gamma, KI = K / Gamma                 (rows = window tokens)
//     A[t][i] = beta_t KG_t . KI_i (i < t),  P[t][i] = QG_t . KI_i (i <= t)
//     [W0; Y0] = [KG; QG] S                                            (the only d_k x d_v work)
//     U = (I + A)^-1 diag(beta) (V - W0),   O = Y0 + P U
// which is the recurrence substituted token by token (u_t needs the state decayed to t and read
// along k_t; every earlier write k_i u_i^T reaches it scaled by Gamma_t / Gamma_i).  Per element of S
// that is two multiply-adds per token instead of four, and no barrier per token.  [KG; QG] S is a
// 16 x 128 x 128 product per (sequence, head): warp w computes value columns 16w .. 16w + 15 with
// mma.sync m16n8k16 bf16, every operand split into a bf16 pair (x = hi + lo, products hi.hi +
// hi.lo + lo.hi with fp32 accumulation: relative error about 2^-16, far below the bf16 outputs'
// rounding).  [KG; QG] and KI are staged as bf16 hi/lo tiles and read with ldmatrix / 32-bit loads;
// the snapshot goes from shared memory straight into split B-fragment registers (rows of the staged
// copy XOR-swizzled in 16-byte pieces so those loads are free of bank conflicts), which frees the
// copy buffer for the next unit early.  The in-window products U and O (K = 8 tokens) stay on the
// split tf32 form.
struct RepVLayout {
    static constexpr int kRow = kRepD + 4;                              // padded fp32 row of the token-row tiles
    static constexpr int kStage = 0;                                    // fp32 [128][128], swizzled
    static constexpr int kRaw = kStage + kRepD * kRepD * 4;             // bf16 [token][q, k, z, v][128]
    static constexpr int kRawBeta = kRaw + kRepGroup * 4 * kRepD * 2;   // fp32 [token]
    static constexpr int kBRow = kRepD + 8;                             // padded bf16 row of the split operand tiles
    static constexpr int kKQhi = kRawBeta + kRepGroup * 4;              // bf16 [16][kBRow]: KG rows 0..7, QG rows 8..15
    static constexpr int kKQlo = kKQhi + 16 * kBRow * 2;                //   (hi; then lo).  Later U fp32 [token][kRow]
    static constexpr int kKI = kKQlo + 16 * kBRow * 2;                  // bf16 [token][kBRow] hi, then lo
    static constexpr int kV = kKI + 2 * kRepGroup * kBRow * 2;          // fp32 [token][128]
    static constexpr int kWY = kV + kRepGroup * kRepD * 4;              // fp32 [16][kRow]: W0 rows 0..7, Y0 rows 8..15;
                                                                        // before that, the base-2 log-decays [token][128]
    static constexpr int kGram = kWY + 16 * kRow * 4;                   // fp32 [warp][16][8]: partial [KG; QG] KI^T
    static constexpr int kGsum = kGram + kRepWarps * 16 * 8 * 4;        // fp32 [16][8]: its sum
    static constexpr int kT = kGsum + 16 * 8 * 4;                       // fp32 [8][8]: (I + A)^-1 diag(beta)
    static constexpr int kBeta = kT + 64 * 4;
    static constexpr int kBytes = kBeta + kRepGroup * 4;
};
static_assert(RepVLayout::kKQhi % 16 == 0 && RepVLayout::kKQlo % 16 == 0 && RepVLayout::kKI % 16 == 0 &&
                  RepVLayout::kV % 16 == 0 && RepVLayout::kWY % 16 == 0 && RepVLayout::kGram % 16 == 0,
              "alignment");
static_assert(kRepGroup * RepVLayout::kRow * 4 <= 16 * RepVLayout::kBRow * 2, "U fits in the KG/QG hi tile");
static_assert(2 * (RepVLayout::kBytes + 1024) <= 228 * 1024, "two CTAs per SM");

// word offset of element (c, j) of the staged snapshot: 16-byte piece j/4 of row c moves to
// (j/4) xor 2 ((c/2) mod 4), so that the B-fragment loads (rows c0 + 2t for t = 0..3, eight
// consecutive columns) hit 32 different banks
__device__ __forceinline__ int vstage_piece(int c, int piece) { return piece ^ (((c >> 1) & 3) << 1); }
__device__ __forceinline__ int vstage_word(int c, int j) { return c * kRepD + ((vstage_piece(c, j >> 2) << 2) | (j & 3)); }

// (x0, x1) = hi + lo as packed bf16 pairs (x0 in the low half)
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 r = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// acc += (ah + al)(bh + bl), dropping al.bl
__device__ __forceinline__ void mma_bf16x3(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                           const uint32_t (&bh)[2], const uint32_t (&bl)[2])
{
    mma_bf16(d, al, bh[0], bh[1]);
    mma_bf16(d, ah, bl[0], bl[1]);
    mma_bf16(d, ah, bh[0], bh[1]);
}

// A fragments (rows 0..15, columns k0 .. k0 + 15) of a row-major bf16 tile with rows `row` elements apart
__device__ __forceinline__ void ldsm_a(const __nv_bfloat16* tile, int row, int k0, int lane, uint32_t (&r)[4])
{
    const __nv_bfloat16* p = tile + ((lane & 7) + 8 * ((lane >> 3) & 1)) * row + k0 + 8 * (lane >> 4);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"((uint32_t)__cvta_generic_to_shared(p)));
}

__device__ __forceinline__ uint32_t to_tf32(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// acc += (hi + lo of A) (b0, b1 split into a tf32 pair), dropping lo.lo
__device__ __forceinline__ void mma_tf32x3(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4], float b0, float b1)
{
    const uint32_t bh0 = to_tf32(b0), bh1 = to_tf32(b1);
    const uint32_t bl0 = to_tf32(b0 - __uint_as_float(bh0)), bl1 = to_tf32(b1 - __uint_as_float(bh1));
    mma_tf32(d, al, bh0, bh1);
    mma_tf32(d, ah, bl0, bl1);
    mma_tf32(d, ah, bh0, bh1);
}

__global__ void __launch_bounds__(kRepThreads, 2) kda_decode_replay_verify_d128_kernel(ReplayArgs a)
{
    constexpr int D = kRepD;
    constexpr int R = RepVLayout::kRow;
    using TIO = __nv_bfloat16;
    extern __shared__ __align__(16) unsigned char smem[];
    float* stage = reinterpret_cast<float*>(smem + RepVLayout::kStage);
    unsigned char* raw = smem + RepVLayout::kRaw;
    float* raw_beta = reinterpret_cast<float*>(smem + RepVLayout::kRawBeta);
    constexpr int BR = RepVLayout::kBRow;
    __nv_bfloat16* s_kqhi = reinterpret_cast<__nv_bfloat16*>(smem + RepVLayout::kKQhi);
    __nv_bfloat16* s_kqlo = reinterpret_cast<__nv_bfloat16*>(smem + RepVLayout::kKQlo);
    __nv_bfloat16* s_kihi = reinterpret_cast<__nv_bfloat16*>(smem + RepVLayout::kKI);
    __nv_bfloat16* s_kilo = s_kihi + kRepGroup * BR;
    float* s_v = reinterpret_cast<float*>(smem + RepVLayout::kV);
    float* s_wy = reinterpret_cast<float*>(smem + RepVLayout::kWY);
    float* s_g2 = s_wy;  // the log-decays live there until the products overwrite them
    float* s_gram = reinterpret_cast<float*>(smem + RepVLayout::kGram);
    float* s_gsum = reinterpret_cast<float*>(smem + RepVLayout::kGsum);
    float* s_T = reinterpret_cast<float*>(smem + RepVLayout::kT);
    float* s_beta = reinterpret_cast<float*>(smem + RepVLayout::kBeta);

    const int tid = threadIdx.x;
    const int w = tid >> 5;
    const int l = tid & 31;
    const int g8 = l >> 2;  // mma fragment row / column group
    const int t4 = l & 3;   // mma fragment thread in group
    const int L = a.L;
    const int units = a.N * a.H;
    const TIO* qp = static_cast<const TIO*>(a.q);
    const TIO* kp = static_cast<const TIO*>(a.k);
    const TIO* vp = static_cast<const TIO*>(a.v);
    const TIO* zp = static_cast<const TIO*>(a.z);
    TIO* op = static_cast<TIO*>(a.out);
    constexpr float kLog2e = 1.4426950408889634f;
    const float gm2 = kLog2e * a.g_min;

    auto prefetch = [&](int unit) {
        const int n = unit / a.H;
        const int h = unit - n * a.H;
        const float* S = a.state_in + (int64_t)unit * D * D;
#pragma unroll
        for (int i = 0; i < D * D / 4 / kRepThreads; ++i) {
            const int e4 = tid + kRepThreads * i;  // 16-byte piece e4 % 32 of row e4 / 32
            const int c = e4 >> 5;
            cp_async16(stage + c * D + (vstage_piece(c, e4 & 31) << 2), S + 4 * e4);
        }
        constexpr int CH = D * 2 / 16;
        const int64_t tok0 = (int64_t)n * L;
        for (int e = tid; e < L * 4 * CH; e += kRepThreads) {
            const int j = e / (4 * CH);
            const int rem = e - j * 4 * CH;
            const int which = rem / CH;
            const int ch = rem - which * CH;
            const TIO* base = which == 0 ? qp : which == 1 ? kp : which == 2 ? zp : vp;
            cp_async16(raw + (size_t)e * 16, base + ((tok0 + j) * a.H + h) * D + ch * 8);
        }
        if (tid < L) cp_async4(raw_beta + tid, a.beta + (tok0 + tid) * a.H + h);
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    auto raw_at = [&](int t, int which, int c) {
        return __bfloat162float(reinterpret_cast<const TIO*>(raw + (t * 4 + which) * D * 2)[c]);
    };

    int unit = blockIdx.x;
    if (unit >= units) return;
    prefetch(unit);
    for (; unit < units; unit += gridDim.x) {
        const int next = unit + gridDim.x;
        const int n = unit / a.H;
        const int h = unit - n * a.H;
        const float xs = -kLog2e * expf(a.A[h]);  // exp2(xs |z|) = exp(-exp(A_h) |z|)
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();  // (1) this unit's snapshot and tokens are in shared memory

        // the snapshot columns 16w .. 16w + 15 as split B fragments: [k step][n tile][b0, b1]
        // (b0: rows 16 ks + 2 t4, + 1; b1: rows 16 ks + 2 t4 + 8, + 9; column 16 w + 8 nt + g8)
        uint32_t bh[D / 16][2][2], bl[D / 16][2][2];
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int j = 16 * w + 8 * nt + g8;
                const int c0 = 16 * ks + 2 * t4;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int c = c0 + 8 * hf;
                    split_bf16x2(stage[vstage_word(c, j)], stage[vstage_word(c + 1, j)], bh[ks][nt][hf],
                                 bl[ks][nt][hf]);
                }
            }
        // gate of every (token, key channel) in base 2, and v, over all threads
#pragma unroll
        for (int m = 0; m < kRepGroup * D / kRepThreads; ++m) {
            const int e = tid + kRepThreads * m;
            const int t = e / D;
            const int c = e - t * D;
            if (t < L) {
                const float z = raw_at(t, 2, c);
                const float ez = ex2_approx(xs * fabsf(z));  // exp(-exp(A_h) |z|)
                const float r = rcp_approx(1.f + ez);
                s_g2[e] = gm2 * ((z >= 0.f) ? r : ez * r);   // log2 of alpha: g_min sigmoid(exp(A_h) z) / ln 2
                s_v[e] = raw_at(t, 3, c);
            }
        }
        if (tid < L) s_beta[tid] = raw_beta[tid];
        __syncthreads();
        {
            // key channel c, tokens 4 half .. 4 half + 3: cumulative decay and the scaled rows
            const int c = tid & (D - 1);
            const int t0 = (tid >> 7) * 4;
            float G2 = 0.f;
            for (int t = 0; t < t0 && t < L; ++t) G2 += s_g2[t * D + c];
#pragma unroll
            for (int t = t0; t < t0 + 4; ++t) {
                float kg = 0.f, qg = 0.f, ki = 0.f;
                if (t < L) {
                    G2 += s_g2[t * D + c];
                    const float gam = ex2_approx(G2), igam = ex2_approx(-G2);
                    const float kc = raw_at(t, 1, c);
                    kg = kc * gam;
                    qg = raw_at(t, 0, c) * gam;
                    ki = kc * igam;
                }
                const __nv_bfloat16 kh = __float2bfloat16_rn(kg), qh = __float2bfloat16_rn(qg);
                const __nv_bfloat16 ih = __float2bfloat16_rn(ki);
                s_kqhi[t * BR + c] = kh;
                s_kqlo[t * BR + c] = __float2bfloat16_rn(kg - __bfloat162float(kh));
                s_kqhi[(8 + t) * BR + c] = qh;
                s_kqlo[(8 + t) * BR + c] = __float2bfloat16_rn(qg - __bfloat162float(qh));
                s_kihi[t * BR + c] = ih;
                s_kilo[t * BR + c] = __float2bfloat16_rn(ki - __bfloat162float(ih));
            }
        }
        __syncthreads();  // (2) staged; the copy buffers are free for the next unit
        if (next < units) prefetch(next);

        // [W0; Y0] = [KG; QG] S for value columns 16w .. 16w + 15, and this warp's two k steps of
        // [KG; QG] KI^T (the in-window Gram block: A and P)
        float acc[2][4], gacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t ah[4], al[4];
            ldsm_a(s_kqhi, BR, 16 * ks, l, ah);
            ldsm_a(s_kqlo, BR, 16 * ks, l, al);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma_bf16x3(acc[nt], ah, al, bh[ks][nt], bl[ks][nt]);
            if (ks == w) {  // this warp's k step of the Gram block: B[k][n] = KI[token n][channel k]
                const int k0 = 16 * ks + 2 * t4;
                const uint32_t gh[2] = {*reinterpret_cast<const uint32_t*>(s_kihi + g8 * BR + k0),
                                        *reinterpret_cast<const uint32_t*>(s_kihi + g8 * BR + k0 + 8)};
                const uint32_t gl[2] = {*reinterpret_cast<const uint32_t*>(s_kilo + g8 * BR + k0),
                                        *reinterpret_cast<const uint32_t*>(s_kilo + g8 * BR + k0 + 8)};
                mma_bf16x3(gacc, ah, al, gh, gl);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int j = 16 * w + 8 * nt + 2 * t4;
            *reinterpret_cast<float2*>(s_wy + g8 * R + j) = make_float2(acc[nt][0], acc[nt][1]);
            *reinterpret_cast<float2*>(s_wy + (g8 + 8) * R + j) = make_float2(acc[nt][2], acc[nt][3]);
        }
        *reinterpret_cast<float2*>(s_gram + (w * 16 + g8) * 8 + 2 * t4) = make_float2(gacc[0], gacc[1]);
        *reinterpret_cast<float2*>(s_gram + (w * 16 + g8 + 8) * 8 + 2 * t4) = make_float2(gacc[2], gacc[3]);
        __syncthreads();  // (3) W0, Y0 and the partial Gram blocks complete

        if (w == 0) {
            // Gram block [KG; QG] KI^T = sum of the eight warps' k slices
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int e = l + 32 * m;
                float x = 0.f;
#pragma unroll
                for (int ww = 0; ww < kRepWarps; ++ww) x += s_gram[ww * 128 + e];
                s_gsum[e] = x;
            }
            __syncwarp();
            if (l < L) {
                // column l of T = (I + A)^-1 with A[t][m] = beta_t KG_t . KI_m (m < t), then scaled by beta_l
                float col[kRepGroup];
#pragma unroll
                for (int t = 0; t < kRepGroup; ++t) {
                    float x = (t == l) ? 1.f : 0.f;
                    if (t > l && t < L) {
                        float sum = 0.f;
#pragma unroll
                        for (int m = 0; m < t; ++m)
                            if (m >= l) sum += s_gsum[t * 8 + m] * col[m];
                        x = -s_beta[t] * sum;
                    }
                    col[t] = x;
                }
                const float bl = s_beta[l];
#pragma unroll
                for (int t = 0; t < kRepGroup; ++t)
                    if (t < L) s_T[t * 8 + l] = col[t] * bl;
            }
        }
        __syncthreads();  // (4) T' complete

        {
            // U = T' (V - W0) and O = Y0 + P U (P[t][i] = QG_t . KI_i, i <= t) for this warp's value
            // columns, as two more split-tf32 products with M = tokens (rows 8..15 zero), K = 8 tokens.
            // Entries outside t < L, i <= t are zeroed so that stale rows never enter.
            const bool row_ok = g8 < L;
            const float tA0 = (row_ok && t4 <= g8) ? s_T[g8 * 8 + t4] : 0.f;
            const float tA2 = (row_ok && t4 + 4 <= g8) ? s_T[g8 * 8 + t4 + 4] : 0.f;
            const float pA0 = (row_ok && t4 <= g8) ? s_gsum[(8 + g8) * 8 + t4] : 0.f;
            const float pA2 = (row_ok && t4 + 4 <= g8) ? s_gsum[(8 + g8) * 8 + t4 + 4] : 0.f;
            uint32_t th[4] = {to_tf32(tA0), 0u, to_tf32(tA2), 0u};
            uint32_t tl[4] = {to_tf32(tA0 - __uint_as_float(th[0])), 0u, to_tf32(tA2 - __uint_as_float(th[2])), 0u};
            uint32_t ph[4] = {to_tf32(pA0), 0u, to_tf32(pA2), 0u};
            uint32_t pl[4] = {to_tf32(pA0 - __uint_as_float(ph[0])), 0u, to_tf32(pA2 - __uint_as_float(ph[2])), 0u};
            float* s_u = reinterpret_cast<float*>(s_kqhi);  // [token][kRow]; the operand tiles are no longer read
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int jb = 16 * w + 8 * nt + g8;  // B-fragment column
                const float x0 = (t4 < L) ? s_v[t4 * D + jb] - s_wy[t4 * R + jb] : 0.f;
                const float x1 = (t4 + 4 < L) ? s_v[(t4 + 4) * D + jb] - s_wy[(t4 + 4) * R + jb] : 0.f;
                float u4[4] = {0.f, 0.f, 0.f, 0.f};
                mma_tf32x3(u4, th, tl, x0, x1);
                const int jd = 16 * w + 8 * nt + 2 * t4;  // D-fragment columns jd, jd + 1
                *reinterpret_cast<float2*>(s_u + g8 * R + jd) = make_float2(u4[0], u4[1]);
            }
            __syncwarp();
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int jb = 16 * w + 8 * nt + g8;
                const int jd = 16 * w + 8 * nt + 2 * t4;
                const float2 y = *reinterpret_cast<const float2*>(s_wy + (8 + g8) * R + jd);
                float o4[4] = {y.x, y.y, 0.f, 0.f};
                mma_tf32x3(o4, ph, pl, s_u[t4 * R + jb], s_u[(t4 + 4) * R + jb]);
                if (row_ok)
                    *reinterpret_cast<__nv_bfloat162*>(op + (((int64_t)n * L + g8) * a.H + h) * D + jd) =
                        __floats2bfloat162_rn(o4[0], o4[1]);
            }
        }
    }
}

static cudaError_t launch_replay_verify_d128(const ReplayArgs& a, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(kda_decode_replay_verify_d128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         RepVLayout::kBytes);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)a.N * a.H;
    const unsigned grid = (unsigned)(units < 2LL * sm_count_of_current_device() ? units : 2LL * sm_count_of_current_device());
    kda_decode_replay_verify_d128_kernel<<<grid, kRepThreads, RepVLayout::kBytes, s>>>(a);
    return cudaGetLastError();
}

template <bool OUT>
static cudaError_t launch_replay_d128(const ReplayArgs& a, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(kda_decode_replay_d128_kernel<OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         RepLayout::kBytes);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)a.N * a.H;
    const unsigned grid = (unsigned)(units < 2LL * sm_count_of_current_device() ? units : 2LL * sm_count_of_current_device());
    kda_decode_replay_d128_kernel<OUT><<<grid, kRepThreads, RepLayout::kBytes, s>>>(a);
    return cudaGetLastError();
}

template <typename TIO, bool OUT>
static cudaError_t launch_replay_out(const ReplayArgs& a, int dk, int dv, cudaStream_t s)
{
    const unsigned grid = (unsigned)((int64_t)a.N * a.H);
#define KDA_REP_CASE(DKv, DVv)                                                              \
    if (dk == DKv && dv == DVv) {                                                            \
        kda_decode_replay_kernel<TIO, DKv, DVv, OUT><<<grid, kRepThreads, 0, s>>>(a);        \
        return cudaGetLastError();                                                           \
    }
    KDA_REP_CASE(32, 32) KDA_REP_CASE(32, 64) KDA_REP_CASE(32, 128)
    KDA_REP_CASE(64, 32) KDA_REP_CASE(64, 64) KDA_REP_CASE(64, 128)
    KDA_REP_CASE(128, 32) KDA_REP_CASE(128, 64) KDA_REP_CASE(128, 128)
#undef KDA_REP_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_replay(const ReplayArgs& a, int dk, int dv, kda_dtype_t dt, cudaStream_t s)
{
    const bool out = a.out != nullptr;
    if (dt == KDA_BF16 && dk == kRepD && dv == kRepD && a.L <= kRepGroup) {
        if (out && a.state_out == nullptr) return launch_replay_verify_d128(a, s);
        return out ? launch_replay_d128<true>(a, s) : launch_replay_d128<false>(a, s);
    }
    if (dt == KDA_BF16)
        return out ? launch_replay_out<__nv_bfloat16, true>(a, dk, dv, s) : launch_replay_out<__nv_bfloat16, false>(a, dk, dv, s);
    return out ? launch_replay_out<float, true>(a, dk, dv, s) : launch_replay_out<float, false>(a, dk, dv, s);
}

}  // namespace kda
