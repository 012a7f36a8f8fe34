// kda_internal.cuh -- declarations shared by the libkda.so translation units (not installed).
//
// Workspace layout of kda_forward (every region 256-byte aligned, offsets from the base):
//   [0, 256)   device check word (uint32) written by the kernels, read by kda_workspace_status
// and, for the fp32 SIMT path only (the fused tensor-core path keeps these on chip):
//   G          fp32 [T_tot, H, d_k]   in-chunk inclusive cumulative log-decay (kda_gate)
//   W          fp32 [T_tot, H, d_k]   WY-transformed keys T diag(beta) (K*Gamma)   (kda_ut_wy)
//   Ut         fp32 [T_tot, H, d_v]   UT-transformed values T diag(beta) V         (kda_ut_wy)
// and, for the bf16 d = 128 tensor-core path:
//   blocks     per-step operand blocks [T_tot / 32 + N + 1 slots][H][kBlockBytes] (kda_chunk_prep_tc),
//              present when the workspace holds them ("split" plan; otherwise the fused kernel runs)
//   seg_in, seg_st           fp32 [N][H][max_seg][d_k][d_v] per-segment states (segmented plans)
//   seg_mt                   [N][H][max_seg] transitions M, 64 KB each in the scan's operand format
//                            (seg_m_off below)
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <utility>

#include "kda.h"

namespace kda {

constexpr int kChunk = 16;  // tokens per chunk: a chunk's log-decay stays in [16 g_min, 0]

// Device check word bits.
constexpr uint32_t kCheckBadSeqlens = 1u;
constexpr uint32_t kCheckTimeout = 2u;

// Tries (of up to 20 us each) of a bounded wait in the tensor-core kernels: ~2.6 s at most.
constexpr uint32_t kWaitTries = 1u << 17;
// Default tries of the split plan's state-pass hand-off waits (one warp role waiting for another).
constexpr uint32_t kHandoffTries = kWaitTries;

struct ForwardLayout {
    size_t status_off, g_off, w_off, ut_off, blocks_off, seg_in_off, seg_st_off, seg_mt_off, total;
    int32_t seg_chunks, max_seg;
    bool split;  // tensor-core path: parallel chunk preparation + state pass (else the fused kernel)
};

// Bytes of one operand block (the state pass's input for one 32-token step; see kda_tc_chunk.cuh).
constexpr size_t kBlockBytes = 53760;
constexpr int kPair = 2 * kChunk;  // tokens per state step of the split tensor-core plan

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Steepest log-decay floor the tensor-core kernels take.  They scale a 16-token chunk's keys and
// queries by Gamma and 1/Gamma referred to the chunk's first token and carry the small ones as
// bf16 hi/lo pairs; with g_min >= -5 (K3's floor) Gamma >= e^-80 = 2^-115.4 keeps every hi and,
// but for corrections below 2^-10.6 of the value, every lo part a normal number (the hardware
// exp2 and the products flush subnormals), and 1/Gamma <= e^80 stays far from overflow.
// Steeper floors run on the fp32 path, which forms every pairwise decay exp(G_r - G_i) <= 1.
constexpr float kChunkGminLimit = -5.0f;
// The backward's chunk factors are plain fp32 numbers (no hi/lo pairs, no flushing): with
// g_min >= -5.4, Gamma >= e^-86.4 stays normal and 1/Gamma <= e^86.4 finite.
constexpr float kBackwardGminLimit = -5.4f;

// bf16 inputs with d_k = d_v = 128 run on the tensor-core kernels (they scale keys and queries by
// Gamma and 1/Gamma of one chunk); other problems, and steeper floors, on the fp32 path, which
// forms every pairwise decay exp(G_r - G_i) <= 1 directly.
inline bool use_tensor_core_path(const kda_problem_t& p)
{
    return p.io_dtype == KDA_BF16 && p.d_k == 128 && p.d_v == 128 && p.total_tokens > 0 &&
           p.total_tokens < (int64_t(1) << 31) && p.g_min >= kChunkGminLimit;
}

// Chunks of the longest sequence allowed by the descriptor (max_seqlen, at most T_tot).
inline int64_t max_chunks_of(const kda_problem_t& p)
{
    const int64_t L = p.max_seqlen < p.total_tokens ? p.max_seqlen : p.total_tokens;
    return (L + kChunk - 1) / kChunk;
}

// Operand-block slots of the split tensor-core plan: 32-token step s of sequence n uses slot
// cu[n] / 32 + n + s.
inline size_t block_bytes_of(const kda_problem_t& p)
{
    const size_t slots = (size_t)(p.total_tokens / kPair) + (size_t)p.num_seqs + 1;
    return slots * (size_t)p.num_heads * kBlockBytes;
}

// Segmentation of the tensor-core path.  A sequence is cut into segments of seg_chunks chunks;
// segment k's end state is S_end = M_k S_in + S~_k (its transition applied to the incoming state,
// plus its end state from a zero start), so the segments' (M_k, S~_k) are computed in parallel,
// scanned, and the segments re-run from their true incoming states.  The plan minimises a
// wave-count model of the passes (`split`: two state-pass CTAs per SM, else the fused kernel's
// one).  The environment variable KDA_SEGMENT_CHUNKS=<n> forces n chunks per segment
// (0: no segmentation; the split plan rounds n up to an even count, its state steps being
// pairs of chunks).  Only plans whose per-segment state buffers fit in `budget_bytes` count.
void segment_plan(const kda_problem_t& p, size_t budget_bytes, bool split, int32_t& seg_chunks, int32_t& max_seg);

// Workspace layout for a problem given `available` bytes of workspace.  Tensor-core path: the split
// plan (operand blocks) with the fastest segmentation that fits, else the fused kernel with the
// fastest segmentation that fits (none if only the minimum fits).  forward_layout(p, SIZE_MAX).total
// is the size kda_forward_workspace_bytes reports; forward_layout(p, 0).total is the minimum.
inline ForwardLayout forward_layout(const kda_problem_t& p, size_t available)
{
    ForwardLayout L{};
    const bool tcp = use_tensor_core_path(p);
    const size_t th = tcp ? 0 : (size_t)p.total_tokens * (size_t)p.num_heads;
    L.status_off = 0;
    L.g_off = 256;
    L.w_off = align_up(L.g_off + th * p.d_k * sizeof(float), 256);
    L.ut_off = align_up(L.w_off + th * p.d_k * sizeof(float), 256);
    const size_t end = align_up(L.ut_off + th * p.d_v * sizeof(float), 256);
    L.seg_chunks = 0;
    L.max_seg = 1;
    L.split = false;
    L.blocks_off = end;
    size_t seg_start = end;
    // segment buffers are whole multiples of 256 bytes, so a plan fits iff its three buffers do
    if (tcp) {
        const size_t bb = align_up(block_bytes_of(p), 256);
        // KDA_TC_PLAN=fused keeps the fused kernel even when the operand blocks would fit
        const char* plan = getenv("KDA_TC_PLAN");
        const bool fused_only = plan != nullptr && strcmp(plan, "fused") == 0;
        if (!fused_only && available >= end + bb) {
            L.split = true;
            seg_start = end + bb;
            segment_plan(p, available - seg_start, true, L.seg_chunks, L.max_seg);
        } else if (available > end) {
            segment_plan(p, available - end, false, L.seg_chunks, L.max_seg);
        }
    }
    const size_t seg_bytes = L.max_seg > 1 ? (size_t)p.num_seqs * p.num_heads * L.max_seg * p.d_k * p.d_v * sizeof(float) : 0;
    L.seg_in_off = seg_start;
    L.seg_st_off = align_up(L.seg_in_off + seg_bytes, 256);
    L.seg_mt_off = align_up(L.seg_st_off + seg_bytes, 256);
    L.total = align_up(L.seg_mt_off + seg_bytes, 256);
    return L;
}

// Arguments common to the prefill kernels.
struct PrefillArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* z;
    const float* A;
    const float* beta;
    const float* s0;          // may be null
    const int32_t* cu;        // may be null (equal lengths)
    void* out;
    float* s_final;           // may be null
    float* G;                 // workspace
    float* W;                 // workspace
    float* Ut;                // workspace
    uint32_t* check;          // workspace
    int64_t T_tot;
    int32_t N, H, dk, dv, max_seqlen, chunks_per_seq;
    float g_min;
    // sequence segmentation of the tensor-core path (seg_chunks == 0: one segment per sequence)
    int32_t seg_chunks;       // chunks per segment
    int32_t max_seg;          // segments of the longest sequence
    int32_t seg_mode;         // 0: outputs; 1: end state from zero (S~); 2: transition (M)
    int32_t prep_run;         // preparation kernel: 32-token steps per CTA (set by its launcher)
    uint32_t handoff_tries;   // state pass: tries of a hand-off wait before it gives up (kHandoffTries;
                              // KDA_DEBUG_HANDOFF_TRIES lowers it to exercise the timeout path)
    float* seg_in;            // [N][H][max_seg][d][d] incoming state of every segment (scan output)
    float* seg_st;            // [N][H][max_seg][d][d] S~ of every segment
    float* seg_mt;            // [N][H][max_seg] M of every segment, seg_m_off format (64 KB each)
    unsigned char* blocks;    // per-chunk operand blocks of the split tensor-core plan
};

// A segment's transition M (d = 128; M[c][j]: the coefficient of incoming state row j in outgoing
// row c) as the scan's mma.sync A operand: bf16 hi and lo planes of the row-major [c][j] matrix,
// lo = bf16(M - hi), 32 KB each, the 16-byte chunks of every 256-byte row permuted by XOR with
// c mod 8 so that the rows of an 8 x 8 ldmatrix tile fall on distinct banks.
constexpr uint32_t kSegMPlane = 128 * 128 * 2;
__host__ __device__ __forceinline__ uint32_t seg_m_off(int c, int j)
{
    return (uint32_t)(c * 256 + ((((j >> 3) ^ (c & 7))) << 4) + (j & 7) * 2);
}
__device__ __forceinline__ void store_seg_m(float* seg, int c, int j, float x)
{
    const __nv_bfloat16 hi = __float2bfloat16_rn(x);
    const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
    unsigned char* base = reinterpret_cast<unsigned char*>(seg);
    *reinterpret_cast<__nv_bfloat16*>(base + seg_m_off(c, j)) = hi;
    *reinterpret_cast<__nv_bfloat16*>(base + kSegMPlane + seg_m_off(c, j)) = lo;
}

// ---------------------------------------------------------------- backward (kda_backward)
//
// Workspace of kda_backward (every region 256-byte aligned, offsets from the base):
//   [0, 256)  check word
//   G, W, Ut  fp32 [T_tot, H, d]   the forward path's per-chunk G, W and U~ (kda_gate, kda_ut_wy)
//   P         fp32 [T_tot, H, 16]  row r of each chunk's tril_incl((Q Gamma)(K / Gamma)^T)
//   QG, Kt    fp32 [T_tot, H, d_k] Q Gamma and K Gamma_C / Gamma of every chunk
//   U, dU     fp32 [T_tot, H, d_v] U = U~ - W S_in and its gradient
//   S_chunk   fp32 [slots][H][d_k][d_v]  state entering each chunk
//   dS_chunk  fp32 [slots][H][d_k][d_v]  gradient reaching the state after each chunk
//   dA_part   fp32 [slots][H]            per-chunk partial sums of dA
// Chunk ci of sequence n uses slot cu[n] / 16 + n + ci (slots = T_tot / 16 + N + 1), so the slots
// of consecutive sequences never overlap.
struct BackwardLayout {
    size_t g_off, w_off, ut_off, p_off, qg_off, kt_off, u_off, du_off, s_off, ds_off, da_off, total, slots;
};

inline BackwardLayout backward_layout(const kda_problem_t& p)
{
    BackwardLayout L{};
    const size_t th = (size_t)p.total_tokens * (size_t)p.num_heads;
    L.slots = (size_t)(p.total_tokens / kChunk) + (size_t)p.num_seqs + 1;
    const size_t state = (size_t)p.d_k * p.d_v * sizeof(float);
    L.g_off = 256;
    L.w_off = align_up(L.g_off + th * p.d_k * sizeof(float), 256);
    L.ut_off = align_up(L.w_off + th * p.d_k * sizeof(float), 256);
    L.p_off = align_up(L.ut_off + th * p.d_v * sizeof(float), 256);
    L.qg_off = align_up(L.p_off + th * kChunk * sizeof(float), 256);
    L.kt_off = align_up(L.qg_off + th * p.d_k * sizeof(float), 256);
    L.u_off = align_up(L.kt_off + th * p.d_k * sizeof(float), 256);
    L.du_off = align_up(L.u_off + th * p.d_v * sizeof(float), 256);
    L.s_off = align_up(L.du_off + th * p.d_v * sizeof(float), 256);
    L.ds_off = align_up(L.s_off + L.slots * p.num_heads * state, 256);
    L.da_off = align_up(L.ds_off + L.slots * p.num_heads * state, 256);
    L.total = align_up(L.da_off + L.slots * p.num_heads * sizeof(float), 256);
    return L;
}

struct BackwardArgs {
    PrefillArgs f;            // forward inputs, sizes, check word and the G / W / Ut workspace regions
    const void* dout;         // [T][H][d_v] io dtype
    const float* dS_final;    // [N][H][d_k][d_v] or null (zero)
    void* dq;                 // [T][H][d_k] io dtype
    void* dk;                 // [T][H][d_k] io dtype
    void* dv;                 // [T][H][d_v] io dtype
    void* dz;                 // [T][H][d_k] io dtype
    float* dA;                // [H]
    float* dbeta;             // [T][H]
    float* dS0;               // [N][H][d_k][d_v] or null (not written)
    float* P;                 // workspace regions (see backward_layout)
    float* QG;
    float* Kt;
    float* U;
    float* dU;
    float* S_chunk;
    float* dS_chunk;
    float* dA_part;
    int64_t slots;
};

cudaError_t launch_backward(const BackwardArgs& b, kda_dtype_t dt, cudaStream_t s);

// Context-parallel pieces (kda_kcp.cu): identity states [units][dk][dk]; and the scan
// out = fold_{i < count} (S -> M_i S + S~_i) applied to S0 (null: zeros), M [count][N][H][dk][dk],
// S~ [count][N][H][dk][dv].
cudaError_t launch_identity_states(float* S, int64_t units, int dk, cudaStream_t s);
cudaError_t launch_state_scan(const float* M, const float* St, const float* S0, float* out, int N, int H, int dk, int dv,
                              int count, cudaStream_t s);

// Workspace of kda_forward_summary: a kda_forward workspace large enough for both of its runs (the
// problem itself for S~, and the problem with d_v = d_k for M), then zero values [T][H][d_k] (io
// dtype), identity states [N][H][d_k][d_k] fp32 and discarded outputs [T][H][max(d_k, d_v)] (io).
struct SummaryLayout {
    size_t fwd_bytes, zeros_off, eye_off, out_off, total;
    kda_problem_t pm;  // the problem of the transition run
};

inline SummaryLayout summary_layout(const kda_problem_t& p)
{
    SummaryLayout L{};
    L.pm = p;
    L.pm.d_v = p.d_k;
    const size_t a = forward_layout(p, SIZE_MAX).total, b = forward_layout(L.pm, SIZE_MAX).total;
    const size_t io = p.io_dtype == KDA_BF16 ? 2 : 4;
    const size_t th = (size_t)p.total_tokens * p.num_heads;
    L.fwd_bytes = align_up(a > b ? a : b, 256);
    L.zeros_off = L.fwd_bytes;
    L.eye_off = align_up(L.zeros_off + th * p.d_k * io, 256);
    L.out_off = align_up(L.eye_off + (size_t)p.num_seqs * p.num_heads * p.d_k * p.d_k * sizeof(float), 256);
    const int dmax = p.d_k > p.d_v ? p.d_k : p.d_v;
    L.total = align_up(L.out_off + th * dmax * io, 256);
    return L;
}

struct DecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* z;
    const float* A;
    const float* beta;
    float* state;
    void* out;
    int32_t N, H;
    float g_min;
};

// A window of L tokens for each of N sequences from a state snapshot (kda_decode_replay).
struct ReplayArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* z;
    const float* A;
    const float* beta;
    const float* state_in;    // [N][H][d_k][d_v], read only unless state_out is the same pointer
    const int32_t* accepted;  // [N] or null (all L)
    float* state_out;         // [N][H][d_k][d_v] or null
    void* out;                // [N*L][H][d_v] or null
    int32_t N, H, L;
    float g_min;
};

// Layer prologue / epilogue (kda_prologue, kda_epilogue).
constexpr int kMaxConv = 4;  // widest short convolution supported
struct PrologueArgs {
    const void* x[3];      // q, k, v projections [T][H][d_k | d_k | d_v]
    const float* w[3];     // depthwise convolution weights [H][d][K]
    void* y[3];            // prepared q, k, v
    const int32_t* cu;     // [N + 1] or null (N equal lengths)
    int64_t T;
    int32_t N, H, dk, dv, K;
};
struct EpilogueArgs {
    const void* o;         // [rows][d_v]
    const void* gate;      // [rows][d_v]
    const float* weight;   // [d_v]
    void* y;               // [rows][d_v], may be o
    int64_t rows;          // T * H
    float eps;
};

// Launchers (each returns the cudaError_t of its launch).
cudaError_t launch_gate(const PrefillArgs& a, kda_dtype_t dt, cudaStream_t s);
cudaError_t launch_ut_wy(const PrefillArgs& a, kda_dtype_t dt, cudaStream_t s);
cudaError_t launch_chunk_fwd(const PrefillArgs& a, kda_dtype_t dt, cudaStream_t s);
cudaError_t launch_chunk_fwd_tc(const PrefillArgs& a, cudaStream_t s);      // fused kernel, all passes
cudaError_t launch_chunk_prep_tc(const PrefillArgs& a, cudaStream_t s);     // operand blocks
cudaError_t launch_prefill_split_tc(const PrefillArgs& a, cudaStream_t s);  // blocks + state pass, all passes
cudaError_t launch_segment_scan(const PrefillArgs& a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, int dk, int dv, kda_dtype_t dt, cudaStream_t s);
cudaError_t launch_replay(const ReplayArgs& a, int dk, int dv, kda_dtype_t dt, cudaStream_t s);
cudaError_t launch_prologue(const PrologueArgs& a, kda_dtype_t dt, cudaStream_t s);
cudaError_t launch_epilogue(const EpilogueArgs& a, int dv, kda_dtype_t dt, cudaStream_t s);

// SM count of the current device (cached per device; 152 if it cannot be queried).
int sm_count_of_current_device();

// Optional per-kernel timing around launches (no-ops unless kda_profile_enable(1)).
void prof_start(const char* name, cudaStream_t s);
void prof_stop(cudaStream_t s);

// ---------------------------------------------------------------- programmatic dependent launch

// The kernels of one prefill run back to back on one stream.  Each signals at its start that the
// next kernel may be scheduled (it can then only start once every CTA of this grid has started, so
// it never takes resources this grid still needs); a kernel launched with launch_dependent() waits
// in griddep_wait() until the previous grid has completed and its writes are visible, and does its
// set-up (tensor-memory allocation, barrier initialisation) before that.
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                    Args&&... args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- device helpers

__device__ __forceinline__ float ld_io(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_io(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_io(float* p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_io(__nv_bfloat16* p, int64_t i, float x) { p[i] = __float2bfloat16_rn(x); }

// Token range [t0, t1) of sequence n.  Returns false (and raises the check bit) when the offsets
// are inconsistent with the descriptor, in which case the sequence is skipped.
__device__ __forceinline__ bool seq_range(const PrefillArgs& a, int n, int64_t& t0, int64_t& t1)
{
    if (a.cu == nullptr) {
        const int64_t L = a.T_tot / a.N;
        t0 = (int64_t)n * L;
        t1 = t0 + L;
        return true;
    }
    t0 = a.cu[n];
    t1 = a.cu[n + 1];
    const bool ok = (t0 >= 0) && (t1 >= t0) && (t1 <= a.T_tot) && (t1 - t0 <= (int64_t)a.max_seqlen) &&
                    (n != 0 || t0 == 0) && (n != a.N - 1 || t1 == a.T_tot);
    if (!ok) {
        atomicOr(a.check, kCheckBadSeqlens);
    }
    return ok;
}

// Equation 5: log-decay for logit z with per-head scale e^{A_h}.  Uses the CUDA math library.
__device__ __forceinline__ float log_decay(float z, float expA, float g_min)
{
    const float x = expA * z;
    // logistic in the overflow-free form for both signs
    const float e = expf(-fabsf(x));
    const float sig = (x >= 0.f) ? 1.f / (1.f + e) : e / (1.f + e);
    return g_min * sig;
}

}  // namespace kda
