/*
 * kda.h -- C ABI of libkda.so: Kimi Delta Attention (KDA) prefill and decode on one GB300 GPU.
 *
 * The operation (per sequence n and head h; "Kimi K3: the paper and proofs side by side",
 * section 2.1.1, Equations 1 and 5; "Kimi K3: architecture, derivations and a pinned-source
 * audit", section 4.3):
 *
 *   g_t     = g_min * sigmoid(exp(A_h) * z_t)           per key channel, g_min = -5 in K3
 *   alpha_t = exp(g_t)                                   retention in (exp(g_min), 1)
 *   S_t     = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *   o_t     = S_t^T q_t                                  read after the update
 *
 * S is d_k x d_v with rows = key channels and columns = value channels.  No 1/sqrt(d_k) scale is
 * applied to q (the pages write o = S^T q); callers normalise q and k themselves.  o_t is the
 * recurrence output before any head-wise norm or output gate.
 *
 * Conventions for every entry point
 *   - Layouts are row-major and token-major packed:
 *       q, k, z     [T_tot, H, d_k]      (io dtype)
 *       v, out      [T_tot, H, d_v]      (io dtype)
 *       beta        [T_tot, H]           fp32
 *       A           [H]                  fp32
 *       states      [N, H, d_k, d_v]     fp32
 *       cu_seqlens  [N + 1]              int32, cu_seqlens[0] = 0, non-decreasing, last = T_tot
 *   - All tensor pointers are DEVICE pointers (device or managed memory of the current device,
 *     or mapped pinned host memory), 16-byte aligned.  The problem descriptor is a host pointer.
 *   - The caller owns every buffer.  The library keeps no allocation between calls; forward's
 *     scratch memory is the caller's `workspace`.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only enqueue work and
 *     return without synchronising; launch failures are reported as KDA_ERR_CUDA, asynchronous
 *     faults surface at the caller's next synchronisation.
 *   - Argument errors are detected on the host before anything is launched, and nothing is
 *     written in that case.  No C++ exception crosses this boundary.
 *   - Supported sizes: d_k, d_v in {32, 64, 128}; 1 <= H <= 65535; io dtype fp32 or bf16.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* null/misaligned/host-only pointer, bad descriptor, aliasing   */
    KDA_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement (e.g. d_k = 96)  */
    KDA_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed                   */
    KDA_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up (reported via the status) */
    KDA_ERR_WORKSPACE = 5,    /* workspace missing, misaligned or smaller than required        */
    KDA_ERR_DEVICE_CHECK = 6  /* a device-side input check failed (e.g. bad cu_seqlens)       */
} kda_status_t;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype_t;

/* Problem descriptor (host memory). */
typedef struct {
    int32_t num_seqs;      /* N: number of packed sequences (batch size for equal lengths)      */
    int64_t total_tokens;  /* T_tot = sum of sequence lengths (= N for a decode step)            */
    int32_t max_seqlen;    /* host-known upper bound on any sequence length (grid sizing)       */
    int32_t num_heads;     /* H                                                                  */
    int32_t d_k;           /* key/query channels: 32, 64 or 128                                  */
    int32_t d_v;           /* value channels: 32, 64 or 128                                      */
    kda_dtype_t io_dtype;  /* dtype of q, k, v, z and out; A, beta and states are always fp32   */
    float g_min;           /* log-decay floor, < 0 (-5 in K3)                                    */
} kda_problem_t;

/*
 * Bytes of device workspace kda_forward needs for this problem (0 if the descriptor is invalid).
 * The requirement depends only on the descriptor's sizes, never on the data.
 */
size_t kda_forward_workspace_bytes(const kda_problem_t* problem);

/* The execution plan kda_forward picks for a problem and a workspace size. */
typedef struct {
    int32_t split;         /* 1: parallel chunk preparation + state pass; 0: fused kernel or the
                              fp32 three-kernel path                                              */
    int32_t seg_chunks;    /* chunks per sequence segment, 0 when sequences are not segmented   */
    int32_t num_segments;  /* segments of the longest sequence (1 when not segmented)           */
    int32_t reserved;      /* 0                                                                  */
} kda_plan_t;

/*
 * Fills *plan with the plan kda_forward would use for `problem` with `workspace_bytes` of
 * workspace (SIZE_MAX: the plan of kda_forward_workspace_bytes(problem) bytes).  The plan depends
 * only on the descriptor, the workspace size, the SM count of the current device and the
 * environment overrides documented at kda_forward.  The library has no counterpart of this call
 * on the pages; it exists so that callers can size workspaces and read measurements.
 * Returns KDA_ERR_INVALID_ARG for a NULL plan or an invalid descriptor, KDA_ERR_WORKSPACE if the
 * workspace is below the minimum, else KDA_OK.  Host only; launches nothing.
 */
kda_status_t kda_forward_plan(const kda_problem_t* problem, size_t workspace_bytes, kda_plan_t* plan);

/*
 * Chunkwise-parallel prefill over packed sequences (Equation 1 for every token, in 16-token
 * chunks; the chunk form is an exact regrouping of the token recurrence, "Kimi K3:
 * architecture, derivations and a pinned-source audit", section 4.5, and the bounded gate keeps
 * a chunk's accumulated log-decay in [16 g_min, 0], "Kimi K3" reading notes, section 2).
 *
 *   q, k, z, v, A, beta : inputs as laid out above.
 *   initial_state : [N,H,d_k,d_v] fp32, or NULL for zero states.
 *   cu_seqlens    : [N+1] int32 on the device, or NULL for N equal lengths T_tot / N
 *                   (then T_tot must be a multiple of N).  Chunks restart at every sequence
 *                   start; a zero-length sequence copies its initial state to its final state.
 *                   Every length must be <= max_seqlen and the offsets must be non-decreasing
 *                   and end at T_tot; violations are detected on the device, the offending
 *                   sequence is skipped, and kda_workspace_status() reports KDA_ERR_DEVICE_CHECK.
 *   out           : [T_tot,H,d_v] io dtype.  Must not overlap any input.
 *   final_state   : [N,H,d_k,d_v] fp32, or NULL (not written).  May be the same pointer as
 *                   initial_state (in-place carry); any other overlap is rejected.
 *   workspace     : device scratch, 256-byte aligned, not shared with a concurrently running
 *                   call.  kda_forward_workspace_bytes(problem) bytes allow the fastest plan.  For
 *                   bf16 inputs with d_k = d_v = 128 and g_min >= -5 (steeper floors run on the
 *                   fp32 path, whose workspace holds 4 (2 d_k + d_v) bytes per token and head)
 *                   that plan first prepares the
 *                   state-independent operands of every pair of chunks in parallel (52.5 KB per
 *                   32 tokens and head, held in the workspace) and then runs the sequential state
 *                   pass in 32-token steps; a workspace too
 *                   small for those blocks selects a fused kernel that prepares each chunk on the
 *                   fly.  A smaller workspace also makes long sequences use fewer parallel
 *                   segments (down to none); one below the unsegmented minimum is rejected
 *                   (KDA_ERR_WORKSPACE).  Results do not depend on the plan beyond rounding.
 *                   Environment overrides, read on every call: KDA_TC_PLAN=fused keeps the fused
 *                   kernel; KDA_SEGMENT_CHUNKS=<n> forces n chunks per segment (0: unsegmented;
 *                   the pair-step plan rounds n up to an even count).  KDA_DEBUG_HANDOFF_TRIES=<n>
 *                   (a debugging aid, off unless set) gives the split plan's state-pass hand-off
 *                   waits n tries of up to 20 us instead of ~2.6 s; with n = 0 every such wait gives
 *                   up at once, the kernels stop early without touching memory they do not own, and
 *                   the status readers report KDA_ERR_TIMEOUT (outputs and final states are then
 *                   unspecified).
 *
 * Returns KDA_OK once all kernels are enqueued on `stream`.
 */
kda_status_t kda_forward(const void* q, const void* k, const void* v, const void* z,
                         const float* A, const float* beta, const float* initial_state,
                         const int32_t* cu_seqlens, void* out, float* final_state,
                         const kda_problem_t* problem, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * One recurrent decode step: every one of the N sequences advances by exactly one token
 * (KDA.step: update the state, then read it with the query; "Kimi K3: the paper and proofs side
 * by side", section "A recurrent step and its return type").
 *
 *   q, k, z : [N,H,d_k] io dtype;  v : [N,H,d_v] io dtype;  beta : [N,H] fp32;  A : [H] fp32.
 *   state   : [N,H,d_k,d_v] fp32, read and overwritten in place with the new state.
 *   out     : [N,H,d_v] io dtype; must not overlap any input or the state.
 *   problem : total_tokens must equal num_seqs (cu_seqlens is not used).
 */
kda_status_t kda_decode_step(const void* q, const void* k, const void* v, const void* z,
                             const float* A, const float* beta, float* state, void* out,
                             const kda_problem_t* problem, void* stream);

/*
 * Context-parallel prefill (KCP) for sequences split across ranks ("Kimi K3" reading notes, section 7,
 * "Scaling to 1M Tokens: NoPE and KDA Context Parallelism": every rank summarises its token range,
 * the summaries are exchanged once, and a prefix scan gives every rank the state its range starts
 * from; "Kimi K3: architecture, derivations and a pinned-source audit", section 4.5: a range of
 * tokens acts on the state as an affine map, and such maps compose associatively).  A range maps an
 * incoming state S to M S + S~, with M (d_k x d_k) the range's end state from the identity when
 * every value is zero and S~ (d_k x d_v) its end state from zero.  The flow on rank r of R:
 *     kda_forward_summary(own range)        -> (M_r, S~_r)
 *     all-gather (M, S~) across the ranks   (the caller's collective; 4 d_k (d_k + d_v) bytes per
 *                                            sequence and head and rank)
 *     kda_state_scan(count = r)             -> the state the rank's range starts from
 *     kda_forward(own range, that state)    -> outputs; on rank R - 1 the final state
 */
size_t kda_forward_summary_workspace_bytes(const kda_problem_t* problem);

/*
 * The affine summary of every sequence's token range ("Kimi K3" reading notes, section 7):
 *   transition      : [N,H,d_k,d_k] fp32 output M (M[c][j]: weight of incoming state row j in row c
 *                     of the end state).
 *   state_from_zero : [N,H,d_k,d_v] fp32 output S~.
 * Inputs, layouts and cu_seqlens as for kda_forward (the initial state plays no part).  Runs
 * kda_forward twice inside (S~ from zero; M from identity states with zero values and d_v = d_k),
 * so every kda_forward plan, precision and device check applies; the check word is read with
 * kda_workspace_status(workspace, ...).  workspace: kda_forward_summary_workspace_bytes(problem)
 * bytes, 256-byte aligned.  Outputs must not overlap the inputs, each other or the workspace.
 */
kda_status_t kda_forward_summary(const void* q, const void* k, const void* v, const void* z, const float* A,
                                 const float* beta, const int32_t* cu_seqlens, float* transition, float* state_from_zero,
                                 const kda_problem_t* problem, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The prefix scan of KCP ("Kimi K3" reading notes, section 7): starting from initial_state
 * ([N,H,d_k,d_v] fp32, NULL: zeros), applies S <- M_i S + S~_i for i = 0 .. count - 1 and writes
 * the result to state_out ([N,H,d_k,d_v] fp32; may be initial_state itself, no other overlap).
 *   transition      : [count][N,H,d_k,d_k] fp32 (the gathered M of the ranks before this one, in order)
 *   state_from_zero : [count][N,H,d_k,d_v] fp32 (their S~)
 * count = 0 copies the initial state.  problem: num_seqs, num_heads, d_k, d_v (the rest unused).
 * fp32 arithmetic.
 */
kda_status_t kda_state_scan(const float* transition, const float* state_from_zero, const float* initial_state,
                            int32_t count, float* state_out, const kda_problem_t* problem, void* stream);

/*
 * Bytes of device workspace kda_backward needs for this problem (0 if the descriptor is invalid):
 * per token and head 4 (4 d_k + 3 d_v + 16) bytes, plus two fp32 d_k x d_v states (the state
 * entering each 16-token chunk and the gradient reaching its end) per chunk slot and head, with
 * T_tot / 16 + N + 1 slots -- about 11.6 KiB per token and head at d_k = d_v = 128.
 */
size_t kda_backward_workspace_bytes(const kda_problem_t* problem);

/*
 * Gradients of kda_forward for training: given dL/d(out) and dL/d(final_state), the gradients of
 * L with respect to q, k, v, z, A, beta and the initial state.  The derivative is the analytic one
 * of the recurrence (Equation 1 with the gate of Equation 5, "Kimi K3: the paper and proofs side
 * by side", section 2.1.1) taken chunk by chunk in reverse; the pages check the same analytic
 * derivative against finite differences ("Kimi K3: architecture, derivations and a pinned-source
 * audit", section "CPU laboratory") and name comparing "sequence outputs and gradients" as the
 * test of a kernel (same page, section "Pinned evidence and execution boundary").
 *
 *   q, k, v, z, A, beta, initial_state, cu_seqlens : the forward call's inputs, as for kda_forward
 *                   (initial_state NULL: zeros).
 *   d_out         : [T_tot,H,d_v] io dtype, dL/d(out).
 *   d_final_state : [N,H,d_k,d_v] fp32, dL/d(final_state), or NULL (zero).
 *   dq, dk, dz    : [T_tot,H,d_k] io dtype outputs;  dv : [T_tot,H,d_v] io dtype output.
 *   dA            : [H] fp32 output (summed over all tokens, key channels and sequences).
 *   dbeta         : [T_tot,H] fp32 output.
 *   d_initial_state : [N,H,d_k,d_v] fp32 output, or NULL (not written).
 *   workspace     : kda_backward_workspace_bytes(problem) bytes of device scratch, 256-byte
 *                   aligned, not shared with a concurrently running call.
 * Outputs must not overlap any input, each other or the workspace.  Supported: every d_k, d_v and io
 * dtype of kda_forward with g_min >= -5.4 (a 16-token chunk's 1/Gamma stays a finite fp32 number;
 * steeper floors return KDA_ERR_UNSUPPORTED).  The forward pass is recomputed inside the call (only
 * the inputs are needed).  Arithmetic is fp32 throughout; gradients are rounded to the io dtype once.
 * Invalid cu_seqlens are reported through kda_workspace_status() as for kda_forward.
 */
kda_status_t kda_backward(const void* q, const void* k, const void* v, const void* z, const float* A,
                          const float* beta, const float* initial_state, const int32_t* cu_seqlens,
                          const void* d_out, const float* d_final_state, void* dq, void* dk, void* dv, void* dz,
                          float* dA, float* dbeta, float* d_initial_state, const kda_problem_t* problem,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Speculative-decode state replay: a window of L drafted tokens for each of N sequences, run from a
 * state snapshot ("Kimi K3: architecture, derivations and a pinned-source audit", section 10.3 "KDA
 * state replay for speculative decoding": a speculating server keeps only its drafts' per-token
 * inputs and, once it knows which drafts survived, moves the saved state forward over them on chip
 * in one launch, so no rejected draft ever has to be undone).  Every token is one decode step of the recurrence (as kda_decode_step computes it); one
 * launch reads each (sequence, head) state once, keeps it on chip across the window and writes at
 * most one state.  Typical use, per speculation round:
 *   verify : out given, state_out NULL -- o_t of every drafted token, no state is written, so the
 *            snapshot stays valid whatever is accepted;
 *   commit : accepted given, state_out == state_in, out NULL -- the snapshot advances over each
 *            sequence's accepted prefix; rejected drafts are never applied.
 * With accepted NULL and both outputs given it is an L-token decode step.
 *
 *   q, k, z   : [N*L, H, d_k] io dtype, token t of sequence n at row n*L + t (kda_forward's packed
 *               layout with N equal lengths L);  v : [N*L, H, d_v] io dtype;  beta : [N*L, H] fp32;
 *               A : [H] fp32.
 *   state_in  : [N, H, d_k, d_v] fp32 snapshot; only read (unless state_out is the same pointer).
 *   accepted  : [N] int32 on the device, the number of window tokens of sequence n to keep, or NULL
 *               for all L.  Values outside [0, L] are clamped to it.
 *   state_out : [N, H, d_k, d_v] fp32, the state after the first accepted[n] tokens (the snapshot's
 *               values where accepted[n] = 0), or NULL (not written).  May be state_in itself
 *               (in place); any other overlap with an argument is rejected.
 *   out       : [N*L, H, d_v] io dtype, o_t = S_t^T q_t of every window token from the snapshot,
 *               whatever is accepted; or NULL (not written).  Must not overlap any argument.
 *   problem   : num_seqs = N and total_tokens = N*L with L >= 1; max_seqlen and cu_seqlens are
 *               not used.
 * At least one of out and state_out must be given.  Argument errors as for kda_decode_step.
 */
kda_status_t kda_decode_replay(const void* q, const void* k, const void* v, const void* z,
                               const float* A, const float* beta, const float* state_in,
                               const int32_t* accepted, float* state_out, void* out,
                               const kda_problem_t* problem, void* stream);

/*
 * Layer prologue: the recurrence's q, k, v from their projections, per head ("Kimi K3: the paper
 * and proofs side by side", section 2.1.1, "Preparing the queries, keys, values, and decay";
 * "Kimi K3: architecture, derivations and a pinned-source audit", section 4.3):
 *     y_t = sum_{i < conv_width} w[h][c][i] x_{t-i}   causal depthwise short convolution; tokens
 *                                                      before the sequence start count as zero
 *     y_t = y_t * sigmoid(y_t)                         Swish
 *     y_t = y_t / sqrt(sum_c y_t[c]^2 + 1e-6)          regularised L2 normalisation, q and k only
 *
 *   xq, xk : [T_tot, H, d_k] io dtype;  xv : [T_tot, H, d_v] io dtype  (the projections).
 *   wq, wk : [H, d_k, conv_width] fp32;  wv : [H, d_v, conv_width] fp32  (w[..., 0] weighs the
 *            current token, w[..., i] the token i places earlier).
 *   conv_width : 1 .. 4.
 *   cu_seqlens : as for kda_forward (device [N+1], or NULL for N equal lengths).  Offsets are not
 *            validated on the device here: invalid offsets give unspecified outputs (never an
 *            access outside the tensors).
 *   q, k, v : outputs, shaped like xq, xk, xv; must not overlap any input or each other.
 *   problem : num_seqs, total_tokens, num_heads, d_k, d_v, io_dtype as for kda_forward.
 */
kda_status_t kda_prologue(const void* xq, const void* xk, const void* xv, const float* wq,
                          const float* wk, const float* wv, int32_t conv_width,
                          const int32_t* cu_seqlens, void* q, void* k, void* v,
                          const kda_problem_t* problem, void* stream);

/*
 * Layer epilogue: head-wise RMSNorm of the recurrence output and the sigmoid output gate
 * ("Kimi K3: architecture, derivations and a pinned-source audit", section 4.3; the output gate of
 * Equation 6 in "Kimi K3: the paper and proofs side by side", section 2.1.1):
 *     y = o / sqrt(mean_c o[c]^2 + eps) * weight * sigmoid(gate)
 *
 *   o, gate : [T_tot, H, d_v] io dtype (gate: the output-gate projection, before the sigmoid).
 *   weight  : [d_v] fp32, the RMSNorm weight shared by the heads.
 *   eps     : >= 0, finite (the pages name no value for the RMSNorm stabiliser).  With eps = 0 an
 *             all-zero row has no defined output (0 / 0), as in the formula.
 *   y       : [T_tot, H, d_v] io dtype; may be o itself (in place); any other overlap is rejected.
 */
kda_status_t kda_epilogue(const void* o, const void* gate, const float* weight, float eps, void* y,
                          const kda_problem_t* problem, void* stream);

/*
 * kda_forward for callers that cannot allocate device memory: a library or plugin that runs
 * inside a host application which owns every device allocation (its own pool or arena) and gives
 * the plugin no allocator, or a latency-critical path that must not enter the driver's allocator.
 * Such callers still provide every input and output buffer; only the scratch is taken care of.
 *
 * The paper has no counterpart to this entry point: it is a memory-management convenience.
 *
 * Scratch comes from one array of KDA_STATIC_SCRATCH_BYTES that the library keeps in device
 * memory of every GPU that loads it, for the life of the process.  The call allocates nothing and
 * calls no allocating routine.  Arguments, layouts and results are those of kda_forward (same
 * kernels), without `workspace` / `workspace_bytes`.
 *   - A problem whose smallest workspace exceeds KDA_STATIC_SCRATCH_BYTES is rejected on the host
 *     with KDA_ERR_WORKSPACE before anything is launched.  (bf16 problems with d_k = d_v = 128
 *     need only a few hundred bytes, and use as many parallel sequence segments as the array
 *     holds; the fp32 path needs 4 (2 d_k + d_v) bytes per token and head.)
 *   - Every call looks up the array's address in the caller's current context (a lookup, no
 *     allocation); the first call in a context also loads the library's device code there, so make
 *     that first call before any stream capture.  The address is never cached across calls, so it
 *     stays right after cudaDeviceReset or when the caller switches contexts.
 *   - All calls on a device share the one array, and it keeps the last call's contents (the
 *     check word is cleared at the start of every call).  Calls whose GPU work overlaps -- on
 *     different streams, or from different host threads -- race on it; serialise them.
 *   - The device-side check word of the last call (bad cu_seqlens, a bounded wait that gave up) is
 *     read with kda_static_scratch_status(), not kda_workspace_status().
 */
#define KDA_STATIC_SCRATCH_BYTES ((size_t)8 << 20)
kda_status_t kda_forward_static_scratch(const void* q, const void* k, const void* v, const void* z,
                                        const float* A, const float* beta, const float* initial_state,
                                        const int32_t* cu_seqlens, void* out, float* final_state,
                                        const kda_problem_t* problem, void* stream);

/*
 * Synchronises `stream` and reads the check word of the last kda_forward_static_scratch call in the
 * current context (the word at the start of the library's scratch array): KDA_OK,
 * KDA_ERR_DEVICE_CHECK or KDA_ERR_TIMEOUT as for kda_workspace_status.  Allocates nothing.
 * The paper has no counterpart to this call.
 */
kda_status_t kda_static_scratch_status(void* stream);

/*
 * Synchronises `stream` and reads the device-side check word that kda_forward keeps in its
 * workspace: KDA_OK, or KDA_ERR_DEVICE_CHECK if a sequence was skipped because its cu_seqlens
 * entries were invalid, or KDA_ERR_TIMEOUT if a bounded device wait gave up.  The word is
 * cleared by the next kda_forward on that workspace.
 */
kda_status_t kda_workspace_status(const void* workspace, size_t workspace_bytes, void* stream);

/* Static, human-readable name of a status code. */
const char* kda_status_string(kda_status_t status);

/*
 * Per-kernel device timing, for measurement tools.  While enabled, every kernel launched by
 * kda_forward / kda_backward / kda_decode_step / kda_decode_replay / kda_prologue / kda_epilogue is bracketed by two CUDA events recorded on the call's stream;
 * kda_profile_read synchronises on those events and returns, per kernel name, the number of
 * launches and their summed device time.  Enabling (or disabling) discards earlier records.
 * Events are host-side objects: no device memory is allocated.  Not thread-safe against
 * concurrent calls on other threads while enabled.
 */
typedef struct {
    char name[32];        /* kernel name, NUL-terminated                    */
    int64_t launches;     /* launches recorded since the last enable        */
    double total_ms;      /* summed device time of those launches (ms)      */
} kda_kernel_time_t;

kda_status_t kda_profile_enable(int enable);

/* Fills up to max_entries records; returns the number of distinct kernels (or -1 on error). */
int32_t kda_profile_read(kda_kernel_time_t* out, int32_t max_entries);

/* ABI version of this header: (major << 16) | minor. */
uint32_t kda_abi_version(void);

#define KDA_ABI_VERSION ((1u << 16) | 5u)

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
