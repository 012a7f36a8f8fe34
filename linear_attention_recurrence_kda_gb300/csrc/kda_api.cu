// kda_api.cu -- the C ABI of libkda.so (declared in include/kda.h): argument checks and launches.
//
// Every check that can be made without the data runs on the host before anything is enqueued,
// in this order: descriptor, required pointers, alignment, overlap, workspace, and finally the
// CUDA pointer attributes (device-accessible memory of the current device).  The first four need
// no GPU.  Nothing here synchronises except kda_workspace_status.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "kda_internal.cuh"

using kda::ForwardLayout;

namespace {

bool supported_dim(int32_t d) { return d == 32 || d == 64 || d == 128; }

size_t io_size(kda_dtype_t dt) { return dt == KDA_BF16 ? 2 : 4; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

Range range_of(const void* p, size_t bytes)
{
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + bytes};
}

bool overlaps(Range a, Range b)
{
    if (a.lo == a.hi || b.lo == b.hi || a.lo == 0 || b.lo == 0) return false;
    return a.lo < b.hi && b.lo < a.hi;
}

enum class Call { Forward, Decode, Replay };

kda_status_t check_descriptor(const kda_problem_t* p, Call call)
{
    if (p == nullptr) return KDA_ERR_INVALID_ARG;
    if (p->num_seqs < 1 || p->total_tokens < 0 || p->num_heads < 1 || p->num_heads > 65535) return KDA_ERR_INVALID_ARG;
    if (p->d_k <= 0 || p->d_v <= 0) return KDA_ERR_INVALID_ARG;
    if (p->io_dtype != KDA_F32 && p->io_dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
    if (!(p->g_min < 0.f) || !std::isfinite(p->g_min)) return KDA_ERR_INVALID_ARG;
    if (!supported_dim(p->d_k) || !supported_dim(p->d_v)) return KDA_ERR_UNSUPPORTED;
    // element counts must stay far from overflow: T_tot * H * d <= 2^40
    const double elems = (double)p->total_tokens * p->num_heads * (p->d_k > p->d_v ? p->d_k : p->d_v);
    if (elems > 1099511627776.0) return KDA_ERR_UNSUPPORTED;
    if ((double)p->num_seqs * p->num_heads * p->d_k * p->d_v > 1099511627776.0) return KDA_ERR_UNSUPPORTED;
    if (call == Call::Decode) {
        if (p->total_tokens != p->num_seqs) return KDA_ERR_INVALID_ARG;
    } else if (call == Call::Replay) {
        // a window of L >= 1 tokens per sequence, L < 2^31
        if (p->total_tokens < p->num_seqs || p->total_tokens % p->num_seqs != 0) return KDA_ERR_INVALID_ARG;
        if (p->total_tokens / p->num_seqs > 2147483647LL) return KDA_ERR_UNSUPPORTED;
    } else {
        if (p->max_seqlen < 0) return KDA_ERR_INVALID_ARG;
    }
    return KDA_OK;
}

// Device-accessible memory of the current device (or mapped pinned host memory).
kda_status_t check_device_pointer(const void* p)
{
    if (p == nullptr) return KDA_OK;
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return e == cudaErrorInvalidValue ? KDA_ERR_INVALID_ARG : KDA_ERR_CUDA;
    }
    if (attr.devicePointer == nullptr) return KDA_ERR_INVALID_ARG;
    if (attr.type == cudaMemoryTypeDevice) {
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
        if (attr.device != dev) return KDA_ERR_INVALID_ARG;
    }
    return KDA_OK;
}

int sm_count_cached()
{
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return 152;
    }
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            n = 152;
        }
        cached[dev] = n;
    }
    return cached[dev];
}

}  // namespace

namespace kda {

int sm_count_of_current_device() { return sm_count_cached(); }

void segment_plan(const kda_problem_t& p, size_t budget_bytes, bool split, int32_t& seg_chunks, int32_t& max_seg)
{
    const int64_t chunks = max_chunks_of(p);
    // the split plan advances the state by pairs of chunks, so its segments hold an even number
    const int64_t gran = split ? 2 : 1;
    seg_chunks = 0;
    max_seg = 1;
    if (chunks <= gran) return;
    if (const char* env = std::getenv("KDA_SEGMENT_CHUNKS")) {
        long v = std::strtol(env, nullptr, 10);
        if (v > 0) v = (long)(((int64_t)v + gran - 1) / gran * gran);
        const int64_t ns = v > 0 ? (chunks + v - 1) / v : 1;
        const double need = (double)p.num_seqs * p.num_heads * p.d_k * p.d_v * 12.0 * (double)ns;
        if (v > 0 && v < chunks && need <= (double)budget_bytes) {
            seg_chunks = (int32_t)v;
            max_seg = (int32_t)ns;
        }
        return;
    }
    // cost in units of one state step of a chain running alone on an SM (a chunk, or a pair of
    // chunks in the split plan).  A pass of c chains of sc steps takes sc steps per wave plus a
    // start-up of about OVH steps per wave (launch, first operand block, initial state); the split
    // plan's state pass fits two chains per SM at about 1.1 times the time per step (the fused
    // kernel: one chain per SM).  Pass 3 runs one chain per segment, pass 1 two (S~ and M) per
    // segment but the last; one step of the scan costs about scan_step state steps.
    const int64_t steps = (chunks + gran - 1) / gran;
    const double sms = (double)sm_count_of_current_device();
    const double scan_step = split ? 0.6 : 0.8;
    constexpr double OVH = 4.0;
    const double units = (double)p.num_seqs * p.num_heads;
    const double per_seg = units * p.d_k * p.d_v * 4.0 * 3.0;  // S_in, S~ and M of one segment
    auto pass = [&](double ctas, double sc) -> double {
        if (ctas <= sms) return sc + OVH;
        const double nw = split ? std::ceil(ctas / (2.0 * sms)) : std::ceil(ctas / sms);
        return nw * ((split ? 1.1 : 1.0) * sc + OVH);
    };
    const double unsegmented = pass(units, (double)steps);
    double best = unsegmented;
    for (int64_t sc = 1; sc < steps; ++sc) {  // steps per segment
        const int64_t ns = (steps + sc - 1) / sc;
        if (ns < 2 || ns > 64) continue;
        if (per_seg * (double)ns > (double)budget_bytes || per_seg * (double)ns > 2.0e9) continue;
        // pass 3: when only the last segment's chains overflow the SMs, they share SMs with full
        // chains, which run about 20 % slower while both run (the last segment's steps)
        const int64_t last = steps - (ns - 1) * sc;
        const double ctas3 = units * ns;
        const double pass3 = (split && ctas3 > sms && units * (ns - 1) <= sms && ctas3 <= 2.0 * sms)
                                 ? (double)sc + 0.2 * (double)last + OVH
                                 : pass(ctas3, (double)sc);
        const double cost = pass3 + pass(2.0 * units * (ns - 1), (double)sc) + scan_step * (double)(ns - 1);
        if (cost < best && cost < 0.9 * unsegmented) {
            best = cost;
            seg_chunks = (int32_t)(sc * gran);
            max_seg = (int32_t)ns;
        }
    }
}

}  // namespace kda

namespace {

int32_t chunks_per_seq(const kda_problem_t& p) { return (int32_t)kda::max_chunks_of(p); }

}  // namespace

extern "C" {

uint32_t kda_abi_version(void) { return KDA_ABI_VERSION; }

const char* kda_status_string(kda_status_t s)
{
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: unsupported size or type";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA runtime error";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: a bounded device wait gave up";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case KDA_ERR_DEVICE_CHECK: return "KDA_ERR_DEVICE_CHECK: device-side input check failed";
    }
    return "KDA: unknown status";
}

size_t kda_forward_workspace_bytes(const kda_problem_t* problem)
{
    if (check_descriptor(problem, Call::Forward) != KDA_OK) return 0;
    return kda::forward_layout(*problem, SIZE_MAX).total;
}

kda_status_t kda_forward_plan(const kda_problem_t* problem, size_t workspace_bytes, kda_plan_t* plan)
{
    if (plan == nullptr) return KDA_ERR_INVALID_ARG;
    const kda_status_t st = check_descriptor(problem, Call::Forward);
    if (st != KDA_OK) return st;
    const ForwardLayout L = kda::forward_layout(*problem, workspace_bytes);
    if (workspace_bytes < L.total) return KDA_ERR_WORKSPACE;
    plan->split = L.split ? 1 : 0;
    plan->seg_chunks = L.max_seg > 1 ? L.seg_chunks : 0;
    plan->num_segments = L.max_seg > 1 ? L.max_seg : 1;
    plan->reserved = 0;
    return KDA_OK;
}

kda_status_t kda_forward(const void* q, const void* k, const void* v, const void* z, const float* A,
                         const float* beta, const float* initial_state, const int32_t* cu_seqlens,
                         void* out, float* final_state, const kda_problem_t* problem, void* workspace,
                         size_t workspace_bytes, void* stream)
{
    kda_status_t st = check_descriptor(problem, Call::Forward);
    if (st != KDA_OK) return st;
    const kda_problem_t& p = *problem;
    const bool equal = cu_seqlens == nullptr;
    if (equal && (p.total_tokens % p.num_seqs) != 0) return KDA_ERR_INVALID_ARG;
    // with equal lengths every sequence has T_tot / N tokens, which max_seqlen must bound
    if (equal && (int64_t)p.max_seqlen < p.total_tokens / p.num_seqs) return KDA_ERR_INVALID_ARG;
    const int64_t cps = chunks_per_seq(p);
    if ((int64_t)p.num_seqs * (cps > 0 ? cps : 1) > 2147483647LL) return KDA_ERR_UNSUPPORTED;

    const bool has_tokens = p.total_tokens > 0;
    if (A == nullptr) return KDA_ERR_INVALID_ARG;
    if (has_tokens && (!q || !k || !v || !z || !beta || !out)) return KDA_ERR_INVALID_ARG;

    const size_t io = io_size(p.io_dtype);
    const size_t tk = (size_t)p.total_tokens * p.num_heads * p.d_k;
    const size_t tv = (size_t)p.total_tokens * p.num_heads * p.d_v;
    const size_t sb = (size_t)p.num_seqs * p.num_heads * p.d_k * p.d_v * sizeof(float);
    for (const void* ptr : {q, k, v, z, (const void*)out, (const void*)initial_state, (const void*)final_state}) {
        if (!aligned(ptr, 16)) return KDA_ERR_INVALID_ARG;
    }
    if (!aligned(A, 4) || !aligned(beta, 4) || !aligned(cu_seqlens, 4)) return KDA_ERR_INVALID_ARG;

    const Range rq = range_of(q, tk * io), rk = range_of(k, tk * io), rz = range_of(z, tk * io);
    const Range rv = range_of(v, tv * io), ro = range_of(out, tv * io);
    const Range ra = range_of(A, p.num_heads * sizeof(float));
    const Range rb = range_of(beta, (size_t)p.total_tokens * p.num_heads * sizeof(float));
    const Range ri = range_of(initial_state, sb), rf = range_of(final_state, sb);
    const Range rc = range_of(cu_seqlens, cu_seqlens ? (size_t)(p.num_seqs + 1) * sizeof(int32_t) : 0);
    for (Range r : {rq, rk, rz, rv, ra, rb, ri, rf, rc}) {
        if (overlaps(ro, r)) return KDA_ERR_INVALID_ARG;
    }
    for (Range r : {rq, rk, rz, rv, ra, rb, rc}) {
        if (overlaps(rf, r)) return KDA_ERR_INVALID_ARG;
    }
    if (overlaps(rf, ri) && final_state != initial_state) return KDA_ERR_INVALID_ARG;

    // the fastest plan whose segment buffers fit in the workspace given (down to no segmentation)
    const ForwardLayout L = kda::forward_layout(p, workspace_bytes);
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < L.total) return KDA_ERR_WORKSPACE;
    const Range rw = range_of(workspace, L.total);
    for (Range r : {rq, rk, rz, rv, ra, rb, ri, rf, rc, ro}) {
        if (overlaps(rw, r)) return KDA_ERR_INVALID_ARG;
    }

    for (const void* ptr : {q, k, v, z, (const void*)A, (const void*)beta, (const void*)initial_state,
                            (const void*)cu_seqlens, (const void*)out, (const void*)final_state,
                            (const void*)workspace}) {
        st = check_device_pointer(ptr);
        if (st != KDA_OK) return st;
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    kda::PrefillArgs a{};
    a.q = q; a.k = k; a.v = v; a.z = z; a.A = A; a.beta = beta;
    a.s0 = initial_state; a.cu = cu_seqlens; a.out = out; a.s_final = final_state;
    a.check = reinterpret_cast<uint32_t*>(ws + L.status_off);
    a.G = reinterpret_cast<float*>(ws + L.g_off);
    a.W = reinterpret_cast<float*>(ws + L.w_off);
    a.Ut = reinterpret_cast<float*>(ws + L.ut_off);
    a.T_tot = p.total_tokens; a.N = p.num_seqs; a.H = p.num_heads; a.dk = p.d_k; a.dv = p.d_v;
    a.max_seqlen = equal ? (int32_t)(p.total_tokens / p.num_seqs) : p.max_seqlen;
    a.chunks_per_seq = (int32_t)cps;
    a.g_min = p.g_min;
    a.seg_chunks = L.seg_chunks;
    a.max_seg = L.max_seg;
    a.seg_mode = 0;
    a.handoff_tries = kda::kHandoffTries;
    if (const char* env = std::getenv("KDA_DEBUG_HANDOFF_TRIES")) {
        // debugging aid, off unless set: fewer tries make the state pass's hand-off waits give up,
        // which exercises the timeout path (reported as KDA_ERR_TIMEOUT by the status readers)
        char* end = nullptr;
        const unsigned long v = std::strtoul(env, &end, 10);
        if (end != env && *end == '\0' && v < kda::kHandoffTries) a.handoff_tries = (uint32_t)v;
    }
    a.seg_in = reinterpret_cast<float*>(ws + L.seg_in_off);
    a.seg_st = reinterpret_cast<float*>(ws + L.seg_st_off);
    a.seg_mt = reinterpret_cast<float*>(ws + L.seg_mt_off);
    a.blocks = ws + L.blocks_off;

    if (cudaMemsetAsync(a.check, 0, sizeof(uint32_t), s) != cudaSuccess) return KDA_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    if (kda::use_tensor_core_path(p)) {
        // every pass is timed by the profiling hooks inside the launchers
        e = L.split ? kda::launch_prefill_split_tc(a, s) : kda::launch_chunk_fwd_tc(a, s);
        return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    }
    if (cps > 0) {
        kda::prof_start("kda_gate", s);
        e = kda::launch_gate(a, p.io_dtype, s);
        kda::prof_stop(s);
        if (e != cudaSuccess) return KDA_ERR_CUDA;
        kda::prof_start("kda_ut_wy", s);
        e = kda::launch_ut_wy(a, p.io_dtype, s);
        kda::prof_stop(s);
        if (e != cudaSuccess) return KDA_ERR_CUDA;
    }
    kda::prof_start("kda_chunk_fwd", s);
    e = kda::launch_chunk_fwd(a, p.io_dtype, s);
    kda::prof_stop(s);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

size_t kda_backward_workspace_bytes(const kda_problem_t* problem)
{
    if (check_descriptor(problem, Call::Forward) != KDA_OK) return 0;
    return kda::backward_layout(*problem).total;
}

kda_status_t kda_backward(const void* q, const void* k, const void* v, const void* z, const float* A,
                          const float* beta, const float* initial_state, const int32_t* cu_seqlens,
                          const void* d_out, const float* d_final_state, void* dq, void* dk, void* dv, void* dz,
                          float* dA, float* dbeta, float* d_initial_state, const kda_problem_t* problem,
                          void* workspace, size_t workspace_bytes, void* stream)
{
    kda_status_t st = check_descriptor(problem, Call::Forward);
    if (st != KDA_OK) return st;
    const kda_problem_t& p = *problem;
    if (p.g_min < kda::kBackwardGminLimit) return KDA_ERR_UNSUPPORTED;
    const bool equal = cu_seqlens == nullptr;
    if (equal && (p.total_tokens % p.num_seqs) != 0) return KDA_ERR_INVALID_ARG;
    if (equal && (int64_t)p.max_seqlen < p.total_tokens / p.num_seqs) return KDA_ERR_INVALID_ARG;
    const int64_t cps = chunks_per_seq(p);
    if ((int64_t)p.num_seqs * (cps > 0 ? cps : 1) > 2147483647LL) return KDA_ERR_UNSUPPORTED;
    const bool has_tokens = p.total_tokens > 0;
    if (A == nullptr || dA == nullptr) return KDA_ERR_INVALID_ARG;
    if (has_tokens && (!q || !k || !v || !z || !beta || !d_out || !dq || !dk || !dv || !dz || !dbeta))
        return KDA_ERR_INVALID_ARG;

    const size_t io = io_size(p.io_dtype);
    const size_t tk = (size_t)p.total_tokens * p.num_heads * p.d_k;
    const size_t tv = (size_t)p.total_tokens * p.num_heads * p.d_v;
    const size_t th = (size_t)p.total_tokens * p.num_heads;
    const size_t sb = (size_t)p.num_seqs * p.num_heads * p.d_k * p.d_v * sizeof(float);
    for (const void* ptr : {q, k, v, z, d_out, (const void*)dq, (const void*)dk, (const void*)dv, (const void*)dz,
                            (const void*)initial_state, (const void*)d_final_state, (const void*)d_initial_state}) {
        if (!aligned(ptr, 16)) return KDA_ERR_INVALID_ARG;
    }
    for (const void* ptr : {(const void*)A, (const void*)beta, (const void*)cu_seqlens, (const void*)dA,
                            (const void*)dbeta}) {
        if (!aligned(ptr, 4)) return KDA_ERR_INVALID_ARG;
    }
    const Range in[10] = {range_of(q, tk * io), range_of(k, tk * io), range_of(z, tk * io), range_of(v, tv * io),
                          range_of(A, p.num_heads * sizeof(float)), range_of(beta, th * sizeof(float)),
                          range_of(initial_state, sb),
                          range_of(cu_seqlens, cu_seqlens ? (size_t)(p.num_seqs + 1) * sizeof(int32_t) : 0),
                          range_of(d_out, tv * io), range_of(d_final_state, sb)};
    const Range out[7] = {range_of(dq, tk * io), range_of(dk, tk * io), range_of(dv, tv * io), range_of(dz, tk * io),
                          range_of(dA, p.num_heads * sizeof(float)), range_of(dbeta, th * sizeof(float)),
                          range_of(d_initial_state, sb)};
    for (int i = 0; i < 7; ++i) {
        for (const Range& r : in) {
            if (overlaps(out[i], r)) return KDA_ERR_INVALID_ARG;
        }
        for (int j = 0; j < i; ++j) {
            if (overlaps(out[i], out[j])) return KDA_ERR_INVALID_ARG;
        }
    }
    const kda::BackwardLayout L = kda::backward_layout(p);
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < L.total) return KDA_ERR_WORKSPACE;
    const Range rw = range_of(workspace, L.total);
    for (const Range& r : in) {
        if (overlaps(rw, r)) return KDA_ERR_INVALID_ARG;
    }
    for (const Range& r : out) {
        if (overlaps(rw, r)) return KDA_ERR_INVALID_ARG;
    }
    for (const void* ptr : {q, k, v, z, (const void*)A, (const void*)beta, (const void*)initial_state,
                            (const void*)cu_seqlens, d_out, (const void*)d_final_state, (const void*)dq, (const void*)dk,
                            (const void*)dv, (const void*)dz, (const void*)dA, (const void*)dbeta,
                            (const void*)d_initial_state, (const void*)workspace}) {
        st = check_device_pointer(ptr);
        if (st != KDA_OK) return st;
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    kda::BackwardArgs b{};
    kda::PrefillArgs& a = b.f;
    a.q = q; a.k = k; a.v = v; a.z = z; a.A = A; a.beta = beta;
    a.s0 = initial_state; a.cu = cu_seqlens; a.out = nullptr; a.s_final = nullptr;
    a.check = reinterpret_cast<uint32_t*>(ws);
    a.G = reinterpret_cast<float*>(ws + L.g_off);
    a.W = reinterpret_cast<float*>(ws + L.w_off);
    a.Ut = reinterpret_cast<float*>(ws + L.ut_off);
    a.T_tot = p.total_tokens; a.N = p.num_seqs; a.H = p.num_heads; a.dk = p.d_k; a.dv = p.d_v;
    a.max_seqlen = equal ? (int32_t)(p.total_tokens / p.num_seqs) : p.max_seqlen;
    a.chunks_per_seq = (int32_t)cps;
    a.g_min = p.g_min;
    a.max_seg = 1;
    a.handoff_tries = kda::kHandoffTries;
    b.dout = d_out; b.dS_final = d_final_state;
    b.dq = dq; b.dk = dk; b.dv = dv; b.dz = dz; b.dA = dA; b.dbeta = dbeta; b.dS0 = d_initial_state;
    b.P = reinterpret_cast<float*>(ws + L.p_off);
    b.QG = reinterpret_cast<float*>(ws + L.qg_off);
    b.Kt = reinterpret_cast<float*>(ws + L.kt_off);
    b.U = reinterpret_cast<float*>(ws + L.u_off);
    b.dU = reinterpret_cast<float*>(ws + L.du_off);
    b.S_chunk = reinterpret_cast<float*>(ws + L.s_off);
    b.dS_chunk = reinterpret_cast<float*>(ws + L.ds_off);
    b.dA_part = reinterpret_cast<float*>(ws + L.da_off);
    b.slots = (int64_t)L.slots;
    if (cudaMemsetAsync(a.check, 0, sizeof(uint32_t), s) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaMemsetAsync(b.dA_part, 0, L.slots * p.num_heads * sizeof(float), s) != cudaSuccess) return KDA_ERR_CUDA;
    const cudaError_t e = kda::launch_backward(b, p.io_dtype, s);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

size_t kda_forward_summary_workspace_bytes(const kda_problem_t* problem)
{
    if (check_descriptor(problem, Call::Forward) != KDA_OK) return 0;
    return kda::summary_layout(*problem).total;
}

kda_status_t kda_forward_summary(const void* q, const void* k, const void* v, const void* z, const float* A,
                                 const float* beta, const int32_t* cu_seqlens, float* transition, float* state_from_zero,
                                 const kda_problem_t* problem, void* workspace, size_t workspace_bytes, void* stream)
{
    kda_status_t st = check_descriptor(problem, Call::Forward);
    if (st != KDA_OK) return st;
    const kda_problem_t& p = *problem;
    if (transition == nullptr || state_from_zero == nullptr) return KDA_ERR_INVALID_ARG;
    if (!aligned(transition, 16) || !aligned(state_from_zero, 16)) return KDA_ERR_INVALID_ARG;
    const kda::SummaryLayout L = kda::summary_layout(p);
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < L.total) return KDA_ERR_WORKSPACE;
    const size_t io = io_size(p.io_dtype);
    const size_t tk = (size_t)p.total_tokens * p.num_heads * p.d_k;
    const size_t tv = (size_t)p.total_tokens * p.num_heads * p.d_v;
    const size_t units = (size_t)p.num_seqs * p.num_heads;
    const Range rm = range_of(transition, units * p.d_k * p.d_k * sizeof(float));
    const Range rs = range_of(state_from_zero, units * p.d_k * p.d_v * sizeof(float));
    const Range ins[7] = {range_of(q, tk * io), range_of(k, tk * io), range_of(z, tk * io), range_of(v, tv * io),
                          range_of(A, p.num_heads * sizeof(float)),
                          range_of(beta, (size_t)p.total_tokens * p.num_heads * sizeof(float)),
                          range_of(cu_seqlens, cu_seqlens ? (size_t)(p.num_seqs + 1) * sizeof(int32_t) : 0)};
    const Range rw = range_of(workspace, L.total);
    for (const Range& r : ins) {
        if (overlaps(rm, r) || overlaps(rs, r) || overlaps(rw, r)) return KDA_ERR_INVALID_ARG;
    }
    if (overlaps(rm, rs) || overlaps(rw, rm) || overlaps(rw, rs)) return KDA_ERR_INVALID_ARG;
    if ((st = check_device_pointer(workspace)) != KDA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    void* zeros = ws + L.zeros_off;
    float* eye = reinterpret_cast<float*>(ws + L.eye_off);
    void* out = ws + L.out_off;
    // S~: the range from a zero state
    st = kda_forward(q, k, v, z, A, beta, nullptr, cu_seqlens, out, state_from_zero, problem, ws, L.fwd_bytes, stream);
    if (st != KDA_OK) return st;
    // M: the range from the identity with every value zero (the columns of M evolve like state columns)
    if (p.total_tokens > 0 && cudaMemsetAsync(zeros, 0, tk * io, s) != cudaSuccess) return KDA_ERR_CUDA;
    if (kda::launch_identity_states(eye, (int64_t)units, p.d_k, s) != cudaSuccess) return KDA_ERR_CUDA;
    return kda_forward(q, k, zeros, z, A, beta, eye, cu_seqlens, out, transition, &L.pm, ws, L.fwd_bytes, stream);
}

kda_status_t kda_state_scan(const float* transition, const float* state_from_zero, const float* initial_state,
                            int32_t count, float* state_out, const kda_problem_t* problem, void* stream)
{
    kda_status_t st = check_descriptor(problem, Call::Forward);
    if (st != KDA_OK) return st;
    const kda_problem_t& p = *problem;
    if (count < 0 || state_out == nullptr) return KDA_ERR_INVALID_ARG;
    if (count > 0 && (transition == nullptr || state_from_zero == nullptr)) return KDA_ERR_INVALID_ARG;
    for (const void* ptr : {(const void*)transition, (const void*)state_from_zero, (const void*)initial_state,
                            (const void*)state_out}) {
        if (!aligned(ptr, 16)) return KDA_ERR_INVALID_ARG;
    }
    if ((int64_t)p.num_seqs * p.num_heads > 2147483647LL) return KDA_ERR_UNSUPPORTED;
    const size_t units = (size_t)p.num_seqs * p.num_heads;
    const Range rm = range_of(transition, (size_t)count * units * p.d_k * p.d_k * sizeof(float));
    const Range rt = range_of(state_from_zero, (size_t)count * units * p.d_k * p.d_v * sizeof(float));
    const Range ri = range_of(initial_state, units * p.d_k * p.d_v * sizeof(float));
    const Range ro = range_of(state_out, units * p.d_k * p.d_v * sizeof(float));
    if (overlaps(ro, rm) || overlaps(ro, rt)) return KDA_ERR_INVALID_ARG;
    // in place (state_out == initial_state) is allowed: every CTA reads its slice before writing it
    if (state_out != initial_state && overlaps(ro, ri)) return KDA_ERR_INVALID_ARG;
    for (const void* ptr : {(const void*)transition, (const void*)state_from_zero, (const void*)initial_state,
                            (const void*)state_out}) {
        if ((st = check_device_pointer(ptr)) != KDA_OK) return st;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kda::prof_start("kda_state_scan", s);
    const cudaError_t e = kda::launch_state_scan(transition, state_from_zero, initial_state, state_out, p.num_seqs,
                                                 p.num_heads, p.d_k, p.d_v, count, s);
    kda::prof_stop(s);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_decode_step(const void* q, const void* k, const void* v, const void* z, const float* A,
                             const float* beta, float* state, void* out, const kda_problem_t* problem,
                             void* stream)
{
    kda_status_t st = check_descriptor(problem, Call::Decode);
    if (st != KDA_OK) return st;
    const kda_problem_t& p = *problem;
    if (!q || !k || !v || !z || !A || !beta || !state || !out) return KDA_ERR_INVALID_ARG;
    for (const void* ptr : {q, k, v, z, (const void*)state, (const void*)out}) {
        if (!aligned(ptr, 16)) return KDA_ERR_INVALID_ARG;
    }
    if (!aligned(A, 4) || !aligned(beta, 4)) return KDA_ERR_INVALID_ARG;
    if ((int64_t)p.num_seqs * p.num_heads > 2147483647LL) return KDA_ERR_UNSUPPORTED;
    const size_t io = io_size(p.io_dtype);
    const size_t nh = (size_t)p.num_seqs * p.num_heads;
    const Range rq = range_of(q, nh * p.d_k * io), rk = range_of(k, nh * p.d_k * io);
    const Range rz = range_of(z, nh * p.d_k * io), rv = range_of(v, nh * p.d_v * io);
    const Range ra = range_of(A, p.num_heads * sizeof(float)), rb = range_of(beta, nh * sizeof(float));
    const Range rs = range_of(state, nh * p.d_k * p.d_v * sizeof(float));
    const Range ro = range_of(out, nh * p.d_v * io);
    for (Range r : {rq, rk, rz, rv, ra, rb, rs}) {
        if (overlaps(ro, r)) return KDA_ERR_INVALID_ARG;
    }
    for (Range r : {rq, rk, rz, rv, ra, rb}) {
        if (overlaps(rs, r)) return KDA_ERR_INVALID_ARG;
    }
    for (const void* ptr : {q, k, v, z, (const void*)A, (const void*)beta, (const void*)state, (const void*)out}) {
        st = check_device_pointer(ptr);
        if (st != KDA_OK) return st;
    }
    kda::DecodeArgs a{};
    a.q = q; a.k = k; a.v = v; a.z = z; a.A = A; a.beta = beta; a.state = state; a.out = out;
    a.N = p.num_seqs; a.H = p.num_heads; a.g_min = p.g_min;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kda::prof_start("kda_decode_step", s);
    const cudaError_t e = kda::launch_decode(a, p.d_k, p.d_v, p.io_dtype, s);
    kda::prof_stop(s);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_decode_replay(const void* q, const void* k, const void* v, const void* z, const float* A,
                               const float* beta, const float* state_in, const int32_t* accepted, float* state_out,
                               void* out, const kda_problem_t* problem, void* stream)
{
    kda_status_t st = check_descriptor(problem, Call::Replay);
    if (st != KDA_OK) return st;
    const kda_problem_t& p = *problem;
    if (!q || !k || !v || !z || !A || !beta || !state_in) return KDA_ERR_INVALID_ARG;
    if (!out && !state_out) return KDA_ERR_INVALID_ARG;
    for (const void* ptr : {q, k, v, z, (const void*)state_in, (const void*)state_out, (const void*)out}) {
        if (!aligned(ptr, 16)) return KDA_ERR_INVALID_ARG;
    }
    if (!aligned(A, 4) || !aligned(beta, 4) || !aligned(accepted, 4)) return KDA_ERR_INVALID_ARG;
    if ((int64_t)p.num_seqs * p.num_heads > 2147483647LL) return KDA_ERR_UNSUPPORTED;
    const size_t io = io_size(p.io_dtype);
    const size_t th = (size_t)p.total_tokens * p.num_heads;
    const size_t nh = (size_t)p.num_seqs * p.num_heads;
    const Range rq = range_of(q, th * p.d_k * io), rk = range_of(k, th * p.d_k * io);
    const Range rz = range_of(z, th * p.d_k * io), rv = range_of(v, th * p.d_v * io);
    const Range ra = range_of(A, p.num_heads * sizeof(float)), rb = range_of(beta, th * sizeof(float));
    const Range racc = range_of(accepted, (size_t)p.num_seqs * sizeof(int32_t));
    const Range rsi = range_of(state_in, nh * p.d_k * p.d_v * sizeof(float));
    const Range rso = range_of(state_out, nh * p.d_k * p.d_v * sizeof(float));
    const Range ro = range_of(out, th * p.d_v * io);
    for (Range r : {rq, rk, rz, rv, ra, rb, racc, rsi, rso}) {
        if (overlaps(ro, r)) return KDA_ERR_INVALID_ARG;
    }
    for (Range r : {rq, rk, rz, rv, ra, rb, racc}) {
        if (overlaps(rso, r)) return KDA_ERR_INVALID_ARG;
    }
    // state_out may be state_in itself (each CTA reads its whole state before writing it), nothing else
    if (state_out != state_in && overlaps(rso, rsi)) return KDA_ERR_INVALID_ARG;
    for (const void* ptr : {q, k, v, z, (const void*)A, (const void*)beta, (const void*)state_in,
                            (const void*)accepted, (const void*)state_out, (const void*)out}) {
        st = check_device_pointer(ptr);
        if (st != KDA_OK) return st;
    }
    kda::ReplayArgs a{};
    a.q = q; a.k = k; a.v = v; a.z = z; a.A = A; a.beta = beta;
    a.state_in = state_in; a.accepted = accepted; a.state_out = state_out; a.out = out;
    a.N = p.num_seqs; a.H = p.num_heads; a.L = (int32_t)(p.total_tokens / p.num_seqs); a.g_min = p.g_min;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kda::prof_start("kda_decode_replay", s);
    const cudaError_t e = kda::launch_replay(a, p.d_k, p.d_v, p.io_dtype, s);
    kda::prof_stop(s);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_prologue(const void* xq, const void* xk, const void* xv, const float* wq, const float* wk,
                          const float* wv, int32_t conv_width, const int32_t* cu_seqlens, void* q, void* k, void* v,
                          const kda_problem_t* problem, void* stream)
{
    kda_status_t st = check_descriptor(problem, Call::Forward);
    if (st != KDA_OK) return st;
    const kda_problem_t& p = *problem;
    if (conv_width < 1 || conv_width > kda::kMaxConv) return KDA_ERR_UNSUPPORTED;
    if (!xq || !xk || !xv || !wq || !wk || !wv || !q || !k || !v) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr && p.total_tokens % p.num_seqs != 0) return KDA_ERR_INVALID_ARG;
    for (const void* ptr : {xq, xk, xv, (const void*)q, (const void*)k, (const void*)v}) {
        if (!aligned(ptr, 16)) return KDA_ERR_INVALID_ARG;
    }
    for (const void* ptr : {(const void*)wq, (const void*)wk, (const void*)wv, (const void*)cu_seqlens}) {
        if (!aligned(ptr, 4)) return KDA_ERR_INVALID_ARG;
    }
    const size_t io = io_size(p.io_dtype);
    const size_t th = (size_t)p.total_tokens * p.num_heads;
    const Range in[7] = {range_of(xq, th * p.d_k * io), range_of(xk, th * p.d_k * io), range_of(xv, th * p.d_v * io),
                         range_of(wq, (size_t)p.num_heads * p.d_k * conv_width * 4),
                         range_of(wk, (size_t)p.num_heads * p.d_k * conv_width * 4),
                         range_of(wv, (size_t)p.num_heads * p.d_v * conv_width * 4),
                         range_of(cu_seqlens, ((size_t)p.num_seqs + 1) * 4)};
    const Range out[3] = {range_of(q, th * p.d_k * io), range_of(k, th * p.d_k * io), range_of(v, th * p.d_v * io)};
    for (int i = 0; i < 3; ++i) {
        for (const Range& r : in) {
            if (overlaps(out[i], r)) return KDA_ERR_INVALID_ARG;
        }
        for (int j = 0; j < i; ++j) {
            if (overlaps(out[i], out[j])) return KDA_ERR_INVALID_ARG;
        }
    }
    for (const void* ptr : {xq, xk, xv, (const void*)wq, (const void*)wk, (const void*)wv, (const void*)cu_seqlens,
                            (const void*)q, (const void*)k, (const void*)v}) {
        st = check_device_pointer(ptr);
        if (st != KDA_OK) return st;
    }
    kda::PrologueArgs a{};
    a.x[0] = xq; a.x[1] = xk; a.x[2] = xv;
    a.w[0] = wq; a.w[1] = wk; a.w[2] = wv;
    a.y[0] = q; a.y[1] = k; a.y[2] = v;
    a.cu = cu_seqlens;
    a.T = p.total_tokens; a.N = p.num_seqs; a.H = p.num_heads; a.dk = p.d_k; a.dv = p.d_v; a.K = conv_width;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kda::prof_start("kda_prologue", s);
    const cudaError_t e = kda::launch_prologue(a, p.io_dtype, s);
    kda::prof_stop(s);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_epilogue(const void* o, const void* gate, const float* weight, float eps, void* y,
                          const kda_problem_t* problem, void* stream)
{
    kda_status_t st = check_descriptor(problem, Call::Forward);
    if (st != KDA_OK) return st;
    const kda_problem_t& p = *problem;
    if (!o || !gate || !weight || !y) return KDA_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return KDA_ERR_INVALID_ARG;
    for (const void* ptr : {o, gate, (const void*)y}) {
        if (!aligned(ptr, 16)) return KDA_ERR_INVALID_ARG;
    }
    if (!aligned(weight, 4)) return KDA_ERR_INVALID_ARG;
    const size_t io = io_size(p.io_dtype);
    const size_t bytes = (size_t)p.total_tokens * p.num_heads * p.d_v * io;
    const Range ro = range_of(o, bytes), rg = range_of(gate, bytes), rw = range_of(weight, (size_t)p.d_v * 4);
    const Range ry = range_of(y, bytes);
    if (overlaps(ry, rg) || overlaps(ry, rw)) return KDA_ERR_INVALID_ARG;
    if (y != o && overlaps(ry, ro)) return KDA_ERR_INVALID_ARG;  // in place, or apart
    for (const void* ptr : {o, gate, (const void*)weight, (const void*)y}) {
        st = check_device_pointer(ptr);
        if (st != KDA_OK) return st;
    }
    kda::EpilogueArgs a{};
    a.o = o; a.gate = gate; a.weight = weight; a.y = y;
    a.rows = p.total_tokens * p.num_heads; a.eps = eps;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kda::prof_start("kda_epilogue", s);
    const cudaError_t e = kda::launch_epilogue(a, p.d_v, p.io_dtype, s);
    kda::prof_stop(s);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_workspace_status(const void* workspace, size_t workspace_bytes, void* stream)
{
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < 256) return KDA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return KDA_ERR_CUDA;
    if (word & kda::kCheckTimeout) return KDA_ERR_TIMEOUT;
    if (word & kda::kCheckBadSeqlens) return KDA_ERR_DEVICE_CHECK;
    return KDA_OK;
}

}  // extern "C"
