// kda_static_scratch.cu -- kda_forward for callers that cannot allocate device memory.
//
// The scratch lives in one file-scope device array (KDA_STATIC_SCRATCH_BYTES, 256-byte aligned)
// that every device loading the library holds for the life of the process.  Host code cannot use
// the array's name as a device address, so every call looks the address up with
// cudaGetSymbolAddress in the caller's current context (the lookup allocates nothing; on a
// context's first call it loads the library's module there).  Looking it up each time, rather than
// caching it per device, keeps the address right after cudaDeviceReset or when the caller switches
// between contexts of one device, where the module -- and the array -- is loaded again elsewhere.
// The entry point allocates nothing: it checks the problem's scratch requirement against the
// array's size and hands the array to kda_forward as its workspace.
#include "kda_internal.cuh"

static __device__ __align__(256) unsigned char g_kda_static_scratch[KDA_STATIC_SCRATCH_BYTES];

namespace {

// Device address of the scratch array in the current context.
kda_status_t scratch_for_current_context(void** out)
{
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kda_static_scratch) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    *out = p;
    return KDA_OK;
}

}  // namespace

extern "C" kda_status_t kda_forward_static_scratch(const void* q, const void* k, const void* v, const void* z,
                                                   const float* A, const float* beta, const float* initial_state,
                                                   const int32_t* cu_seqlens, void* out, float* final_state,
                                                   const kda_problem_t* problem, void* stream)
{
    if (problem == nullptr) return KDA_ERR_INVALID_ARG;
    // the smallest workspace kda_forward can run with (it uses fewer sequence segments, or none,
    // when the scratch is smaller than the fastest plan wants)
    if (kda_forward_workspace_bytes(problem) == 0) return KDA_ERR_INVALID_ARG;
    if (kda::forward_layout(*problem, 0).total > KDA_STATIC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;
    void* scratch = nullptr;
    const kda_status_t st = scratch_for_current_context(&scratch);
    if (st != KDA_OK) return st;
    return kda_forward(q, k, v, z, A, beta, initial_state, cu_seqlens, out, final_state, problem, scratch,
                       KDA_STATIC_SCRATCH_BYTES, stream);
}

extern "C" kda_status_t kda_static_scratch_status(void* stream)
{
    void* scratch = nullptr;
    const kda_status_t st = scratch_for_current_context(&scratch);
    if (st != KDA_OK) return st;
    return kda_workspace_status(scratch, KDA_STATIC_SCRATCH_BYTES, stream);
}
