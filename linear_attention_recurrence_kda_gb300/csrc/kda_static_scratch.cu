// kda_static_scratch.cu -- kda_forward for callers that cannot allocate device memory.
//
// The scratch lives in one file-scope device array (KDA_STATIC_SCRATCH_BYTES, 256-byte aligned)
// that every device loading the library holds for the life of the process.  Host code cannot use
// the array's name as a device address, so the address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached.  The entry point allocates nothing:
// it checks the problem's scratch requirement against the array's size and hands the array to
// kda_forward as its workspace.
#include <mutex>

#include "kda_internal.cuh"

static __device__ __align__(256) unsigned char g_kda_static_scratch[KDA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's copy of the scratch array (looked up on first use).
kda_status_t scratch_for_current_device(void** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kda_static_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return KDA_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
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
    const kda_status_t st = scratch_for_current_device(&scratch);
    if (st != KDA_OK) return st;
    return kda_forward(q, k, v, z, A, beta, initial_state, cu_seqlens, out, final_state, problem, scratch,
                       KDA_STATIC_SCRATCH_BYTES, stream);
}
