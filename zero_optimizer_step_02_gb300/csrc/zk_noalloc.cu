// zk_noalloc.cu -- zero_step_fused_noalloc: the fused step for callers that
// cannot allocate a workspace.  The workspace becomes one scratch array that
// lives in this library (file scope, __device__), so the call allocates
// nothing.  Contract and limits: include/zero.h.
#include <cuda_runtime.h>

#include "zero.h"

namespace {

constexpr size_t kScratchBytes = ZERO_NOALLOC_SCRATCH_BYTES;

// The scratch: per-CTA partial sums first (32 KB), then the fp32 reduced
// gradient of a clipped step.  Host code must not pass this name to a kernel
// (on the host it is a stand-in, not a device address); it uses the address
// looked up below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
int g_scratch_ready[kMaxDevices];

// Device address of g_scratch on the current device, looked up once per
// device (the first call on a device does it with that device current).
zero_status scratch_address(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ZERO_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ZERO_ERR_BOUNDS;
    if (!__atomic_load_n(&g_scratch_ready[dev], __ATOMIC_ACQUIRE)) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess || p == nullptr) return ZERO_ERR_CUDA;
        g_scratch_addr[dev] = p;
        __atomic_store_n(&g_scratch_ready[dev], 1, __ATOMIC_RELEASE);
    }
    *out = g_scratch_addr[dev];
    return ZERO_OK;
}

}  // namespace

extern "C" ZERO_API zero_status zero_step_fused_noalloc(const zero_plan* plan, const zero_hparams* hp,
                                                        const void* const* rank_grads, const float* master_in,
                                                        const float* m_in, const float* v_in, float* master_out,
                                                        float* m_out, float* v_out, void* lp_out,
                                                        zero_dev_scalars* scalars_dev, void* stream)
{
    if (plan == nullptr || hp == nullptr) return ZERO_ERR_INVALID_ARG;
    // refuse, before touching the device, what the fixed scratch cannot hold
    if (zero_workspace_bytes(plan, hp) > kScratchBytes) return ZERO_ERR_BOUNDS;
    void* ws = nullptr;
    const zero_status s = scratch_address(&ws);
    if (s != ZERO_OK) return s;
    return zero_step_fused(plan, hp, rank_grads, master_in, m_in, v_in, master_out, m_out, v_out, lp_out,
                           scalars_dev, ws, stream);
}
