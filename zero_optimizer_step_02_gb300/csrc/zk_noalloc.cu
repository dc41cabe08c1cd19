// zk_noalloc.cu -- zero_step_fused_noalloc: the fused step for callers that
// cannot allocate a workspace.  The workspace becomes one scratch array that
// lives in this library (file scope, __device__), so the call allocates
// nothing.  Contract and limits: include/zero.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "zero.h"

namespace {

constexpr size_t kScratchBytes = ZERO_NOALLOC_SCRATCH_BYTES;

// The scratch: per-CTA partial sums first (32 KB), then the fp32 reduced
// gradient of a clipped step.  Host code must not pass this name to a kernel
// (on the host it is a stand-in, not a device address); it uses the address
// looked up below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// The scratch's device address belongs to the context the library's module
// was loaded into: a device reset (cudaDeviceReset, or the primary context
// destroyed and made again) loads the module anew and may move it.  So the
// address is kept per device together with the id of the context it was
// looked up in (context ids are never reused within a process), and looked
// up again when the current context is another one.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct DriverFns {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver_fns()
{
    static DriverFns fns;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fns.get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fns.get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    return fns;
}

// id of the calling thread's current context; 0 when there is none (or the
// driver cannot say)
unsigned long long current_context_id()
{
    const DriverFns& d = driver_fns();
    if (d.get_current == nullptr || d.get_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    if (d.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    unsigned long long id = 0;
    if (d.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

constexpr int kMaxDevices = 64;
struct ScratchEntry {
    unsigned long long ctx_id;  // context the address was looked up in (0: none yet)
    void* addr;
};
ScratchEntry g_entry[kMaxDevices];
std::mutex g_entry_mutex;

// Device address of g_scratch on the current device, looked up once per
// device and context (with that device current).
zero_status scratch_address(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ZERO_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ZERO_ERR_BOUNDS;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_entry_mutex);
    ScratchEntry& e = g_entry[dev];
    if (e.addr == nullptr || ctx == 0 || ctx != e.ctx_id) {
        void* p = nullptr;
        const cudaError_t err = cudaGetSymbolAddress(&p, g_scratch);
        if (err != cudaSuccess || p == nullptr) return ZERO_ERR_CUDA;
        e.addr = p;
        // the lookup makes the device's primary context current if it was not
        e.ctx_id = ctx != 0 ? ctx : current_context_id();
    }
    *out = e.addr;
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
