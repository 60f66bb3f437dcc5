// kvc_noalloc.cu -- kvc_decode_noalloc: split-K paged decode whose partials live in scratch
// memory owned by this library, for callers that cannot allocate device memory (they are
// given only input and output buffers, or may not call cudaMalloc while serving).
//
// The scratch is one file-scope device array.  In host code its name is only a host-side
// stand-in, so the device address is looked up with cudaGetSymbolAddress once per device
// (with that device current) and that address is what the kernels receive.  The address
// belongs to the device's current context: it is kept together with that context's id
// (unique for the life of the process), and looked up again when a device reset has replaced
// the context, since the array may then live elsewhere.
#include <cudaTypedefs.h>
#include <stdio.h>

#include <mutex>

#include "kvc.h"
#include "kvc_launch.h"

namespace {

constexpr size_t kScratchBytes = KVC_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Split partials of kvc_decode_noalloc; shared by every call on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
struct ScratchSlot {
    unsigned long long context_id;   // id of the context the address was looked up in
    void *address;                   // device address of g_noalloc_scratch there
};
ScratchSlot g_scratch[kMaxDevices];

// Id of the calling thread's current context (0 if the driver cannot say): the driver's own
// entry points, fetched once through the runtime.
unsigned long long current_context_id()
{
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS ||
        ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array on the current device (looked up on first use, and
// again once the device's context has been replaced).
kvc_status scratch_on_current_device(void **address)
{
    int device = 0;
    cudaError_t err = cudaGetDevice(&device);
    if (err != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "cudaGetDevice: %s", cudaGetErrorString(err));
        return static_cast<kvc_status>(kvc::set_last_error(KVC_ERR_CUDA, msg));
    }
    if (device < 0 || device >= kMaxDevices)
        return static_cast<kvc_status>(
            kvc::set_last_error(KVC_ERR_UNSUPPORTED, "device index beyond 63"));
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    ScratchSlot &slot = g_scratch[device];
    if (slot.address == nullptr || slot.context_id == 0 ||
        slot.context_id != current_context_id()) {
        // cudaGetSymbolAddress also makes the device's context current if it is not yet, so
        // the context id is read after it
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess || p == nullptr) {
            char msg[256];
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the scratch array: %s",
                     cudaGetErrorString(err));
            return static_cast<kvc_status>(kvc::set_last_error(KVC_ERR_CUDA, msg));
        }
        slot.address = p;
        slot.context_id = current_context_id();
    }
    *address = slot.address;
    return KVC_OK;
}

}  // namespace

extern "C" kvc_status kvc_decode_noalloc(void *out, int32_t out_dtype, const void *q,
                                         const void *k_pool, const void *v_pool,
                                         kvc_pool_desc pool, const int32_t *block_table,
                                         int32_t bt_stride, const int32_t *context_lens,
                                         int32_t num_seqs, int32_t max_ctx, int32_t q_heads,
                                         float scale, int32_t num_splits, void *stream)
{
    int32_t splits = 0;
    size_t needed = 0;
    kvc_status st = kvc_decode_plan(num_seqs, q_heads, pool, max_ctx, num_splits, &splits,
                                    nullptr, &needed);
    if (st != KVC_OK)
        return st;
    if (needed > kScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "kvc_decode_noalloc: %d splits need %zu bytes of partials, more than the "
                 "library's %zu-byte scratch; ask for fewer splits or use kvc_decode",
                 splits, needed, kScratchBytes);
        return static_cast<kvc_status>(kvc::set_last_error(KVC_ERR_WORKSPACE, msg));
    }
    void *scratch = nullptr;
    if ((st = scratch_on_current_device(&scratch)) != KVC_OK)
        return st;
    return kvc_decode(out, out_dtype, q, k_pool, v_pool, pool, block_table, bt_stride,
                      context_lens, num_seqs, max_ctx, q_heads, scale, num_splits, scratch,
                      kScratchBytes, stream);
}
