// kvc_noalloc.cu -- kvc_decode_noalloc: split-K paged decode whose partials live in scratch
// memory owned by this library, for callers that cannot allocate device memory (they are
// given only input and output buffers, or may not call cudaMalloc while serving).
//
// The scratch is one file-scope device array.  In host code its name is only a host-side
// stand-in, so the device address is looked up with cudaGetSymbolAddress once per device
// (with that device current) and that address is what the kernels receive.
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
void *g_scratch_address[kMaxDevices];   // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device (looked up on first use).
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
    if (g_scratch_address[device] == nullptr) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess || p == nullptr) {
            char msg[256];
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the scratch array: %s",
                     cudaGetErrorString(err));
            return static_cast<kvc_status>(kvc::set_last_error(KVC_ERR_CUDA, msg));
        }
        g_scratch_address[device] = p;
    }
    *address = g_scratch_address[device];
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
