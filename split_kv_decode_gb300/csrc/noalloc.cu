// decode_attn_splitk_noalloc: the split-KV decode for callers that cannot
// allocate device memory.
//
// The partials (the only scratch the split and combine kernels need) live in
// a fixed-size array inside this library instead of a caller workspace, so a
// call allocates nothing. Every GPU that loads the library reserves the array
// until the process exits.
#include <cstdio>
#include <mutex>

#include "internal.h"

namespace skv {
int set_error(int code, const char *phase, const char *msg); // api.cpp
}

namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20; // 16 MiB

// Shared by every decode_attn_splitk_noalloc call on a device; it keeps the
// last call's contents (the kernels need none of it zeroed: the split kernel
// resets the status word itself and overwrites every partial it reads back).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices]; // device address per ordinal, set up once

// The array's name in host code is only a host-side stand-in; the device
// address comes from cudaGetSymbolAddress with the device current.
int scratch_for_current_device(void **addr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return skv::set_error(DA_ECUDA, "noalloc", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return skv::set_error(DA_EUNSUPPORTED, "noalloc", "device ordinal beyond 63");
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            char msg[256];
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static scratch failed: %s",
                     cudaGetErrorString(e));
            return skv::set_error(DA_ECUDA, "noalloc", msg);
        }
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return DA_OK;
}

} // namespace

extern "C" int decode_attn_splitk_noalloc(const da_args_t *args, const da_plan_t *plan,
                                          const float *q, const void *k_cache,
                                          const void *v_cache, void *out, da_stream_t stream)
{
    if (!args || !plan) return skv::set_error(DA_EINVAL, "args", "args or plan is NULL");
    // the partials stay in the library's private array, so a split-only call
    // would hand the caller nothing: refuse it instead of returning DA_OK
    if (args->flags & DA_FLAG_NO_COMBINE)
        return skv::set_error(DA_EINVAL, "noalloc",
                              "DA_FLAG_NO_COMBINE is refused here: the partials live in the "
                              "library's private array and could not be combined later");
    if (plan->workspace_bytes < 0 || (size_t)plan->workspace_bytes > kNoallocScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "this plan needs %lld bytes of partials; the static scratch holds %zu bytes "
                 "(use decode_attn_splitk_ex with a caller workspace)",
                 (long long)plan->workspace_bytes, kNoallocScratchBytes);
        return skv::set_error(DA_ENOSPACE, "noalloc", msg);
    }
    void *ws = nullptr;
    int rc = scratch_for_current_device(&ws);
    if (rc) return rc;
    return decode_attn_splitk_ex(args, plan, q, k_cache, v_cache, out, ws, kNoallocScratchBytes,
                                 stream);
}
