// k6_noalloc.cu -- a forward pass for callers that cannot allocate device
// memory.
//
// k6attn_forward needs caller-provided scratch (the rotated q/k copies and,
// with several K/V chunks, the per-chunk partial outputs).  Some callers have
// no way to provide it: a plugin inside a host framework that owns every
// device allocation and forbids its guests from calling cudaMalloc, a
// deployment held to a fixed memory budget set at start-up, or a binding that
// only sees tensors handed to it.  For them this file holds the scratch
// itself, in one statically sized device array that every GPU loading the
// library reserves until the process exits, so the entry point below never
// allocates.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "k6attn.h"
#include "k6_internal.h"

namespace k6 {

// The scratch shared by every call of k6attn_forward_static_scratch on a
// device.  In host code this name is only a stand-in for the device symbol;
// its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[K6ATTN_STATIC_SCRATCH_BYTES];

namespace {
struct ScratchAddr {
    unsigned long long ctx;  // unique id of the CUDA context the address belongs to
    void *ptr;
};
std::mutex g_scratch_mu;
std::vector<ScratchAddr> g_scratch_addr;  // one entry per context that has made a call
}  // namespace

// Set-up, once per CUDA context, with that context current: look up the device
// address of the static array.  Allocates nothing.  The address is cached per
// context, not per device ordinal: cudaDeviceReset replaces a device's primary
// context, the module (and the array) is loaded anew in the next one, and the
// old address would be stale there.
static k6attn_status static_scratch_address(void **out) {
    unsigned long long id = current_context_id();
    if (id) {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        for (const ScratchAddr &e : g_scratch_addr)
            if (e.ctx == id) {
                *out = e.ptr;
                return K6ATTN_OK;
            }
    }
    void *p = nullptr;
    k6attn_status s = cuda_check(cudaGetSymbolAddress(&p, g_static_scratch), "forward_static_scratch: scratch address");
    if (s != K6ATTN_OK) return s;
    id = current_context_id();  // the lookup above made the device's context current if none was
    if (id) {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        g_scratch_addr.push_back({id, p});
    }
    *out = p;
    return K6ATTN_OK;
}

}  // namespace k6

extern "C" k6attn_status k6attn_forward_static_scratch(k6attn_t h, const void *q, const void *k, const void *v,
                                                       const void *joint_k, const void *joint_v,
                                                       const void *rope_tables, int n_chunks, void *out, float *lse,
                                                       void *stream) {
    using namespace k6;
    k6attn_status hs = check_handle("forward_static_scratch", h);
    if (hs != K6ATTN_OK) return hs;
    if (n_chunks < 1) return set_error(K6ATTN_ERR_INVALID_ARG, "forward_static_scratch: n_chunks must be >= 1");
    const size_t need = k6attn_workspace_bytes(h, n_chunks, rope_tables != nullptr);
    if (need > (size_t)K6ATTN_STATIC_SCRATCH_BYTES)
        return set_error(K6ATTN_ERR_WORKSPACE,
                         "forward_static_scratch: this problem needs %zu bytes of scratch, the static array holds "
                         "%zu; use k6attn_forward with a caller workspace",
                         need, (size_t)K6ATTN_STATIC_SCRATCH_BYTES);
    void *scratch = nullptr;
    if (need) {
        k6attn_status s = static_scratch_address(&scratch);
        if (s != K6ATTN_OK) return s;
    }
    // Every byte of scratch the forward pass reads it has written first in the
    // same call (rotated copies, then partials, then the merge), so nothing
    // needs clearing between calls.
    return k6attn_forward(h, q, k, v, joint_k, joint_v, rope_tables, n_chunks, out, lse, scratch, need, stream);
}
