// k6_host.cu -- host-side helpers shared by the tensor-core launchers: the
// driver entry points (tensor-map encoding, context identity), the tensor map
// over a BSHD tensor, and the per-context opt-in to large dynamic shared
// memory.
//
// Kernel attributes and module globals belong to a CUDA context, not to a
// process: a second device, or the same device after cudaDeviceReset, has a
// context of its own in which nothing has been set up yet.  So every cache
// here is keyed by the context's unique id (cuCtxGetId), never by a
// process-wide once-flag or by the device ordinal.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <utility>
#include <vector>

#include "k6_internal.h"

namespace k6 {

namespace {
struct DriverFns {
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    PFN_cuCtxGetCurrent_v4000 ctx_current = nullptr;
    PFN_cuCtxGetId_v12000 ctx_id = nullptr;
};

template <typename F>
F entry_point(const char *name, int version) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<F>(fn);
    return nullptr;
}

const DriverFns &driver() {
    static DriverFns f;
    static std::once_flag once;
    std::call_once(once, [] {
        f.encode = entry_point<PFN_cuTensorMapEncodeTiled_v12000>("cuTensorMapEncodeTiled", 12000);
        f.ctx_current = entry_point<PFN_cuCtxGetCurrent_v4000>("cuCtxGetCurrent", 4000);
        f.ctx_id = entry_point<PFN_cuCtxGetId_v12000>("cuCtxGetId", 12000);
    });
    return f;
}
}  // namespace

unsigned long long current_context_id() {
    const DriverFns &f = driver();
    if (!f.ctx_current || !f.ctx_id) return 0;
    CUcontext ctx = nullptr;
    if (f.ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (f.ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

bool make_bshd_map(CUtensorMap *m, const void *base, long rows, int H, int B, bool f16, const char **why,
                   int elem_bytes) {
    const DriverFns &f = driver();
    if (!f.encode) {
        if (why) *why = "cuTensorMapEncodeTiled is not available from the driver";
        return false;
    }
    constexpr int D = 128;
    const cuuint64_t eb = (cuuint64_t)elem_bytes;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)D * eb, (cuuint64_t)H * D * eb, (cuuint64_t)rows * H * D * eb};
    // one 128-byte row of the swizzle atom per box row: 64 2-byte or 128 1-byte elements
    cuuint32_t box[4] = {elem_bytes == 1 ? 128u : 64u, 1, 128, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType type = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                     : f16          ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (f.encode(m, type, 4,
                 const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
        if (why) *why = "cuTensorMapEncodeTiled rejected a tensor";
        return false;
    }
    return true;
}

cudaError_t set_max_dynamic_smem(const void *func, int bytes) {
    static std::mutex mu;
    static std::vector<std::pair<const void *, unsigned long long>> done;  // (kernel, context id) set up
    unsigned long long id = current_context_id();
    if (id) {
        std::lock_guard<std::mutex> lock(mu);
        for (const auto &e : done)
            if (e.first == func && e.second == id) return cudaSuccess;
    }
    cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    id = current_context_id();  // the call above made the device's context current if none was
    if (id) {
        std::lock_guard<std::mutex> lock(mu);
        done.emplace_back(func, id);
    }
    return cudaSuccess;
}

int chunk_group(const Geom &g, int n_chunks) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // CTAs per chunk and (batch, head): one per 128-row Q tile (the single-tile
    // kernel, which runs 16-bit q/k)
    const long q_units = (g.Sq + 127) / 128;
    const long units = (long)g.B * g.H * n_chunks * q_units;
    for (int gsz = 4; gsz > 1; gsz--)
        if (n_chunks % gsz == 0 && units / gsz >= 4L * sms) return gsz;
    return 1;
}

}  // namespace k6
