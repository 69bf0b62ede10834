// status.cu -- status strings and the launch counter of libpagedkv.
#include <nvtx3/nvToolsExt.h>

#include <atomic>

#include "pkv_common.cuh"

namespace pkv {
static std::atomic<unsigned long long> g_launches{0};
void note_launches(int n) { g_launches.fetch_add(static_cast<unsigned long long>(n)); }

constexpr unsigned long long kDefaultWaitLimitNs = 1000000000ull;
static std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};
unsigned long long wait_limit_ns() { return g_wait_limit_ns.load(); }

static nvtxDomainHandle_t nvtx_domain() {
    static nvtxDomainHandle_t d = nvtxDomainCreateA("pagedkv");
    return d;
}
CallRange::CallRange(const char *name) {
    nvtxEventAttributes_t a = {};
    a.version = NVTX_VERSION;
    a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    a.messageType = NVTX_MESSAGE_TYPE_ASCII;
    a.message.ascii = name;
    nvtxDomainRangePushEx(nvtx_domain(), &a);
}
CallRange::~CallRange() { nvtxDomainRangePop(nvtx_domain()); }
}  // namespace pkv

extern "C" unsigned long long pkv_set_wait_limit_ns(unsigned long long ns) {
    return pkv::g_wait_limit_ns.exchange(ns ? ns : pkv::kDefaultWaitLimitNs);
}

extern "C" const char *pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_NULL: return "a required pointer is NULL";
        case PKV_ERR_INVALID_ARG: return "invalid argument (enum, size, head ratio or alignment)";
        case PKV_ERR_UNSUPPORTED: return "unsupported configuration (head dim, page size or group)";
        case PKV_ERR_WORKSPACE: return "workspace too small";
        case PKV_ERR_CUDA: return "CUDA launch failed";
        default: return "unknown status";
    }
}

extern "C" unsigned long long pkv_kernel_launches(void) { return pkv::g_launches.load(); }

extern "C" int pkv_debug_bounds(void) { return pkv::kDebugBounds ? 1 : 0; }

// ---- tensor-map encoding through the driver entry point (no libcuda link) ----
#include <mutex>

#include "sm103_ptx.cuh"

namespace pkv {

static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool encode_tmap(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int rank,
                 const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box) {
    auto fn = tmap_encoder();
    if (!fn) return false;
    cuuint64_t gdim[5], gstride[4];
    cuuint32_t bdim[5], estride[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estride[i] = 1;
        if (i < rank - 1) gstride[i] = strides_bytes[i];
    }
    CUresult r = fn(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void *>(base), gdim, gstride,
                    bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace pkv
