// status.cu -- status strings and the launch counter of libpagedkv.
#include <atomic>

#include "pkv_common.cuh"

namespace pkv {
static std::atomic<unsigned long long> g_launches{0};
void note_launches(int n) { g_launches.fetch_add(static_cast<unsigned long long>(n)); }
}  // namespace pkv

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
