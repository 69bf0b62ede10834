// pkv_common.cuh -- device and host helpers shared by the library's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

// ---- host side -------------------------------------------------------------

// Count `n` kernel launches (diagnostics; see pkv_kernel_launches).
void note_launches(int n);

// Time limit of every bounded pipeline wait in kernels launched from now on
// (nanoseconds; see pkv_set_wait_limit_ns).
unsigned long long wait_limit_ns();

// Programmatic dependent launch between the kernels of one call: the second
// kernel is launched with programmatic stream serialisation, may start while
// the first finishes, and waits (griddepcontrol.wait) for the first grid's
// completion and memory before it reads what that grid wrote.  Both
// instructions are no-ops in a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
template <typename... Params, typename... Args>
static cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// An NVTX range named after one entry point, in the "pagedkv" domain, open
// for the whole call: a profiler's timeline nests the call's launches inside
// it, and ncu --nvtx can select them by it.  With no tool attached, the push
// and the pop are each a call through a no-op pointer.
class CallRange {
  public:
    explicit CallRange(const char *name);
    ~CallRange();
    CallRange(const CallRange &) = delete;
    CallRange &operator=(const CallRange &) = delete;
};

// PKV_OK if the launches just made succeeded, PKV_ERR_CUDA otherwise.
inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int ilog2_exact(int x) {  // -1 unless x is a power of two
    if (x <= 0 || (x & (x - 1))) return -1;
    int s = 0;
    while ((1 << s) < x) ++s;
    return s;
}

inline int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
    return n;
}

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---- device side -----------------------------------------------------------

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void set_err(int32_t *err, int bits) {
    if (err) atomicOr(err, bits);
}

// Range checks of derived offsets, compiled in by -DPKV_DEBUG_BOUNDS=1 (the
// debug build of the library).  dbg_in(off, n, extent, err) is true when the
// elements [off, off + n) lie inside [0, extent); otherwise it sets
// PKV_DEV_ERR_BOUNDS and the caller skips the access.  In the release build
// it is the constant true and costs nothing: there only the indices read
// from device memory (page ids, batch indices, positions, lengths) are
// checked, since every offset derived from a checked index is in range by
// construction -- which the debug build verifies.
#ifndef PKV_DEBUG_BOUNDS
#define PKV_DEBUG_BOUNDS 0
#endif
constexpr bool kDebugBounds = PKV_DEBUG_BOUNDS != 0;
__device__ __forceinline__ bool dbg_in(int64_t off, int64_t n, int64_t extent, int32_t *err) {
    if constexpr (!kDebugBounds) return true;
    if (off >= 0 && n >= 0 && off + n <= extent) return true;
    set_err(err, PKV_DEV_ERR_BOUNDS);
    return false;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared copy that bypasses L1; pred false writes zeros and
// reads nothing.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, bool pred) {
    int n = pred ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D(16x8, fp32) += A(16x16, row) * B(16x8, col) with 16-bit inputs of type T.
template <typename T>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&d)[4], const uint32_t (&a)[4],
                                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__half>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                 uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two floats -> packed pair of T (round to nearest even), low half = a.
template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Two E4M3 values (low byte first) widened exactly to a 16-bit pair: every
// E4M3 value is an fp16 and a bf16 value.  To bf16 through fp16 and fp32,
// each step exact.
template <typename T>
__device__ __forceinline__ uint32_t widen_e4m3x2(uint32_t two);
template <>
__device__ __forceinline__ uint32_t widen_e4m3x2<__half>(uint32_t two) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(h) : "h"(static_cast<unsigned short>(two)));
    return h;
}
template <>
__device__ __forceinline__ uint32_t widen_e4m3x2<__nv_bfloat16>(uint32_t two) {
    const uint32_t h = widen_e4m3x2<__half>(two);
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    return pack2<__nv_bfloat16>(f.x, f.y);
}

// 2^x on the special-function unit (PTX ex2.approx; -inf -> 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}
// log2(x) on the special-function unit (PTX lg2.approx).
__device__ __forceinline__ float fast_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// Byte offset of 16-byte chunk `c` of row `r` in a row-major smem tile whose
// rows are `row_bytes` long: chunks are XOR-swizzled within each group of 8
// so that 8 consecutive rows at the same logical chunk hit distinct banks.
__device__ __forceinline__ uint32_t swz(int r, int c, int row_bytes) {
    return static_cast<uint32_t>(r * row_bytes + ((c ^ (r & 7)) << 4));
}

// Element offset of (page, head, slot) row start inside one cache tensor.
template <int LAYOUT>
__device__ __forceinline__ int64_t kv_row_offset(int64_t page, int64_t page_stride, int head,
                                                 int slot, int num_heads, int page_size,
                                                 int head_dim) {
    if (LAYOUT == PKV_HND)
        return page * page_stride + (static_cast<int64_t>(head) * page_size + slot) * head_dim;
    return page * page_stride + (static_cast<int64_t>(slot) * num_heads + head) * head_dim;
}

}  // namespace pkv
