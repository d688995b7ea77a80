// Shared host/device helpers of the spec_tree library: error reporting,
// argument checks, the traced launch wrapper, element conversions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <utility>

#include "spec_tree.h"

namespace spec {

// ---------------------------------------------------------------- errors (host)

void set_error(const char* fmt, ...);
void clear_error();

// Record a message and return the status, for `return fail(SPEC_EINVAL, "...")`.
spec_status fail(spec_status st, const char* fmt, ...);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Checks of a spec_tree passed by a caller (host fields and device pointers).
spec_status check_tree(const spec_tree* t);

// Workspace header: the first 16 bytes of every workspace hold the device status word.
constexpr size_t kWsHeader = 256;
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Reset the device status word of a workspace (queued on the stream).
cudaError_t reset_device_status(void* ws, cudaStream_t s);

// ---------------------------------------------------------------- traced launches

void trace_before(cudaStream_t s);
void trace_after(cudaStream_t s, const char* name);
void count_launch();

// Launch `kernel` on stream `s`, bracketed by trace events when tracing is on.
template <typename... KArgs, typename... Args>
inline cudaError_t launch(const char* name, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                          size_t smem, cudaStream_t s, Args&&... args) {
    trace_before(s);
    kernel<<<grid, block, smem, s>>>(std::forward<Args>(args)...);
    cudaError_t e = cudaGetLastError();
    trace_after(s, name);
    count_launch();
    return e;
}

bool trace_active();

// Launch with cudaLaunchKernelEx; `pdl` allows programmatic dependent launch
// (the kernel may start while the previous kernel on the stream drains; it must
// call griddep_wait() before touching that kernel's results).  Tracing turns
// the overlap off so each kernel's events bracket it alone.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(const char* name, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    const bool use_pdl = pdl && !trace_active();
    cfg.attrs = use_pdl ? attr : nullptr;
    cfg.numAttrs = use_pdl ? 1 : 0;
    trace_before(s);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    trace_after(s, name);
    count_launch();
    return e;
}

// launch_ex with a thread-block cluster shape (cluster.x * y * z CTAs, at most 8).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_cluster(const char* name, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t s, bool pdl, dim3 cluster, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster.x;
    attr[0].val.clusterDim.y = cluster.y;
    attr[0].val.clusterDim.z = cluster.z;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl && !trace_active() ? 2 : 1;
    trace_before(s);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    trace_after(s, name);
    count_launch();
    return e;
}

#define SPEC_CUDA_TRY(expr)                                                              \
    do {                                                                                 \
        cudaError_t _e = (expr);                                                         \
        if (_e != cudaSuccess)                                                           \
            return ::spec::fail(SPEC_ECUDA, "%s: %s", #expr, cudaGetErrorString(_e));    \
    } while (0)

// ---------------------------------------------------------------- device helpers

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Load 4 consecutive elements (16 bytes of fp32 or 8 bytes of bf16) as floats.
__device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
    float4 t = *reinterpret_cast<const float4*>(p);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
    uint2 t = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(t.x << 16); v[1] = __uint_as_float(t.x & 0xFFFF0000u);
    v[2] = __uint_as_float(t.y << 16); v[3] = __uint_as_float(t.y & 0xFFFF0000u);
}

__device__ __forceinline__ float warp_max(float v) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_min(float v) {
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Programmatic dependent launch: wait for the preceding kernel's results /
// allow the next kernel to start launching.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// A 32-bit key that orders like the float (NaN below -inf, -0 equal to +0), and back.
__device__ __forceinline__ unsigned order_key(float v) {
    if (v != v) return 0u;
    if (v == 0.f) v = 0.f;
    const unsigned b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Record a device-detected failure in a workspace's status word (largest code wins).
__device__ __forceinline__ void flag_status(void* ws, int code) { atomicMax(static_cast<int*>(ws), code); }

// Clear a call's status words from the call's first kernel (instead of a memset
// before it): thread 0 of block 0 stores and fences, then the block meets at a
// barrier, and only after that does the kernel trigger its dependents.  So no
// later kernel of the call can flag before the clear; the first kernel itself
// must flag only from block 0 after this call, or not at all.
__device__ __forceinline__ void clear_status_then_trigger(void* ws) {
    if (ws && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) {
        if (threadIdx.x == 0) {
            *static_cast<int4*>(ws) = make_int4(0, 0, 0, 0);
            __threadfence();
        }
        __syncthreads();
    }
    griddep_launch();
}

// Merge two (max, sum of exp(x - max)) pairs.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) { m = m2; s = s2; return; }
    if (m2 > m) { s = s * expf(m - m2) + s2; m = m2; }
    else { s = s + s2 * expf(m2 - m); }
}

}  // namespace spec
