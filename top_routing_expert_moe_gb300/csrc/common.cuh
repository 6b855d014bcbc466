// common.cuh -- helpers shared by the sm_103a kernels of the MoE layer.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

// ---- host bookkeeping (defined in moe_abi.cu) ----
void note_launch(int n = 1);        // count kernels launched by this library
int* device_status_ptr();           // device address of the status word (current device)
int num_sms();                      // SM count of the current device

#define MOE_CUDA_TRY(expr)                                  \
    do {                                                    \
        cudaError_t _e = (expr);                            \
        if (_e != cudaSuccess) return MOE_ERR_CUDA;         \
    } while (0)

#define MOE_LAUNCH_CHECK()                                  \
    do {                                                    \
        ::moe::note_launch();                               \
        if (cudaPeekAtLastError() != cudaSuccess) {         \
            (void)cudaGetLastError();                       \
            return MOE_ERR_CUDA;                            \
        }                                                   \
    } while (0)

// ---- programmatic dependent launch ----
// Every kernel of the library is launched with programmatic stream
// serialization: it may be scheduled while the kernel before it on the stream
// is still finishing.  Each kernel therefore calls pdl_wait() before its first
// global-memory access (it returns once the preceding grid has completed and
// its writes are visible), then pdl_trigger() to let the next kernel be
// scheduled early in turn.  Set-up that touches no global memory (barrier
// init, TMEM allocation, tensor-map prefetch) may come before the wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

inline cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                     cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// launch with arguments converted to the kernel's parameter types
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(grid, block, smem, st, attr);
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch a kernel whose single parameter is a const __grid_constant__ struct
template <typename P>
inline cudaError_t launch_pdl_param(void (*kernel)(const P), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t st, const P& param) {
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(grid, block, smem, st, attr);
    void* args[] = {const_cast<P*>(&param)};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(kernel), args);
}

// launch, count the launch, and turn a failure into MOE_ERR_CUDA
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) for `kernel` on the current
// device, once per device (function attributes belong to a device's context;
// `done` is the call site's static per-device flags)
template <class F>
inline int smem_attr_once(F* kernel, size_t bytes, bool (&done)[64]) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev >= 0 && dev < 64 && done[dev]) return MOE_OK;
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(kernel),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    if (dev >= 0 && dev < 64) done[dev] = true;
    return MOE_OK;
}

#define MOE_LAUNCH(...)                                                  \
    do {                                                                 \
        const cudaError_t _le = ::moe::launch_pdl(__VA_ARGS__);          \
        ::moe::note_launch();                                            \
        if (_le != cudaSuccess) {                                        \
            (void)cudaGetLastError();                                    \
            return MOE_ERR_CUDA;                                         \
        }                                                                \
    } while (0)

#define MOE_LAUNCH_PARAM(...)                                            \
    do {                                                                 \
        const cudaError_t _le = ::moe::launch_pdl_param(__VA_ARGS__);    \
        ::moe::note_launch();                                            \
        if (_le != cudaSuccess) {                                        \
            (void)cudaGetLastError();                                    \
            return MOE_ERR_CUDA;                                         \
        }                                                                \
    } while (0)

// ---- element access (fp32 or bf16 stored as __nv_bfloat16) ----
template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// 16-byte vector of elements: 4 fp32 or 8 bf16
template <typename T> struct Vec16 { static constexpr int N = 16 / sizeof(T); };

template <typename T>
__device__ __forceinline__ void load16_f(const T* p, float* out) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    if constexpr (sizeof(T) == 4) {
        out[0] = __uint_as_float(u.x); out[1] = __uint_as_float(u.y);
        out[2] = __uint_as_float(u.z); out[3] = __uint_as_float(u.w);
    } else {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            out[2 * i] = __uint_as_float(w[i] << 16);
            out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
}

template <typename T>
__device__ __forceinline__ void store16_f(T* p, const float* v) {
    uint4 u;
    if constexpr (sizeof(T) == 4) {
        u.x = __float_as_uint(v[0]); u.y = __float_as_uint(v[1]);
        u.z = __float_as_uint(v[2]); u.w = __float_as_uint(v[3]);
    } else {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&b);
        }
        u = make_uint4(w[0], w[1], w[2], w[3]);
    }
    *reinterpret_cast<uint4*>(p) = u;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }
__device__ __forceinline__ float dsilu_f(float z) {
    float s = 1.0f / (1.0f + expf(-z));
    return s * (1.0f + z * (1.0f - s));
}

// record the first device-side error (others keep the first)
__device__ __forceinline__ void set_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

}  // namespace moe
