// common.cuh -- helpers shared by the sm_103a kernels of the MoE layer.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

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
