// kernels.h -- internal launchers of the MoE layer (not part of the C ABI).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

inline size_t align_up(size_t b, size_t a = 256) { return (b + a - 1) / a * a; }

int capacity_of(const moe_config& c);      // per-expert capacity (T when unlimited)
int64_t rows_cap_of(const moe_config& c);  // worst-case permuted rows
int64_t shared_rows_of(const moe_config& c);  // rows of the shared FFN's buffers (0: none)

// route.cu
size_t route_ws_bytes(const moe_config& c);
int launch_route(const moe_config& c, const void* x, const void* Wr, const float* bias,
                 const float* noise, const uint8_t* mask, float* logits, int32_t* topk,
                 float* gate, int32_t* counts, float* stats, void* ws, cudaStream_t st);

// permute.cu
size_t permute_ws_bytes(const moe_config& c);
int launch_permute(const moe_config& c, const void* x, const int32_t* topk, void* x_perm,
                   int32_t* perm_token, int32_t* slot_of, int32_t* kept, int32_t* offsets,
                   float* stats, void* ws, cudaStream_t st);

// combine.cu
int launch_combine(const moe_config& c, const void* y_perm, const int32_t* slot_of,
                   const float* gate, const void* y_shared, void* out, cudaStream_t st);
int launch_combine_backward(const moe_config& c, const void* dout, const void* y_perm,
                            const float* gate, const int32_t* slot_of, const int32_t* perm_token,
                            const int32_t* offsets, void* dy_perm, float* dgate, cudaStream_t st);
size_t router_bwd_ws_bytes(const moe_config& c);
int launch_router_backward(const moe_config& c, const void* x, const void* Wr,
                           const float* logits, const int32_t* topk, const float* gate,
                           const int32_t* slot_of, const float* dgate, const void* dx_perm,
                           const void* dx_shared, const float* stats, void* dx, void* dWr,
                           float* dbias, float* dlogits, void* ws, cudaStream_t st);

// ffn.cu (grouped GEMMs: tcgen05 path for bf16, SIMT path for fp32)
size_t ffn_ws_bytes(const moe_config& c);
int launch_ffn_forward(const moe_config& c, const void* x_perm, const int32_t* offsets,
                       const void* W_up, const void* W_gate, const void* W_down, void* h_saved,
                       void* act, void* y_perm, const moe_shared_ffn* shared, void* ws,
                       cudaStream_t st);
int launch_ffn_backward(const moe_config& c, const void* x_perm, const int32_t* offsets,
                        const void* W_up, const void* W_gate, const void* W_down,
                        const void* h_saved, const void* act, const void* dy_perm, void* dh,
                        void* dx_perm, void* dW_up, void* dW_gate, void* dW_down,
                        const moe_shared_ffn* shared, void* ws, cudaStream_t st);

}  // namespace moe
