// gemm_tc.h -- tcgen05 grouped GEMM launchers for the bf16 expert FFN.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

#include "../../include/moe.h"

namespace moe {

int tc_ffn_forward(const moe_config& c, const void* x_perm, const int32_t* offsets,
                   const void* W_up, const void* W_gate, const void* W_down, void* h_saved,
                   void* act, void* y_perm, const moe_shared_ffn* shared, cudaStream_t st);
int tc_ffn_backward(const moe_config& c, const void* x_perm, const int32_t* offsets,
                    const void* W_up, const void* W_gate, const void* W_down,
                    const void* h_saved, const void* act, const void* dy_perm, void* dh,
                    void* dx_perm, void* dW_up, void* dW_gate, void* dW_down,
                    const moe_shared_ffn* shared, cudaStream_t st);

}  // namespace moe
