// route_noalloc.cu -- the router entry point for callers that cannot allocate.
//
// moe_route needs a caller-provided workspace (per-CTA partial statistics and
// the transposed router weights).  Some callers cannot obtain one: code that
// runs inside a host framework which owns all device memory through its own
// pool and forbids side allocations once it has started, or code on a latency
// path that cannot afford cudaMalloc's cost and implicit device
// synchronisation.  moe_route_noalloc serves them with the same kernels, its
// scratch taken from one file-scope __device__ array of fixed size.
//
// The array lives on every GPU that loads this library until the process
// exits.  Host code may not use its name as a device address (the host symbol
// is only a stand-in): the device address is fetched once per device with
// cudaGetSymbolAddress, with that device current, on the first call there.
// All calls share the array and it keeps the previous call's contents; the
// router kernels write every scratch word before reading it, so nothing needs
// clearing.  Two calls whose kernels overlap on the GPU (different streams,
// same device) race on the array.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

static __device__ __align__(256) uint8_t g_route_scratch[MOE_ROUTE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDev] = {};

// Device address of g_route_scratch on the current device (looked up once).
int route_scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDev) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" int moe_route_noalloc(const moe_config* c, const void* x, const void* W_r,
                                 const float* bias, const float* noise, const uint8_t* token_mask,
                                 float* logits, int32_t* topk_idx, float* gate, int32_t* counts,
                                 float* stats, moe_stream_t stream) {
    using namespace moe;
    int r = moe_check_config(c);
    if (r) return r;
    if (route_ws_bytes(*c) > (size_t)MOE_ROUTE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_SCRATCH_LIMIT;
    auto ok = [](const void* p) { return p != nullptr && aligned16(p); };
    auto opt = [](const void* p) { return p == nullptr || aligned16(p); };
    if (!ok(x) || !ok(W_r) || !opt(bias) || !opt(noise) || !opt(token_mask) || !ok(logits) ||
        !ok(topk_idx) || !ok(gate) || !ok(counts) || !opt(stats))
        return MOE_ERR_INVALID_ARG;
    void* scratch = nullptr;
    if ((r = route_scratch_address(&scratch))) return r;
    return launch_route(*c, x, W_r, bias, noise, token_mask, logits, topk_idx, gate, counts, stats,
                        scratch, (cudaStream_t)stream);
}
