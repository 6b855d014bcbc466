// moe_abi.cu -- the extern "C" entry points: argument checks, workspace
// layout, and the order of kernel launches for each step of the layer.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
__device__ int g_device_status;  // first device-side error since the last read
std::atomic<uint64_t> g_launches{0};
constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::mutex g_dev_mu;

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    return dev;
}
}  // namespace

void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int* device_status_ptr() {
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) == cudaSuccess) g_status_ptr[dev] = static_cast<int*>(p);
    }
    return g_status_ptr[dev];
}

int num_sms() {
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

int capacity_of(const moe_config& c) {
    if (!(c.capacity_factor > 0.0f)) return c.T;
    const double v = std::ceil((double)c.capacity_factor * (double)c.T * (double)c.k / (double)c.E);
    return v > (double)c.T ? c.T : (int)v;
}

int64_t rows_cap_of(const moe_config& c) {
    const int64_t a = (int64_t)c.T * c.k;
    const int64_t b = (int64_t)c.E * capacity_of(c);
    return (a < b ? a : b) + (int64_t)c.E * (c.pad_m - 1);
}

int64_t shared_rows_of(const moe_config& c) {
    if (c.f_shared <= 0) return 0;
    return c.dtype == MOE_DTYPE_BF16 ? ((int64_t)c.T + 127) / 128 * 128 : (int64_t)c.T;
}

}  // namespace moe

using namespace moe;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }
bool ok_opt(const void* p) { return p == nullptr || aligned16(p); }
size_t esize(const moe_config& c) { return c.dtype == MOE_DTYPE_BF16 ? 2 : 4; }
int nh_of(const moe_config& c) { return c.ffn == MOE_FFN_SWIGLU ? 2 : 1; }

// The shared-experts block: present iff f_shared > 0; the fields each entry
// point uses must be set and 16-byte aligned.
enum SharedUse { SH_FWD, SH_COMBINE, SH_BWD, SH_ROUTER_BWD };
bool shared_ok(const moe_config& c, const moe_shared_ffn* s, SharedUse use) {
    if (c.f_shared <= 0) return s == nullptr;
    if (!s) return false;
    const bool sw = c.ffn == MOE_FFN_SWIGLU;
    switch (use) {
        case SH_FWD:
            return ok_ptr(s->x) && ok_ptr(s->W_up) && ok_ptr(s->W_down) &&
                   (sw ? ok_ptr(s->W_gate) : ok_opt(s->W_gate)) && ok_ptr(s->h) &&
                   ok_ptr(s->act) && ok_ptr(s->y);
        case SH_COMBINE:
            return ok_ptr(s->y);
        case SH_BWD:
            return ok_ptr(s->x) && ok_ptr(s->W_up) && ok_ptr(s->W_down) &&
                   (sw ? ok_ptr(s->W_gate) : ok_opt(s->W_gate)) && ok_ptr(s->h) &&
                   ok_ptr(s->act) && ok_ptr(s->dout) && ok_ptr(s->dh) && ok_ptr(s->dx) &&
                   ok_ptr(s->dW_up) && (sw ? ok_ptr(s->dW_gate) : ok_opt(s->dW_gate)) &&
                   ok_ptr(s->dW_down);
        case SH_ROUTER_BWD:
            return ok_ptr(s->dx);
    }
    return false;
}

// intermediate buffers of moe_backward, carved from the workspace
struct BwdLayout {
    size_t dy, dgate, dh, dxp, dlogits, sdh, sdx, rest, total;
};
BwdLayout bwd_layout(const moe_config& c) {
    const size_t rc = (size_t)rows_cap_of(c), es = esize(c), ts = (size_t)shared_rows_of(c);
    BwdLayout L;
    size_t o = 0;
    L.dy = o; o += align_up(rc * c.d * es);
    L.dgate = o; o += align_up((size_t)c.T * c.k * 4);
    L.dh = o; o += align_up((size_t)nh_of(c) * rc * c.f * es);
    L.dxp = o; o += align_up(rc * c.d * es);
    L.dlogits = o; o += align_up((size_t)c.T * c.E * 4);
    L.sdh = o; o += align_up((size_t)nh_of(c) * ts * (c.f_shared > 0 ? c.f_shared : 0) * es);
    L.sdx = o; o += align_up(ts * c.d * es);
    L.rest = o;
    size_t r = ffn_ws_bytes(c);
    size_t rb = router_bwd_ws_bytes(c);
    o += align_up(r > rb ? r : rb);
    L.total = o;
    return L;
}

}  // namespace

extern "C" {

int moe_check_config(const moe_config* c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->T < 1 || c->d < 1 || c->f < 1 || c->E < 1 || c->k < 1 || c->k > c->E || c->pad_m < 1)
        return MOE_ERR_INVALID_ARG;
    if (c->dtype != MOE_DTYPE_F32 && c->dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
    if (c->ffn != MOE_FFN_SILU && c->ffn != MOE_FFN_SWIGLU) return MOE_ERR_INVALID_ARG;
    if (c->normalize_gates != 0 && c->normalize_gates != 1) return MOE_ERR_INVALID_ARG;
    if (std::isnan(c->capacity_factor) || std::isinf(c->capacity_factor)) return MOE_ERR_INVALID_ARG;
    if (!std::isfinite(c->aux_coef)) return MOE_ERR_INVALID_ARG;
    if (!std::isfinite(c->temperature) || c->temperature < 0.0f) return MOE_ERR_INVALID_ARG;
    if (c->straight_through != 0 && c->straight_through != 1) return MOE_ERR_INVALID_ARG;
    if (c->f_shared < 0) return MOE_ERR_INVALID_ARG;
    if (c->f_shared % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (c->dtype == MOE_DTYPE_BF16 && c->f_shared % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (c->E > 64 || c->k > 8) return MOE_ERR_UNSUPPORTED;
    if (c->d % 8 != 0 || c->f % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (c->dtype == MOE_DTYPE_BF16 && (c->d % 128 != 0 || c->f % 128 != 0 || c->pad_m % 128 != 0))
        return MOE_ERR_UNSUPPORTED;
    // 32-bit row and element indices on the device
    const int64_t rc = rows_cap_of(*c);
    if ((int64_t)c->T * c->k > (1LL << 30) || rc > (1LL << 30) || (int64_t)c->pad_m > (1 << 20))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

int moe_capacity(const moe_config* c, int32_t* capacity) {
    int r = moe_check_config(c);
    if (r) return r;
    if (!capacity) return MOE_ERR_INVALID_ARG;
    *capacity = capacity_of(*c);
    return MOE_OK;
}

int moe_rows_capacity(const moe_config* c, int64_t* rows) {
    int r = moe_check_config(c);
    if (r) return r;
    if (!rows) return MOE_ERR_INVALID_ARG;
    *rows = rows_cap_of(*c);
    return MOE_OK;
}

int moe_shared_rows(const moe_config* c, int64_t* rows) {
    int r = moe_check_config(c);
    if (r) return r;
    if (!rows) return MOE_ERR_INVALID_ARG;
    *rows = shared_rows_of(*c);
    return MOE_OK;
}

int moe_workspace_size(const moe_config* c, size_t* bytes) {
    int r = moe_check_config(c);
    if (r) return r;
    if (!bytes) return MOE_ERR_INVALID_ARG;
    size_t b = route_ws_bytes(*c);
    b = std::max(b, permute_ws_bytes(*c));
    b = std::max(b, ffn_ws_bytes(*c));
    b = std::max(b, router_bwd_ws_bytes(*c));
    b = std::max(b, bwd_layout(*c).total);
    *bytes = b;
    return MOE_OK;
}

int moe_route(const moe_config* c, const void* x, const void* W_r, const float* bias,
              const float* noise, const uint8_t* token_mask, float* logits, int32_t* topk_idx,
              float* gate, int32_t* counts, float* stats, void* ws, moe_stream_t stream) {
    int r = moe_check_config(c);
    if (r) return r;
    if (!ok_ptr(x) || !ok_ptr(W_r) || !ok_opt(bias) || !ok_opt(noise) || !ok_opt(token_mask) ||
        !ok_ptr(logits) || !ok_ptr(topk_idx) || !ok_ptr(gate) || !ok_ptr(counts) ||
        !ok_opt(stats) || !ok_ptr(ws))
        return MOE_ERR_INVALID_ARG;
    return launch_route(*c, x, W_r, bias, noise, token_mask, logits, topk_idx, gate, counts,
                        stats, ws, (cudaStream_t)stream);
}

int moe_permute(const moe_config* c, const void* x, const int32_t* topk_idx, void* x_perm,
                int32_t* perm_token, int32_t* slot_of, int32_t* kept, int32_t* offsets,
                float* stats, void* ws, moe_stream_t stream) {
    int r = moe_check_config(c);
    if (r) return r;
    if (!ok_ptr(x) || !ok_ptr(topk_idx) || !ok_ptr(x_perm) || !ok_ptr(perm_token) ||
        !ok_ptr(slot_of) || !ok_ptr(kept) || !ok_ptr(offsets) || !ok_opt(stats) || !ok_ptr(ws))
        return MOE_ERR_INVALID_ARG;
    return launch_permute(*c, x, topk_idx, x_perm, perm_token, slot_of, kept, offsets, stats, ws,
                          (cudaStream_t)stream);
}

int moe_grouped_ffn(const moe_config* c, const void* x_perm, const int32_t* offsets,
                    const void* W_up, const void* W_gate, const void* W_down, void* h_saved,
                    void* act, void* y_perm, const moe_shared_ffn* shared, void* ws,
                    moe_stream_t stream) {
    int r = moe_check_config(c);
    if (r) return r;
    const bool sw = c->ffn == MOE_FFN_SWIGLU;
    if (!ok_ptr(x_perm) || !ok_ptr(offsets) || !ok_ptr(W_up) || !ok_ptr(W_down) ||
        (sw ? !ok_ptr(W_gate) : !ok_opt(W_gate)) || !ok_ptr(h_saved) || !ok_ptr(act) ||
        !ok_ptr(y_perm) || !ok_opt(ws) || !shared_ok(*c, shared, SH_FWD))
        return MOE_ERR_INVALID_ARG;
    if (ffn_ws_bytes(*c) > 0 && !ws) return MOE_ERR_INVALID_ARG;
    return launch_ffn_forward(*c, x_perm, offsets, W_up, W_gate, W_down, h_saved, act, y_perm,
                              shared, ws, (cudaStream_t)stream);
}

int moe_combine(const moe_config* c, const void* y_perm, const int32_t* slot_of, const float* gate,
                const moe_shared_ffn* shared, void* out, moe_stream_t stream) {
    int r = moe_check_config(c);
    if (r) return r;
    if (!ok_ptr(y_perm) || !ok_ptr(slot_of) || !ok_ptr(gate) || !ok_ptr(out) ||
        !shared_ok(*c, shared, SH_COMBINE))
        return MOE_ERR_INVALID_ARG;
    return launch_combine(*c, y_perm, slot_of, gate, shared ? shared->y : nullptr, out,
                          (cudaStream_t)stream);
}

int moe_combine_backward(const moe_config* c, const void* dout, const void* y_perm,
                         const float* gate, const int32_t* slot_of, const int32_t* perm_token,
                         const int32_t* offsets, void* dy_perm, float* dgate, moe_stream_t stream) {
    int r = moe_check_config(c);
    if (r) return r;
    if (!ok_ptr(dout) || !ok_ptr(y_perm) || !ok_ptr(gate) || !ok_ptr(slot_of) || !ok_ptr(perm_token) ||
        !ok_ptr(offsets) || !ok_ptr(dy_perm) || !ok_ptr(dgate))
        return MOE_ERR_INVALID_ARG;
    return launch_combine_backward(*c, dout, y_perm, gate, slot_of, perm_token, offsets, dy_perm,
                                   dgate, (cudaStream_t)stream);
}

int moe_grouped_ffn_backward(const moe_config* c, const void* x_perm, const int32_t* offsets,
                             const void* W_up, const void* W_gate, const void* W_down,
                             const void* h_saved, const void* act, const void* dy_perm, void* dh,
                             void* dx_perm, void* dW_up, void* dW_gate, void* dW_down,
                             const moe_shared_ffn* shared, void* ws, moe_stream_t stream) {
    int r = moe_check_config(c);
    if (r) return r;
    const bool sw = c->ffn == MOE_FFN_SWIGLU;
    if (!ok_ptr(x_perm) || !ok_ptr(offsets) || !ok_ptr(W_up) || !ok_ptr(W_down) ||
        (sw ? !ok_ptr(W_gate) : !ok_opt(W_gate)) || !ok_ptr(h_saved) || !ok_ptr(act) ||
        !ok_ptr(dy_perm) || !ok_ptr(dh) || !ok_ptr(dx_perm) || !ok_ptr(dW_up) ||
        (sw ? !ok_ptr(dW_gate) : !ok_opt(dW_gate)) || !ok_ptr(dW_down) || !ok_opt(ws) ||
        !shared_ok(*c, shared, SH_BWD))
        return MOE_ERR_INVALID_ARG;
    if (ffn_ws_bytes(*c) > 0 && !ws) return MOE_ERR_INVALID_ARG;
    return launch_ffn_backward(*c, x_perm, offsets, W_up, W_gate, W_down, h_saved, act, dy_perm, dh,
                               dx_perm, dW_up, dW_gate, dW_down, shared, ws, (cudaStream_t)stream);
}

int moe_router_backward(const moe_config* c, const void* x, const void* W_r, const float* logits,
                        const int32_t* topk_idx, const float* gate, const int32_t* slot_of,
                        const float* dgate, const void* dx_perm, const moe_shared_ffn* shared,
                        const float* stats, void* dx, void* dW_r, float* dbias, float* dlogits,
                        void* ws, moe_stream_t stream) {
    int r = moe_check_config(c);
    if (r) return r;
    if (!ok_ptr(x) || !ok_ptr(W_r) || !ok_ptr(logits) || !ok_ptr(topk_idx) || !ok_ptr(gate) ||
        !ok_ptr(slot_of) || !ok_ptr(dgate) || !ok_ptr(dx_perm) || !ok_opt(stats) || !ok_ptr(dx) ||
        !ok_ptr(dW_r) || !ok_opt(dbias) || !ok_opt(dlogits) || !ok_ptr(ws) ||
        !shared_ok(*c, shared, SH_ROUTER_BWD))
        return MOE_ERR_INVALID_ARG;
    if (c->aux_coef != 0.0f && !stats) return MOE_ERR_INVALID_ARG;
    return launch_router_backward(*c, x, W_r, logits, topk_idx, gate, slot_of, dgate, dx_perm,
                                  shared ? shared->dx : nullptr, stats, dx, dW_r, dbias, dlogits,
                                  ws, (cudaStream_t)stream);
}

int moe_backward(const moe_config* c, const void* x, const void* W_r, const void* W_up,
                 const void* W_gate, const void* W_down, const float* logits,
                 const int32_t* topk_idx, const float* gate, const int32_t* slot_of,
                 const int32_t* perm_token, const int32_t* offsets, const void* x_perm,
                 const void* h_saved, const void* act, const void* y_perm, const float* stats,
                 const void* dout, void* dx, void* dW_r, float* dbias, void* dW_up, void* dW_gate,
                 void* dW_down, const moe_shared_ffn* shared, void* ws, moe_stream_t stream) {
    int r = moe_check_config(c);
    if (r) return r;
    if (!ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
    if ((c->f_shared > 0) != (shared != nullptr)) return MOE_ERR_INVALID_ARG;
    const BwdLayout L = bwd_layout(*c);
    uint8_t* w = static_cast<uint8_t*>(ws);
    void* dy = w + L.dy;
    float* dgate = reinterpret_cast<float*>(w + L.dgate);
    void* dh = w + L.dh;
    void* dxp = w + L.dxp;
    float* dlogits = reinterpret_cast<float*>(w + L.dlogits);
    void* rest = w + L.rest;
    moe_shared_ffn sh;
    if (shared) {                     // the shared FFN's dy is the layer's dout (weight 1)
        sh = *shared;
        sh.dout = dout;
        if (!sh.dh) sh.dh = w + L.sdh;
        if (!sh.dx) sh.dx = w + L.sdx;
    }
    const moe_shared_ffn* shp = shared ? &sh : nullptr;
    if ((r = moe_combine_backward(c, dout, y_perm, gate, slot_of, perm_token, offsets, dy, dgate, stream)))
        return r;
    if ((r = moe_grouped_ffn_backward(c, x_perm, offsets, W_up, W_gate, W_down, h_saved, act, dy, dh,
                                      dxp, dW_up, dW_gate, dW_down, shp, rest, stream)))
        return r;
    return moe_router_backward(c, x, W_r, logits, topk_idx, gate, slot_of, dgate, dxp, shp, stats,
                               dx, dW_r, dbias, dlogits, rest, stream);
}

const char* moe_error_string(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument (shape, null or misaligned pointer)";
        case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_TIMEOUT: return "device: a bounded wait timed out";
        case MOE_ERR_NONFINITE: return "device: non-finite router logits";
        case MOE_ERR_DEVICE_BOUNDS: return "device: index out of range";
        case MOE_ERR_SCRATCH_LIMIT: return "configuration exceeds the no-allocation router's static scratch";
        default: return "unknown status";
    }
}

int moe_last_device_status(moe_stream_t stream, int* status) {
    if (!status) return MOE_ERR_INVALID_ARG;
    int* p = device_status_ptr();
    if (!p) return MOE_ERR_CUDA;
    MOE_CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
    int v = 0;
    MOE_CUDA_TRY(cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost));
    const int zero = 0;
    MOE_CUDA_TRY(cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice));
    *status = v;
    return MOE_OK;
}

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
