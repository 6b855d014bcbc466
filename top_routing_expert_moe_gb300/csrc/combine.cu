// combine.cu -- gate-weighted combine, its backward, and the router backward.
//
// [LLaMA4-MoE] §2.4: each token's output is the weighted sum of its selected
// experts' outputs, the weight being the post-softmax routing score; the
// gradient must flow through those weights into the router (no detach).
// [ZeRO3-MoE] §3.2: variance-form aux loss on the mean routing probability.
//
// All kernels are HBM-bound row streams: one warp per row, 16-byte vectors,
// fp32 accumulation, fixed summation order (deterministic).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// out[t] = sum_j gate[t,j] * y_perm[slot_of[t,j]] (kept slots, j ascending)
template <typename T>
__global__ void __launch_bounds__(256) combine_kernel(const T* __restrict__ y_perm,
                                                      const int32_t* __restrict__ slot_of,
                                                      const float* __restrict__ gate, int Tn,
                                                      int d, int k, T* __restrict__ out)
{
    constexpr int V = 16 / sizeof(T);
    const int nv = d / V;
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < Tn; t += warps) {
        int slot[8];
        float g[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            slot[j] = j < k ? slot_of[(size_t)t * k + j] : -1;
            g[j] = j < k ? gate[(size_t)t * k + j] : 0.f;
        }
        for (int v = lane; v < nv; v += 32) {
            float acc[V];
#pragma unroll
            for (int q = 0; q < V; ++q) acc[q] = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (slot[j] < 0) continue;
                float y[V];
                load16_f<T>(y_perm + (size_t)slot[j] * d + v * V, y);
#pragma unroll
                for (int q = 0; q < V; ++q) acc[q] = fmaf(g[j], y[q], acc[q]);
            }
            store16_f<T>(out + (size_t)t * d + v * V, acc);
        }
    }
}

// Row r of the permuted layout: dy_perm[r] = gate * dout[t]; dgate = <dout[t], y_perm[r]>.
template <typename T>
__global__ void __launch_bounds__(256) combine_bwd_kernel(
    const T* __restrict__ dout, const T* __restrict__ y_perm, const float* __restrict__ gate,
    const int32_t* __restrict__ slot_of, const int32_t* __restrict__ perm_token,
    const int32_t* __restrict__ offsets, int E, int d, int k, T* __restrict__ dy_perm,
    float* __restrict__ dgate)
{
    constexpr int V = 16 / sizeof(T);
    const int rows = offsets[E];
    const int nv = d / V;
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        const int t = perm_token[r];
        T* dst = dy_perm + (size_t)r * d;
        if (t < 0) {
            for (int v = lane; v < nv; v += 32)
                reinterpret_cast<uint4*>(dst)[v] = make_uint4(0, 0, 0, 0);
            continue;
        }
        int j = 0;
        while (j < k - 1 && slot_of[(size_t)t * k + j] != r) ++j;
        const float gt = gate[(size_t)t * k + j];
        float dot = 0.f;
        for (int v = lane; v < nv; v += 32) {
            float go[V], y[V], o[V];
            load16_f<T>(dout + (size_t)t * d + v * V, go);
            load16_f<T>(y_perm + (size_t)r * d + v * V, y);
#pragma unroll
            for (int q = 0; q < V; ++q) {
                dot = fmaf(go[q], y[q], dot);
                o[q] = gt * go[q];
            }
            store16_f<T>(dst + v * V, o);
        }
        dot = warp_sum(dot);
        if (lane == 0) dgate[(size_t)t * k + j] = dot;
    }
}

// dgate of dropped slots is zero
__global__ void zero_dropped_dgate_kernel(const int32_t* __restrict__ slot_of, int n,
                                          float* __restrict__ dgate)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        if (slot_of[i] < 0) dgate[i] = 0.f;
}

// W_r [d,E] -> W_rT [E,d] fp32 (router-backward operand)
template <typename T>
__global__ void transpose_wr_f32_kernel(const T* __restrict__ Wr, float* __restrict__ WrT, int d,
                                        int E)
{
    const size_t n = (size_t)E * d;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < n;
         idx += (size_t)gridDim.x * blockDim.x) {
        int e = (int)(idx / d), i = (int)(idx % d);
        WrT[idx] = to_f<T>(Wr[(size_t)i * E + e]);
    }
}

// One warp per token: dlogits (gate Jacobian + aux term), then
// dx[t] = sum_kept dx_perm[slot] + dlogits[t] . W_r^T.
template <typename T>
__global__ void __launch_bounds__(256) router_bwd_token_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ topk,
    const float* __restrict__ gate, const int32_t* __restrict__ slot_of,
    const float* __restrict__ dgate, const float* __restrict__ stats,
    const T* __restrict__ dx_perm, const float* __restrict__ WrT, int Tn, int d, int E, int k,
    int normalize, float aux_coef, float* __restrict__ dlogits, T* __restrict__ dx)
{
    constexpr int V = 16 / sizeof(T);
    __shared__ float s_dl[8][64];
    const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nv = d / V;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int t = blockIdx.x * (blockDim.x >> 5) + wib; t < Tn; t += warps) {
        // lanes hold experts e = lane and lane + 32
        float l0 = lane < E ? logits[(size_t)t * E + lane] : -INFINITY;
        float l1 = lane + 32 < E ? logits[(size_t)t * E + lane + 32] : -INFINITY;
        const float m = warp_max(fmaxf(l0, l1));
        float p0 = lane < E ? expf(l0 - m) : 0.f;
        float p1 = lane + 32 < E ? expf(l1 - m) : 0.f;
        const float z = warp_sum(p0 + p1);
        p0 /= z;
        p1 /= z;
        float dl0 = 0.f, dl1 = 0.f;
        if (normalize) {
            float s = 0.f;
            for (int j = 0; j < k; ++j) {
                float dg = slot_of[(size_t)t * k + j] >= 0 ? dgate[(size_t)t * k + j] : 0.f;
                s += gate[(size_t)t * k + j] * dg;
            }
            for (int j = 0; j < k; ++j) {
                float dg = slot_of[(size_t)t * k + j] >= 0 ? dgate[(size_t)t * k + j] : 0.f;
                const int e = topk[(size_t)t * k + j];
                const float v = gate[(size_t)t * k + j] * (dg - s);
                if (e == lane) dl0 += v;
                if (e == lane + 32) dl1 += v;
            }
        } else {
            float s = 0.f;
            for (int j = 0; j < k; ++j) {
                float dg = slot_of[(size_t)t * k + j] >= 0 ? dgate[(size_t)t * k + j] : 0.f;
                const int e = topk[(size_t)t * k + j];
                const float pe = __shfl_sync(0xffffffffu, e < 32 ? p0 : p1, e & 31);
                s += dg * pe;
                if (e == lane) dl0 += dg * p0;
                if (e == lane + 32) dl1 += dg * p1;
            }
            dl0 -= p0 * s;
            dl1 -= p1 * s;
        }
        if (aux_coef != 0.f) {
            const float invE = 1.0f / (float)E, sc = aux_coef * 2.0f / (float)Tn;
            const float c0 = lane < E ? sc * (stats[MOE_STAT_PBAR + lane] - invE) : 0.f;
            const float c1 = lane + 32 < E ? sc * (stats[MOE_STAT_PBAR + lane + 32] - invE) : 0.f;
            const float s2 = warp_sum(p0 * c0 + p1 * c1);
            dl0 += p0 * (c0 - s2);
            dl1 += p1 * (c1 - s2);
        }
        if (lane < E) { dlogits[(size_t)t * E + lane] = dl0; s_dl[wib][lane] = dl0; }
        if (lane + 32 < E) { dlogits[(size_t)t * E + lane + 32] = dl1; s_dl[wib][lane + 32] = dl1; }
        __syncwarp();
        int slot[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) slot[j] = j < k ? slot_of[(size_t)t * k + j] : -1;
        for (int v = lane; v < nv; v += 32) {
            float acc[V];
#pragma unroll
            for (int q = 0; q < V; ++q) acc[q] = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (slot[j] < 0) continue;
                float y[V];
                load16_f<T>(dx_perm + (size_t)slot[j] * d + v * V, y);
#pragma unroll
                for (int q = 0; q < V; ++q) acc[q] += y[q];
            }
            for (int e = 0; e < E; ++e) {
                const float de = s_dl[wib][e];
                const float* w = WrT + (size_t)e * d + v * V;
#pragma unroll
                for (int q = 0; q < V; q += 4) {
                    float4 wv = __ldg(reinterpret_cast<const float4*>(w + q));
                    acc[q] = fmaf(de, wv.x, acc[q]);
                    acc[q + 1] = fmaf(de, wv.y, acc[q + 1]);
                    acc[q + 2] = fmaf(de, wv.z, acc[q + 2]);
                    acc[q + 3] = fmaf(de, wv.w, acc[q + 3]);
                }
            }
            store16_f<T>(dx + (size_t)t * d + v * V, acc);
        }
        __syncwarp();
    }
}

// Partial dW_r over a token chunk: part[s][i][e] = sum_{t in chunk s} x[t,i] dlogits[t,e].
// CTA = 32 column vectors (16 bytes each) x 8 token lanes; each thread keeps
// V x EB accumulators (V columns of one vector, EB experts of this CTA's expert
// group) while streaming its token lane's x rows with 16-byte loads; the 8 token
// lanes are summed in a fixed order through shared memory.
template <typename T, int EB>
__global__ void __launch_bounds__(256) dwr_partial_kernel(const T* __restrict__ x,
                                                          const float* __restrict__ dlogits,
                                                          int Tn, int d, int E, int chunk,
                                                          float* __restrict__ part,
                                                          float* __restrict__ part_db)
{
    constexpr int V = 16 / sizeof(T);
    extern __shared__ __align__(16) float red[];          // [8][32][V*EB]
    const int tid = threadIdx.x, tl = tid >> 5, cv = tid & 31;
    const int col0 = (blockIdx.x * 32 + cv) * V;
    const int e0 = blockIdx.z * EB;
    const int s = blockIdx.y;
    const int tbeg = s * chunk, tend = min(Tn, tbeg + chunk);
    const bool colok = col0 < d;
    float acc[V][EB];
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
        for (int e = 0; e < EB; ++e) acc[v][e] = 0.f;
    for (int t = tbeg + tl; t < tend; t += 8) {
        float xv[V];
        if (colok) load16_f<T>(x + (size_t)t * d + col0, xv);
        else {
#pragma unroll
            for (int v = 0; v < V; ++v) xv[v] = 0.f;
        }
        float dl[EB];
#pragma unroll
        for (int e = 0; e < EB; ++e) dl[e] = (e0 + e < E) ? __ldg(dlogits + (size_t)t * E + e0 + e) : 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v)
#pragma unroll
            for (int e = 0; e < EB; ++e) acc[v][e] = fmaf(xv[v], dl[e], acc[v][e]);
    }
    float* mine = red + ((size_t)tl * 32 + cv) * (V * EB);
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
        for (int e = 0; e < EB; ++e) mine[v * EB + e] = acc[v][e];
    __syncthreads();
    for (int i = tid; i < 32 * V * EB; i += 256) {
        const int c = i / (V * EB), r = i % (V * EB);
        const int v = r / EB, e = r % EB;
        float a = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) a += red[((size_t)q * 32 + c) * (V * EB) + r];
        const int col = (blockIdx.x * 32 + c) * V + v;
        if (col < d && e0 + e < E) part[((size_t)s * d + col) * E + e0 + e] = a;
    }
    if (blockIdx.x == 0 && blockIdx.z == 0 && tid < E) {
        float a = 0.f;
        for (int t = tbeg; t < tend; ++t) a += dlogits[(size_t)t * E + tid];
        part_db[(size_t)s * E + tid] = a;
    }
}

template <typename T>
__global__ void dwr_reduce_kernel(const float* __restrict__ part, const float* __restrict__ part_db,
                                  int nsplit, int d, int E, T* __restrict__ dWr,
                                  float* __restrict__ dbias)
{
    const size_t n = (size_t)d * E;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        float a = 0.f;
        for (int s = 0; s < nsplit; ++s) a += part[(size_t)s * n + i];
        dWr[i] = from_f<T>(a);
    }
    if (dbias && blockIdx.x == 0 && threadIdx.x < E) {
        float a = 0.f;
        for (int s = 0; s < nsplit; ++s) a += part_db[(size_t)s * E + threadIdx.x];
        dbias[threadIdx.x] = a;
    }
}

constexpr int DWR_EB = 8;  // experts per CTA of dwr_partial_kernel

dim3 dwr_grid_xz(const moe_config& c) {
    const int V = c.dtype == MOE_DTYPE_BF16 ? 8 : 4;
    return dim3((c.d + 32 * V - 1) / (32 * V), 1, (c.E + DWR_EB - 1) / DWR_EB);
}

// token chunks: enough CTAs for about four per SM
int dwr_nsplit(const moe_config& c) {
    const dim3 g = dwr_grid_xz(c);
    const int per = (int)(g.x * g.z);
    int ns = std::max(1, (4 * num_sms() + per - 1) / per);
    return std::min(ns, std::max(1, (c.T + 63) / 64));
}

int row_grid(int64_t rows) {
    return (int)std::max<int64_t>(1, std::min<int64_t>((rows + 7) / 8, (int64_t)num_sms() * 16));
}

}  // namespace

int launch_combine(const moe_config& c, const void* y_perm, const int32_t* slot_of,
                   const float* gate, void* out, cudaStream_t st)
{
    const int grid = row_grid(c.T);
    if (c.dtype == MOE_DTYPE_BF16)
        combine_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
            static_cast<const __nv_bfloat16*>(y_perm), slot_of, gate, c.T, c.d, c.k,
            static_cast<__nv_bfloat16*>(out));
    else
        combine_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(y_perm), slot_of,
                                                    gate, c.T, c.d, c.k, static_cast<float*>(out));
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

int launch_combine_backward(const moe_config& c, const void* dout, const void* y_perm,
                            const float* gate, const int32_t* slot_of, const int32_t* perm_token,
                            const int32_t* offsets, void* dy_perm, float* dgate, cudaStream_t st)
{
    const int n = c.T * c.k;
    zero_dropped_dgate_kernel<<<std::min(1024, (n + 255) / 256), 256, 0, st>>>(slot_of, n, dgate);
    MOE_LAUNCH_CHECK();
    const int grid = row_grid(rows_cap_of(c));
    if (c.dtype == MOE_DTYPE_BF16)
        combine_bwd_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
            static_cast<const __nv_bfloat16*>(dout), static_cast<const __nv_bfloat16*>(y_perm),
            gate, slot_of, perm_token, offsets, c.E, c.d, c.k,
            static_cast<__nv_bfloat16*>(dy_perm), dgate);
    else
        combine_bwd_kernel<float><<<grid, 256, 0, st>>>(
            static_cast<const float*>(dout), static_cast<const float*>(y_perm), gate, slot_of,
            perm_token, offsets, c.E, c.d, c.k, static_cast<float*>(dy_perm), dgate);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

size_t router_bwd_ws_bytes(const moe_config& c) {
    const int ns = dwr_nsplit(c);
    return align_up((size_t)c.E * c.d * 4) + align_up((size_t)ns * c.d * c.E * 4) +
           align_up((size_t)ns * c.E * 4) + align_up((size_t)c.T * c.E * 4);
}

int launch_router_backward(const moe_config& c, const void* x, const void* Wr,
                           const float* logits, const int32_t* topk, const float* gate,
                           const int32_t* slot_of, const float* dgate, const void* dx_perm,
                           const float* stats, void* dx, void* dWr, float* dbias, float* dlogits,
                           void* ws, cudaStream_t st)
{
    const int ns = dwr_nsplit(c);
    uint8_t* w = static_cast<uint8_t*>(ws);
    float* WrT = reinterpret_cast<float*>(w); w += align_up((size_t)c.E * c.d * 4);
    float* part = reinterpret_cast<float*>(w); w += align_up((size_t)ns * c.d * c.E * 4);
    float* part_db = reinterpret_cast<float*>(w); w += align_up((size_t)ns * c.E * 4);
    if (!dlogits) dlogits = reinterpret_cast<float*>(w);
    const int chunk = (c.T + ns - 1) / ns;
    const int grid = row_grid(c.T);
    dim3 pgrid = dwr_grid_xz(c);
    pgrid.y = ns;
    // reduction buffer: 8 token lanes x 32 vectors x (V * EB) floats, V = 16 / sizeof(T)
    const size_t dwr_smem = (size_t)8 * 32 * (c.dtype == MOE_DTYPE_BF16 ? 8 : 4) * DWR_EB * sizeof(float);
    if (c.dtype == MOE_DTYPE_BF16) {
        static bool attr = false;
        if (!attr) {
            MOE_CUDA_TRY(cudaFuncSetAttribute(dwr_partial_kernel<__nv_bfloat16, DWR_EB>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dwr_smem));
            attr = true;
        }
    } else {
        static bool attr = false;
        if (!attr) {
            MOE_CUDA_TRY(cudaFuncSetAttribute(dwr_partial_kernel<float, DWR_EB>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dwr_smem));
            attr = true;
        }
    }
    if (c.dtype == MOE_DTYPE_BF16) {
        using T = __nv_bfloat16;
        transpose_wr_f32_kernel<T><<<64, 256, 0, st>>>(static_cast<const T*>(Wr), WrT, c.d, c.E);
        MOE_LAUNCH_CHECK();
        router_bwd_token_kernel<T><<<grid, 256, 0, st>>>(
            logits, topk, gate, slot_of, dgate, stats, static_cast<const T*>(dx_perm), WrT, c.T,
            c.d, c.E, c.k, c.normalize_gates, c.aux_coef, dlogits, static_cast<T*>(dx));
        MOE_LAUNCH_CHECK();
        dwr_partial_kernel<T, DWR_EB><<<pgrid, 256, dwr_smem, st>>>(static_cast<const T*>(x), dlogits,
                                                                   c.T, c.d, c.E, chunk, part, part_db);
        MOE_LAUNCH_CHECK();
        dwr_reduce_kernel<T><<<std::min(1024, (c.d * c.E + 255) / 256), 256, 0, st>>>(
            part, part_db, ns, c.d, c.E, static_cast<T*>(dWr), dbias);
        MOE_LAUNCH_CHECK();
    } else {
        using T = float;
        transpose_wr_f32_kernel<T><<<64, 256, 0, st>>>(static_cast<const T*>(Wr), WrT, c.d, c.E);
        MOE_LAUNCH_CHECK();
        router_bwd_token_kernel<T><<<grid, 256, 0, st>>>(
            logits, topk, gate, slot_of, dgate, stats, static_cast<const T*>(dx_perm), WrT, c.T,
            c.d, c.E, c.k, c.normalize_gates, c.aux_coef, dlogits, static_cast<T*>(dx));
        MOE_LAUNCH_CHECK();
        dwr_partial_kernel<T, DWR_EB><<<pgrid, 256, dwr_smem, st>>>(static_cast<const T*>(x), dlogits,
                                                                   c.T, c.d, c.E, chunk, part, part_db);
        MOE_LAUNCH_CHECK();
        dwr_reduce_kernel<T><<<std::min(1024, (c.d * c.E + 255) / 256), 256, 0, st>>>(
            part, part_db, ns, c.d, c.E, static_cast<T*>(dWr), dbias);
        MOE_LAUNCH_CHECK();
    }
    return MOE_OK;
}

}  // namespace moe
