// combine.cu -- gate-weighted combine, its backward, and the router backward.
//
// [LLaMA4-MoE] §2.4: each token's output is the weighted sum of its selected
// experts' outputs, the weight being the post-softmax routing score; the
// gradient must flow through those weights into the router (no detach).
// [ZeRO3-MoE] §3.2: variance-form aux loss on the mean routing probability.
//
// All kernels are HBM-bound with fp32 accumulation in a fixed order
// (deterministic): the combine and its backward stream rows (one warp per row,
// 16-byte vectors); the router backward forms dlogits with a few lanes per token,
// then dX and the dW_r partials on mma.sync tiles, reduced in one more pass.
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

__host__ __device__ constexpr size_t align_up_dev(size_t b) { return (b + 255) / 256 * 256; }

// out[t] = sum_j gate[t,j] * y_perm[slot_of[t,j]] (kept slots, j ascending),
// plus y_shared[t] (the shared experts, weight 1) when given.
// One warp per token; for each group of U 16-byte vectors per lane the loads of
// all k slots are issued before any is used (k * U = 8 loads in flight per
// lane), then summed in slot order.
template <typename T, int KMAX, int U>
__global__ void __launch_bounds__(256) combine_kernel(const T* __restrict__ y_perm,
                                                      const int32_t* __restrict__ slot_of,
                                                      const float* __restrict__ gate,
                                                      const T* __restrict__ y_shared, int Tn,
                                                      int d, int k, T* __restrict__ out)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    constexpr int V = 16 / sizeof(T);
    const int nv = d / V;
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < Tn; t += warps) {
        int slot[KMAX];
        float g[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            slot[j] = j < k ? slot_of[(size_t)t * k + j] : -1;
            g[j] = j < k ? gate[(size_t)t * k + j] : 0.f;
        }
        for (int v0 = lane; v0 < nv; v0 += 32 * U) {
            uint4 raw[KMAX][U];
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
#pragma unroll
                for (int u = 0; u < U; ++u)
                    raw[j][u] = (slot[j] >= 0 && v0 + 32 * u < nv)
                                    ? __ldg(reinterpret_cast<const uint4*>(y_perm + (size_t)slot[j] * d) + v0 + 32 * u)
                                    : make_uint4(0, 0, 0, 0);
            float acc[U][V];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int q = 0; q < V; ++q) acc[u][q] = 0.f;
            if (y_shared) {
                const T* row = y_shared + (size_t)t * d;
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (v0 + 32 * u < nv) load16_f<T>(row + (v0 + 32 * u) * V, acc[u]);
            }
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (slot[j] < 0) continue;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    float y[V];
                    load16_f<T>(reinterpret_cast<const T*>(&raw[j][u]), y);
#pragma unroll
                    for (int q = 0; q < V; ++q) acc[u][q] = fmaf(g[j], y[q], acc[u][q]);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (v0 + 32 * u < nv) store16_f<T>(out + (size_t)t * d + (v0 + 32 * u) * V, acc[u]);
        }
    }
}

// Row r of the permuted layout: dy_perm[r] = gate * dout[t]; dgate = <dout[t], y_perm[r]>.
// Slots without a row (dropped or padding tokens) get dgate = 0 in a first
// grid-stride pass over the Tn * k slots.
template <typename T>
__global__ void __launch_bounds__(256) combine_bwd_kernel(
    const T* __restrict__ dout, const T* __restrict__ y_perm, const float* __restrict__ gate,
    const int32_t* __restrict__ slot_of, const int32_t* __restrict__ perm_token,
    const int32_t* __restrict__ offsets, int Tn, int E, int d, int k, T* __restrict__ dy_perm,
    float* __restrict__ dgate)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < Tn * k; i += gridDim.x * blockDim.x)
        if (slot_of[i] < 0) dgate[i] = 0.f;
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

// W_r [d,E] -> W_rT [E,d] fp32 (router-backward operand)
template <typename T>
__global__ void transpose_wr_f32_kernel(const T* __restrict__ Wr, float* __restrict__ WrT, int d,
                                        int E)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    const size_t n = (size_t)E * d;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < n;
         idx += (size_t)gridDim.x * blockDim.x) {
        int e = (int)(idx / d), i = (int)(idx % d);
        WrT[idx] = to_f<T>(Wr[(size_t)i * E + e]);
    }
}

// The fp32 path's router backward, one warp per token: dlogits (gate Jacobian +
// aux term); with WITH_DX also dx[t] = sum_kept dx_perm[slot] + dlogits[t] . W_r^T.
// (The bf16 path forms dlogits in router_dlogits_kernel and dx in
// router_dx_dwr_kernel on the tensor cores.)
template <typename T, bool WITH_DX>
__global__ void __launch_bounds__(256) router_bwd_token_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ topk,
    const float* __restrict__ gate, const int32_t* __restrict__ slot_of,
    const float* __restrict__ dgate, const float* __restrict__ stats,
    const T* __restrict__ dx_perm, const T* __restrict__ dx_shared, const float* __restrict__ WrT,
    int Tn, int d, int E, int k, int normalize, int st, float inv_tau, float aux_coef,
    float* __restrict__ dlogits, T* __restrict__ dx)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    constexpr int V = 16 / sizeof(T);
    __shared__ float s_dl[8][64];
    const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nv = d / V;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int t = blockIdx.x * (blockDim.x >> 5) + wib; t < Tn; t += warps) {
        // lanes hold experts e = lane and lane + 32
        // p = softmax(l / tau); every derivative through it carries 1 / tau
        float l0 = lane < E ? logits[(size_t)t * E + lane] * inv_tau : -INFINITY;
        float l1 = lane + 32 < E ? logits[(size_t)t * E + lane + 32] * inv_tau : -INFINITY;
        const float m = warp_max(fmaxf(l0, l1));
        float p0 = lane < E ? expf(l0 - m) : 0.f;
        float p1 = lane + 32 < E ? expf(l1 - m) : 0.f;
        const float z = warp_sum(p0 + p1);
        p0 /= z;
        p1 /= z;
        float dl0 = 0.f, dl1 = 0.f;
        const bool routed = topk[(size_t)t * k] >= 0;   // padding tokens: no gradient
        if (!routed) {
        } else if (normalize && !st) {
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
            // raw probabilities, and the straight-through estimator (gates 1 forward,
            // gradient through p of the selected experts)
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
        if (routed && aux_coef != 0.f) {
            const float invE = 1.0f / (float)E;
            const float sc = aux_coef * 2.0f / fmaxf(stats[MOE_STAT_TOKENS], 1.0f);
            const float c0 = lane < E ? sc * (stats[MOE_STAT_PBAR + lane] - invE) : 0.f;
            const float c1 = lane + 32 < E ? sc * (stats[MOE_STAT_PBAR + lane + 32] - invE) : 0.f;
            const float s2 = warp_sum(p0 * c0 + p1 * c1);
            dl0 += p0 * (c0 - s2);
            dl1 += p1 * (c1 - s2);
        }
        dl0 *= inv_tau;
        dl1 *= inv_tau;
        if (lane < E) { dlogits[(size_t)t * E + lane] = dl0; s_dl[wib][lane] = dl0; }
        if (lane + 32 < E) { dlogits[(size_t)t * E + lane + 32] = dl1; s_dl[wib][lane + 32] = dl1; }
        if (!WITH_DX) continue;
        __syncwarp();
        int slot[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) slot[j] = j < k ? slot_of[(size_t)t * k + j] : -1;
        for (int v = lane; v < nv; v += 32) {
            float acc[V];
#pragma unroll
            for (int q = 0; q < V; ++q) acc[q] = 0.f;
            if (dx_shared) load16_f<T>(dx_shared + (size_t)t * d + v * V, acc);
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

// dlogits for the bf16 path (dX and dW_r follow on the tensor cores): G lanes per
// token (G = the expert count rounded up to a power of two, at most 32; a lane holds
// experts sub and sub + G), 32 / G tokens per warp.  Every load of a token (logits,
// its k picks, gates, slots and dgates) is issued before any is used, and the
// softmax, gate Jacobian and aux term reduce over the token's G lanes; the token
// loop and every shuffle are uniform across the warp.
template <int G>
__global__ void __launch_bounds__(256) router_dlogits_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ topk,
    const float* __restrict__ gate, const int32_t* __restrict__ slot_of,
    const float* __restrict__ dgate, const float* __restrict__ stats, int Tn, int E, int k,
    int normalize, int st, float inv_tau, float aux_coef, float* __restrict__ dlogits)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    constexpr int TPW = 32 / G;
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31, sub = lane % G, gbase = lane - sub;
    const int e0 = sub, e1 = sub + G;
    // the aux term's per-expert coefficients (the statistics are final)
    float c0 = 0.f, c1 = 0.f;
    if (aux_coef != 0.f) {
        const float invE = 1.0f / (float)E;
        const float sc = aux_coef * 2.0f / fmaxf(stats[MOE_STAT_TOKENS], 1.0f);
        if (e0 < E) c0 = sc * (stats[MOE_STAT_PBAR + e0] - invE);
        if (e1 < E) c1 = sc * (stats[MOE_STAT_PBAR + e1] - invE);
    }
    const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nw = (int)((gridDim.x * blockDim.x) >> 5);
    for (int tw = gw * TPW; tw < Tn; tw += nw * TPW) {      // uniform per warp
        const int t = tw + lane / G;
        const bool valid = t < Tn;
        const size_t tb = (size_t)(valid ? t : 0);
        const float x0 = (valid && e0 < E) ? logits[tb * E + e0] : 0.f;
        const float x1 = (valid && e1 < E) ? logits[tb * E + e1] : 0.f;
        int tk[8], so[8];
        float gt[8], dgr[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const bool in = valid && j < k;
            tk[j] = in ? topk[tb * k + j] : -1;
            so[j] = in ? slot_of[tb * k + j] : -1;
            gt[j] = in ? gate[tb * k + j] : 0.f;
            dgr[j] = in ? dgate[tb * k + j] : 0.f;
        }
        // p = softmax(l / tau); every derivative through it carries 1 / tau
        const float l0 = e0 < E ? x0 * inv_tau : -INFINITY;
        const float l1 = e1 < E ? x1 * inv_tau : -INFINITY;
        float m = fmaxf(l0, l1);
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(full, m, off));
        float p0 = e0 < E ? expf(l0 - m) : 0.f;
        float p1 = e1 < E ? expf(l1 - m) : 0.f;
        float z = p0 + p1;
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) z += __shfl_xor_sync(full, z, off);
        p0 /= z;
        p1 /= z;
        const bool routed = valid && tk[0] >= 0;   // padding tokens: no gradient
        float dl0 = 0.f, dl1 = 0.f;
        if (normalize && !st) {
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float dg = so[j] >= 0 ? dgr[j] : 0.f;
                s += gt[j] * dg;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (j >= k) break;
                const float dg = so[j] >= 0 ? dgr[j] : 0.f;
                const float v = gt[j] * (dg - s);
                if (tk[j] == e0) dl0 += v;
                if (tk[j] == e1) dl1 += v;
            }
        } else {
            // raw probabilities, and the straight-through estimator (gates 1 forward,
            // gradient through p of the selected experts); p of a pick comes from the
            // lane that holds it (every lane shuffles, whatever its token)
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (j >= k) break;
                const int e = tk[j] >= 0 ? tk[j] : 0;
                const int src = gbase + (e % G);
                const float pa = __shfl_sync(full, p0, src);
                const float pb = __shfl_sync(full, p1, src);
                const float dg = so[j] >= 0 ? dgr[j] : 0.f;
                s += dg * (e < G ? pa : pb);
                if (tk[j] == e0) dl0 += dg * p0;
                if (tk[j] == e1) dl1 += dg * p1;
            }
            dl0 -= p0 * s;
            dl1 -= p1 * s;
        }
        float s2 = p0 * c0 + p1 * c1;
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) s2 += __shfl_xor_sync(full, s2, off);
        if (aux_coef != 0.f) {
            dl0 += p0 * (c0 - s2);
            dl1 += p1 * (c1 - s2);
        }
        if (!routed) dl0 = dl1 = 0.f;
        if (valid && e0 < E) dlogits[tb * E + e0] = dl0 * inv_tau;
        if (valid && e1 < E) dlogits[tb * E + e1] = dl1 * inv_tau;
    }
}

// dx for the bf16 path: dx[t] = sum_kept dx_perm[slot] + dlogits[t] . W_r^T.
// The router term is a [T, E] x [E, d] contraction with K = E (<= 64): it runs
// on the tensor cores (mma.sync m16n8k16, bf16 operands, fp32 accumulate)
// with the CTA's 128 columns of W_r staged once in shared memory, so W_r is
// not re-read per token.  CTA = 8 warps sharing one 128-column chunk; a warp
// takes 16-token tiles: 16 MMA n-tiles write the router term to its smem
// tile, then half-warps add the kept dx_perm rows (16-byte vectors) and store.
constexpr int RDX_CW = 128;  // columns per CTA

// CTA (bx, by) of a gx x gy grid: column chunk bx, 16-token tiles by, by + gy, ...
template <int KS>  // KS = ceil(E / 16) k-steps
__device__ __forceinline__ void router_dx_body(
    const float* __restrict__ dlogits, const __nv_bfloat16* __restrict__ Wr,
    const int32_t* __restrict__ slot_of, const __nv_bfloat16* __restrict__ dx_perm,
    const __nv_bfloat16* __restrict__ dx_shared, int Tn, int d, int E, int k,
    __nv_bfloat16* __restrict__ dx, int bx, int by, int gy, uint8_t* smem_raw)
{
    constexpr int E16 = KS * 16, LDW = E16 + 2, LDO = RDX_CW + 4;
    __nv_bfloat16* sW = reinterpret_cast<__nv_bfloat16*>(smem_raw);                 // [128][LDW]
    float* sOut = reinterpret_cast<float*>(smem_raw + align_up_dev(RDX_CW * LDW * 2)); // [8][16][LDO]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int hl = lane & 15, hw = lane >> 4;
    const int c0 = bx * RDX_CW;
    const int col = c0 + hl * 8;
    for (int i = tid; i < RDX_CW * E16; i += 256) {
        const int cc = i / E16, e = i % E16;
        sW[cc * LDW + e] = (e < E && c0 + cc < d) ? Wr[(size_t)(c0 + cc) * E + e]
                                                  : __float2bfloat16_rn(0.f);
    }
    __syncthreads();
    float* so = sOut + warp * 16 * LDO;
    const int ntiles = (Tn + 15) / 16;
    for (int wt = by * 8 + warp; wt < ntiles; wt += gy * 8) {
        const int t0 = wt * 16;
        // round trip 1: this tile's dlogits (A fragments) and the half-warp's
        // first two slot indices for its 8 tokens, all independent loads
        auto dl_pair = [&](int row, int e) -> uint32_t {
            const int t = t0 + row;
            const float lo = (t < Tn && e < E) ? __ldg(dlogits + (size_t)t * E + e) : 0.f;
            const float hi = (t < Tn && e + 1 < E) ? __ldg(dlogits + (size_t)t * E + e + 1) : 0.f;
            __nv_bfloat162 bb = __floats2bfloat162_rn(lo, hi);
            return *reinterpret_cast<uint32_t*>(&bb);
        };
        uint32_t a[KS][4];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            a[ks][0] = dl_pair(g, ks * 16 + 2 * tq);
            a[ks][1] = dl_pair(g + 8, ks * 16 + 2 * tq);
            a[ks][2] = dl_pair(g, ks * 16 + 2 * tq + 8);
            a[ks][3] = dl_pair(g + 8, ks * 16 + 2 * tq + 8);
        }
        int sl[2][8];
        auto load_slots = [&](int j0) {
#pragma unroll
            for (int jj = 0; jj < 2; ++jj)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int t = t0 + hw + 2 * i;
                    sl[jj][i] = (t < Tn && j0 + jj < k) ? __ldg(slot_of + (size_t)t * k + j0 + jj) : -1;
                }
        };
        load_slots(0);
        // router term of the 16 tokens x 128 columns on the tensor cores
#pragma unroll 4
        for (int nt = 0; nt < RDX_CW / 8; ++nt) {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            const __nv_bfloat16* wrow = sW + (nt * 8 + g) * LDW;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(wrow + ks * 16 + 2 * tq);
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(wrow + ks * 16 + 2 * tq + 8);
                asm volatile(
                    "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                    "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                    : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                    : "r"(a[ks][0]), "r"(a[ks][1]), "r"(a[ks][2]), "r"(a[ks][3]), "r"(b0), "r"(b1));
            }
            so[g * LDO + nt * 8 + 2 * tq] = c[0];
            so[g * LDO + nt * 8 + 2 * tq + 1] = c[1];
            so[(g + 8) * LDO + nt * 8 + 2 * tq] = c[2];
            so[(g + 8) * LDO + nt * 8 + 2 * tq + 1] = c[3];
        }
        __syncwarp();
        // round trip 2 (per pair of slots): 16 row loads in flight per lane (and the
        // shared experts' rows with the last pair); a half-warp covers the chunk's
        // 128 columns for 8 tokens.  The router term waits in shared memory, so
        // only the loads occupy registers; partial sums of k > 2 go back there.
        if (col < d) {
            for (int j0 = 0; j0 < k; j0 += 2) {
                if (j0 > 0) load_slots(j0);
                const bool last = j0 + 2 >= k;
                uint4 y[2][8], ys[8];
#pragma unroll
                for (int jj = 0; jj < 2; ++jj)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        y[jj][i] = sl[jj][i] >= 0
                                       ? __ldg(reinterpret_cast<const uint4*>(dx_perm + (size_t)sl[jj][i] * d + col))
                                       : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int t = t0 + hw + 2 * i;
                    ys[i] = (last && dx_shared && t < Tn)
                                ? __ldg(reinterpret_cast<const uint4*>(dx_shared + (size_t)t * d + col))
                                : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = hw + 2 * i;
                    float* sp = so + r * LDO + hl * 8;
                    const float4 s0 = *reinterpret_cast<const float4*>(sp);
                    const float4 s1 = *reinterpret_cast<const float4*>(sp + 4);
                    float a8[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                    const uint4 src[3] = {y[0][i], y[1][i], ys[i]};
#pragma unroll
                    for (int m = 0; m < 3; ++m) {
                        const uint32_t w4[4] = {src[m].x, src[m].y, src[m].z, src[m].w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            a8[2 * q] += __uint_as_float(w4[q] << 16);
                            a8[2 * q + 1] += __uint_as_float(w4[q] & 0xFFFF0000u);
                        }
                    }
                    if (last) {
                        const int t = t0 + r;
                        if (t < Tn) store16_f<__nv_bfloat16>(dx + (size_t)t * d + col, a8);
                    } else {
                        *reinterpret_cast<float4*>(sp) = make_float4(a8[0], a8[1], a8[2], a8[3]);
                        *reinterpret_cast<float4*>(sp + 4) = make_float4(a8[4], a8[5], a8[6], a8[7]);
                    }
                }
            }
        }
        __syncwarp();
    }
}

// dW_r on the tensor cores (bf16 path): part[s][i][e] = sum over the token chunk s
// of x[t,i] dlogits[t,e], as the [E16 x 16 tokens] x [16 tokens x 8 cols] MMAs
// dl^T x.  CTA = 4 warps on a 128-column chunk (32 columns each); 16-token x
// tiles stream through a 4-stage cp.async ring; dlogits are staged transposed
// (tokens contiguous) so the A fragments are plain 32-bit loads; B fragments come
// from ldmatrix.trans of the row-major x tile.  Column-chunk-0 CTAs also sum
// dlogits over the chunk for dbias.
constexpr int DWM_STAGES = 4, DWM_LDX = 128 + 8;

// shared memory of one 128-thread dW_r unit: x ring, dlogits ring, dbias partials
template <int MT>
constexpr size_t dwr_unit_smem() {
    return (size_t)DWM_STAGES * 16 * DWM_LDX * 2 + (size_t)DWM_STAGES * 16 * MT * 16 * 4 + 128 * 4;
}

// 128 threads (tid 0..127, named barrier `bar`) on column chunk bx, token chunk by
template <int MT>  // MT = ceil(E / 16) expert m-tiles
__device__ __forceinline__ void dwr_mma_body(const __nv_bfloat16* __restrict__ x,
                                             const float* __restrict__ dlogits, int Tn, int d, int E,
                                             int chunk, float* __restrict__ part,
                                             float* __restrict__ part_db, int bx, int by, int tid,
                                             uint8_t* smem, int bar)
{
    constexpr int E16 = MT * 16;
    auto sX = reinterpret_cast<__nv_bfloat16 (*)[16][DWM_LDX]>(smem);
    auto sDf = reinterpret_cast<float (*)[16][E16]>(smem + (size_t)DWM_STAGES * 16 * DWM_LDX * 2);  // [token][expert]
    float* sDb = reinterpret_cast<float*>(smem + (size_t)DWM_STAGES * 16 * DWM_LDX * 2 +
                                          (size_t)DWM_STAGES * 16 * E16 * 4);
    auto hsync = [bar]() {   // immediate barrier ids: the CTA uses barriers 0-2 only
        if (bar == 1) asm volatile("bar.sync 1, 128;" ::: "memory");
        else asm volatile("bar.sync 2, 128;" ::: "memory");
    };
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int c0 = bx * 128;
    const int tbeg = by * chunk, tend = min(Tn, tbeg + chunk);
    const int nblk16 = (tend - tbeg + 15) / 16;
    // dlogits rows stream with cp.async too when they are 16-byte granular (E % 4
    // == 0), so no synchronous load stalls the ring; columns E..E16 stay zero
    const bool async_dl = (E & 3) == 0;
    for (int i = tid; i < DWM_STAGES * 16 * E16; i += 128) (&sDf[0][0][0])[i] = 0.f;
    hsync();
    float db = 0.f;  // this thread's dbias share (expert tid, tid < E16), column chunk 0 only
    auto load = [&](int b, int st) {
        const int t0 = tbeg + b * 16;
        // x tile: 16 rows x 128 columns = 256 vectors of 16 bytes, two per thread
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int v = tid + r * 128;
            const int row = v >> 4, cv = v & 15;
            const int t = t0 + row, cc = c0 + cv * 8;
            const bool ok = t < tend && cc < d;
            const __nv_bfloat16* src = ok ? x + (size_t)t * d + cc : x;
            const uint32_t dst = (uint32_t)__cvta_generic_to_shared(&sX[st][row][cv * 8]);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                         "r"(ok ? 16 : 0));
        }
        if (async_dl) {
            const int q4 = E >> 2;                       // 16-byte pieces per token row
            for (int i = tid; i < 16 * q4; i += 128) {
                const int row = i / q4, c4 = i % q4;
                const int t = t0 + row;
                const bool ok = t < tend;
                const float* src = ok ? dlogits + (size_t)t * E + c4 * 4 : dlogits;
                const uint32_t dst = (uint32_t)__cvta_generic_to_shared(&sDf[st][row][c4 * 4]);
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                             "r"(ok ? 16 : 0));
            }
        } else {
            for (int i = tid; i < 16 * E; i += 128) {
                const int row = i / E, e = i % E;
                const int t = t0 + row;
                sDf[st][row][e] = t < tend ? __ldg(dlogits + (size_t)t * E + e) : 0.f;
            }
        }
    };
    auto pack2 = [](float lo, float hi) -> uint32_t {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&b2);
    };
    float acc[MT][4][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n) acc[m][n][0] = acc[m][n][1] = acc[m][n][2] = acc[m][n][3] = 0.f;
#pragma unroll
    for (int s = 0; s < DWM_STAGES - 1; ++s) {
        if (s < nblk16) load(s, s);
        asm volatile("cp.async.commit_group;\n" ::);
    }
    for (int b = 0; b < nblk16; ++b) {
        asm volatile("cp.async.wait_group %0;\n" ::"n"(DWM_STAGES - 2));
        hsync();
        const int st = b % DWM_STAGES;
        // A = dlogits^T (rows experts, k = tokens), bf16 pairs of consecutive tokens
        uint32_t af[MT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const int e0 = m * 16 + g;
            af[m][0] = pack2(sDf[st][2 * tq][e0], sDf[st][2 * tq + 1][e0]);
            af[m][1] = pack2(sDf[st][2 * tq][e0 + 8], sDf[st][2 * tq + 1][e0 + 8]);
            af[m][2] = pack2(sDf[st][2 * tq + 8][e0], sDf[st][2 * tq + 9][e0]);
            af[m][3] = pack2(sDf[st][2 * tq + 8][e0 + 8], sDf[st][2 * tq + 9][e0 + 8]);
        }
        if (bx == 0 && tid < E16)
#pragma unroll
            for (int r = 0; r < 16; ++r) db += sDf[st][r][tid];
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            // B (k = token, n = column) from the row-major [token][col] tile
            const int ncol = warp * 32 + n * 8;
            const uint32_t addr = (uint32_t)__cvta_generic_to_shared(&sX[st][lane & 15][ncol]);
            uint32_t b0, b1;
            asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];\n"
                         : "=r"(b0), "=r"(b1) : "r"(addr));
#pragma unroll
            for (int m = 0; m < MT; ++m)
                asm volatile(
                    "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                    "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                    : "+f"(acc[m][n][0]), "+f"(acc[m][n][1]), "+f"(acc[m][n][2]), "+f"(acc[m][n][3])
                    : "r"(af[m][0]), "r"(af[m][1]), "r"(af[m][2]), "r"(af[m][3]), "r"(b0), "r"(b1));
        }
        // the refill targets the stage read in the previous iteration (all threads
        // passed this iteration's barrier after reading it)
        const int nxt = b + DWM_STAGES - 1;
        if (nxt < nblk16) load(nxt, nxt % DWM_STAGES);
        asm volatile("cp.async.commit_group;\n" ::);
    }
    asm volatile("cp.async.wait_group 0;\n" ::);
    // C fragment: rows = experts (g, g+8 of m-tile m), cols = 2tq, 2tq+1 of n-tile n
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const int colb = c0 + warp * 32 + n * 8 + 2 * tq;
            const int e_lo = m * 16 + g, e_hi = e_lo + 8;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int cc = colb + h;
                if (cc >= d) continue;
                float* dst = part + ((size_t)by * d + cc) * E;
                if (e_lo < E) dst[e_lo] = acc[m][n][h];
                if (e_hi < E) dst[e_hi] = acc[m][n][2 + h];
            }
        }
    if (bx == 0) {
        sDb[tid] = db;
        hsync();
        if (tid < E) {
            float a = 0.f;
            for (int i = tid; i < 128; i += E16) a += sDb[i];
            part_db[(size_t)by * E + tid] = a;
        }
    }
}

// dX and the dW_r partials in one launch (both read dlogits only; they run side
// by side): CTAs 0 .. n_dx - 1 form the gx x gy grid of the dX body, the rest run
// two 128-thread dW_r units each over the gxm x ns grid of (column, token) chunks.
template <int KS>
__global__ void __launch_bounds__(256, 2) router_dx_dwr_kernel(
    const float* __restrict__ dlogits, const __nv_bfloat16* __restrict__ Wr,
    const int32_t* __restrict__ slot_of, const __nv_bfloat16* __restrict__ dx_perm,
    const __nv_bfloat16* __restrict__ dx_shared, const __nv_bfloat16* __restrict__ x, int Tn,
    int d, int E, int k, __nv_bfloat16* __restrict__ dx, int gx, int gy, int chunk, int gxm,
    int ns, float* __restrict__ part, float* __restrict__ part_db)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int bid = blockIdx.x, n_dx = gx * gy;
    if (bid < n_dx) {
        router_dx_body<KS>(dlogits, Wr, slot_of, dx_perm, dx_shared, Tn, d, E, k, dx, bid % gx,
                           bid / gx, gy, smem_raw);
        return;
    }
    const int half = threadIdx.x >> 7;
    const int u = 2 * (bid - n_dx) + half;   // this unit's (column chunk, token chunk)
    if (u >= gxm * ns) return;               // (its barrier is its own: the other unit runs on)
    dwr_mma_body<KS>(x, dlogits, Tn, d, E, chunk, part, part_db, u % gxm, u / gxm, threadIdx.x & 127,
                     smem_raw + half * dwr_unit_smem<KS>(), 1 + half);
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
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    constexpr int V = 16 / sizeof(T);
    extern __shared__ __align__(16) float red[];          // [8][32][V*EB]
    // grid: x = expert group (fastest, so the groups of one x tile run together and
    // the later ones read it from L2), y = column block, z = token chunk
    const int tid = threadIdx.x, tl = tid >> 5, cv = tid & 31;
    const int col0 = (blockIdx.y * 32 + cv) * V;
    const int e0 = blockIdx.x * EB;
    const int s = blockIdx.z;
    const int tbeg = s * chunk, tend = min(Tn, tbeg + chunk);
    const bool colok = col0 < d;
    float acc[V][EB];
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
        for (int e = 0; e < EB; ++e) acc[v][e] = 0.f;
    auto consume = [&](const float* xv, int t) {
        float dl[EB];
#pragma unroll
        for (int e = 0; e < EB; ++e) dl[e] = (e0 + e < E) ? __ldg(dlogits + (size_t)t * E + e0 + e) : 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v)
#pragma unroll
            for (int e = 0; e < EB; ++e) acc[v][e] = fmaf(xv[v], dl[e], acc[v][e]);
    };
    int t = tbeg + tl;
    if (colok) {
        for (; t + 24 < tend; t += 32) {   // four rows of this lane in flight
            float xa[V], xb[V], xc[V], xd[V];
            load16_f<T>(x + (size_t)t * d + col0, xa);
            load16_f<T>(x + (size_t)(t + 8) * d + col0, xb);
            load16_f<T>(x + (size_t)(t + 16) * d + col0, xc);
            load16_f<T>(x + (size_t)(t + 24) * d + col0, xd);
            consume(xa, t);
            consume(xb, t + 8);
            consume(xc, t + 16);
            consume(xd, t + 24);
        }
        for (; t < tend; t += 8) {
            float xa[V];
            load16_f<T>(x + (size_t)t * d + col0, xa);
            consume(xa, t);
        }
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
        const int col = (blockIdx.y * 32 + c) * V + v;
        if (col < d && e0 + e < E) part[((size_t)s * d + col) * E + e0 + e] = a;
    }
    if (blockIdx.x == 0 && blockIdx.y == 0 && tid < E) {
        float a = 0.f;
        for (int t = tbeg; t < tend; ++t) a += dlogits[(size_t)t * E + tid];
        part_db[(size_t)s * E + tid] = a;
    }
}

// dW_r = sum of the nsplit token-chunk partials (and dbias likewise).  A CTA
// covers 64 four-column vectors with 4 groups of lanes; each group sums every
// fourth partial with all of its loads independent (one memory round trip for
// up to 32 partials), then the 4 group sums are added in a fixed order.
constexpr int DWR_RED_COLS = 64, DWR_RED_GROUPS = 4;

template <typename T>
__global__ void __launch_bounds__(DWR_RED_COLS * DWR_RED_GROUPS) dwr_reduce_kernel(
    const float* __restrict__ part, const float* __restrict__ part_db, int nsplit, int d, int E,
    T* __restrict__ dWr, float* __restrict__ dbias)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    __shared__ float4 s_acc[DWR_RED_GROUPS][DWR_RED_COLS];
    const int n4 = d * E / 4;                    // d * E is a multiple of 4 (d % 8 == 0)
    const int col = threadIdx.x % DWR_RED_COLS, grp = threadIdx.x / DWR_RED_COLS;
    const int i4 = blockIdx.x * DWR_RED_COLS + col;
    const float4* p4 = reinterpret_cast<const float4*>(part);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i4 < n4) {
        int s0 = grp;
        for (; s0 + 7 * DWR_RED_GROUPS < nsplit; s0 += 8 * DWR_RED_GROUPS) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldg(p4 + (size_t)(s0 + u * DWR_RED_GROUPS) * n4 + i4);
#pragma unroll
            for (int u = 0; u < 8; ++u) { a.x += v[u].x; a.y += v[u].y; a.z += v[u].z; a.w += v[u].w; }
        }
        for (; s0 < nsplit; s0 += DWR_RED_GROUPS) {
            const float4 v = __ldg(p4 + (size_t)s0 * n4 + i4);
            a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
        }
    }
    s_acc[grp][col] = a;
    __syncthreads();
    if (grp == 0 && i4 < n4) {
#pragma unroll
        for (int g = 1; g < DWR_RED_GROUPS; ++g) {
            const float4 b = s_acc[g][col];
            a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
        }
        const float o[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) dWr[(size_t)i4 * 4 + q] = from_f<T>(o[q]);
    }
    if (dbias && blockIdx.x == 0 && threadIdx.x < E) {
        float b = 0.f;
        for (int s = 0; s < nsplit; ++s) b += part_db[(size_t)s * E + threadIdx.x];
        dbias[threadIdx.x] = b;
    }
}

constexpr int DWR_EB = 8;  // experts per CTA of dwr_partial_kernel

// grid of dwr_partial_kernel without the token-chunk dimension (z)
dim3 dwr_grid_xy(const moe_config& c) {
    const int V = c.dtype == MOE_DTYPE_BF16 ? 8 : 4;
    return dim3((c.E + DWR_EB - 1) / DWR_EB, (c.d + 32 * V - 1) / (32 * V), 1);
}

// token chunks of the dW_r partial kernels: enough CTAs to fill the GPU, at most
// 32 chunks so the final fixed-order reduction stays short
int dwr_nsplit(const moe_config& c) {
    if (c.dtype == MOE_DTYPE_BF16) {
        const int per = (c.d + 127) / 128;
        const int ns = (8 * num_sms() + per - 1) / per;
        return std::max(1, std::min(std::min(ns, 32), (c.T + 15) / 16));
    }
    const dim3 g = dwr_grid_xy(c);
    const int per = (int)(g.x * g.y);
    int ns = std::max(1, (4 * num_sms() + per - 1) / per);
    return std::min(ns, std::max(1, (c.T + 63) / 64));
}

int dwr_chunk(const moe_config& c, int ns) {
    const int ch = (c.T + ns - 1) / ns;
    return c.dtype == MOE_DTYPE_BF16 ? (ch + 15) / 16 * 16 : ch;
}

int row_grid(int64_t rows) {
    return (int)std::max<int64_t>(1, std::min<int64_t>((rows + 7) / 8, (int64_t)num_sms() * 16));
}

}  // namespace

template <typename T, int KMAX, int U>
int launch_combine_t(const moe_config& c, const void* y_perm, const int32_t* slot_of,
                     const float* gate, const void* y_shared, void* out, cudaStream_t st) {
    MOE_LAUNCH(combine_kernel<T, KMAX, U>, row_grid(c.T), 256, 0, st, static_cast<const T*>(y_perm),
               slot_of, gate, static_cast<const T*>(y_shared), c.T, c.d, c.k, static_cast<T*>(out));
    return MOE_OK;
}

template <typename T>
int launch_combine_k(const moe_config& c, const void* y_perm, const int32_t* slot_of,
                     const float* gate, const void* y_shared, void* out, cudaStream_t st) {
    if (c.k <= 1) return launch_combine_t<T, 1, 8>(c, y_perm, slot_of, gate, y_shared, out, st);
    if (c.k <= 2) return launch_combine_t<T, 2, 4>(c, y_perm, slot_of, gate, y_shared, out, st);
    if (c.k <= 4) return launch_combine_t<T, 4, 2>(c, y_perm, slot_of, gate, y_shared, out, st);
    return launch_combine_t<T, 8, 1>(c, y_perm, slot_of, gate, y_shared, out, st);
}

int launch_combine(const moe_config& c, const void* y_perm, const int32_t* slot_of,
                   const float* gate, const void* y_shared, void* out, cudaStream_t st)
{
    if (c.dtype == MOE_DTYPE_BF16)
        return launch_combine_k<__nv_bfloat16>(c, y_perm, slot_of, gate, y_shared, out, st);
    return launch_combine_k<float>(c, y_perm, slot_of, gate, y_shared, out, st);
}

int launch_combine_backward(const moe_config& c, const void* dout, const void* y_perm,
                            const float* gate, const int32_t* slot_of, const int32_t* perm_token,
                            const int32_t* offsets, void* dy_perm, float* dgate, cudaStream_t st)
{
    const int grid = row_grid(rows_cap_of(c));
    if (c.dtype == MOE_DTYPE_BF16)
        MOE_LAUNCH(combine_bwd_kernel<__nv_bfloat16>, grid, 256, 0, st, static_cast<const __nv_bfloat16*>(dout), static_cast<const __nv_bfloat16*>(y_perm),
            gate, slot_of, perm_token, offsets, c.T, c.E, c.d, c.k,
            static_cast<__nv_bfloat16*>(dy_perm), dgate);
    else
        MOE_LAUNCH(combine_bwd_kernel<float>, grid, 256, 0, st, static_cast<const float*>(dout), static_cast<const float*>(y_perm), gate, slot_of,
            perm_token, offsets, c.T, c.E, c.d, c.k, static_cast<float*>(dy_perm), dgate);
    return MOE_OK;
}

#define MOE_TRY_R(x)                   \
    do {                               \
        int _r = (x);                  \
        if (_r != MOE_OK) return _r;   \
    } while (0)

namespace {
// dX and the dW_r partials (bf16): one launch of router_dx_dwr_kernel
template <int KS>
int launch_router_dx_dwr_ks(const moe_config& c, const float* dl, const __nv_bfloat16* Wr,
                            const int32_t* slot_of, const __nv_bfloat16* dxp,
                            const __nv_bfloat16* dxs, const __nv_bfloat16* x, __nv_bfloat16* dx,
                            int chunk, int ns, float* part, float* part_db, cudaStream_t st) {
    constexpr int LDW = KS * 16 + 2;
    const size_t smem_dx = align_up_dev((size_t)RDX_CW * LDW * 2) + (size_t)8 * 16 * (RDX_CW + 4) * 4;
    const size_t smem = std::max(smem_dx, 2 * dwr_unit_smem<KS>());
    static bool attr[64] = {};
    if (const int r = smem_attr_once(router_dx_dwr_kernel<KS>, smem, attr)) return r;
    const int gx = (c.d + RDX_CW - 1) / RDX_CW;
    const int tiles = (c.T + 15) / 16;
    // the dX part: one wave of the resident CTA slots (2 per SM) at most
    const int gy = std::max(1, std::min((tiles + 7) / 8, (2 * num_sms()) / gx));
    const int gxm = (c.d + 127) / 128;
    const int n_dwr = (gxm * ns + 1) / 2;   // two dW_r units per CTA
    MOE_LAUNCH(router_dx_dwr_kernel<KS>, gx * gy + n_dwr, 256, smem, st, dl, Wr, slot_of, dxp, dxs, x,
               c.T, c.d, c.E, c.k, dx, gx, gy, chunk, gxm, ns, part, part_db);
    return MOE_OK;
}
}  // namespace

size_t router_bwd_ws_bytes(const moe_config& c) {
    const int ns = dwr_nsplit(c);
    return align_up((size_t)c.E * c.d * 4) + align_up((size_t)ns * c.d * c.E * 4) +
           align_up((size_t)ns * c.E * 4) + align_up((size_t)c.T * c.E * 4);
}

int launch_router_backward(const moe_config& c, const void* x, const void* Wr,
                           const float* logits, const int32_t* topk, const float* gate,
                           const int32_t* slot_of, const float* dgate, const void* dx_perm,
                           const void* dx_shared, const float* stats, void* dx, void* dWr,
                           float* dbias, float* dlogits, void* ws, cudaStream_t st)
{
    const int ns = dwr_nsplit(c);
    uint8_t* w = static_cast<uint8_t*>(ws);
    float* WrT = reinterpret_cast<float*>(w); w += align_up((size_t)c.E * c.d * 4);
    float* part = reinterpret_cast<float*>(w); w += align_up((size_t)ns * c.d * c.E * 4);
    float* part_db = reinterpret_cast<float*>(w); w += align_up((size_t)ns * c.E * 4);
    if (!dlogits) dlogits = reinterpret_cast<float*>(w);
    const int chunk = dwr_chunk(c, ns);
    const int grid = row_grid(c.T);
    const float inv_tau = c.temperature > 0.f ? 1.0f / c.temperature : 1.0f;
    dim3 pgrid = dwr_grid_xy(c);
    pgrid.z = ns;
    // reduction buffer: 8 token lanes x 32 vectors x (V * EB) floats, V = 16 / sizeof(T)
    const size_t dwr_smem = (size_t)8 * 32 * (c.dtype == MOE_DTYPE_BF16 ? 8 : 4) * DWR_EB * sizeof(float);
    if (c.dtype == MOE_DTYPE_BF16) {
        static bool attr[64] = {};
        if (const int r = smem_attr_once(dwr_partial_kernel<__nv_bfloat16, DWR_EB>, dwr_smem, attr)) return r;
    } else {
        static bool attr[64] = {};
        if (const int r = smem_attr_once(dwr_partial_kernel<float, DWR_EB>, dwr_smem, attr)) return r;
    }
    if (c.dtype == MOE_DTYPE_BF16) {
        using T = __nv_bfloat16;
        {
            const int g = c.E <= 2 ? 2 : c.E <= 4 ? 4 : c.E <= 8 ? 8 : c.E <= 16 ? 16 : 32;
            const int tok_per_cta = 8 * (32 / g);
            const int grid_dl = std::max(1, std::min((c.T + tok_per_cta - 1) / tok_per_cta, 8 * num_sms()));
#define MOE_DL(GG)                                                                                   \
    MOE_LAUNCH(router_dlogits_kernel<GG>, grid_dl, 256, 0, st, logits, topk, gate, slot_of, dgate,   \
               stats, c.T, c.E, c.k, c.normalize_gates, c.straight_through, inv_tau, c.aux_coef, \
               dlogits)
            if (g == 2) MOE_DL(2);
            else if (g == 4) MOE_DL(4);
            else if (g == 8) MOE_DL(8);
            else if (g == 16) MOE_DL(16);
            else MOE_DL(32);
#undef MOE_DL
        }
        const T* Wr_ = static_cast<const T*>(Wr);
        const T* dxp_ = static_cast<const T*>(dx_perm);
        const T* dxs_ = static_cast<const T*>(dx_shared);
        const T* x_ = static_cast<const T*>(x);
        T* dx_ = static_cast<T*>(dx);
        if (c.E <= 16)
            MOE_TRY_R(launch_router_dx_dwr_ks<1>(c, dlogits, Wr_, slot_of, dxp_, dxs_, x_, dx_, chunk, ns, part, part_db, st));
        else if (c.E <= 32)
            MOE_TRY_R(launch_router_dx_dwr_ks<2>(c, dlogits, Wr_, slot_of, dxp_, dxs_, x_, dx_, chunk, ns, part, part_db, st));
        else
            MOE_TRY_R(launch_router_dx_dwr_ks<4>(c, dlogits, Wr_, slot_of, dxp_, dxs_, x_, dx_, chunk, ns, part, part_db, st));
        MOE_LAUNCH(dwr_reduce_kernel<T>, (c.d * c.E / 4 + DWR_RED_COLS - 1) / DWR_RED_COLS, DWR_RED_COLS * DWR_RED_GROUPS, 0, st, part, part_db, ns, c.d, c.E, static_cast<T*>(dWr), dbias);
    } else {
        using T = float;
        MOE_LAUNCH(transpose_wr_f32_kernel<T>, 64, 256, 0, st, static_cast<const T*>(Wr), WrT, c.d, c.E);
        MOE_LAUNCH(router_bwd_token_kernel<T, true>, grid, 256, 0, st, logits, topk, gate, slot_of, dgate, stats, static_cast<const T*>(dx_perm),
            static_cast<const T*>(dx_shared), WrT, c.T, c.d, c.E, c.k, c.normalize_gates,
            c.straight_through, inv_tau, c.aux_coef, dlogits, static_cast<T*>(dx));
        MOE_LAUNCH(dwr_partial_kernel<T, DWR_EB>, pgrid, 256, dwr_smem, st, static_cast<const T*>(x), dlogits,
                                                                   c.T, c.d, c.E, chunk, part, part_db);
        MOE_LAUNCH(dwr_reduce_kernel<T>, (c.d * c.E / 4 + DWR_RED_COLS - 1) / DWR_RED_COLS, DWR_RED_COLS * DWR_RED_GROUPS, 0, st, part, part_db, ns, c.d, c.E, static_cast<T*>(dWr), dbias);
    }
    return MOE_OK;
}

}  // namespace moe
