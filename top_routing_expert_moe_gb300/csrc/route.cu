// route.cu -- router GEMM + softmax + top-k + gates + per-expert statistics.
//
// [LLaMA4-MoE] §2.4: a linear router with softmax scores over the experts,
// a [B,K] top-K index, outputs weighted by the post-softmax score.
// [ZeRO3-MoE] §5.3: gating in fp32 even for half-precision models.
//
// bf16: one CTA per TT tokens (16..128, chosen so the grid covers the GPU),
// 8 warps splitting each stage's 128 rows into (k-slice, 16 tokens); the x
// tile streams through a 4-stage cp.async ring (HBM-bound: x is read once);
// the router contraction runs on the tensor cores (mma.sync m16n8k16, fp32
// accumulate) so that the E flops/byte never throttle the HBM stream.  The
// logits tile lands in shared memory and one thread per token finishes the
// row: bias, noise, softmax, top-k, gates.  Per-CTA partial statistics are
// reduced in a fixed order by a one-CTA finalize kernel (deterministic).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int RT_TOK = 128;      // tokens per CTA
constexpr int RT_BK = 64;        // k-chunk (elements)
constexpr int RT_LDS = RT_BK + 8;  // smem row stride (bf16 elements), conflict-free
constexpr int RT_STAGES = 4;

struct RouteOut {
    int T, d, E, k, normalize;
    const float* bias;
    const float* noise;
    float* logits;
    int32_t* topk;
    float* gate;
    int32_t* part_counts;  // [nblk][E]
    float* part_psum;      // [nblk][E]
    float* part_ent;       // [nblk]
    int32_t* part_bad;     // [nblk]
};

// a ranks above b: larger logit; a NaN ranks below any number; then lower id
__device__ __forceinline__ bool ranks_above(float la, int a, float lb, int b) {
    bool na = isnan(la), nb = isnan(lb);
    if (na != nb) return nb;
    if (!na && la != lb) return la > lb;
    return a < b;
}

// Finish a tile of raw router sums held in sLog[tok][ldl]: one thread per
// token, then fixed-order column sums for the per-CTA statistics.
// sSel needs RT_TOK * k ints, sEnt/sBad RT_TOK entries.
__device__ void finish_tile(float* sLog, int ldl, int* sSel, float* sEnt, int* sBad,
                            int t0, int ntok, const RouteOut& o)
{
    const int E = o.E, k = o.k;
    const int i = threadIdx.x;
    if (i < ntok) {
        const int t = t0 + i;
        float* l = sLog + i * ldl;
        bool bad = false;
        float m = -INFINITY;
        for (int e = 0; e < E; ++e) {
            float v = l[e];
            if (o.bias) v += o.bias[e];
            if (o.noise) v += o.noise[(size_t)t * E + e];
            l[e] = v;
            o.logits[(size_t)t * E + e] = v;
            bad |= !isfinite(v);
            m = fmaxf(m, v);  // fmaxf ignores NaN
        }
        // top-k: k passes of "best not yet taken"
        int* sel = sSel + i * k;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            float bl = 0.f;
            for (int e = 0; e < E; ++e) {
                bool taken = false;
                for (int q = 0; q < j; ++q) taken |= (sel[q] == e);
                if (taken) continue;
                if (best < 0 || ranks_above(l[e], e, bl, best)) { best = e; bl = l[e]; }
            }
            sel[j] = best;
            o.topk[(size_t)t * k + j] = best;
        }
        // softmax (fp32)
        float z = 0.f;
        for (int e = 0; e < E; ++e) z += expf(l[e] - m);
        const float inv = 1.0f / z;
        if (o.normalize) {
            const float ms = l[sel[0]];
            float zs = 0.f;
            for (int j = 0; j < k; ++j) zs += expf(l[sel[j]] - ms);
            for (int j = 0; j < k; ++j) o.gate[(size_t)t * k + j] = expf(l[sel[j]] - ms) / zs;
        } else {
            for (int j = 0; j < k; ++j) o.gate[(size_t)t * k + j] = expf(l[sel[j]] - m) * inv;
        }
        float h = 0.f;
        for (int e = 0; e < E; ++e) {
            float p = expf(l[e] - m) * inv;
            l[e] = p;  // the tile now holds probabilities
            if (p > 0.f) h -= p * logf(p);
        }
        sEnt[i] = h;
        sBad[i] = bad ? 1 : 0;
    }
    __syncthreads();
    if (i < E) {
        float ps = 0.f;
        int cnt = 0;
        for (int r = 0; r < ntok; ++r) {
            ps += sLog[r * ldl + i];
            for (int j = 0; j < k; ++j) cnt += (sSel[r * k + j] == i);
        }
        o.part_psum[(size_t)blockIdx.x * E + i] = ps;
        o.part_counts[(size_t)blockIdx.x * E + i] = cnt;
    }
    if (i == blockDim.x - 1) {
        float h = 0.f;
        int b = 0;
        for (int r = 0; r < ntok; ++r) { h += sEnt[r]; b += sBad[r]; }
        o.part_ent[blockIdx.x] = h;
        o.part_bad[blockIdx.x] = b;
    }
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool pred) {
    uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    int n = pred ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// W_r [d,E] bf16 -> WrT [E_pad, d] bf16 (zero rows for e >= E)
__global__ void transpose_router_kernel(const __nv_bfloat16* __restrict__ Wr,
                                        __nv_bfloat16* __restrict__ WrT, int d, int E, int E_pad)
{
    const size_t n = (size_t)E_pad * d;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < n;
         idx += (size_t)gridDim.x * blockDim.x) {
        int e = (int)(idx / d), i = (int)(idx % d);
        WrT[idx] = e < E ? Wr[(size_t)i * E + e] : __float2bfloat16_rn(0.f);
    }
}

// One CTA = TT tokens.  The 8 warps split the 128 rows of each smem stage as
// (k-slice, token): with NKS = 128 / TT k-slices, a stage holds NKS x 64 columns
// of x for the CTA's TT tokens, so small token counts still spread over many
// CTAs (split-K across warps); the k-slice partials are summed in a fixed order.
template <int NT, int TT>  // NT = E_pad / 8 tensor-core n-tiles; TT tokens per CTA
__global__ void __launch_bounds__(256) route_bf16_kernel(const __nv_bfloat16* __restrict__ x,
                                                         const __nv_bfloat16* __restrict__ WrT,
                                                         RouteOut o)
{
    constexpr int E_PAD = NT * 8;
    constexpr int NKS = RT_TOK / TT;            // k-slices per stage
    constexpr int LDL = E_PAD + 1;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __nv_bfloat16* sX = reinterpret_cast<__nv_bfloat16*>(smem_raw);      // [S][128][LDS]
    __nv_bfloat16* sW = sX + RT_STAGES * RT_TOK * RT_LDS;                // [S][NKS*E_PAD][LDS]
    float* sLog = reinterpret_cast<float*>(sW + RT_STAGES * NKS * E_PAD * RT_LDS);  // [TT][LDL]
    int* sSel = reinterpret_cast<int*>(sLog + TT * LDL);
    float* sEnt = reinterpret_cast<float*>(sSel + TT * 8);
    int* sBad = reinterpret_cast<int*>(sEnt + TT);
    float* sRed = reinterpret_cast<float*>(smem_raw);                    // reuses the ring

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int t0 = blockIdx.x * TT;
    const int ntok = min(TT, o.T - t0);
    const int d = o.d;
    const int kw = RT_BK * NKS;                  // columns per stage
    const int nk = d / kw;

    auto load_stage = [&](int kc, int st) {
        const int k0 = kc * kw;
        __nv_bfloat16* dX = sX + st * RT_TOK * RT_LDS;
#pragma unroll
        for (int r = 0; r < (RT_TOK * RT_BK / 8) / 256; ++r) {
            const int s = tid + r * 256;
            const int row = s >> 3, c = s & 7;
            const int ks = row / TT, tok = row % TT;
            const bool ok = tok < ntok;
            const __nv_bfloat16* src = ok ? x + (size_t)(t0 + tok) * d + k0 + ks * RT_BK + c * 8 : x;
            cp_async16(dX + row * RT_LDS + c * 8, src, ok);
        }
        __nv_bfloat16* dW = sW + st * NKS * E_PAD * RT_LDS;
        for (int s = tid; s < NKS * E_PAD * 8; s += 256) {
            const int row = s >> 3, c = s & 7;   // row = ks * E_PAD + e
            const int ks = row / E_PAD, e = row % E_PAD;
            cp_async16(dW + row * RT_LDS + c * 8, WrT + (size_t)e * d + k0 + ks * RT_BK + c * 8, true);
        }
    };

    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    const int my_ks = (warp * 16) / TT;

#pragma unroll
    for (int s = 0; s < RT_STAGES - 1; ++s) {
        if (s < nk) load_stage(s, s);
        cp_async_commit();
    }
    for (int kc = 0; kc < nk; ++kc) {
        cp_async_wait<RT_STAGES - 2>();
        __syncthreads();
        const int st = kc % RT_STAGES;
        const __nv_bfloat16* A = sX + st * RT_TOK * RT_LDS + (warp * 16) * RT_LDS;
        const __nv_bfloat16* B = sW + (st * NKS + my_ks) * E_PAD * RT_LDS;
#pragma unroll
        for (int ks = 0; ks < RT_BK / 16; ++ks) {
            const int kk = ks * 16 + 2 * tq;
            uint32_t a0 = *reinterpret_cast<const uint32_t*>(A + g * RT_LDS + kk);
            uint32_t a1 = *reinterpret_cast<const uint32_t*>(A + (g + 8) * RT_LDS + kk);
            uint32_t a2 = *reinterpret_cast<const uint32_t*>(A + g * RT_LDS + kk + 8);
            uint32_t a3 = *reinterpret_cast<const uint32_t*>(A + (g + 8) * RT_LDS + kk + 8);
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                uint32_t b0 = *reinterpret_cast<const uint32_t*>(B + (n * 8 + g) * RT_LDS + kk);
                uint32_t b1 = *reinterpret_cast<const uint32_t*>(B + (n * 8 + g) * RT_LDS + kk + 8);
                asm volatile(
                    "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                    "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                    : "+f"(acc[n][0]), "+f"(acc[n][1]), "+f"(acc[n][2]), "+f"(acc[n][3])
                    : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
            }
        }
        const int nxt = kc + RT_STAGES - 1;
        if (nxt < nk) load_stage(nxt, nxt % RT_STAGES);
        cp_async_commit();
    }
    cp_async_wait<0>();
    __syncthreads();                             // ring no longer read: reuse it
    // partial sums of this warp's k-slice: sRed[ks][tok][E_PAD]
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const int r0 = warp * 16 + g, c0 = n * 8 + 2 * tq;   // r0 = ks * TT + tok
        sRed[r0 * E_PAD + c0] = acc[n][0];
        sRed[r0 * E_PAD + c0 + 1] = acc[n][1];
        sRed[(r0 + 8) * E_PAD + c0] = acc[n][2];
        sRed[(r0 + 8) * E_PAD + c0 + 1] = acc[n][3];
    }
    __syncthreads();
    for (int i = tid; i < TT * E_PAD; i += 256) {
        const int tok = i / E_PAD, e = i % E_PAD;
        float v = 0.f;
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) v += sRed[(ks * TT + tok) * E_PAD + e];
        sLog[tok * LDL + e] = v;
    }
    __syncthreads();
    finish_tile(sLog, LDL, sSel, sEnt, sBad, t0, ntok, o);
}

// fp32: plain FMA, 128 tokens per CTA, k-chunks of 32 staged in smem.
__global__ void __launch_bounds__(256) route_f32_kernel(const float* __restrict__ x,
                                                        const float* __restrict__ Wr, RouteOut o)
{
    constexpr int BK = 32;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int E = o.E, d = o.d;
    const int ldl = E + 1;
    float* sX = reinterpret_cast<float*>(smem_raw);            // [128][BK+1]
    float* sW = sX + RT_TOK * (BK + 1);                         // [BK][E]
    float* sLog = sW + BK * E;                                  // [128][E+1]
    int* sSel = reinterpret_cast<int*>(sLog + RT_TOK * ldl);
    float* sEnt = reinterpret_cast<float*>(sSel + RT_TOK * 8);
    int* sBad = reinterpret_cast<int*>(sEnt + RT_TOK);
    const int tid = threadIdx.x;
    const int t0 = blockIdx.x * RT_TOK;
    const int ntok = min(RT_TOK, o.T - t0);
    const int tok = tid & 127, half = tid >> 7;
    const int e_begin = half * ((E + 1) / 2), e_end = min(E, e_begin + (E + 1) / 2);
    float acc[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) acc[q] = 0.f;
    for (int k0 = 0; k0 < d; k0 += BK) {
        const int kw = min(BK, d - k0);
        for (int s = tid; s < RT_TOK * BK; s += 256) {
            int r = s / BK, c = s % BK;
            sX[r * (BK + 1) + c] = (r < ntok && c < kw) ? x[(size_t)(t0 + r) * d + k0 + c] : 0.f;
        }
        for (int s = tid; s < BK * E; s += 256) {
            int r = s / E, c = s % E;
            sW[s] = r < kw ? Wr[(size_t)(k0 + r) * E + c] : 0.f;
        }
        __syncthreads();
        for (int c = 0; c < kw; ++c) {
            const float xv = sX[tok * (BK + 1) + c];
#pragma unroll
            for (int q = 0; q < 32; ++q)
                if (e_begin + q < e_end) acc[q] = fmaf(xv, sW[c * E + e_begin + q], acc[q]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int q = 0; q < 32; ++q)
        if (e_begin + q < e_end) sLog[tok * ldl + e_begin + q] = acc[q];
    __syncthreads();
    finish_tile(sLog, ldl, sSel, sEnt, sBad, t0, ntok, o);
}

// Sum the per-CTA partials (a warp per expert, lane-strided, then a fixed
// shuffle tree: deterministic); derive the statistics.  1024 threads.
__global__ void __launch_bounds__(1024) route_finalize_kernel(
    int nblk, int T, int E, int k, float aux_coef, const int32_t* __restrict__ part_counts,
    const float* __restrict__ part_psum, const float* __restrict__ part_ent,
    const int32_t* __restrict__ part_bad, int32_t* __restrict__ counts, float* __restrict__ stats,
    int* status)
{
    __shared__ float s_pbar[64];
    __shared__ int s_cnt[64];
    __shared__ float s_h[32];
    __shared__ int s_b[32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int e = warp; e < E; e += 32) {
        int c = 0;
        float ps = 0.f;
        for (int b = lane; b < nblk; b += 32) {
            c += part_counts[(size_t)b * E + e];
            ps += part_psum[(size_t)b * E + e];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            c += __shfl_xor_sync(0xffffffffu, c, o);
            ps += __shfl_xor_sync(0xffffffffu, ps, o);
        }
        if (lane == 0) {
            counts[e] = c;
            s_cnt[e] = c;
            s_pbar[e] = ps / (float)T;
            if (stats) stats[MOE_STAT_PBAR + e] = ps / (float)T;
        }
    }
    float h = 0.f;
    int bad = 0;
    for (int b = tid; b < nblk; b += blockDim.x) { h += part_ent[b]; bad += part_bad[b]; }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        h += __shfl_xor_sync(0xffffffffu, h, o);
        bad += __shfl_xor_sync(0xffffffffu, bad, o);
    }
    if (lane == 0) { s_h[warp] = h; s_b[warp] = bad; }
    __syncthreads();
    if (tid == 0) {
        h = 0.f;
        bad = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) { h += s_h[w]; bad += s_b[w]; }
        float aux = 0.f, sw = 0.f, cmean = 0.f, cmax = 0.f;
        for (int q = 0; q < E; ++q) {
            float dq = s_pbar[q] - 1.0f / (float)E;
            aux += dq * dq;
            sw += ((float)s_cnt[q] / ((float)T * (float)k)) * s_pbar[q];
            cmean += (float)s_cnt[q];
            cmax = fmaxf(cmax, (float)s_cnt[q]);
        }
        cmean /= (float)E;
        float var = 0.f;
        for (int q = 0; q < E; ++q) var += ((float)s_cnt[q] - cmean) * ((float)s_cnt[q] - cmean);
        if (stats) {
            stats[MOE_STAT_AUX_LOSS] = aux_coef * aux;
            stats[MOE_STAT_AUX_SWITCH] = (float)E * sw;
            stats[MOE_STAT_ENTROPY] = h / (float)T;
            stats[MOE_STAT_NONFINITE] = (float)bad;
            stats[MOE_STAT_DROPPED] = 0.f;
            stats[MOE_STAT_MAX_OVER_MEAN_KEPT] = 0.f;
            stats[MOE_STAT_COUNT_CV] = cmean > 0.f ? sqrtf(var / (float)E) / cmean : 0.f;
            stats[MOE_STAT_MAX_OVER_MEAN_COUNT] = cmean > 0.f ? cmax / cmean : 0.f;
        }
        if (bad) set_status(status, MOE_ERR_NONFINITE);
    }
}

}  // namespace

// Tokens per CTA of the bf16 router: the largest TT whose grid still covers two
// waves of the GPU, else the smallest legal TT.  TT must keep a stage's router
// columns within 64 rows (NKS * E_pad <= 64) and split d evenly into NKS slices.
int route_tile_tokens(const moe_config& c) {
    if (c.dtype != MOE_DTYPE_BF16) return RT_TOK;
    const int e_pad = c.E <= 8 ? 8 : c.E <= 16 ? 16 : c.E <= 32 ? 32 : 64;
    int best = -1, smallest = -1;
    for (int tt = 16; tt <= RT_TOK; tt *= 2) {
        const int nks = RT_TOK / tt;
        if (nks * e_pad > 64 || (c.d / RT_BK) % nks != 0) continue;
        if (smallest < 0) smallest = tt;
        if ((c.T + tt - 1) / tt >= 2 * num_sms()) best = tt;
    }
    return best > 0 ? best : smallest;
}

size_t route_ws_bytes(const moe_config& c) {
    const int tt = route_tile_tokens(c);
    const size_t nblk = (size_t)(c.T + tt - 1) / tt;
    const int e_pad = c.E <= 8 ? 8 : c.E <= 16 ? 16 : c.E <= 32 ? 32 : 64;
    size_t b = 0;
    b += align_up(nblk * c.E * 4);          // counts
    b += align_up(nblk * c.E * 4);          // psum
    b += align_up(nblk * 4);                // ent
    b += align_up(nblk * 4);                // bad
    if (c.dtype == MOE_DTYPE_BF16) b += align_up((size_t)e_pad * c.d * 2);  // W_r^T
    return b;
}

namespace {
int finalize_route(const moe_config& c, const RouteOut& o, int nblk, int32_t* counts,
                   float* stats, cudaStream_t st) {
    route_finalize_kernel<<<1, 1024, 0, st>>>(nblk, c.T, c.E, c.k, c.aux_coef, o.part_counts,
                                            o.part_psum, o.part_ent, o.part_bad, counts, stats,
                                            device_status_ptr());
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

template <int NT, int TT>
int launch_route_bf16(const __nv_bfloat16* x, const __nv_bfloat16* WrT, const RouteOut& o,
                      int nblk, cudaStream_t st) {
    constexpr int E_PAD = NT * 8, NKS = RT_TOK / TT;
    const size_t smem = (size_t)RT_STAGES * (RT_TOK + NKS * E_PAD) * RT_LDS * 2 +
                        (size_t)TT * (E_PAD + 1) * 4 + (size_t)TT * 8 * 4 + (size_t)TT * 4 * 2;
    static bool attr_set = false;  // the size is fixed per instantiation
    if (!attr_set) {
        MOE_CUDA_TRY(cudaFuncSetAttribute(route_bf16_kernel<NT, TT>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        attr_set = true;
    }
    route_bf16_kernel<NT, TT><<<nblk, 256, smem, st>>>(x, WrT, o);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}
}  // namespace

int launch_route(const moe_config& c, const void* x, const void* Wr, const float* bias,
                 const float* noise, float* logits, int32_t* topk, float* gate, int32_t* counts,
                 float* stats, void* ws, cudaStream_t st)
{
    const int tt = route_tile_tokens(c);
    const int nblk = (c.T + tt - 1) / tt;
    const int e_pad = c.E <= 8 ? 8 : c.E <= 16 ? 16 : c.E <= 32 ? 32 : 64;
    uint8_t* w = static_cast<uint8_t*>(ws);
    RouteOut o;
    o.T = c.T; o.d = c.d; o.E = c.E; o.k = c.k; o.normalize = c.normalize_gates;
    o.bias = bias; o.noise = noise; o.logits = logits; o.topk = topk; o.gate = gate;
    o.part_counts = reinterpret_cast<int32_t*>(w); w += align_up((size_t)nblk * c.E * 4);
    o.part_psum = reinterpret_cast<float*>(w); w += align_up((size_t)nblk * c.E * 4);
    o.part_ent = reinterpret_cast<float*>(w); w += align_up((size_t)nblk * 4);
    o.part_bad = reinterpret_cast<int32_t*>(w); w += align_up((size_t)nblk * 4);

    if (c.dtype == MOE_DTYPE_BF16) {
        __nv_bfloat16* WrT = reinterpret_cast<__nv_bfloat16*>(w);
        transpose_router_kernel<<<64, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(Wr), WrT,
                                                    c.d, c.E, e_pad);
        MOE_LAUNCH_CHECK();
        const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
        const int key = (e_pad / 8) * 1000 + tt;
        int r = MOE_OK;
        switch (key) {
            case 1016: r = launch_route_bf16<1, 16>(xb, WrT, o, nblk, st); break;
            case 1032: r = launch_route_bf16<1, 32>(xb, WrT, o, nblk, st); break;
            case 1064: r = launch_route_bf16<1, 64>(xb, WrT, o, nblk, st); break;
            case 1128: r = launch_route_bf16<1, 128>(xb, WrT, o, nblk, st); break;
            case 2032: r = launch_route_bf16<2, 32>(xb, WrT, o, nblk, st); break;
            case 2064: r = launch_route_bf16<2, 64>(xb, WrT, o, nblk, st); break;
            case 2128: r = launch_route_bf16<2, 128>(xb, WrT, o, nblk, st); break;
            case 4064: r = launch_route_bf16<4, 64>(xb, WrT, o, nblk, st); break;
            case 4128: r = launch_route_bf16<4, 128>(xb, WrT, o, nblk, st); break;
            case 8128: r = launch_route_bf16<8, 128>(xb, WrT, o, nblk, st); break;
            default: return MOE_ERR_UNSUPPORTED;
        }
        return r != MOE_OK ? r : finalize_route(c, o, nblk, counts, stats, st);
    }
    const size_t tail = (RT_TOK * 8) * 4 + RT_TOK * 4 * 2;  // sSel, sEnt, sBad
    const size_t smem = (size_t)RT_TOK * 33 * 4 + (size_t)32 * c.E * 4 +
                        (size_t)RT_TOK * (c.E + 1) * 4 + tail;
    MOE_CUDA_TRY(cudaFuncSetAttribute(route_f32_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    route_f32_kernel<<<nblk, 256, smem, st>>>(static_cast<const float*>(x),
                                              static_cast<const float*>(Wr), o);
    MOE_LAUNCH_CHECK();
    return finalize_route(c, o, nblk, counts, stats, st);
}

}  // namespace moe
