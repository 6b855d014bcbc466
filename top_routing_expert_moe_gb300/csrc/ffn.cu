// ffn.cu -- grouped expert FFN, forward and backward, over device-resident
// expert segments ([LLaMA4-MoE] §2.4: every expert a two-layer FFN; tokens
// sorted by expert id and split into per-expert intervals).
//
// bf16 runs on the tcgen05 grouped GEMM (gemm_tc.cu) with the activation and
// its derivative fused into the GEMM epilogues.  fp32 runs on a plain SIMT
// segmented GEMM (fp32 FMA, no TF32, so results stay within 1e-5 of fp64),
// with separate elementwise activation kernels.
#include <algorithm>

#include "common.cuh"
#include "gemm_tc.h"
#include "kernels.h"

namespace moe {

namespace {

// C[m,n] (+)= sum_k A(m,k) B(n,k) over expert segments.
//   SEG_ROWS: rows m in [offsets[e], offsets[e+1]); B advanced by e*b_se.
//   SEG_K   : k in [offsets[e], offsets[e+1]) (weight gradient); C advanced by e*c_se.
// Without offsets there is one segment [0, fixed) (the shared experts' FFN).
enum SegMode { SEG_ROWS = 0, SEG_K = 1 };

struct SimtGemm {
    const void* A; long long a_sm, a_sk;
    const void* B; long long b_sn, b_sk, b_se;
    void* C; long long c_sm, c_sn, c_se;
    int M, N, K;      // extents of the non-segmented dimensions
    int mode;
    const int32_t* offsets;
    int fixed;
    int accumulate;
};

constexpr int SG_BM = 64, SG_BN = 64, SG_BK = 16;

template <typename T>
__global__ void __launch_bounds__(256) simt_seg_gemm_kernel(SimtGemm g)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    __shared__ float As[SG_BK][SG_BM + 4];
    __shared__ float Bs[SG_BK][SG_BN + 4];
    const int e = blockIdx.z;
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    int m_lo, m_hi, k_lo, k_hi;
    const T* A = static_cast<const T*>(g.A);
    const T* B = static_cast<const T*>(g.B);
    T* C = static_cast<T*>(g.C);
    const int s_lo = g.offsets ? g.offsets[e] : 0;
    const int s_hi = g.offsets ? g.offsets[e + 1] : g.fixed;
    if (g.mode == SEG_ROWS) {
        m_lo = s_lo + blockIdx.y * SG_BM;
        m_hi = s_hi;
        if (m_lo >= m_hi) return;
        k_lo = 0; k_hi = g.K;
        B += (long long)e * g.b_se;
    } else {
        m_lo = blockIdx.y * SG_BM;
        m_hi = g.M;
        k_lo = s_lo; k_hi = s_hi;
        C += (long long)e * g.c_se;
    }
    const int n0 = blockIdx.x * SG_BN;
    float acc[4][4] = {};
    for (int k0 = k_lo; k0 < k_hi; k0 += SG_BK) {
        for (int i = tid; i < SG_BK * SG_BM; i += 256) {
            int kk = i / SG_BM, mm = i % SG_BM;
            int m = m_lo + mm, k = k0 + kk;
            As[kk][mm] = (m < m_hi && k < k_hi) ? to_f<T>(A[m * g.a_sm + k * g.a_sk]) : 0.f;
            int n = n0 + mm;
            Bs[kk][mm] = (n < g.N && k < k_hi) ? to_f<T>(B[n * g.b_sn + k * g.b_sk]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < SG_BK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) { a[i] = As[kk][ty * 4 + i]; b[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m_lo + ty * 4 + i;
        if (m >= m_hi) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= g.N) continue;
            T* p = C + m * g.c_sm + n * g.c_sn;
            float v = acc[i][j];
            if (g.accumulate) v += to_f<T>(*p);
            *p = from_f<T>(v);
        }
    }
}

// act = silu(h)  or  silu(g) * u, on rows [0, offsets[E]) (or [0, rows) without offsets)
template <typename T>
__global__ void act_fwd_kernel(const T* __restrict__ h0, const T* __restrict__ h1, T* __restrict__ act,
                               const int32_t* __restrict__ offsets, int E, int rows, int f,
                               int swiglu)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    const long long n = (long long)(offsets ? offsets[E] : rows) * f;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        float z = to_f<T>(h0[i]);
        float a = silu_f(z);
        if (swiglu) a *= to_f<T>(h1[i]);
        act[i] = from_f<T>(a);
    }
}

// SiLU  : dh0 = dact * silu'(h)                 (dact held in dh0)
// SwiGLU: dg = dact * u * silu'(g), du = dact * silu(g)   (dact held in dh1)
template <typename T>
__global__ void act_bwd_kernel(const T* __restrict__ h0, const T* __restrict__ h1, T* dh0, T* dh1,
                               const int32_t* __restrict__ offsets, int E, int rows, int f,
                               int swiglu)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    const long long n = (long long)(offsets ? offsets[E] : rows) * f;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const float z = to_f<T>(h0[i]);
        if (swiglu) {
            const float da = to_f<T>(dh1[i]);
            const float u = to_f<T>(h1[i]);
            dh0[i] = from_f<T>(da * u * dsilu_f(z));
            dh1[i] = from_f<T>(da * silu_f(z));
        } else {
            dh0[i] = from_f<T>(to_f<T>(dh0[i]) * dsilu_f(z));
        }
    }
}

template <typename T>
int simt_gemm(const SimtGemm& g, int E, int max_seg_rows, cudaStream_t st)
{
    dim3 grid((g.N + SG_BN - 1) / SG_BN,
              g.mode == SEG_ROWS ? (max_seg_rows + SG_BM - 1) / SG_BM : (g.M + SG_BM - 1) / SG_BM,
              E);
    MOE_LAUNCH(simt_seg_gemm_kernel<T>, grid, 256, 0, st, g);
    return MOE_OK;
}

SimtGemm rows_gemm(const void* A, long long lda, const void* B, long long b_sn, long long b_sk,
                   long long b_se, void* C, long long ldc, int N, int K, const int32_t* off,
                   int accumulate, int fixed = 0)
{
    SimtGemm g{};
    g.fixed = fixed;
    g.A = A; g.a_sm = lda; g.a_sk = 1;
    g.B = B; g.b_sn = b_sn; g.b_sk = b_sk; g.b_se = b_se;
    g.C = C; g.c_sm = ldc; g.c_sn = 1; g.c_se = 0;
    g.M = 0; g.N = N; g.K = K; g.mode = SEG_ROWS; g.offsets = off; g.accumulate = accumulate;
    return g;
}

// dW[e][m][n] = sum_{rows r of e} A[r][m] B[r][n]
SimtGemm wgrad_gemm(const void* A, long long lda, const void* B, long long ldb, void* C, int M,
                    int N, const int32_t* off, int fixed = 0)
{
    SimtGemm g{};
    g.fixed = fixed;
    g.A = A; g.a_sm = 1; g.a_sk = lda;
    g.B = B; g.b_sn = 1; g.b_sk = ldb; g.b_se = 0;
    g.C = C; g.c_sm = N; g.c_sn = 1; g.c_se = (long long)M * N;
    g.M = M; g.N = N; g.K = 0; g.mode = SEG_K; g.offsets = off; g.accumulate = 0;
    return g;
}

int max_seg_rows(const moe_config& c) {
    return std::min(c.T, capacity_of(c)) + c.pad_m - 1;
}

int ew_grid(long long n) {
    return (int)std::max<long long>(1, std::min<long long>((n + 255) / 256, num_sms() * 8LL));
}
int ew_grid(const moe_config& c) { return ew_grid(rows_cap_of(c) * (long long)c.f); }

int ffn_forward_f32(const moe_config& c, const float* xp, const int32_t* off, const float* Wu,
                    const float* Wg, const float* Wd, float* h, float* act, float* y,
                    cudaStream_t st)
{
    const int d = c.d, f = c.f, E = c.E, msr = max_seg_rows(c);
    const long long rc = rows_cap_of(c);
    const bool sw = c.ffn == MOE_FFN_SWIGLU;
    float* h0 = h;
    float* h1 = sw ? h + rc * f : nullptr;
    int r;
    if (sw) {
        if ((r = simt_gemm<float>(rows_gemm(xp, d, Wg, 1, f, (long long)d * f, h0, f, f, d, off, 0), E, msr, st))) return r;
        if ((r = simt_gemm<float>(rows_gemm(xp, d, Wu, 1, f, (long long)d * f, h1, f, f, d, off, 0), E, msr, st))) return r;
    } else {
        if ((r = simt_gemm<float>(rows_gemm(xp, d, Wu, 1, f, (long long)d * f, h0, f, f, d, off, 0), E, msr, st))) return r;
    }
    MOE_LAUNCH(act_fwd_kernel<float>, ew_grid(c), 256, 0, st, h0, h1, act, off, E, 0, f, sw);
    return simt_gemm<float>(rows_gemm(act, f, Wd, 1, d, (long long)f * d, y, d, d, f, off, 0), E, msr, st);
}

int ffn_backward_f32(const moe_config& c, const float* xp, const int32_t* off, const float* Wu,
                     const float* Wg, const float* Wd, const float* h, const float* act,
                     const float* dy, float* dh, float* dxp, float* dWu, float* dWg, float* dWd,
                     cudaStream_t st)
{
    const int d = c.d, f = c.f, E = c.E, msr = max_seg_rows(c);
    const long long rc = rows_cap_of(c);
    const bool sw = c.ffn == MOE_FFN_SWIGLU;
    const float* h0 = h;
    const float* h1 = sw ? h + rc * f : nullptr;
    float* dh0 = dh;
    float* dh1 = sw ? dh + rc * f : nullptr;
    float* dact = sw ? dh1 : dh0;
    int r;
    // dact = dy W_down^T   (B(n=j,k=i) = W_down[j][i])
    if ((r = simt_gemm<float>(rows_gemm(dy, d, Wd, d, 1, (long long)f * d, dact, f, f, d, off, 0), E, msr, st))) return r;
    MOE_LAUNCH(act_bwd_kernel<float>, ew_grid(c), 256, 0, st, h0, h1, dh0, dh1, off, E, 0, f, sw);
    // weight gradients
    if ((r = simt_gemm<float>(wgrad_gemm(act, f, dy, d, dWd, f, d, off), E, 0, st))) return r;
    if (sw) {
        if ((r = simt_gemm<float>(wgrad_gemm(xp, d, dh1, f, dWu, d, f, off), E, 0, st))) return r;
        if ((r = simt_gemm<float>(wgrad_gemm(xp, d, dh0, f, dWg, d, f, off), E, 0, st))) return r;
    } else {
        if ((r = simt_gemm<float>(wgrad_gemm(xp, d, dh0, f, dWu, d, f, off), E, 0, st))) return r;
    }
    // dx_perm = dh W_up^T (+ dg W_gate^T)   (B(n=i,k=j) = W[i][j])
    if (sw) {
        if ((r = simt_gemm<float>(rows_gemm(dh1, f, Wu, f, 1, (long long)d * f, dxp, d, d, f, off, 0), E, msr, st))) return r;
        return simt_gemm<float>(rows_gemm(dh0, f, Wg, f, 1, (long long)d * f, dxp, d, d, f, off, 1), E, msr, st);
    }
    return simt_gemm<float>(rows_gemm(dh0, f, Wu, f, 1, (long long)d * f, dxp, d, d, f, off, 0), E, msr, st);
}

// The shared experts' FFN in fp32: the same GEMMs over one segment of T rows.
int shared_forward_f32(const moe_config& c, const moe_shared_ffn& s, cudaStream_t st)
{
    const int d = c.d, f = c.f_shared, T = c.T;
    const bool sw = c.ffn == MOE_FFN_SWIGLU;
    const float* x = static_cast<const float*>(s.x);
    float* h0 = static_cast<float*>(s.h);
    float* h1 = sw ? h0 + (long long)T * f : nullptr;
    float* act = static_cast<float*>(s.act);
    int r;
    if (sw) {
        if ((r = simt_gemm<float>(rows_gemm(x, d, s.W_gate, 1, f, 0, h0, f, f, d, nullptr, 0, T), 1, T, st))) return r;
        if ((r = simt_gemm<float>(rows_gemm(x, d, s.W_up, 1, f, 0, h1, f, f, d, nullptr, 0, T), 1, T, st))) return r;
    } else {
        if ((r = simt_gemm<float>(rows_gemm(x, d, s.W_up, 1, f, 0, h0, f, f, d, nullptr, 0, T), 1, T, st))) return r;
    }
    MOE_LAUNCH(act_fwd_kernel<float>, ew_grid((long long)T * f), 256, 0, st, h0, h1, act, nullptr, 0, T, f, sw);
    return simt_gemm<float>(rows_gemm(act, f, s.W_down, 1, d, 0, s.y, d, d, f, nullptr, 0, T), 1, T, st);
}

int shared_backward_f32(const moe_config& c, const moe_shared_ffn& s, cudaStream_t st)
{
    const int d = c.d, f = c.f_shared, T = c.T;
    const bool sw = c.ffn == MOE_FFN_SWIGLU;
    const float* x = static_cast<const float*>(s.x);
    const float* dy = static_cast<const float*>(s.dout);
    const float* h0 = static_cast<const float*>(s.h);
    const float* h1 = sw ? h0 + (long long)T * f : nullptr;
    float* dh0 = static_cast<float*>(s.dh);
    float* dh1 = sw ? dh0 + (long long)T * f : nullptr;
    float* dact = sw ? dh1 : dh0;
    int r;
    if ((r = simt_gemm<float>(rows_gemm(dy, d, s.W_down, d, 1, 0, dact, f, f, d, nullptr, 0, T), 1, T, st))) return r;
    MOE_LAUNCH(act_bwd_kernel<float>, ew_grid((long long)T * f), 256, 0, st, h0, h1, dh0, dh1, nullptr, 0, T, f, sw);
    if ((r = simt_gemm<float>(wgrad_gemm(s.act, f, dy, d, s.dW_down, f, d, nullptr, T), 1, 0, st))) return r;
    if (sw) {
        if ((r = simt_gemm<float>(wgrad_gemm(x, d, dh1, f, s.dW_up, d, f, nullptr, T), 1, 0, st))) return r;
        if ((r = simt_gemm<float>(wgrad_gemm(x, d, dh0, f, s.dW_gate, d, f, nullptr, T), 1, 0, st))) return r;
        if ((r = simt_gemm<float>(rows_gemm(dh1, f, s.W_up, f, 1, 0, s.dx, d, d, f, nullptr, 0, T), 1, T, st))) return r;
        return simt_gemm<float>(rows_gemm(dh0, f, s.W_gate, f, 1, 0, s.dx, d, d, f, nullptr, 1, T), 1, T, st);
    }
    if ((r = simt_gemm<float>(wgrad_gemm(x, d, dh0, f, s.dW_up, d, f, nullptr, T), 1, 0, st))) return r;
    return simt_gemm<float>(rows_gemm(dh0, f, s.W_up, f, 1, 0, s.dx, d, d, f, nullptr, 0, T), 1, T, st);
}

}  // namespace

size_t ffn_ws_bytes(const moe_config&) { return 0; }   // the expert FFN needs no scratch

int launch_ffn_forward(const moe_config& c, const void* x_perm, const int32_t* offsets,
                       const void* W_up, const void* W_gate, const void* W_down, void* h_saved,
                       void* act, void* y_perm, const moe_shared_ffn* shared, void* ws,
                       cudaStream_t st)
{
    if (c.dtype == MOE_DTYPE_BF16)
        return tc_ffn_forward(c, x_perm, offsets, W_up, W_gate, W_down, h_saved, act, y_perm,
                              shared, st);
    int r = ffn_forward_f32(c, static_cast<const float*>(x_perm), offsets,
                            static_cast<const float*>(W_up), static_cast<const float*>(W_gate),
                            static_cast<const float*>(W_down), static_cast<float*>(h_saved),
                            static_cast<float*>(act), static_cast<float*>(y_perm), st);
    if (r || !shared) return r;
    return shared_forward_f32(c, *shared, st);
}

int launch_ffn_backward(const moe_config& c, const void* x_perm, const int32_t* offsets,
                        const void* W_up, const void* W_gate, const void* W_down,
                        const void* h_saved, const void* act, const void* dy_perm, void* dh,
                        void* dx_perm, void* dW_up, void* dW_gate, void* dW_down,
                        const moe_shared_ffn* shared, void* ws, cudaStream_t st)
{
    if (c.dtype == MOE_DTYPE_BF16)
        return tc_ffn_backward(c, x_perm, offsets, W_up, W_gate, W_down, h_saved, act, dy_perm,
                               dh, dx_perm, dW_up, dW_gate, dW_down, shared, st);
    int r = ffn_backward_f32(c, static_cast<const float*>(x_perm), offsets,
                            static_cast<const float*>(W_up), static_cast<const float*>(W_gate),
                            static_cast<const float*>(W_down), static_cast<const float*>(h_saved),
                            static_cast<const float*>(act), static_cast<const float*>(dy_perm),
                            static_cast<float*>(dh), static_cast<float*>(dx_perm),
                            static_cast<float*>(dW_up), static_cast<float*>(dW_gate),
                            static_cast<float*>(dW_down), st);
    if (r || !shared) return r;
    return shared_backward_f32(c, *shared, st);
}

}  // namespace moe
