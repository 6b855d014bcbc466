// permute.cu -- capacity dropping and the expert-contiguous permutation.
//
// [LLaMA4-MoE] §2.4: sort the [B,K] index by expert id, take each expert's
// token-count interval, split, run each expert.  [ZeRO3-MoE] §3.1/§3.4:
// a per-expert capacity (capacity_factor) caps the tokens an expert takes.
//
// A stable counting sort, deterministic (no order-dependent atomics):
//   1. tile histogram: per 256-token tile, selections per expert;
//   2. per tile (one CTA each): the expert's tokens in earlier tiles and in all
//      tiles (every CTA sums the small histogram itself, so no separate scan
//      launch), the capacity and the padded segments (offsets); then warp
//      ballots give each assignment its rank among the expert's assignments in
//      token order; rank < C keeps it at row offsets[e] + rank; padding rows
//      are marked, each CTA a strided share of them;
//   3. gather: one warp per destination row copies the token's x row with
//      16-byte vectors (zeros on padding rows), rows read from device offsets.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int PT_TOK = 256;  // tokens per tile (one per thread)

__global__ void __launch_bounds__(PT_TOK) tile_hist_kernel(const int32_t* __restrict__ topk,
                                                           int T, int E, int k,
                                                           int32_t* __restrict__ tile_counts,
                                                           int* status)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    __shared__ int h[64];
    if (threadIdx.x < E) h[threadIdx.x] = 0;
    __syncthreads();
    const int t = blockIdx.x * PT_TOK + threadIdx.x;
    if (t < T)
        for (int j = 0; j < k; ++j) {
            int e = topk[(size_t)t * k + j];
            if (e >= 0 && e < E) atomicAdd(&h[e], 1);  // integer count: order-free
            else if (e != -1) set_status(status, MOE_ERR_DEVICE_BOUNDS);  // -1: masked token
        }
    __syncthreads();
    if (threadIdx.x < E) tile_counts[(size_t)blockIdx.x * E + threadIdx.x] = h[threadIdx.x];
}

// One CTA per 256-token tile.  A warp per expert sums the expert's counts over
// the earlier tiles (this tile's first rank) and over all tiles; thread 0 then
// applies the capacity and lays out the padded segments (every CTA finds the
// same layout; CTA 0 writes offsets, kept and the statistics).
__global__ void __launch_bounds__(PT_TOK) scan_assign_kernel(
    const int32_t* __restrict__ topk, int T, int E, int k, int C, int pad_m,
    const int32_t* __restrict__ tile_counts, int ntiles, int32_t* __restrict__ kept,
    int32_t* __restrict__ offsets, int32_t* __restrict__ slot_of, int32_t* __restrict__ perm_token,
    float* __restrict__ stats)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    __shared__ int s_base[64], s_total[64], s_off[65];
    __shared__ int wcount[PT_TOK / 32][64];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int blk = blockIdx.x;
    for (int e = warp; e < E; e += PT_TOK / 32) {
        int before = 0, total = 0;
        for (int b = lane; b < ntiles; b += 32) {
            const int v = tile_counts[(size_t)b * E + e];
            total += v;
            if (b < blk) before += v;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            before += __shfl_xor_sync(0xffffffffu, before, o);
            total += __shfl_xor_sync(0xffffffffu, total, o);
        }
        if (lane == 0) {
            s_base[e] = before;
            s_total[e] = total;
        }
    }
    __syncthreads();
    if (tid == 0) {
        int off = 0, kmax = 0;
        long ksum = 0, dropped = 0;
        for (int e = 0; e < E; ++e) {
            const int ke = min(s_total[e], C);
            s_off[e] = off;
            if (blk == 0) {
                offsets[e] = off;
                kept[e] = ke;
            }
            off += (ke + pad_m - 1) / pad_m * pad_m;
            kmax = max(kmax, ke);
            ksum += ke;
            dropped += s_total[e] - ke;
        }
        s_off[E] = off;
        if (blk == 0) {
            offsets[E] = off;
            if (stats) {
                stats[MOE_STAT_DROPPED] = (float)dropped;
                stats[MOE_STAT_MAX_OVER_MEAN_KEPT] =
                    ksum > 0 ? (float)kmax / ((float)ksum / (float)E) : 0.f;
            }
        }
    }
    __syncthreads();
    // padding rows carry token -1 (this CTA: every ntiles-th group of 256 rows)
    for (int e = 0; e < E; ++e) {
        const int end = s_off[e + 1];
        for (int r = s_off[e] + min(s_total[e], C) + blk * PT_TOK + tid; r < end; r += ntiles * PT_TOK)
            perm_token[r] = -1;
    }
    // ranks within the tile: per expert, a ballot over each warp's tokens
    const int t = blk * PT_TOK + tid;
    int sel[8];
    int inrank[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        sel[j] = (j < k && t < T) ? topk[(size_t)t * k + j] : -1;
        inrank[j] = 0;
    }
    const unsigned lt = (1u << lane) - 1u;
    for (int e = 0; e < E; ++e) {
        bool mine = false;
#pragma unroll
        for (int j = 0; j < 8; ++j) mine |= (sel[j] == e);
        const unsigned bal = __ballot_sync(0xffffffffu, mine);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (sel[j] == e) inrank[j] = __popc(bal & lt);
        if (lane == 0) wcount[warp][e] = __popc(bal);
    }
    __syncthreads();
    if (t >= T) return;
    for (int j = 0; j < k; ++j) {
        const int e = sel[j];
        if (e < 0 || e >= E) { slot_of[(size_t)t * k + j] = -1; continue; }
        int r = s_base[e] + inrank[j];
        for (int w = 0; w < warp; ++w) r += wcount[w][e];
        if (r < C) {
            const int row = s_off[e] + r;
            slot_of[(size_t)t * k + j] = row;
            perm_token[row] = t;
        } else {
            slot_of[(size_t)t * k + j] = -1;
        }
    }
}

// one warp per destination row; 16-byte vectors; the row count is read on the device
template <typename T>
__global__ void __launch_bounds__(256) gather_rows_kernel(const T* __restrict__ x,
                                                          const int32_t* __restrict__ perm_token,
                                                          const int32_t* __restrict__ offsets,
                                                          int E, int d, T* __restrict__ x_perm)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    constexpr int V = 16 / sizeof(T);
    const int rows = offsets[E];
    const int nv = d / V;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        const int t = perm_token[r];
        uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)r * d);
        if (t < 0) {
            for (int v = threadIdx.x & 31; v < nv; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
        } else {
            const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
            int v = threadIdx.x & 31;
            for (; v + 96 < nv; v += 128) {
                uint4 a = __ldg(src + v), b = __ldg(src + v + 32), c = __ldg(src + v + 64),
                      e = __ldg(src + v + 96);
                dst[v] = a; dst[v + 32] = b; dst[v + 64] = c; dst[v + 96] = e;
            }
            for (; v < nv; v += 32) dst[v] = __ldg(src + v);
        }
    }
}

}  // namespace

size_t permute_ws_bytes(const moe_config& c) {
    const size_t ntiles = (size_t)(c.T + PT_TOK - 1) / PT_TOK;
    return align_up(ntiles * c.E * 4);
}

int launch_permute(const moe_config& c, const void* x, const int32_t* topk, void* x_perm,
                   int32_t* perm_token, int32_t* slot_of, int32_t* kept, int32_t* offsets,
                   float* stats, void* ws, cudaStream_t st)
{
    const int ntiles = (c.T + PT_TOK - 1) / PT_TOK;
    int32_t* tile_counts = static_cast<int32_t*>(ws);
    const int C = capacity_of(c);
    MOE_LAUNCH(tile_hist_kernel, ntiles, PT_TOK, 0, st, topk, c.T, c.E, c.k, tile_counts,
                                                device_status_ptr());
    MOE_LAUNCH(scan_assign_kernel, ntiles, PT_TOK, 0, st, topk, c.T, c.E, c.k, C, c.pad_m, tile_counts,
               ntiles, kept, offsets, slot_of, perm_token, stats);
    const int64_t rows = rows_cap_of(c);
    const int grid = (int)std::min<int64_t>((rows + 7) / 8, (int64_t)num_sms() * 8);
    if (c.dtype == MOE_DTYPE_BF16)
        MOE_LAUNCH(gather_rows_kernel<__nv_bfloat16>, grid, 256, 0, st, static_cast<const __nv_bfloat16*>(x), perm_token, offsets, c.E, c.d,
            static_cast<__nv_bfloat16*>(x_perm));
    else
        MOE_LAUNCH(gather_rows_kernel<float>, grid, 256, 0, st, static_cast<const float*>(x), perm_token,
                                                        offsets, c.E, c.d,
                                                        static_cast<float*>(x_perm));
    return MOE_OK;
}

}  // namespace moe
