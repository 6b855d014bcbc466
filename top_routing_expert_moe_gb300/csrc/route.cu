// route.cu -- router GEMM + softmax + top-k + gates + per-expert statistics.
//
// [LLaMA4-MoE] §2.4: a linear router with softmax scores over the experts,
// a [B,K] top-K index, outputs weighted by the post-softmax score; §3.2 gate
// noise; §4.1 padding tokens kept out of expert selection.  [ZeRO3-MoE] §5.3:
// gating in fp32 even for half-precision models.  [Twinkle] §3.1: softmax with
// a temperature, and Gumbel top-k with a straight-through estimator.
//
// bf16: a persistent CTA per SM walks tiles of TT tokens (16..64, the largest
// that still gives every SM a tile).  Warp 8 streams x (and the transposed
// router weights) with TMA into a ring of 128-row stages (mbarrier transaction
// counts); warps 0-7 split each stage's rows into (k-slice, 16 tokens) and run
// the router contraction on the tensor cores (mma.sync m16n8k16, fp32
// accumulate, fragments fetched from the swizzled boxes with ldmatrix), so the
// E flops/byte never throttle the HBM stream even at a power-capped clock;
// warps 9-12 take the finished logit tile (double-buffered, so the next tile's
// loads and MMAs overlap) and finish it with G lanes per token: bias, noise,
// softmax of logits / tau, top-k, gates, entropy (each lane's expert loops
// unrolled to the padded expert count).  Each CTA sums its tiles' statistics;
// the last CTA to finish (an atomic ticket) reduces all CTAs' sums in CTA
// order (deterministic), so no separate reduction launch follows.
// fp32: plain FMA over 128-token tiles (k-chunks staged in shared memory),
// finished by the same per-token code, then a one-CTA reduction kernel.
#include "common.cuh"
#include "kernels.h"
#include "tma.cuh"

namespace moe {

namespace {

constexpr int RT_TOK = 128;      // tokens per CTA
constexpr int RT_BK = 64;        // k-chunk (elements)

struct RouteOut {
    int T, d, E, k, normalize;
    int st;                // straight-through: noise enters the selection key only, gates 1
    float inv_tau;         // 1 / softmax temperature
    const float* bias;
    const float* noise;
    const uint8_t* mask;   // 0 = padding token (or NULL)
    float* logits;
    int32_t* topk;
    float* gate;
    int32_t* part_counts;  // [nblk][E]
    float* part_psum;      // [nblk][E]
    float* part_ent;       // [nblk]
    int32_t* part_bad;     // [nblk]
    int32_t* part_real;    // [nblk] routed (unmasked) tokens
    int* ticket;           // CTAs done (zeroed before the bf16 kernel); the last one reduces
    int32_t* counts;       // [E] selections per expert (bf16 kernel's last CTA writes)
    float* stats;          // statistics vector or NULL (idem)
};

// a ranks above b: larger logit; a NaN ranks below any number; then lower id
__device__ __forceinline__ bool ranks_above(float la, int a, float lb, int b) {
    bool na = isnan(la), nb = isnan(lb);
    if (na != nb) return nb;
    if (!na && la != lb) return la > lb;
    return a < b;
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Finish a tile of raw router sums held in sLog[tok][ldl], by nthr threads
// (index i) sharing named barrier bar_id.  G = nthr / TT consecutive lanes
// (a power of two, at most 32) work on one token: each lane takes experts
// e = sub, sub + G, ..., and the lanes combine the row's max, sums, entropy
// and each top-k pick with butterfly shuffles (exact, fixed order).  Then
// fixed-order column sums give the tile's partial statistics: written to the
// partials at index pidx, or, when acc (shared memory, ACC_FLOATS words) is
// given, added to the running sums of this CTA's tiles.
constexpr int ACC_FLOATS = 64 + 64 + 4;   // psum[64], counts[64] (int), h, bad (int), real (int)

// EP > 0: E <= EP is known at compile time, so each lane's expert loops (at most
// EP / G slots) unroll and their loads and exponentials overlap; EP = 0: runtime loops.
template <int G, int EP>
__device__ void finish_tile_seg(float* sLog, int ldl, int* sSel, float* sEnt, int* sBad, int t0,
                                int ntok, int TT, int pidx, const RouteOut& o, int i, int nthr,
                                int bar_id, float* acc)
{
    constexpr int QMAX = EP > 0 ? (EP + G - 1) / G : 64;   // expert slots of one lane
    constexpr int UNR = EP > 0 ? QMAX : 1;
    const int E = o.E, k = o.k;
    const int sub = i % G, per_pass = nthr / G;
    const unsigned mask = 0xffffffffu;
    const float itau = o.inv_tau;
    for (int tok = i / G; tok < TT; tok += per_pass) {      // uniform trip count per G-group
        const bool valid = tok < ntok;
        const int t = t0 + tok;
        const bool routed = valid && !(o.mask && o.mask[t] == 0);
        float* l = sLog + tok * ldl;
        bool bad = false;
        float m = -INFINITY;
        uint64_t taken = 0;                                  // my experts already selected
#pragma unroll UNR
        for (int q = 0; q < QMAX; ++q) {
            const int e = sub + q * G;
            if (e >= E) break;
            float v = l[e];
            if (o.bias) v += o.bias[e];
            if (o.noise && valid && !o.st) v += o.noise[(size_t)t * E + e];  // gate noise
            l[e] = v;
            if (valid) o.logits[(size_t)t * E + e] = v;
            bad |= !isfinite(v);
            m = fmaxf(m, v);
        }
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) {
            m = fmaxf(m, __shfl_xor_sync(mask, m, off));
            bad |= __shfl_xor_sync(mask, (int)bad, off) != 0;
        }
        // z = sum exp((l - m) / tau); zl = sum exp((l - m) / tau) (l - m) / tau gives the
        // entropy without a logarithm per expert: -sum p log p = log z - zl / z
        float z = 0.f, zl = 0.f;
#pragma unroll UNR
        for (int q = 0; q < QMAX; ++q) {
            const int e = sub + q * G;
            if (e >= E) break;
            const float dl = (l[e] - m) * itau;
            const float ex = __expf(dl);
            z += ex;
            zl += ex * dl;
        }
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) {
            z += __shfl_xor_sync(mask, z, off);
            zl += __shfl_xor_sync(mask, zl, off);
        }
        const float inv = __fdividef(1.0f, z);
        // top-k: k rounds; each lane proposes its best unselected expert, the
        // group keeps the one that ranks highest (larger key, NaN lowest, lower id).
        // The key is the logit, or logit + Gumbel draw in straight-through mode.
        int sel[8];
        float lsel[8];
        for (int j = 0; j < k; ++j) {
            int be = -1;
            float bv = 0.f;
#pragma unroll UNR
            for (int q = 0; q < QMAX; ++q) {
                const int e = sub + q * G;
                if (e >= E) break;
                if ((taken >> q) & 1ull) continue;
                const float key = (o.st && o.noise && valid) ? l[e] + o.noise[(size_t)t * E + e] : l[e];
                if (be < 0 || ranks_above(key, e, bv, be)) { be = e; bv = key; }
            }
#pragma unroll
            for (int off = G / 2; off > 0; off >>= 1) {
                const int oe = __shfl_xor_sync(mask, be, off);
                const float ov = __shfl_xor_sync(mask, bv, off);
                if (oe >= 0 && (be < 0 || ranks_above(ov, oe, bv, be))) { be = oe; bv = ov; }
            }
            sel[j] = be;
            if (be % G == sub) taken |= 1ull << (be / G);
        }
        // selected logits (noise-free), gathered from the owning lanes
        // (each lane reads back only its own smem writes; the owner's value is shuffled)
        const int gbase = (int)(threadIdx.x & 31) & ~(G - 1);
        for (int j = 0; j < k; ++j) lsel[j] = __shfl_sync(mask, l[sel[j]], gbase + sel[j] % G);
        if (sub == 0 && valid)
            for (int j = 0; j < k; ++j) {
                sSel[tok * k + j] = routed ? sel[j] : -1;
                o.topk[(size_t)t * k + j] = routed ? sel[j] : -1;
            }
        if (sub == 0 && valid) {
            if (!routed) {
                for (int j = 0; j < k; ++j) o.gate[(size_t)t * k + j] = 0.f;
            } else if (o.st) {
                for (int j = 0; j < k; ++j) o.gate[(size_t)t * k + j] = 1.0f;
            } else if (o.normalize) {
                float ms = lsel[0];
                for (int j = 1; j < k; ++j) ms = fmaxf(ms, lsel[j]);
                float zs = 0.f;
                for (int j = 0; j < k; ++j) zs += __expf((lsel[j] - ms) * itau);
                const float izs = __fdividef(1.0f, zs);
                for (int j = 0; j < k; ++j) o.gate[(size_t)t * k + j] = __expf((lsel[j] - ms) * itau) * izs;
            } else {
                for (int j = 0; j < k; ++j) o.gate[(size_t)t * k + j] = __expf((lsel[j] - m) * itau) * inv;
            }
        }
#pragma unroll UNR
        for (int q = 0; q < QMAX; ++q) {   // the tile now holds probabilities (0 for padding tokens)
            const int e = sub + q * G;
            if (e >= E) break;
            l[e] = routed ? __expf((l[e] - m) * itau) * inv : 0.f;
        }
        const float h = (routed && !bad) ? __logf(z) - zl * inv : 0.f;   // non-finite rows: none
        if (sub == 0) {
            sEnt[tok] = routed ? h : 0.f;
            sBad[tok] = (routed && bad) ? 1 : 0;
        }
    }
    named_sync(bar_id, nthr);
    // The tile's per-expert column sums (probabilities, selections): R lanes of
    // one warp per expert, each over rows r, r + R, ..., then a shuffle tree
    // (a fixed order: deterministic).  nthr is a multiple of 32.
    {
        int R = 32;
        while (R > 1 && R * E > nthr) R >>= 1;
        const int e = i / R, r = i % R;
        float ps = 0.f;
        int cnt = 0;
        if (e < E)
            for (int row = r; row < ntok; row += R) {
                ps += sLog[row * ldl + e];
                for (int j = 0; j < k; ++j) cnt += (sSel[row * k + j] == e);
            }
        for (int off = R / 2; off > 0; off >>= 1) {
            ps += __shfl_xor_sync(0xffffffffu, ps, off);
            cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
        }
        if (e < E && r == 0) {
            if (acc) {
                acc[e] += ps;
                reinterpret_cast<int*>(acc + 64)[e] += cnt;
            } else {
                o.part_psum[(size_t)pidx * E + e] = ps;
                o.part_counts[(size_t)pidx * E + e] = cnt;
            }
        }
    }
    // the tile's entropy, non-finite and routed-token counts: the first warp
    if (i < 32) {
        float h = 0.f;
        int b = 0, real = 0;
        for (int row = i; row < ntok; row += 32) {
            h += sEnt[row];
            b += sBad[row];
            real += sSel[row * k] >= 0;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            h += __shfl_xor_sync(0xffffffffu, h, off);
            b += __shfl_xor_sync(0xffffffffu, b, off);
            real += __shfl_xor_sync(0xffffffffu, real, off);
        }
        if (i == 0) {
            if (acc) {
                acc[128] += h;
                reinterpret_cast<int*>(acc)[129] += b;
                reinterpret_cast<int*>(acc)[130] += real;
            } else {
                o.part_ent[pidx] = h;
                o.part_bad[pidx] = b;
                o.part_real[pidx] = real;
            }
        }
    }
}

// G lanes per token for TT tokens on nthr threads (G <= 32, a power of two)
template <int EP>
__device__ __forceinline__ void finish_tile(float* sLog, int ldl, int* sSel, float* sEnt, int* sBad,
                                            int t0, int ntok, int TT, int pidx, const RouteOut& o,
                                            int i, int nthr, int bar_id, float* acc = nullptr)
{
    const int G = nthr / TT;
    if (G >= 8) finish_tile_seg<8, EP>(sLog, ldl, sSel, sEnt, sBad, t0, ntok, TT, pidx, o, i, nthr, bar_id, acc);
    else if (G >= 4) finish_tile_seg<4, EP>(sLog, ldl, sSel, sEnt, sBad, t0, ntok, TT, pidx, o, i, nthr, bar_id, acc);
    else if (G >= 2) finish_tile_seg<2, EP>(sLog, ldl, sSel, sEnt, sBad, t0, ntok, TT, pidx, o, i, nthr, bar_id, acc);
    else finish_tile_seg<1, EP>(sLog, ldl, sSel, sEnt, sBad, t0, ntok, TT, pidx, o, i, nthr, bar_id, acc);
}

// Reduce the per-tile (or per-CTA) partials into counts and the statistics,
// by nthr threads (index tid, a multiple of 32) sharing named barrier bar_id.
// All partial loads are issued in one pass (R lanes of a warp per expert, up
// to 16 independent loads each) so the reduction costs about one memory
// round trip; every sum runs in a fixed order (deterministic).  Partials are
// read with L1-bypassing loads: other CTAs wrote them.
__device__ void finalize_stats(int nblk, int E, int k, float aux_coef,
                               const int32_t* __restrict__ part_counts,
                               const float* __restrict__ part_psum,
                               const float* __restrict__ part_ent,
                               const int32_t* __restrict__ part_bad,
                               const int32_t* __restrict__ part_real, int32_t* __restrict__ counts,
                               float* __restrict__ stats, int* status, int tid, int nthr,
                               int bar_id)
{
    __shared__ float s_psum[64];
    __shared__ int s_cnt[64];
    __shared__ float s_h[32];
    __shared__ int s_b[32], s_r[32];
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    // every load of the pass issued before any is used: per-tile scalars (routed
    // tokens, entropy, non-finite tokens) for up to 4 partials per thread, and
    // per expert R lanes x 16 partials
    int R = 32;
    while (R > 1 && R * E > nthr) R >>= 1;
    const int e = tid / R, r = tid % R;
    int rl = 0, bad = 0, c = 0;
    float h = 0.f, ps = 0.f;
    {   // first round: every load in flight at once
        int rv[4], bv[4];
        float hv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int b = tid + u * nthr;
            rv[u] = b < nblk ? __ldcg(part_real + b) : 0;
            hv[u] = b < nblk ? __ldcg(part_ent + b) : 0.f;
            bv[u] = b < nblk ? __ldcg(part_bad + b) : 0;
        }
        float pv[16];
        int cv[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int bb = r + u * R;
            const bool in = e < E && bb < nblk;
            pv[u] = in ? __ldcg(part_psum + (size_t)bb * E + e) : 0.f;
            cv[u] = in ? __ldcg(part_counts + (size_t)bb * E + e) : 0;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) { rl += rv[u]; h += hv[u]; bad += bv[u]; }
#pragma unroll
        for (int u = 0; u < 16; ++u) { ps += pv[u]; c += cv[u]; }
    }
    // more partials than one round covers
    for (int b = tid + 4 * nthr; b < nblk; b += nthr) {
        rl += __ldcg(part_real + b);
        h += __ldcg(part_ent + b);
        bad += __ldcg(part_bad + b);
    }
    if (e < E)
        for (int bb = r + 16 * R; bb < nblk; bb += R) {
            ps += __ldcg(part_psum + (size_t)bb * E + e);
            c += __ldcg(part_counts + (size_t)bb * E + e);
        }
    for (int off = R / 2; off > 0; off >>= 1) {
        ps += __shfl_xor_sync(0xffffffffu, ps, off);
        c += __shfl_xor_sync(0xffffffffu, c, off);
    }
    if (e < E && r == 0) { s_psum[e] = ps; s_cnt[e] = c; }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        rl += __shfl_xor_sync(0xffffffffu, rl, o);
        h += __shfl_xor_sync(0xffffffffu, h, o);
        bad += __shfl_xor_sync(0xffffffffu, bad, o);
    }
    if (lane == 0) { s_r[warp] = rl; s_h[warp] = h; s_b[warp] = bad; }
    named_sync(bar_id, nthr);
    // warp 0: lanes e and e + 32 take the experts; fixed shuffle trees (deterministic)
    if (warp == 0) {
        int tr = 0;
        h = 0.f;
        bad = 0;
        for (int w = 0; w < nwarps; ++w) { tr += s_r[w]; h += s_h[w]; bad += s_b[w]; }
        const float Tr = fmaxf((float)tr, 1.0f);   // means over the routed tokens
        float aux = 0.f, sw = 0.f, csum = 0.f, cmax = 0.f;
        float cnt_l[2] = {0.f, 0.f};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int q = lane + 32 * hh;
            if (q < E) {
                const float pbar = s_psum[q] / Tr;
                counts[q] = s_cnt[q];
                if (stats) stats[MOE_STAT_PBAR + q] = pbar;
                const float dq = pbar - 1.0f / (float)E;
                aux += dq * dq;
                sw += ((float)s_cnt[q] / (Tr * (float)k)) * pbar;
                cnt_l[hh] = (float)s_cnt[q];
                csum += cnt_l[hh];
                cmax = fmaxf(cmax, cnt_l[hh]);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            aux += __shfl_xor_sync(0xffffffffu, aux, o);
            sw += __shfl_xor_sync(0xffffffffu, sw, o);
            csum += __shfl_xor_sync(0xffffffffu, csum, o);
            cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
        }
        const float cmean = csum / (float)E;
        float var = 0.f;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
            if (lane + 32 * hh < E) var += (cnt_l[hh] - cmean) * (cnt_l[hh] - cmean);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) var += __shfl_xor_sync(0xffffffffu, var, o);
        if (lane == 0) {
            if (stats) {
                stats[MOE_STAT_TOKENS] = (float)tr;
                stats[MOE_STAT_AUX_LOSS] = aux_coef * aux;
                stats[MOE_STAT_AUX_SWITCH] = (float)E * sw;
                stats[MOE_STAT_ENTROPY] = h / Tr;
                stats[MOE_STAT_NONFINITE] = (float)bad;
                stats[MOE_STAT_DROPPED] = 0.f;
                stats[MOE_STAT_MAX_OVER_MEAN_KEPT] = 0.f;
                stats[MOE_STAT_COUNT_CV] = cmean > 0.f ? sqrtf(var / (float)E) / cmean : 0.f;
                stats[MOE_STAT_MAX_OVER_MEAN_COUNT] = cmean > 0.f ? cmax / cmean : 0.f;
            }
            if (bad) set_status(status, MOE_ERR_NONFINITE);
        }
    }
}

// W_r [d,E] bf16 -> WrT [E_pad, d] bf16 (zero rows for e >= E); also zeroes the
// router kernel's CTA ticket (this kernel runs just before it on the stream)
__global__ void transpose_router_kernel(const __nv_bfloat16* __restrict__ Wr,
                                        __nv_bfloat16* __restrict__ WrT, int d, int E, int E_pad,
                                        int* ticket)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    if (blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0;
    const size_t n = (size_t)E_pad * d;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < n;
         idx += (size_t)gridDim.x * blockDim.x) {
        int e = (int)(idx / d), i = (int)(idx % d);
        WrT[idx] = e < E ? Wr[(size_t)i * E + e] : __float2bfloat16_rn(0.f);
    }
}

// Token tiles of TT tokens; the 8 MMA warps split each tile as (k-slice, 16
// tokens): NKS = 128 / TT k-slices (split-K across warps; slice partials summed
// in a fixed order).  A stage holds NKS x NB consecutive 64-column blocks of x
// for the tile (NB = 1 or 2 blocks per k-slice), so a stage covers NKS*NB*128
// contiguous bytes of each token row (in a plain read probe on GB300, stages of
// 32 KB streamed at 7.1 TB/s and stages of 16 KB at 4.4).
//
// Persistent CTAs (one per SM), three roles:
//   warp 8      TMA producer: 128B-swizzled boxes of x ({64 columns, TT rows}
//               per k-slice) and of W_r^T ({64, E_pad}) stream into a ring of
//               `stages` slots across tile boundaries (mbarrier tx counts);
//   warps 0-7   MMA: mma.sync m16n8k16 (bf16 in, fp32 accumulate) on
//               swizzle-aware fragment loads; at a tile's end they reduce the
//               k-slices into one of two logits buffers and move on;
//   warps 9-12  finish, concurrently with the next tile's streaming: bias,
//               noise, softmax, top-k, gates, the tile's partial statistics.
// The two logits buffers are handed over with mbarriers.  Every wait is
// bounded; after a failed wait a warp keeps its barrier sequence, skipping work.
struct RouteTma {
    CUtensorMap tmX, tmW;
    RouteOut o;
    int* status;
    int stages;
    int nb;          // 64-column blocks per k-slice per stage
    float aux_coef;
};

constexpr int RTMA_THREADS = 13 * 32;   // 8 MMA warps, 1 producer warp, 4 finish warps

template <int NT, int TT>  // NT = E_pad / 8 tensor-core n-tiles; TT tokens per tile
__global__ void __launch_bounds__(RTMA_THREADS, 1) route_bf16_kernel(const __grid_constant__ RouteTma P)
{
    constexpr int E_PAD = NT * 8;
    constexpr int NKS = RT_TOK / TT;                 // k-slices per tile
    constexpr int LDL = E_PAD + 1;
    const int NB = P.nb;
    const uint32_t X_BYTES = (uint32_t)NB * RT_TOK * 128;                        // 16 or 32 KB
    const uint32_t W_BYTES = ((uint32_t)NB * NKS * E_PAD * 128 + 1023) / 1024 * 1024;
    const uint32_t STAGE = X_BYTES + W_BYTES;
    const RouteOut& o = P.o;
    const int S = P.stages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* sRed = reinterpret_cast<float*>(ring + (size_t)S * STAGE);   // [128][E_PAD]
    float* sLogB = sRed + RT_TOK * E_PAD;                                // [2][TT][LDL]
    int* sSel = reinterpret_cast<int*>(sLogB + 2 * TT * LDL);            // [TT*8]
    float* sEnt = reinterpret_cast<float*>(sSel + TT * 8);
    int* sBad = reinterpret_cast<int*>(sEnt + TT);
    float* sAcc = reinterpret_cast<float*>(sBad + TT);                   // [ACC_FLOATS]
    uint64_t* bars = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(sAcc + ACC_FLOATS) + 15) & ~uintptr_t(15));
    uint64_t* full = bars;
    uint64_t* empty = full + S;
    uint64_t* lfull = empty + S;     // [2] logits buffer written (256 arrivals)
    uint64_t* lempty = lfull + 2;    // [2] logits buffer finished (128 arrivals)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(lempty + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = o.d;
    const int nk = d / (RT_BK * NKS * NB);
    const int ntiles = (o.T + TT - 1) / TT;
    const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const uint32_t ring0 = smem_u32(ring);

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 8);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&lfull[b]), 256);
            mbar_init(smem_u32(&lempty[b]), 128);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_wait();      // the preceding kernel's writes (x, W_r^T, the ticket) are visible from here on
    pdl_trigger();
    // a timeout recorded earlier on this device (not yet read by the host): skip the work
    if (tid == 0 && timeout_pending(P.status)) *abort_flag = 1;
    __syncthreads();
    const bool start_live = *abort_flag == 0;

    if (warp == 8) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmX)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmW)) : "memory");
            int it = 0;
            bool ok = start_live;
            for (int i = 0; ok && i < my_tiles; ++i) {
                const int t0 = (blockIdx.x + i * gridDim.x) * TT;
                for (int kc = 0; kc < nk; ++kc, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (uint32_t)(it / S) & 1u;
                    if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1u, abort_flag, P.status)) { ok = false; break; }
                    const uint32_t bar = smem_u32(&full[s]);
                    const uint32_t sx = ring0 + s * STAGE, sw = sx + X_BYTES;
                    mbar_expect_tx(bar, X_BYTES + (uint32_t)NB * NKS * E_PAD * 128);
                    const int k0 = kc * RT_BK * NKS * NB;
                    for (int j = 0; j < NKS * NB; ++j) {   // block j: k-slice j / NB, columns k0 + 64 j
                        tma_load3(&P.tmX, sx + j * TT * 128, bar, k0 + j * RT_BK, t0, 0);
                        tma_load3(&P.tmW, sw + j * E_PAD * 128, bar, k0 + j * RT_BK, 0, 0);
                    }
                }
            }
            for (int j = max(0, it - S); j < it; ++j)     // every issued load lands before exit
                mbar_drain(smem_u32(&full[j % S]), (uint32_t)(j / S) & 1u);
        }
        return;
    }

    if (warp >= 9) {
        // ------------------------------------------------ finish warps
        const int ftid = tid - 9 * 32;   // 0..127
        for (int q = ftid; q < ACC_FLOATS; q += 128) sAcc[q] = 0.f;   // the CTA's running sums
        bool live = start_live;
        for (int i = 0; i < my_tiles; ++i) {
            const int tile = blockIdx.x + i * gridDim.x;
            const int t0 = tile * TT, ntok = min(TT, o.T - t0);
            const int b = i & 1;
            if (live) live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&lfull[b]), (uint32_t)(i >> 1) & 1u,
                                                            abort_flag, P.status));
            if (live) finish_tile<E_PAD>(sLogB + b * TT * LDL, LDL, sSel, sEnt, sBad, t0, ntok, TT, tile, o, ftid, 128, 2, sAcc);
            else named_sync(2, 128);
            named_sync(2, 128);          // sSel / sEnt / sBad read by all before reuse
            mbar_arrive(smem_u32(&lempty[b]));
        }
        named_sync(2, 128);              // every tile's sums are in sAcc
        // one partial per CTA (pidx = blockIdx.x), its tiles summed in tile order
        for (int e = ftid; e < o.E; e += 128) {
            o.part_psum[(size_t)blockIdx.x * o.E + e] = sAcc[e];
            o.part_counts[(size_t)blockIdx.x * o.E + e] = reinterpret_cast<int*>(sAcc + 64)[e];
        }
        if (ftid == 0) {
            o.part_ent[blockIdx.x] = sAcc[128];
            o.part_bad[blockIdx.x] = reinterpret_cast<int*>(sAcc)[129];
            o.part_real[blockIdx.x] = reinterpret_cast<int*>(sAcc)[130];
        }
        // the last CTA to finish reduces every CTA's partials (in CTA order)
        __shared__ int s_last;
        __threadfence();
        named_sync(2, 128);
        if (ftid == 0) s_last = atomicAdd(o.ticket, 1) == (int)gridDim.x - 1;
        named_sync(2, 128);
        if (s_last) {
            __threadfence();
            finalize_stats(gridDim.x, o.E, o.k, P.aux_coef, o.part_counts, o.part_psum, o.part_ent,
                           o.part_bad, o.part_real, o.counts, o.stats, P.status, ftid, 128, 2);
        }
        return;
    }

    // ---------------------------------------------------- MMA warps 0-7
    const int g = lane >> 2, tq = lane & 3;
    const int my_ks = (warp * 16) / TT;
    // ldmatrix row addresses (each 8 x 8 bf16 matrix = 8 rows of 16 bytes of a
    // 128B-swizzled box: chunk c of row r sits at chunk c ^ (r & 7)).
    // A (x4): lanes 0-15 rows 0-15 of the warp's 16 tokens at k 0-7, lanes 16-31 the
    // same rows at k 8-15 -> the m16n8k16 A fragment {a0, a1, a2, a3}.
    const int a_row = (warp * 16) % TT + (lane & 15), a_kh = lane >> 4;
    // B (x4 over n-tiles n, n + 1; x2 for a last odd one): lanes 0-7 / 8-15 rows
    // (experts) of tile n at k 0-7 / 8-15, lanes 16-31 the same for tile n + 1.
    const int b_row = (lane & 7) + ((lane >> 4) << 3), b_kh = (lane >> 3) & 1;
    const uint32_t ring_sa = smem_u32(ring);
    bool live = start_live;
    int it = 0;
    for (int i = 0; i < my_tiles; ++i) {
        float acc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        for (int kc = 0; kc < nk; ++kc, ++it) {
            const int s = it % S;
            const uint32_t ph = (uint32_t)(it / S) & 1u;
            if (live) live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&full[s]), ph, abort_flag, P.status));
            if (!live) continue;
            for (int bb = 0; bb < NB; ++bb) {
                const int j = my_ks * NB + bb;                 // this warp's block of the stage
                const uint32_t Xs = ring_sa + (uint32_t)s * STAGE + (uint32_t)j * TT * 128;
                const uint32_t Ws = ring_sa + (uint32_t)s * STAGE + X_BYTES + (uint32_t)j * E_PAD * 128;
#pragma unroll
                for (int k16 = 0; k16 < RT_BK / 16; ++k16) {
                    uint32_t a0, a1, a2, a3;
                    const uint32_t xa = Xs + (uint32_t)(a_row * 128 + (((k16 * 2 + a_kh) ^ (a_row & 7)) << 4));
                    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(xa));
#pragma unroll
                    for (int n = 0; n < NT; n += 2) {
                        const int row = n * 8 + b_row;
                        const uint32_t wa = Ws + (uint32_t)(row * 128 + (((k16 * 2 + b_kh) ^ (row & 7)) << 4));
                        uint32_t b[4];
                        if (n + 1 < NT)
                            asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                                         : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]) : "r"(wa));
                        else
                            asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];\n"
                                         : "=r"(b[0]), "=r"(b[1]) : "r"(wa));
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            if (n + h >= NT) break;
                            asm volatile(
                                "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                                "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                                : "+f"(acc[n + h][0]), "+f"(acc[n + h][1]), "+f"(acc[n + h][2]), "+f"(acc[n + h][3])
                                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b[2 * h]), "r"(b[2 * h + 1]));
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));   // slot free for the producer
        }
        // ---- the tile is summed: hand its logits to the finish warps
#pragma unroll
        for (int n = 0; n < NT; ++n) {   // this warp's k-slice partials: sRed[ks][tok][e]
            const int r0 = warp * 16 + g, c0 = n * 8 + 2 * tq;   // r0 = ks * TT + tok
            sRed[r0 * E_PAD + c0] = acc[n][0];
            sRed[r0 * E_PAD + c0 + 1] = acc[n][1];
            sRed[(r0 + 8) * E_PAD + c0] = acc[n][2];
            sRed[(r0 + 8) * E_PAD + c0 + 1] = acc[n][3];
        }
        named_sync(1, 256);
        const int b = i & 1;
        if (i >= 2 && live)              // buffer b's previous tile must be finished
            live = __all_sync(0xffffffffu, mbar_wait(smem_u32(&lempty[b]), (uint32_t)((i - 2) >> 1) & 1u,
                                                     abort_flag, P.status));
        float* sLog = sLogB + b * TT * LDL;
        if (live)
            for (int q = tid; q < TT * E_PAD; q += 256) {
                const int tok = q / E_PAD, e = q % E_PAD;
                float v = 0.f;
#pragma unroll
                for (int ks = 0; ks < NKS; ++ks) v += sRed[(ks * TT + tok) * E_PAD + e];
                sLog[tok * LDL + e] = v;
            }
        mbar_arrive(smem_u32(&lfull[b]));    // release: this thread's logits writes
        named_sync(1, 256);                  // sRed free for the next tile
    }
}

// fp32: plain FMA, 128 tokens per CTA, k-chunks of 32 staged in smem.
__global__ void __launch_bounds__(256) route_f32_kernel(const float* __restrict__ x,
                                                        const float* __restrict__ Wr, RouteOut o)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
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
    finish_tile<0>(sLog, ldl, sSel, sEnt, sBad, t0, ntok, RT_TOK, blockIdx.x, o, threadIdx.x, 256, 1);
}

// Sum the per-CTA partials (a warp per expert, lane-strided, then a fixed
// shuffle tree: deterministic); derive the statistics.  1024 threads.
// fp32 path: the reduction as its own one-CTA kernel after the router
__global__ void __launch_bounds__(1024) route_finalize_kernel(
    int nblk, int T, int E, int k, float aux_coef, const int32_t* __restrict__ part_counts,
    const float* __restrict__ part_psum, const float* __restrict__ part_ent,
    const int32_t* __restrict__ part_bad, const int32_t* __restrict__ part_real,
    int32_t* __restrict__ counts, float* __restrict__ stats, int* status)
{
    pdl_wait();      // the preceding kernel's writes are visible from here on
    pdl_trigger();
    finalize_stats(nblk, E, k, aux_coef, part_counts, part_psum, part_ent, part_bad, part_real,
                   counts, stats, status, threadIdx.x, blockDim.x, 1);
}

}  // namespace

// Tokens per tile of the bf16 router (16, 32 or 64): the largest tile that
// still gives every SM at least one tile, else the smallest legal one.  On
// GB300 64-token tiles routed fastest even where they leave the last wave
// uneven (T = 16384, d = 2048, E = 8: 50 us at 64 tokens, 52 at 32, 60 at 16;
// T = 65536, d = 4096, E = 16: 159 / 179 / 233 us).  A tile must split d / 64
// evenly into NKS = 128 / TT k-slices and keep a k-slice's W_r^T block (NKS *
// E_pad rows of 128 B) within 16 KB.
int route_tile_tokens(const moe_config& c) {
    if (c.dtype != MOE_DTYPE_BF16) return RT_TOK;
    const int e_pad = c.E <= 8 ? 8 : c.E <= 16 ? 16 : c.E <= 32 ? 32 : 64;
    int smallest = -1;
    for (int tt = 64; tt >= 16; tt /= 2) {
        const int nks = RT_TOK / tt;
        if (nks * e_pad > 128 || (c.d / RT_BK) % nks != 0) continue;
        if ((c.T + tt - 1) / tt >= num_sms()) return tt;
        smallest = tt;
    }
    return smallest > 0 ? smallest : RT_TOK;
}

// 64-column blocks per k-slice in one stage: 2 (32 KB of x per stage) when d
// splits evenly and the stage's W_r^T blocks stay within 32 KB, else 1.
int route_stage_blocks(const moe_config& c, int tt, int e_pad) {
    const int nks = RT_TOK / tt;
    if ((c.d / RT_BK) % (2 * nks) == 0 && 2 * nks * e_pad <= 256) return 2;
    return 1;
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
    b += align_up(nblk * 4);                // routed tokens
    b += align_up(4);                       // CTA ticket
    if (c.dtype == MOE_DTYPE_BF16) b += align_up((size_t)e_pad * c.d * 2);  // W_r^T
    return b;
}

namespace {
int finalize_route(const moe_config& c, const RouteOut& o, int nblk, int32_t* counts,
                   float* stats, cudaStream_t st) {
    MOE_LAUNCH(route_finalize_kernel, 1, 1024, 0, st, nblk, c.T, c.E, c.k, c.aux_coef, o.part_counts,
                                            o.part_psum, o.part_ent, o.part_bad, o.part_real,
                                            counts, stats,
                                            device_status_ptr());
    return MOE_OK;
}

template <int NT, int TT>
int launch_route_bf16(const moe_config& c, const void* x, const __nv_bfloat16* WrT, int e_pad,
                      const RouteOut& o, int nblk, cudaStream_t st) {
    constexpr int E_PAD = NT * 8, NKS = RT_TOK / TT;
    const int nb = route_stage_blocks(c, TT, E_PAD);
    const size_t STAGE = (size_t)nb * RT_TOK * 128 + ((size_t)nb * NKS * E_PAD * 128 + 1023) / 1024 * 1024;
    const size_t extra = (size_t)RT_TOK * E_PAD * 4 + 2 * (size_t)TT * (E_PAD + 1) * 4 +
                        (size_t)TT * 8 * 4 + (size_t)TT * 4 * 2 + ACC_FLOATS * 4 + 16 + (2 * 16 + 4) * 8 + 64;
    // dynamic shared memory: the 227 KB per-block limit less the kernel's ~1 KB of
    // static shared memory (the statistics reduction), rounded down
    constexpr size_t DYN_SMEM = 225 * 1024;
    const size_t budget = DYN_SMEM - 1024 - extra;
    const int stages = (int)std::min<size_t>(16, budget / STAGE);
    const size_t smem = 1024 + stages * STAGE + extra;
    static bool attr_set[64] = {};  // the largest size is fixed per instantiation
    if (const int ra = smem_attr_once(route_bf16_kernel<NT, TT>, DYN_SMEM, attr_set)) return ra;
    RouteTma P;
    memset(&P, 0, sizeof(P));
    int r = encode_bf16_map(&P.tmX, x, (uint64_t)c.d, (uint64_t)c.T, 1, (uint64_t)c.d * 2,
                            (uint64_t)c.d * 2 * c.T, RT_BK, TT);
    if (r) return r;
    r = encode_bf16_map(&P.tmW, WrT, (uint64_t)c.d, (uint64_t)e_pad, 1, (uint64_t)c.d * 2,
                        (uint64_t)c.d * 2 * e_pad, RT_BK, E_PAD);
    if (r) return r;
    P.o = o;
    P.status = device_status_ptr();
    P.stages = stages;
    P.nb = nb;
    P.aux_coef = c.aux_coef;
    if (stages < 2) return MOE_ERR_UNSUPPORTED;
    // persistent: one CTA per SM walks tiles blockIdx.x, blockIdx.x + gridDim.x, ...
    const int grid = std::min(nblk, num_sms());
    MOE_LAUNCH_PARAM(route_bf16_kernel<NT, TT>, grid, RTMA_THREADS, smem, st, P);
    return MOE_OK;
}
}  // namespace

int launch_route(const moe_config& c, const void* x, const void* Wr, const float* bias,
                 const float* noise, const uint8_t* mask, float* logits, int32_t* topk,
                 float* gate, int32_t* counts, float* stats, void* ws, cudaStream_t st)
{
    const int tt = route_tile_tokens(c);
    const int nblk = (c.T + tt - 1) / tt;
    const int e_pad = c.E <= 8 ? 8 : c.E <= 16 ? 16 : c.E <= 32 ? 32 : 64;
    uint8_t* w = static_cast<uint8_t*>(ws);
    RouteOut o;
    o.T = c.T; o.d = c.d; o.E = c.E; o.k = c.k; o.normalize = c.normalize_gates;
    o.bias = bias; o.noise = noise; o.mask = mask; o.logits = logits; o.topk = topk; o.gate = gate;
    o.st = c.straight_through;
    o.inv_tau = c.temperature > 0.f ? 1.0f / c.temperature : 1.0f;
    o.part_counts = reinterpret_cast<int32_t*>(w); w += align_up((size_t)nblk * c.E * 4);
    o.part_psum = reinterpret_cast<float*>(w); w += align_up((size_t)nblk * c.E * 4);
    o.part_ent = reinterpret_cast<float*>(w); w += align_up((size_t)nblk * 4);
    o.part_bad = reinterpret_cast<int32_t*>(w); w += align_up((size_t)nblk * 4);
    o.part_real = reinterpret_cast<int32_t*>(w); w += align_up((size_t)nblk * 4);
    o.ticket = reinterpret_cast<int*>(w); w += align_up(4);
    o.counts = counts;
    o.stats = stats;

    if (c.dtype == MOE_DTYPE_BF16) {
        __nv_bfloat16* WrT = reinterpret_cast<__nv_bfloat16*>(w);
        MOE_LAUNCH(transpose_router_kernel, 64, 256, 0, st, static_cast<const __nv_bfloat16*>(Wr), WrT,
                                                    c.d, c.E, e_pad, o.ticket);
        const int key = (e_pad / 8) * 1000 + tt;
        int r = MOE_OK;
        switch (key) {
            case 1016: r = launch_route_bf16<1, 16>(c, x, WrT, e_pad, o, nblk, st); break;
            case 1032: r = launch_route_bf16<1, 32>(c, x, WrT, e_pad, o, nblk, st); break;
            case 1064: r = launch_route_bf16<1, 64>(c, x, WrT, e_pad, o, nblk, st); break;
            case 1128: r = launch_route_bf16<1, 128>(c, x, WrT, e_pad, o, nblk, st); break;
            case 2016: r = launch_route_bf16<2, 16>(c, x, WrT, e_pad, o, nblk, st); break;
            case 2032: r = launch_route_bf16<2, 32>(c, x, WrT, e_pad, o, nblk, st); break;
            case 2064: r = launch_route_bf16<2, 64>(c, x, WrT, e_pad, o, nblk, st); break;
            case 2128: r = launch_route_bf16<2, 128>(c, x, WrT, e_pad, o, nblk, st); break;
            case 4032: r = launch_route_bf16<4, 32>(c, x, WrT, e_pad, o, nblk, st); break;
            case 4064: r = launch_route_bf16<4, 64>(c, x, WrT, e_pad, o, nblk, st); break;
            case 4128: r = launch_route_bf16<4, 128>(c, x, WrT, e_pad, o, nblk, st); break;
            case 8064: r = launch_route_bf16<8, 64>(c, x, WrT, e_pad, o, nblk, st); break;
            case 8128: r = launch_route_bf16<8, 128>(c, x, WrT, e_pad, o, nblk, st); break;
            default: return MOE_ERR_UNSUPPORTED;
        }
        return r;   // the kernel's last CTA reduced the statistics
    }
    const size_t tail = (RT_TOK * 8) * 4 + RT_TOK * 4 * 2;  // sSel, sEnt, sBad
    const size_t smem = (size_t)RT_TOK * 33 * 4 + (size_t)32 * c.E * 4 +
                        (size_t)RT_TOK * (c.E + 1) * 4 + tail;
    MOE_CUDA_TRY(cudaFuncSetAttribute(route_f32_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    MOE_LAUNCH(route_f32_kernel, nblk, 256, smem, st, static_cast<const float*>(x),
                                              static_cast<const float*>(Wr), o);
    return finalize_route(c, o, nblk, counts, stats, st);
}

}  // namespace moe
