// gemm_tc.cu -- persistent tcgen05 grouped GEMM over expert segments (sm_103a).
//
// Every expert-FFN contraction of the layer ([LLaMA4-MoE] §2.4: each expert a
// two-layer FFN over the tokens routed to it) is one launch of this kernel:
//   forward   h|g,u = x_perm W_up|W_gate  (activation fused in the epilogue)
//             y     = act W_down
//   backward  dact  = dy W_down^T          (silu' / SwiGLU derivative fused)
//             dW    = x^T dh, act^T dy     (reduction over each expert's rows)
//             dx    = dh W_up^T (+ dg W_gate^T)
//
// Design (clusters of two CTAs -- a pair -- one CTA per SM, 320 threads each):
//   warp 0      TMA producer of each CTA: its 128 rows of A and its half of B's
//               columns, 128B-swizzled, into a ring of three 64 KB stages 128
//               deep in k, one TMA load per operand share; the loads of both
//               CTAs complete on the even CTA's "full" barrier.
//   warp 1      allocates 512 TMEM columns (both CTAs, collectively); the even
//               CTA's thread issues tcgen05.mma.cta_group::2 (M = 256, N = 256,
//               K = 16, bf16 in, fp32 accumulate) and commits, multicast to both
//               CTAs, to the ring's "empty" barriers and to one of two TMEM
//               accumulators' "full" barriers.
//   warps 2-9   epilogue of each CTA's 128 accumulator lanes: two warps per TMEM
//               lane quarter, tcgen05.ld 32 columns at a time, the fused
//               activation (or its derivative), 32 x 32 output boxes written by
//               TMA stores; the accumulator is released to the even CTA so the
//               next tile's MMAs overlap this epilogue.
// A one-CTA variant (M = 128, two 96 KB stages) serves devices that cannot
// hold pairs.  Tiles come from a static persistent schedule whose per-expert
// tile counts are read from the device-side segment offsets, so no host sync
// separates routing from the GEMMs; within an expert, tiles are visited in
// groups of RASTER_GM row blocks so the A rows and B columns in flight stay
// L2-resident.  A launch may hold up to six independent problems (the
// backward's dgrad || weight gradient pairs, the shared experts' FFN).
//
// Shared-memory operand layouts (canonical 128B-swizzle layouts):
//   K-major   rows of 64 bf16 (128 B); 8-row groups 1024 B apart (SBO);
//             the K=16 step advances the start address by 32 B.
//   MN-major  blocks of 64 k-rows x 64 MN-elements (8 KB); 8-k-row groups
//             1024 B apart (SBO); MN blocks 8 KB apart (LBO); the K=16 step
//             advances the start address by 2048 B.
//
// Every mbarrier wait is bounded (globaltimer): on expiry the kernel records
// MOE_ERR_TIMEOUT, tells the other roles to stop, drains its own TMA loads and
// MMAs (again bounded), frees TMEM and returns.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "gemm_tc.h"
#include "kernels.h"
#include "tma.cuh"

namespace moe {

namespace {

constexpr int BM = 128, BK = 128;             // k per stage: two 64-wide k-blocks (128-byte rows)
constexpr int A_BYTES = BM * BK * 2;          // 32 KB
constexpr int RING_BYTES = 192 * 1024;        // 2 stages of 96 KB (one CTA) or 3 of 64 KB (a pair)
constexpr int STAGING_BYTES = 32 * 1024;      // epilogue: two 2 KB output boxes per epilogue warp
constexpr int CTRL_BYTES = 2048;   // barriers, TMEM slot, offsets[65], prefix[6*64+1], slot bases
constexpr int SMEM_BYTES = 1024 + RING_BYTES + STAGING_BYTES + CTRL_BYTES;
static_assert(SMEM_BYTES <= 232448, "227 KB of dynamic shared memory per block");
constexpr int TMEM_COLS = 512;
constexpr int NUM_EPI_WARPS = 8;                   // two per TMEM lane quarter
constexpr int NTHREADS = 64 + 32 * NUM_EPI_WARPS;  // producer warp, MMA warp, epilogue
constexpr int RASTER_GM = 32;
// Every operand share of a stage arrives with one TMA load: each TMA instruction
// the producer issues costs mainloop time, more than the bytes it moves (on the
// Mixtral step one load per share instead of two took the grouped GEMMs about 8 %
// faster, and 128-deep stages, half the loads again, about 7 % more; L2 prefetch
// instructions beside the loads made them slower).  So a stage is 128 deep in k
// -- a share is a {64, 128, 2} box of a block view of the tensor.  Raster groups
// of 32 row blocks: one pass over an expert's weights per 4096 rows (GEMM1 at
// K = d reads 30 % less DRAM than with 16) while a group's A rows fit in L2.
constexpr int SPLIT_MIN_WAVES = 16;   // "many waves of tiles": a launch this long is split by tile length

enum Epi { EPI_STORE = 0, EPI_SILU_FWD = 1, EPI_SWIGLU_FWD = 2, EPI_SILU_BWD = 3, EPI_SWIGLU_BWD = 4 };
enum Sched { SCHED_ROWS = 0, SCHED_KSEG = 1 };

// One GEMM problem of a launch.  A launch runs up to MAX_PROBLEMS independent
// problems, their tiles in one schedule (the backward's dgrad2 || dW_down, then
// dW_up || dW_gate || dgrad1, for the routed experts and the shared FFN).
// A problem either runs over the routed experts' segments (rows taken from
// the device offsets) or over one fixed segment of fixed_rows rows with
// expert index 0 (the shared FFN, which every token passes through).
struct TcProblem {
    CUtensorMap tmA0, tmB0, tmA1, tmB1;
    CUtensorMap tmO[3];     // outputs out0..out2: boxes of 32 rows x 32 columns, 64-byte swizzle
    __nv_bfloat16* out0;
    __nv_bfloat16* out1;
    __nv_bfloat16* out2;
    const __nv_bfloat16* in0;
    const __nv_bfloat16* in1;
    long long out_estride;  // SCHED_KSEG: elements between experts' outputs
    int sched;
    int n_blocks;           // N / bn
    int m_blocks;           // SCHED_KSEG: M / 128
    int k_blocks;           // SCHED_ROWS: K / BK (per operand pair)
    int kconcat;            // SCHED_ROWS: 2 = K loop continues over (A1, B1)
    int a_mn, b_mn;         // operand is MN-major in global memory
    int bn;                 // 128 or 256
    int dual;               // SwiGLU GEMM1: B = [B0 tile | B1 tile], accumulator columns 0..127 / 128..255
    int epi;
    int ldo;
    int fixed_rows;         // > 0: one segment [0, fixed_rows) (a multiple of BM)
};
constexpr int MAX_PROBLEMS = 6;

struct TcParams {
    TcProblem prob[MAX_PROBLEMS];
    const int32_t* offsets;
    int* status;
    int nprob, E;
};
static_assert(sizeof(TcParams) <= 32764, "kernel parameters within the 32 KB launch limit");

// mbarrier / TMA / timer helpers: tma.cuh

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version (sm_100 family)
    d |= (uint64_t)2 << 61;  // 128-byte swizzle
    return d;
}
// kind::f16 instruction descriptor: bf16 x bf16 -> fp32, dense
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// element i (0..31) of 32 consecutive bf16 values held in four 16-byte words
__device__ __forceinline__ float bf16_at(const uint4 (&w)[4], int i) {
    const uint4 q = w[i >> 3];
    const uint32_t x = ((i >> 1) & 3) == 0 ? q.x : ((i >> 1) & 3) == 1 ? q.y : ((i >> 1) & 3) == 2 ? q.z : q.w;
    return __uint_as_float((i & 1) ? (x & 0xFFFF0000u) : (x << 16));
}

// bf16-path activations: fast exp and approximate divide (no slow-path
// branches); errors of a few fp32 ulp vanish in the bf16 outputs.
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }
__device__ __forceinline__ float dsilu_fast(float z) {
    const float s = __fdividef(1.0f, 1.0f + __expf(-z));
    return s * (1.0f + z * (1.0f - s));
}

// ---------------------------------------------------------------- schedule
// A tile is CG * 128 rows (CG = 1: one CTA; CG = 2: a CTA pair, 128 rows each)
// by bn columns.  Tiles are counted in these units; within a pair each CTA
// takes its 128-row half, and a half that falls past the segment (an odd
// number of 128-row blocks) computes but stores nothing.
struct Tile {
    int p, e, m0, n0, krow0, nk;
    int mb;        // index of the tile's first 128-row block within its segment
    int mb_e;      // 128-row blocks of the segment (SCHED_ROWS) or of M (SCHED_KSEG)
};

__device__ __forceinline__ int seg_m_blocks(const TcProblem& q, const int* offs, int e) {
    if (q.sched != SCHED_ROWS) return q.m_blocks;
    return q.fixed_rows ? q.fixed_rows / BM : (offs[e + 1] - offs[e]) / BM;
}

// Slots: problem p's segments (E of them, or 1 for a fixed-rows problem) are
// slots sbase[p] .. sbase[p+1]-1.  prefix[s] = first tile of slot s;
// prefix[sbase[nprob]] = total.  Binary search for the slot holding tile tix.
template <int CG>
__device__ __forceinline__ void decode_tile(const TcParams& P, const int* offs, const int* prefix,
                                            const int* sbase, int tix, Tile& t) {
    int lo = 0, hi = sbase[P.nprob] - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= tix) lo = mid; else hi = mid - 1;
    }
    int pi = 0;
    while (pi + 1 < P.nprob && sbase[pi + 1] <= lo) ++pi;
    const int e = lo - sbase[pi];
    const TcProblem& q = P.prob[pi];
    const int local = tix - prefix[lo];
    const int mb_e = seg_m_blocks(q, offs, e);
    const int mt_e = (mb_e + CG - 1) / CG;                 // tiles along M
    constexpr int RG = RASTER_GM / CG;
    const int gsz = RG * q.n_blocks;
    const int grp = local / gsz;
    const int first = grp * RG;
    const int gm = min(RG, mt_e - first);
    const int r = local - grp * gsz;
    const int mt = first + r % gm, nb = r / gm;
    t.p = pi;
    t.e = e;
    t.n0 = nb * q.bn;
    t.mb = mt * CG;
    t.mb_e = mb_e;
    if (q.sched == SCHED_ROWS) {
        t.m0 = (q.fixed_rows ? 0 : offs[e]) + t.mb * BM;
        t.krow0 = 0;
        t.nk = q.k_blocks * q.kconcat;
    } else {
        t.m0 = t.mb * BM;
        t.krow0 = q.fixed_rows ? 0 : offs[e];
        t.nk = (q.fixed_rows ? q.fixed_rows : offs[e + 1] - offs[e]) / BK;
    }
}

template <int CG>
__device__ __forceinline__ void mma_issue(uint32_t dtmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    if constexpr (CG == 1) {
        asm volatile(
            "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(dtmem),
            "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
    } else {
        asm volatile(
            "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(dtmem),
            "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
    }
}
// arrive on `bar` once the MMAs issued so far complete: in this CTA (CG = 1),
// or at the same offset in both CTAs of the pair (CG = 2)
template <int CG>
__device__ __forceinline__ void mma_commit_all(uint32_t bar) {
    if constexpr (CG == 1) {
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
    } else {
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
            "h"((uint16_t)0x3)
            : "memory");
    }
}
template <int CG>
__device__ __forceinline__ void mma_commit_local(uint32_t bar) {
    if constexpr (CG == 1)
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
    else
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
}

// ---------------------------------------------------------------- kernel
// CG = 1: every CTA works alone on 128 x bn tiles (M = 128 MMAs).
// CG = 2: clusters of two CTAs (a pair) work on 256 x bn tiles with M = 256
// tcgen05.mma.cta_group::2 issued by the even CTA.  Each CTA stages its own
// 128 rows of A and half of B's columns (32 KB per stage instead of 48, so six
// stages fit instead of four and each CTA reads a third less from L2); both
// halves' TMA loads complete on the even CTA's "full" barrier, the MMA
// completions are multicast to both CTAs' "empty" and "accumulator full"
// barriers, and both CTAs' epilogue warps release an accumulator on the even
// CTA's "accumulator empty" barrier.  Each CTA drains its own 128 TMEM lanes.
template <int CG>
__global__ void __launch_bounds__(NTHREADS, 1) tc_grouped_gemm_kernel(const __grid_constant__ TcParams P)
{
    constexpr int S = CG == 1 ? 2 : 3;                       // ring stages
    constexpr int SB = CG == 1 ? 96 * 1024 : 64 * 1024;      // stage bytes per CTA
    static_assert(S * SB == RING_BYTES, "ring size");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ctrl = base + RING_BYTES + STAGING_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
    uint64_t* empty = full + 8;
    uint64_t* tfull = empty + 8;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* offs = reinterpret_cast<int*>(tmem_slot + 2);  // [E+1] segment offsets
    int* prefix = offs + 66;                            // [slots+1] first tile of each slot
    int* sbase = prefix + MAX_PROBLEMS * 64 + 4;        // [nprob+1] first slot of each problem

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = CG == 1 ? 0u : cluster_rank();
    const bool leader = rank == 0;
    const int unit = (int)blockIdx.x / CG, nunits = (int)gridDim.x / CG;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), CG * NUM_EPI_WARPS);
        }
        mbar_init(smem_u32(drain), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if constexpr (CG == 2) cluster_sync_all();   // both CTAs' barriers exist before any cross-CTA use
    pdl_wait();      // the preceding kernel's writes (offsets, operands) are visible from here on
    pdl_trigger();
    if (P.offsets && tid < P.E + 1) offs[tid] = P.offsets[tid];
    if (warp == 1) {
        if constexpr (CG == 1) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                         "r"(TMEM_COLS));
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        } else {   // one warp of each CTA of the pair, collectively
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                         "r"(TMEM_COLS));
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        int acc = 0, sl = 0;
        for (int pi = 0; pi < P.nprob; ++pi) {
            sbase[pi] = sl;
            const int nseg = P.prob[pi].fixed_rows ? 1 : P.E;
            for (int e = 0; e < nseg; ++e, ++sl) {
                prefix[sl] = acc;
                acc += (seg_m_blocks(P.prob[pi], offs, e) + CG - 1) / CG * P.prob[pi].n_blocks;
            }
        }
        sbase[P.nprob] = sl;
        prefix[sl] = acc;
    }
    // a timeout recorded earlier on this device (not yet read by the host): skip the work
    if (tid == 0 && timeout_pending(P.status)) *abort_flag = 1;
    __syncthreads();
    const uint32_t tmem_base = *tmem_slot;
    const int total = prefix[sbase[P.nprob]];
    const uint32_t smem0 = smem_u32(base);
    const bool start_live = *abort_flag == 0;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer (each CTA)
        for (int pi = 0; pi < P.nprob; ++pi) {   // the descriptors this launch uses
            const TcProblem& q = P.prob[pi];
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&q.tmA0)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&q.tmB0)) : "memory");
            if (q.kconcat == 2)
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&q.tmA1)) : "memory");
            if (q.kconcat == 2 || q.dual)
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&q.tmB1)) : "memory");
            const __nv_bfloat16* outs[3] = {q.out0, q.out1, q.out2};
            for (int i = 0; i < 3; ++i)
                if (outs[i])
                    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&q.tmO[i])) : "memory");
        }
        int it = 0;
        bool ok = start_live;
        for (int tix = unit; ok && tix < total; tix += nunits) {
            Tile t;
            decode_tile<CG>(P, offs, prefix, sbase, tix, t);
            // per-tile copies of the problem's fields (registers, not re-read after each
            // "memory"-clobbering wait)
            const TcProblem& q = P.prob[t.p];
            const int q_kseg = q.sched == SCHED_KSEG, q_kb = q.k_blocks, q_dual = q.dual;
            const int q_bmn = q.b_mn;
            const CUtensorMap* tA0 = &q.tmA0;
            const CUtensorMap* tA1 = &q.tmA1;
            const CUtensorMap* tB0 = &q.tmB0;
            const CUtensorMap* tB1 = &q.tmB1;
            // this CTA's rows of A and columns of B
            const int am0 = t.m0 + (int)rank * BM;
            // SwiGLU's gate and up tiles form one 256-column B operand [gate | up]:
            // one CTA stages both (CG = 1), or the even CTA the gate and the odd
            // CTA the up tile (CG = 2)
            const int bcols = (q_dual ? 256 : q.bn) / CG;
            const int bn0 = t.n0 + (q_dual ? 0 : (int)rank * bcols);
            const uint32_t b_bytes = (uint32_t)bcols * BK * 2u;
            const uint32_t stage_tx = CG * ((uint32_t)A_BYTES + b_bytes);   // both CTAs' bytes
            for (int kb = 0; kb < t.nk; ++kb, ++it) {
                const int s = it % S;
                const uint32_t ph = (uint32_t)(it / S) & 1u;
                if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1u, abort_flag, P.status)) { ok = false; break; }
                const uint32_t sA = smem0 + s * SB, sB = sA + A_BYTES;
                uint32_t bar;
                if constexpr (CG == 1) {
                    bar = smem_u32(&full[s]);
                    mbar_expect_tx(bar, stage_tx);
                } else {
                    bar = mapa_shared(smem_u32(&full[s]), 0);
                    if (leader) mbar_expect_tx(smem_u32(&full[s]), stage_tx);
                }
                auto ld = [&](const CUtensorMap* m, uint32_t dst, int c0, int c1, int c2) {
                    if constexpr (CG == 1) tma_load3(m, dst, bar, c0, c1, c2);
                    else tma_load3_pair(m, dst, bar, c0, c1, c2);
                };
                auto ld4 = [&](const CUtensorMap* m, uint32_t dst, int c0, int c1, int c2, int c3) {
                    if constexpr (CG == 1) tma_load4(m, dst, bar, c0, c1, c2, c3);
                    else tma_load4_pair(m, dst, bar, c0, c1, c2, c3);
                };
                // one load per operand share; every view is {64, rows, 64-column blocks[, E]}
                if (q_kseg) {   // both MN-major: 128 k-rows x the share's 64-column blocks
                    const int kr = t.krow0 + kb * BK;
                    ld(tA0, sA, 0, kr, am0 / 64);
                    ld(tB0, sB, 0, kr, bn0 / 64);
                } else {
                    const int phase = kb >= q_kb ? 1 : 0;
                    const int k0 = (kb - phase * q_kb) * BK;
                    ld(phase ? tA1 : tA0, sA, 0, am0, k0 / 64);   // K-major: 128 rows x 2 k-blocks
                    if (q_dual) {   // [gate | up]: two 64-column blocks of one of them per load
                        for (int c = 0; c < 4 / CG; c += 2) {
                            const int g = c + (int)rank * (4 / CG);        // 0: gate; 2: up
                            ld4(g < 2 ? tB0 : tB1, sB + c * (BK * 128), 0, k0, bn0 / 64, t.e);
                        }
                    } else if (q_bmn) {   // MN-major weights: 128 k-rows x the share's blocks
                        ld4(tB0, sB, 0, k0, bn0 / 64, t.e);
                    } else {              // K-major weights: the share's rows of N x 2 k-blocks
                        ld4(phase ? tB1 : tB0, sB, 0, bn0, k0 / 64, t.e);
                    }
                }
            }
        }
        // drain: every load issued has landed before the CTA may exit (for a
        // pair, the even CTA's "full" barriers count both CTAs' loads)
        if (CG == 1 || leader)
            for (int i = max(0, it - S); i < it; ++i) {
                if constexpr (CG == 1) mbar_drain(smem_u32(&full[i % S]), (uint32_t)(i / S) & 1u);
                else mbar_drain_cl(smem_u32(&full[i % S]), (uint32_t)(i / S) & 1u);
            }
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------------------------ MMA issuer (the pair's even CTA)
        int it = 0, tcount = 0;
        bool ok = start_live;
        for (int tix = unit; ok && tix < total; tix += nunits, ++tcount) {
            Tile t;
            decode_tile<CG>(P, offs, prefix, sbase, tix, t);
            const TcProblem& q = P.prob[t.p];
            const int q_dual = q.dual, q_amn = q.a_mn, q_bmn = q.b_mn;
            const uint32_t idesc = idesc_bf16(BM * CG, q_dual ? 256 : q.bn, q_amn, q_bmn);
            // K-major B: stride between the stage's two k-blocks (the CTA's rows of B x 128 B)
            const uint32_t b_kblk = (uint32_t)((q_dual ? 256 : q.bn) / CG) * 128u;
            const int acc = tcount & 1;
            const uint32_t aph = (uint32_t)(tcount >> 1) & 1u;
            const bool got = CG == 1 ? mbar_wait(smem_u32(&tempty[acc]), aph ^ 1u, abort_flag, P.status)
                                     : mbar_wait_cl(smem_u32(&tempty[acc]), aph ^ 1u, abort_flag, P.status);
            if (!got) { ok = false; break; }
            tc_fence_after();
            const uint32_t dt = tmem_base + (uint32_t)(acc * 256);
            uint32_t accum = 0;
            for (int kb = 0; kb < t.nk; ++kb, ++it) {
                const int s = it % S;
                const uint32_t ph = (uint32_t)(it / S) & 1u;
                const bool in = CG == 1 ? mbar_wait(smem_u32(&full[s]), ph, abort_flag, P.status)
                                        : mbar_wait_cl(smem_u32(&full[s]), ph, abort_flag, P.status);
                if (!in) { ok = false; break; }
                tc_fence_after();
                const uint32_t sA = smem0 + s * SB, sB = sA + A_BYTES;
#pragma unroll
                for (int ks = 0; ks < BK / 16; ++ks) {
                    // K-major: 128-byte rows, k-block (ks / 4) at a fixed stride, 32 B per K = 16;
                    // MN-major: 64-column blocks of 128 k-rows (16 KB apart), 2048 B per K = 16
                    const uint64_t ad = q_amn ? sdesc(sA + ks * 2048, 16384, 1024)
                                              : sdesc(sA + (ks >> 2) * (BM * 128) + (ks & 3) * 32, 16, 1024);
                    // (dual: one N = 256 MMA, gate -> columns 0..127, up -> 128..255)
                    const uint64_t bd = (q_bmn || q_dual) ? sdesc(sB + ks * 2048, 16384, 1024)
                                                          : sdesc(sB + (ks >> 2) * b_kblk + (ks & 3) * 32, 16, 1024);
                    mma_issue<CG>(dt, ad, bd, idesc, accum);
                    accum = 1;
                }
                mma_commit_all<CG>(smem_u32(&empty[s]));  // stage free (both CTAs) once these MMAs finish
            }
            if (!ok) break;
            mma_commit_all<CG>(smem_u32(&tfull[acc]));    // accumulator ready (both CTAs)
        }
        mma_commit_local<CG>(smem_u32(drain));
        if constexpr (CG == 1) mbar_drain(smem_u32(drain), 0);
        else mbar_drain_cl(smem_u32(drain), 0);
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue (each CTA, its 128 rows)
        // Each warp drains 32 TMEM lanes (rows) x 32 columns at a time and writes
        // every output box through one of its two 2 KB shared-memory buffers with a
        // TMA store (64-byte swizzle: lane r's 16-byte chunk j goes to chunk
        // j ^ ((r >> 1) & 3), conflict-free), so global writes leave as whole
        // 64-byte row pieces instead of 16-byte partial stores.
        const int qd = warp & 3;                  // TMEM lane quarter this warp may access
        const int half = (warp - 2) / 4;          // which half of the tile's columns
        const int row_in_tile = qd * 32 + lane;
        const uint32_t tempty_leader0 = CG == 1 ? smem_u32(&tempty[0]) : mapa_shared(smem_u32(&tempty[0]), 0);
        uint8_t* stg = base + RING_BYTES + (warp - 2) * 4096;
        int nst = 0;                              // boxes this warp has stored
        auto put = [&](const CUtensorMap* m, const float* v, int c0, int c1, int c2) {
            uint8_t* buf = stg + (nst & 1) * 2048;
            if (nst >= 2) {                       // the store that last used buf has read it
                if (lane == 0) bulk_wait_read<1>();
                __syncwarp();
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
                    w[i] = *reinterpret_cast<uint32_t*>(&b2);
                }
                *reinterpret_cast<uint4*>(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store3(m, smem_u32(buf), c0, c1, c2);
                bulk_commit();
            }
            ++nst;
        };
        int tcount = 0;
        for (int tix = unit; tix < total; tix += nunits, ++tcount) {
            Tile t;
            decode_tile<CG>(P, offs, prefix, sbase, tix, t);
            const TcProblem& q = P.prob[t.p];
            const int width = q.dual ? 128 : q.bn;
            const int c_lo = half * (width / 64), c_hi = c_lo + width / 64;  // 32-column chunks
            const int acc = tcount & 1;
            const uint32_t aph = (uint32_t)(tcount >> 1) & 1u;
            const bool valid = t.mb + (int)rank < t.mb_e;   // this CTA's half lies in the segment
            const long long row = (long long)t.m0 + (long long)rank * BM + row_in_tile;
            const long long obase = (q.sched == SCHED_KSEG ? (long long)t.e * q.out_estride : 0) +
                                    row * q.ldo + t.n0;
            // The backward epilogues' inputs (h, or g and u) do not depend on the
            // accumulator: the first chunk's are fetched before waiting for it, each
            // later chunk's while the one before is processed (kept as packed bf16).
            const int n_in = q.epi == EPI_SWIGLU_BWD ? 2 : (q.epi == EPI_SILU_BWD ? 1 : 0);
            uint4 nxt[2][4];
            auto fetch = [&](int c) {
                const uint4* p0 = reinterpret_cast<const uint4*>(q.in0 + obase + c * 32);
#pragma unroll
                for (int j = 0; j < 4; ++j) nxt[0][j] = p0[j];
                if (n_in == 2) {
                    const uint4* p1 = reinterpret_cast<const uint4*>(q.in1 + obase + c * 32);
#pragma unroll
                    for (int j = 0; j < 4; ++j) nxt[1][j] = p1[j];
                }
            };
            if (valid && n_in) fetch(c_lo);
            // every lane takes the same decision (the box stores below sync the warp)
            const bool got = __all_sync(0xffffffffu,
                                        CG == 1 ? mbar_wait(smem_u32(&tfull[acc]), aph, abort_flag, P.status)
                                                : mbar_wait_cl(smem_u32(&tfull[acc]), aph, abort_flag, P.status));
            if (!got) break;
            tc_fence_after();
            // box coordinates of this warp's 32 rows: (column, row or M index, expert)
            const int brow = t.m0 + (int)rank * BM + qd * 32;
            const int bz = q.sched == SCHED_KSEG ? t.e : 0;
            const uint32_t taddr = tmem_base + (uint32_t)(acc * 256) + ((uint32_t)(qd * 32) << 16);
            for (int c = c_lo; valid && c < c_hi; ++c) {
                const int bcol = t.n0 + c * 32;
                float v[32];
                if (t.nk == 0) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0.f;
                    put(&q.tmO[0], v, bcol, brow, bz);
                    continue;
                }
                tmem_ld32(taddr + c * 32, v);
                if (q.epi == EPI_SWIGLU_FWD) {
                    float u[32];
                    tmem_ld32(taddr + 128 + c * 32, u);
                    tmem_wait_ld();
                    put(&q.tmO[0], v, bcol, brow, bz);
                    put(&q.tmO[1], u, bcol, brow, bz);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = silu_fast(v[i]) * u[i];
                    put(&q.tmO[2], v, bcol, brow, bz);
                    continue;
                }
                uint4 cur[2][4];
#pragma unroll
                for (int j = 0; j < 4; ++j) { cur[0][j] = nxt[0][j]; cur[1][j] = nxt[1][j]; }
                if (n_in && c + 1 < c_hi) fetch(c + 1);
                tmem_wait_ld();
                if (q.epi == EPI_STORE) {
                    put(&q.tmO[0], v, bcol, brow, bz);
                } else if (q.epi == EPI_SILU_FWD) {
                    put(&q.tmO[0], v, bcol, brow, bz);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = silu_fast(v[i]);
                    put(&q.tmO[1], v, bcol, brow, bz);
                } else if (q.epi == EPI_SILU_BWD) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= dsilu_fast(bf16_at(cur[0], i));
                    put(&q.tmO[0], v, bcol, brow, bz);
                } else {  // EPI_SWIGLU_BWD: v = dact; dg = dact u silu'(g), du = dact silu(g)
                    float o[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float g = bf16_at(cur[0], i), u = bf16_at(cur[1], i);
                        const float sg = __fdividef(1.0f, 1.0f + __expf(-g));   // sigmoid(g), once
                        o[i] = v[i] * u * (sg * (1.0f + g * (1.0f - sg)));
                        v[i] = v[i] * (g * sg);
                    }
                    put(&q.tmO[0], o, bcol, brow, bz);
                    put(&q.tmO[1], v, bcol, brow, bz);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {   // release the accumulator (on the even CTA's barrier)
                if constexpr (CG == 1) mbar_arrive(smem_u32(&tempty[acc]));
                else mbar_arrive_remote(tempty_leader0 + (uint32_t)(acc * 8));
            }
        }
        if (lane == 0) bulk_wait_all();           // every output box written before exit
    }
    tc_fence_before();
    __syncthreads();
    // a pair ends together: no CTA leaves while the other may still reach its
    // shared memory (the MMAs read both CTAs' stages; arrivals cross CTAs)
    if constexpr (CG == 2) cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (CG == 1)
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
        else
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
    }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

// 3-D bf16 map with 128-byte swizzle: dims {d0 (contiguous), d1, d2}, byte strides
// {s1, s2}, box {b0, b1, 1}
int encode_bf16_map(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                    uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return MOE_ERR_CUDA;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {b0, b1, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

namespace {

// bf16 map of rank 3 or 4 with 128-byte swizzle: dims[0] contiguous, strides[i] the
// byte stride of dims[i + 1] (any order: the outer dimensions may step by less than
// an inner one, as in the block views below)
int make_map_nd(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                const uint64_t* strides, const uint32_t* box) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return MOE_ERR_CUDA;
    cuuint64_t d[4], st[3];
    cuuint32_t b[4], es[4] = {1, 1, 1, 1};
    for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; }
    for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(ptr), d, st,
                    b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// activations [rows_cap, cols] as the block view {64, rows_cap, cols / 64} (64-column
// blocks 128 B apart).  K-major share: box {64, 128 rows, 2 k-blocks}; MN-major share:
// box {64, 128 k-rows, blocks 64-column blocks}.  Shared memory: the box's blocks one
// after the other, each its rows of 128 B (the canonical 128B-swizzled layouts).
int act_map(CUtensorMap* m, const void* ptr, int64_t rows_cap, int cols, bool mn_major, int blocks) {
    const uint64_t dims[3] = {64, (uint64_t)rows_cap, (uint64_t)cols / 64};
    const uint64_t st[2] = {(uint64_t)cols * 2, 128};
    const uint32_t box[3] = {64, mn_major ? (uint32_t)BK : (uint32_t)BM, mn_major ? (uint32_t)blocks : 2u};
    return make_map_nd(m, ptr, 3, dims, st, box);
}
// expert weights [E, rows, cols] as the view {64, rows, cols / 64, E}.  MN-major (N =
// cols): box {64, 128 k-rows, n_blocks, 1}; K-major (N = rows, K = cols): box {64,
// n_rows, 2 k-blocks, 1}.
int weight_map(CUtensorMap* m, const void* ptr, int E, int rows, int cols, bool mn, int share) {
    const uint64_t dims[4] = {64, (uint64_t)rows, (uint64_t)cols / 64, (uint64_t)E};
    const uint64_t st[3] = {(uint64_t)cols * 2, 128, (uint64_t)cols * 2 * rows};
    const uint32_t b[4] = {64, mn ? (uint32_t)BK : (uint32_t)share, mn ? (uint32_t)share : 2u, 1};
    return make_map_nd(m, ptr, 4, dims, st, b);
}

int max_pairs();
int cta_group() { return max_pairs() > 0 ? 2 : 1; }

int pick_bn(int n) { return n % 256 == 0 ? 256 : 128; }

#define MOE_TRY(x)                \
    do {                          \
        int _r = (x);             \
        if (_r != MOE_OK) return _r; \
    } while (0)

// Upper bound of a problem's tile count in cg * 128-row tiles (grid sizing
// only; the kernel counts the real tiles from the device offsets).
int64_t max_tiles(const moe_config& c, const TcProblem& q, int cg) {
    if (q.sched == SCHED_ROWS) {
        const int64_t mb = q.fixed_rows ? q.fixed_rows / BM : rows_cap_of(c) / BM;
        // each segment may round up by one pair tile
        return ((mb + cg - 1) / cg + (q.fixed_rows ? 0 : (cg - 1) * c.E)) * q.n_blocks;
    }
    return (int64_t)(q.fixed_rows ? 1 : c.E) * ((q.m_blocks + cg - 1) / cg) * q.n_blocks;
}

// CTA pairs the device can hold at once (0: pairs unusable)
int max_pairs() {
    static int cached[64] = {};
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!done[dev]) {
        done[dev] = true;
        if (cudaFuncSetAttribute(tc_grouped_gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES) != cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (num_sms() / 2));
        cfg.blockDim = dim3(NTHREADS);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, tc_grouped_gemm_kernel<2>, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        cached[dev] = std::min(n, num_sms() / 2);
    }
    return cached[dev];
}

int launch_tc(const moe_config& c, const int32_t* offsets, const TcProblem* probs, int nprob,
              cudaStream_t st) {
    static bool attr_done[64] = {};
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 64 && !attr_done[dev]) {
        MOE_CUDA_TRY(cudaFuncSetAttribute(tc_grouped_gemm_kernel<1>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES));
        attr_done[dev] = true;
    }
    if (nprob < 1 || nprob > MAX_PROBLEMS) return MOE_ERR_INVALID_ARG;
    TcParams P;
    memset(&P, 0, sizeof(P));
    for (int i = 0; i < nprob; ++i) P.prob[i] = probs[i];
    P.nprob = nprob;
    P.E = c.E;
    P.offsets = offsets;
    P.status = device_status_ptr();
    const int pairs = max_pairs();
    if (pairs > 0) {   // CTA pairs: 256-row tiles, M = 256 MMAs across the pair
        int64_t tiles = 0;
        for (int i = 0; i < nprob; ++i) tiles += max_tiles(c, probs[i], 2);
        const int units = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, pairs));
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * units);
        cfg.blockDim = dim3(NTHREADS);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        void* args[] = {&P};
        const cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(tc_grouped_gemm_kernel<2>), args);
        note_launch();
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        return MOE_OK;
    }
    int64_t tiles = 0;
    for (int i = 0; i < nprob; ++i) tiles += max_tiles(c, probs[i], 1);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, num_sms()));
    MOE_LAUNCH_PARAM(tc_grouped_gemm_kernel<1>, grid, NTHREADS, SMEM_BYTES, st, P);
    return MOE_OK;
}

// Estimated 64-deep k-steps of one tile of a problem: the routed experts'
// segments at their mean size (their exact sizes are known on the device only).
int64_t est_ksteps(const moe_config& c, const TcProblem& q) {
    if (q.sched == SCHED_ROWS) return (int64_t)q.k_blocks * q.kconcat;
    const int64_t rows = q.fixed_rows ? q.fixed_rows : (int64_t)c.T * c.k / c.E;
    return std::max<int64_t>(1, rows / BK);
}

// The CTA pairs of a persistent launch take tiles in a fixed stride.  When the
// launch mixes problems whose tiles differ in length (the backward's dgrad with
// K = d next to a weight gradient with K = an expert's rows), the pairs cross
// from one problem to the next at different times and stay offset from each
// other by up to a tile.  Tiles that share an operand's k-slices then ask for
// them tens of microseconds apart, longer than L2 keeps them once the launch
// streams from DRAM, and the operands are fetched from DRAM again and again.
// So a launch that holds many waves of tiles is issued as one launch per class
// of tile length (k-steps within a factor of about 1.4), problems in their
// given order; small launches stay whole (a launch's tail costs more there).
int launch_tc_classes(const moe_config& c, const int32_t* offsets, const TcProblem* probs,
                      int nprob, cudaStream_t st) {
    const int cg = max_pairs() > 0 ? 2 : 1;
    const int units = std::max(1, cg == 2 ? max_pairs() : num_sms());
    int64_t tiles = 0;
    for (int i = 0; i < nprob; ++i) tiles += max_tiles(c, probs[i], cg);
    if (nprob < 2 || tiles < (int64_t)SPLIT_MIN_WAVES * units)
        return launch_tc(c, offsets, probs, nprob, st);
    int cls[MAX_PROBLEMS];
    bool done[MAX_PROBLEMS] = {};
    for (int i = 0; i < nprob; ++i) cls[i] = (int)std::lround(std::log2((double)est_ksteps(c, probs[i])));
    for (int i = 0; i < nprob; ++i) {
        if (done[i]) continue;
        TcProblem g[MAX_PROBLEMS];
        int n = 0;
        for (int j = i; j < nprob; ++j)
            if (!done[j] && cls[j] == cls[i]) {
                g[n++] = probs[j];
                done[j] = true;
            }
        const int r = launch_tc(c, offsets, g, n, st);
        if (r != MOE_OK) return r;
    }
    return MOE_OK;
}

TcProblem new_problem() {
    TcProblem q;
    memset(&q, 0, sizeof(q));
    q.kconcat = 1;
    return q;
}

// One family of expert FFNs sharing a row layout: the routed experts (rows of
// the expert-contiguous layout, segments from the device offsets, E weight
// blocks) or the shared FFN (rows = tokens, one fixed segment, one block).
struct Family {
    const void* x;            // GEMM1 input rows
    int64_t x_rows;           // rows of x (the tensor map's extent; TMA zero-fills past it)
    int64_t rows;             // rows of the h / act / y / dh / dx buffers
    int fixed;                // 0: segments from offsets; else the one segment's rows
    int E;                    // weight blocks
    int f;                    // hidden width
    const void *Wu, *Wg, *Wd;
};

// Output maps of a row-segmented problem: out_i [rows_total, ldo], boxes of
// 32 columns x 32 rows with 64-byte swizzle (the epilogue's TMA stores)
int out_maps_rows(TcProblem& q, int64_t rows_total) {
    __nv_bfloat16* outs[3] = {q.out0, q.out1, q.out2};
    for (int i = 0; i < 3; ++i)
        if (outs[i])
            MOE_TRY(encode_bf16_map(&q.tmO[i], outs[i], (uint64_t)q.ldo, (uint64_t)rows_total, 1,
                                    (uint64_t)q.ldo * 2, (uint64_t)q.ldo * 2 * rows_total, 32, 32,
                                    CU_TENSOR_MAP_SWIZZLE_64B));
    return MOE_OK;
}

// Row-segmented problem: C[rows, N] = A[rows, K] (K-major) x B_e (expert weights)
int rows_problem(TcProblem& q, const Family& F, const void* A, int64_t a_rows, int K, int N) {
    q.sched = SCHED_ROWS;
    q.fixed_rows = F.fixed;
    q.k_blocks = K / BK;
    q.bn = pick_bn(N);
    q.n_blocks = N / q.bn;
    q.ldo = N;
    return act_map(&q.tmA0, A, a_rows, K, false, 0);
}

// Weight-gradient problem: out_e[M, N] = A_e^T B_e over the segment's rows (both MN-major)
int wgrad_problem(TcProblem& q, const Family& F, const void* A, int64_t a_rows, int M,
                  const void* B, int64_t b_rows, int N, void* out) {
    q.sched = SCHED_KSEG;
    q.fixed_rows = F.fixed;
    q.a_mn = 1;
    q.b_mn = 1;
    q.bn = pick_bn(N);
    q.m_blocks = M / BM;
    q.n_blocks = N / q.bn;
    q.epi = EPI_STORE;
    q.out0 = static_cast<__nv_bfloat16*>(out);
    q.ldo = N;
    q.out_estride = (long long)M * N;
    MOE_TRY(act_map(&q.tmA0, A, a_rows, M, true, BM / 64));
    MOE_TRY(act_map(&q.tmB0, B, b_rows, N, true, q.bn / cta_group() / 64));
    // out [E][M][N]: boxes of 32 columns x 32 rows of one expert
    return encode_bf16_map(&q.tmO[0], out, (uint64_t)N, (uint64_t)M, (uint64_t)F.E, (uint64_t)N * 2,
                           (uint64_t)N * 2 * M, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

// GEMM1 with the activation fused: h|g,u = x W_up|W_gate; act = silu(h) | silu(g) u
int gemm1_problem(TcProblem& q, const moe_config& c, const Family& F, void* h, void* act) {
    using bf = __nv_bfloat16;
    const int d = c.d, f = F.f;
    MOE_TRY(rows_problem(q, F, F.x, F.x_rows, d, f));
    q.b_mn = 1;
    if (c.ffn == MOE_FFN_SWIGLU) {
        q.dual = 1;
        q.bn = 128;
        q.n_blocks = f / 128;
        // a CTA's load: two 64-column blocks of the gate or of the up tile
        MOE_TRY(weight_map(&q.tmB0, F.Wg, F.E, d, f, true, 2));
        MOE_TRY(weight_map(&q.tmB1, F.Wu, F.E, d, f, true, 2));
        q.epi = EPI_SWIGLU_FWD;
        q.out0 = static_cast<bf*>(h);
        q.out1 = static_cast<bf*>(h) + F.rows * f;
        q.out2 = static_cast<bf*>(act);
    } else {
        MOE_TRY(weight_map(&q.tmB0, F.Wu, F.E, d, f, true, q.bn / cta_group() / 64));
        q.epi = EPI_SILU_FWD;
        q.out0 = static_cast<bf*>(h);
        q.out1 = static_cast<bf*>(act);
    }
    return out_maps_rows(q, F.rows);
}

// GEMM2: y = act W_down
int gemm2_problem(TcProblem& q, const moe_config& c, const Family& F, const void* act, void* y) {
    MOE_TRY(rows_problem(q, F, act, F.rows, F.f, c.d));
    q.b_mn = 1;
    MOE_TRY(weight_map(&q.tmB0, F.Wd, F.E, F.f, c.d, true, q.bn / cta_group() / 64));
    q.epi = EPI_STORE;
    q.out0 = static_cast<__nv_bfloat16*>(y);
    return out_maps_rows(q, F.rows);
}

// dgrad2 with the activation derivative fused: dact = dy W_down^T -> dh (SiLU) or dg, du (SwiGLU)
int dgrad2_problem(TcProblem& q, const moe_config& c, const Family& F, const void* dy,
                   int64_t dy_rows, const void* h, void* dh) {
    using bf = __nv_bfloat16;
    const int f = F.f;
    MOE_TRY(rows_problem(q, F, dy, dy_rows, c.d, f));
    MOE_TRY(weight_map(&q.tmB0, F.Wd, F.E, f, c.d, false, q.bn / cta_group()));
    q.in0 = static_cast<const bf*>(h);
    q.out0 = static_cast<bf*>(dh);
    if (c.ffn == MOE_FFN_SWIGLU) {
        q.epi = EPI_SWIGLU_BWD;
        q.in1 = static_cast<const bf*>(h) + F.rows * f;
        q.out1 = static_cast<bf*>(dh) + F.rows * f;
    } else {
        q.epi = EPI_SILU_BWD;
    }
    return out_maps_rows(q, F.rows);
}

// dgrad1: dx = dh W_up^T  (SwiGLU: du W_up^T + dg W_gate^T, one K loop over both)
int dgrad1_problem(TcProblem& q, const moe_config& c, const Family& F, const void* dh, void* dx) {
    using bf = __nv_bfloat16;
    const bool sw = c.ffn == MOE_FFN_SWIGLU;
    const bf* dh0 = static_cast<const bf*>(dh);
    const bf* dh1 = sw ? dh0 + F.rows * F.f : nullptr;
    MOE_TRY(rows_problem(q, F, sw ? dh1 : dh0, F.rows, F.f, c.d));
    MOE_TRY(weight_map(&q.tmB0, F.Wu, F.E, c.d, F.f, false, q.bn / cta_group()));
    if (sw) {
        q.kconcat = 2;
        MOE_TRY(act_map(&q.tmA1, dh0, F.rows, F.f, false, 0));
        MOE_TRY(weight_map(&q.tmB1, F.Wg, F.E, c.d, F.f, false, q.bn / cta_group()));
    }
    q.epi = EPI_STORE;
    q.out0 = static_cast<bf*>(dx);
    return out_maps_rows(q, F.rows);
}

// weight gradients: dW_down = act^T dy; dW_up = x^T dh (du); dW_gate = x^T dg
int wgrads_down(TcProblem& q, const moe_config& c, const Family& F, const void* act,
                const void* dy, int64_t dy_rows, void* dWd) {
    return wgrad_problem(q, F, act, F.rows, F.f, dy, dy_rows, c.d, dWd);
}

Family routed_family(const moe_config& c, const void* x_perm, const void* Wu, const void* Wg,
                     const void* Wd) {
    const int64_t rc = rows_cap_of(c);
    return Family{x_perm, rc, rc, 0, c.E, c.f, Wu, Wg, Wd};
}

Family shared_family(const moe_config& c, const moe_shared_ffn& s) {
    const int64_t ts = shared_rows_of(c);
    return Family{s.x, c.T, ts, (int)ts, 1, c.f_shared, s.W_up, s.W_gate, s.W_down};
}

}  // namespace

int tc_ffn_forward(const moe_config& c, const void* x_perm, const int32_t* offsets,
                   const void* W_up, const void* W_gate, const void* W_down, void* h_saved,
                   void* act, void* y_perm, const moe_shared_ffn* sh, cudaStream_t st)
{
    const Family R = routed_family(c, x_perm, W_up, W_gate, W_down);
    TcProblem q[2];
    // GEMM1 (+ activation), routed experts || shared FFN
    q[0] = new_problem();
    MOE_TRY(gemm1_problem(q[0], c, R, h_saved, act));
    if (sh) {
        q[1] = new_problem();
        MOE_TRY(gemm1_problem(q[1], c, shared_family(c, *sh), sh->h, sh->act));
    }
    MOE_TRY(launch_tc(c, offsets, q, sh ? 2 : 1, st));
    // GEMM2
    q[0] = new_problem();
    MOE_TRY(gemm2_problem(q[0], c, R, act, y_perm));
    if (sh) {
        q[1] = new_problem();
        MOE_TRY(gemm2_problem(q[1], c, shared_family(c, *sh), sh->act, sh->y));
    }
    return launch_tc(c, offsets, q, sh ? 2 : 1, st);
}

int tc_ffn_backward(const moe_config& c, const void* x_perm, const int32_t* offsets,
                    const void* W_up, const void* W_gate, const void* W_down,
                    const void* h_saved, const void* act, const void* dy_perm, void* dh,
                    void* dx_perm, void* dW_up, void* dW_gate, void* dW_down,
                    const moe_shared_ffn* sh, cudaStream_t st)
{
    using bf = __nv_bfloat16;
    const bool sw = c.ffn == MOE_FFN_SWIGLU;
    const Family R = routed_family(c, x_perm, W_up, W_gate, W_down);
    TcProblem q[MAX_PROBLEMS];
    int n = 0;
    // launch 1: dact = dy W_down^T with the activation derivative fused  ||  dW_down = act^T dy
    // (the shared FFN's dy is the layer's output gradient: it joins with weight 1)
    q[n] = new_problem();
    MOE_TRY(dgrad2_problem(q[n++], c, R, dy_perm, R.rows, h_saved, dh));
    q[n] = new_problem();
    MOE_TRY(wgrads_down(q[n++], c, R, act, dy_perm, R.rows, dW_down));
    if (sh) {
        const Family S = shared_family(c, *sh);
        q[n] = new_problem();
        MOE_TRY(dgrad2_problem(q[n++], c, S, sh->dout, c.T, sh->h, sh->dh));
        q[n] = new_problem();
        MOE_TRY(wgrads_down(q[n++], c, S, sh->act, sh->dout, c.T, sh->dW_down));
    }
    MOE_TRY(launch_tc_classes(c, offsets, q, n, st));
    // launch 2: dW_up = x^T dh (du)  ||  [dW_gate = x^T dg]  ||  dx = dh W_up^T (+ dg W_gate^T)
    n = 0;
    auto second = [&](const Family& F, const void* dhF, void* dWu, void* dWg, void* dx) -> int {
        const bf* dh0 = static_cast<const bf*>(dhF);
        const bf* dh1 = sw ? dh0 + F.rows * F.f : nullptr;
        q[n] = new_problem();
        MOE_TRY(wgrad_problem(q[n++], F, F.x, F.x_rows, c.d, sw ? dh1 : dh0, F.rows, F.f, dWu));
        if (sw) {
            q[n] = new_problem();
            MOE_TRY(wgrad_problem(q[n++], F, F.x, F.x_rows, c.d, dh0, F.rows, F.f, dWg));
        }
        q[n] = new_problem();
        return dgrad1_problem(q[n++], c, F, dhF, dx);
    };
    MOE_TRY(second(R, dh, dW_up, dW_gate, dx_perm));
    if (sh) MOE_TRY(second(shared_family(c, *sh), sh->dh, sh->dW_up, sh->dW_gate, sh->dx));
    return launch_tc_classes(c, offsets, q, n, st);
}

}  // namespace moe
