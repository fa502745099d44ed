// router.cu -- the MoE router on the device: gate logits on the tensor cores
// (bf16 x bf16 -> fp32), sigmoid affinities, bias-steered group-limited
// top-k and the gate values, then the routing tables by a stable counting
// sort of the selections by expert.
//
// What it follows: sigmoid scoring, 8 expert groups of which 4 are kept,
// top-8 of 256, route_scale 2.5 (config block of "671B 参数如何「激活」37B？");
// the per-expert bias enters the selection only, the FFN output keeps the
// original affinities, and no token is dropped (page 2 of the DeepSeek-V3
// notes, section 2-2); gating stays in higher precision than FP8 (section
// 2-4 of the same notes), so the logits come from bf16 operands with fp32
// accumulation.  Where the pages are silent: a group's score is the largest
// biased affinity in it, ties go to the lower index, and the gate values are
// the chosen affinities normalised to sum 1, times route_scale.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "codec.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace {

// ------------------------------------------------------------------ gate
//
// A 128-token tile is taken by CS CTAs of 640 threads (a thread-block
// cluster of 4 when E % 64 == 0, else one CTA), each computing all E logits
// over a quarter of K: warps 0 and 1 TMA producers (x tile 128 x 64 bf16 and
// the E gate-weight rows x 64 bf16 per 128-byte K chunk, 128-byte swizzle, a
// ring of 4 stages; warp 0 the even chunks, warp 1 the odd ones), warps 2 and
// 3 MMA issuers (four tcgen05.mma.kind::f16, M 128, N E, K 16, per chunk; even
// and odd chunks again, each into its own TMEM accumulator; warp 2 owns the
// TMEM allocation), warps 4-19 the epilogue (four warps per TMEM lane
// quarter), which adds the two sums.  With N = E the tensor core reads each
// x chunk once for all the experts.
// Epilogue:
//   1. (cluster) each CTA writes its partial logits, token-major, into its own
//      shared memory; after a cluster barrier cluster rank q adds, for tokens
//      32q .. 32q + 31 of the tile, the CS partials in rank order (16-byte
//      loads through distributed shared memory) and applies the sigmoid.
//      (One CTA) the sums become affinities directly.  Either way the
//      affinities land token-major in the CTA's selection table.
//   2. one warp per token, lane l holding experts l, l + 32, ...: group
//      scores (largest s + bias of each group) by warp max-reductions, the
//      topk_groups best groups (lower index on ties); each lane then sorts
//      its kept candidates once, and top_k rounds take the warp's best head
//      (a max-reduction, then a min-reduction over the expert index for ties,
//      lower expert first) and advance the winning lane's list; the gate
//      values come from the chosen s in rank order.
// Values are compared through an order-preserving map of their fp32 bits
// to unsigned integers, so the hardware warp reductions give exact fp32
// comparisons.  The steps meet at a bounded mbarrier wait (one CTA) or
// cluster barriers.
constexpr int kGateM = 128;
constexpr int kGateK = 64;            // bf16 elements per 128-byte chunk
constexpr int kGateMaxE = 256;
constexpr int kGateMaxGroups = 32;
constexpr int kGateMaxTopK = 16;
constexpr int kGateEpiWarp0 = 4;
constexpr int kGateEpiWarps = 16;
constexpr int kGateThreads = 32 * (kGateEpiWarp0 + kGateEpiWarps);
constexpr int kGateRowStride = 260;   // floats per token row of the partial-logit and selection tables
static_assert(kGateMaxGroups <= 32 && kGateMaxTopK <= 32, "one lane per group and per chosen expert");
static_assert(kGateMaxE <= 8 * 32, "eight experts per lane");

// Shared memory of one CTA.  After the K loop the pipeline stages hold (one
// CTA) the selection table, or (cluster) this CTA's partial logits for all
// 128 tokens and, beside them, the selection table of its 32 tokens -- apart,
// because the peers read the partial logits while the table is written.
template <int CS>
struct GateLayout {
    // Pipeline stages, a multiple of 2: two producer warps and two MMA warps
    // each take every other K chunk, so a warp's chunks always fall on the
    // stages of one parity and the chunk it waits for on a stage is the one
    // right after its own previous chunk there.  (With an odd count the
    // previous chunk on a stage would belong to the other warp and might not
    // have landed yet; a parity wait would then see the phase before it as
    // complete.)
    static constexpr int ST = 4;
    static_assert(ST % 2 == 0, "stages per warp parity");
    static constexpr int A_BYTES = kGateM * 128;
    static constexpr int B_BYTES = kGateMaxE * 128;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = ST * A_BYTES;
    static constexpr int STAGES_END = OFF_B + ST * B_BYTES;
    // (cluster) partial logits [128 tokens][kGateRowStride] fp32; the stride
    // keeps both the per-token-row accesses and the per-expert reads free of
    // bank conflicts and rows 16-byte aligned
    static constexpr int OFF_PART = 0;
    static constexpr int PART_END = CS == 1 ? 0 : kGateM * kGateRowStride * 4;
    // selection table: affinities [NT tokens][kGateRowStride] fp32, then
    // per-warp group keys [16][32] u32
    static constexpr int NT = kGateM / CS;
    static constexpr int OFF_SEL = PART_END;
    static constexpr int OFF_GK = OFF_SEL + NT * kGateRowStride * 4;
    static constexpr int SEL_END = OFF_GK + kGateEpiWarps * kGateMaxGroups * 4;
    static_assert(SEL_END <= STAGES_END, "the tables fit in the pipeline stages");
    // full[ST], empty[ST], done, the epilogue's step barrier
    static constexpr int OFF_BAR = STAGES_END;
    static constexpr int NUM_BARS = 2 * ST + 2;
    static constexpr int OFF_TMEM = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_ABORT = OFF_TMEM + 4;
    static constexpr int OFF_BIAS = (OFF_ABORT + 4 + 15) & ~15;
    static constexpr int BYTES = OFF_BIAS + kGateMaxE * 4;
    static constexpr int ALLOC = BYTES + 1024;
    // two accumulators (even and odd K chunks) of up to E columns
    static constexpr uint32_t ACC_COLS = kGateMaxE;
    static constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;
    static_assert(TMEM_COLS <= 512, "TMEM allocation");
    static_assert(ALLOC <= 227 * 1024, "shared memory per CTA");
};

struct GateParams {
    const float* bias;  // [E] or nullptr
    int32_t* ids;       // [T, top_k]
    float* w;           // [T, top_k]
    int T, KB, E, n_groups, topk_groups, top_k;
    int kps;            // K chunks per cluster rank
    float route_scale;
    unsigned* err;
    uint64_t timeout_ns;
};

// tcgen05.mma kind::f16, fp32 accumulate, A = B = bf16, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Waits on an mbarrier while draining async work before exit: ignores the
// abort flag (the work must land first) but keeps the time limit.
__device__ __forceinline__ bool drain_wait_g(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
    int no_abort = 0;
    WaitCtl c2{&no_abort, ctl.err, ctl.timeout_ns};
    const bool ok = bounded_wait(bar, parity, c2);
    __syncwarp();
    return ok;
}

__device__ __forceinline__ float sigmoid_f32(float v) { return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-v))); }

// Order-preserving map of fp32 bit patterns to unsigned integers: for
// non-NaN a, b, a > b exactly when key(a) > key(b) (with +0 above -0).
// Selection keys are at least 1, so 0 marks an expert that is not (or no
// longer) a candidate.
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(v);
    return max((u & 0x80000000u) ? ~u : (u | 0x80000000u), 1u);
}

// Compare-exchange of a lane's candidate slots a < b (static indices, so the
// lists stay in registers): slot a ends up holding the better candidate,
// the larger key, or on equal keys the lower slot index (the lower expert).
__device__ __forceinline__ void cand_cx(uint32_t& ka, int& ja, uint32_t& kb, int& jb) {
    const bool swap = kb > ka || (kb == ka && jb < ja);
    const uint32_t tk = swap ? kb : ka;
    const int tj = swap ? jb : ja;
    kb = swap ? ka : kb;
    jb = swap ? ja : jb;
    ka = tk;
    ja = tj;
}

// CS: CTAs per 128-token tile (a thread-block cluster when CS > 1).  Each
// takes K chunks [rank * kps, (rank + 1) * kps) of the whole tile and
// selects for 128 / CS tokens.
template <int CS>
__global__ void __launch_bounds__(kGateThreads, 1)
    moe_gate_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ GateParams p) {
    using L = GateLayout<CS>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t bar0 = sbase + L::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (L::ST + s); };
    const uint32_t done_bar = bar0 + 8u * (2 * L::ST);
    const uint32_t step_bar = bar0 + 8u * (2 * L::ST + 1);
    const uint32_t crank = CS > 1 ? cluster_rank() : 0u;
    const int kb0 = static_cast<int>(crank) * p.kps;
    const int nk = max(0, min(p.KB, kb0 + p.kps) - kb0);  // this CTA's K chunks
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_ABORT);
    float* bias_s = reinterpret_cast<float*>(smem + L::OFF_BIAS);

    if (threadIdx.x == 32) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < L::ST; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(done_bar, 2);  // one commit from each MMA warp
        mbar_init(step_bar, kGateEpiWarps);
        *abort_flag = 0;
        fence_barrier_init();
    }
    grid_dependency_wait();
    allow_dependents();
    if (warp == 2) tmem_alloc(sbase + L::OFF_TMEM, L::TMEM_COLS);
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) bias_s[e] = p.bias ? p.bias[e] : 0.0f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::OFF_TMEM);
    const WaitCtl ctl{abort_flag, p.err, p.timeout_ns};
    const int m0 = (blockIdx.x / CS) * kGateM;

    if (warp <= 1) {
        // ------------------------------------------------------------ producers
        // Warp 0 loads the even K chunks, warp 1 the odd ones: a warp's wait
        // on a stage also holds until its own earlier copies have landed, so
        // two producers keep twice the loads in flight.
        const int j = warp;
        const uint32_t tx = static_cast<uint32_t>(L::A_BYTES + p.E * 128);
        int c = j;
        if (lane == 0) {
            for (; c < nk; c += 2) {
                const int s = c % L::ST;
                if (!bounded_wait(empty_bar(s), ((c / L::ST) & 1u) ^ 1u, ctl)) break;
                mbar_arrive_expect_tx(full_bar(s), tx);
                tma_load_2d(sbase + L::OFF_A + s * L::A_BYTES, &tmX, full_bar(s), (kb0 + c) * kGateK, m0);
                tma_load_2d(sbase + L::OFF_B + s * L::B_BYTES, &tmW, full_bar(s), (kb0 + c) * kGateK, 0);
            }
        }
        c = __shfl_sync(0xffffffffu, c, 0);  // one past this warp's last issued chunk
        // every issued load must land before the CTA's shared memory goes
        // away: the last use of each of this warp's stages
        for (int i = j; i < c; i += 2)
            if (i + L::ST >= c) drain_wait_g(full_bar(i % L::ST), (i / L::ST) & 1u, ctl);
    } else if (warp <= 3) {
        // ------------------------------------------------------------ MMA issuers
        // Warp 2 takes the even K chunks, warp 3 the odd ones, each into its
        // own accumulator.  A thread's mbarrier wait does not return before
        // the MMAs it issued earlier have completed, so with one issuer the
        // tensor core would idle at every chunk; with two, one warp's queued
        // chunk covers the other's wait.
        const int j = warp - 2;
        const uint32_t acc = tmem + static_cast<uint32_t>(j) * L::ACC_COLS;
        const uint32_t idesc = idesc_bf16_f32(kGateM, p.E);
        bool issued = false;
        if (lane == 0) {
            for (int c = j; c < nk; c += 2) {
                const int s = c % L::ST;
                if (!bounded_wait(full_bar(s), (c / L::ST) & 1u, ctl)) break;
                tc_fence_after();
                const uint64_t adesc = sdesc_kmajor_sw128(sbase + L::OFF_A + s * L::A_BYTES);
                const uint64_t bdesc = sdesc_kmajor_sw128(sbase + L::OFF_B + s * L::B_BYTES);
#pragma unroll
                for (int k = 0; k < 4; ++k)  // K 16 = 32 bytes = +2 in the address field
                    umma_bf16(acc, adesc + 2u * k, bdesc + 2u * k, idesc, (c > 1 || k > 0) ? 1u : 0u);
                umma_commit(empty_bar(s));
                issued = true;
            }
            // Publish the sums (also after a wait that gave up: the status
            // word then reports the failure and the outputs are not to be used).
            umma_commit(done_bar);
        }
        __syncwarp();
        if (__shfl_sync(0xffffffffu, issued ? 1 : 0, 0)) drain_wait_g(done_bar, 0, ctl);
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - kGateEpiWarp0;
        const int quarter = warp & 3;         // TMEM lane quarter this warp may read
        const int sl = ew >> 2;               // which of the four warps of the quarter
        const int row = quarter * 32 + lane;  // this thread's token (TMEM lane) in the tile
        const uint32_t taddr0 = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        float* S = reinterpret_cast<float*>(smem + L::OFF_SEL);  // [NT][kGateRowStride]
        bool ok = warp_wait(done_bar, 0, ctl);
        tc_fence_after();
        // the stages were last written by TMA (async proxy); the tables
        // overwrite them with ordinary stores
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        // 1. the sums of this warp's 16-column units sl, sl + 4, ...: the
        //    affinities (one CTA) or the partial logits (cluster)
        if (ok) {
            float* dst = reinterpret_cast<float*>(smem + (CS == 1 ? L::OFF_SEL : L::OFF_PART)) + row * kGateRowStride;
            for (int u = sl; u < p.E / 16; u += 4) {
                uint64_t pr[8], po[8];
                if (nk > 0) {
                    tmem_ld_x16_pairs(taddr0 + 16 * u, pr);
                    if (nk > 1) {  // even-chunk sum + odd-chunk sum
                        tmem_ld_x16_pairs(taddr0 + L::ACC_COLS + 16 * u, po);
#pragma unroll
                        for (int i = 0; i < 8; ++i) pr[i] = f2_add(pr[i], po[i]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) pr[i] = 0;  // no chunks in this K slice
                }
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float l = (i & 1) ? hi_f32(pr[i >> 1]) : lo_f32(pr[i >> 1]);
                    v[i] = CS == 1 ? sigmoid_f32(l) : l;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<float4*>(dst + 16 * u + 4 * q) =
                        make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
        }
        if constexpr (CS > 1) {
            // every CTA's partial logits are complete and visible (the other
            // warps reach the same barrier after their loops)
            asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                             "memory");
            // rank crank's tokens: the CS partials added in rank order, four
            // experts at a time, every peer's load in flight together
            const uint32_t part0 = sbase + L::OFF_PART;
            const int groups = p.E / 4;
            const int items = L::NT * groups;
            for (int it = ew * 32 + lane; it < items; it += 32 * kGateEpiWarps) {
                const int t = it / groups, g = it % groups;
                const uint32_t off =
                    static_cast<uint32_t>(((static_cast<int>(crank) * L::NT + t) * kGateRowStride + 4 * g) * 4);
                float4 pv[CS];
#pragma unroll
                for (int q = 0; q < CS; ++q) pv[q] = ld_cluster_v4f32(mapa_rank(part0 + off, static_cast<uint32_t>(q)));
                float4 sum = pv[0];
#pragma unroll
                for (int q = 1; q < CS; ++q) {
                    sum.x = __fadd_rn(sum.x, pv[q].x);
                    sum.y = __fadd_rn(sum.y, pv[q].y);
                    sum.z = __fadd_rn(sum.z, pv[q].z);
                    sum.w = __fadd_rn(sum.w, pv[q].w);
                }
                *reinterpret_cast<float4*>(S + t * kGateRowStride + 4 * g) =
                    make_float4(sigmoid_f32(sum.x), sigmoid_f32(sum.y), sigmoid_f32(sum.z), sigmoid_f32(sum.w));
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(step_bar);
        ok = warp_wait(step_bar, 0, ctl) && ok;
        // 2. selection, one warp per token; lane l holds experts l + 32 j
        if (ok) {
            const int J = (p.E + 31) / 32;
            const int per = p.E / p.n_groups;
            uint32_t* gk = reinterpret_cast<uint32_t*>(smem + L::OFF_GK) + 32 * ew;
            float bias_r[8];
            int grp[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = 32 * j + lane;
                bias_r[j] = e < p.E ? bias_s[e] : 0.0f;
                grp[j] = e < p.E ? e / per : -1;
            }
            const int tok0 = m0 + static_cast<int>(crank) * L::NT;
            for (int t = ew; t < L::NT && tok0 + t < p.T; t += kGateEpiWarps) {
                const float* St = S + t * kGateRowStride;
                uint32_t ck[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    ck[j] = (j < J && grp[j] >= 0) ? order_key(__fadd_rn(St[32 * j + lane], bias_r[j])) : 0u;
                // group scores: one per lane g < n_groups
                uint32_t mine = 0;
                if (per == 32) {  // group j is slot j
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (j < J) {
                            const uint32_t g = __reduce_max_sync(0xffffffffu, ck[j]);
                            if (lane == j) mine = g;
                        }
                    }
                } else {
                    for (int g = 0; g < p.n_groups; ++g) {
                        uint32_t m = 0;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (grp[j] == g) m = max(m, ck[j]);
                        m = __reduce_max_sync(0xffffffffu, m);
                        if (lane == g) mine = m;
                    }
                }
                gk[lane] = mine;
                __syncwarp();
                // group lane is kept when fewer than topk_groups groups beat it
                int better = 0;
                for (int h = 0; h < p.n_groups; ++h) {
                    const uint32_t o = gk[h];
                    better += (o > mine || (o == mine && h < lane)) ? 1 : 0;
                }
                const uint32_t keep = __ballot_sync(0xffffffffu, lane < p.n_groups && better < p.topk_groups);
                __syncwarp();
                int my_id = -1;
                if (per == 32 && p.topk_groups <= 4) {
                    // Groups of 32: this lane holds one expert of each group, so at
                    // most four candidates, reloaded from the table in group order
                    // and sorted with five compare-exchanges (the selection is
                    // bound by the integer pipe: fewer candidates, fewer selects).
                    uint32_t kk = keep;
                    uint32_t c4[4];
                    int j4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (kk != 0u) {
                            const int g = __ffs(kk) - 1;
                            kk &= kk - 1u;
                            c4[i] = order_key(__fadd_rn(St[32 * g + lane], bias_s[32 * g + lane]));
                            j4[i] = g;
                        } else {
                            c4[i] = 0u;
                            j4[i] = 8 + i;
                        }
                    }
                    cand_cx(c4[0], j4[0], c4[1], j4[1]);
                    cand_cx(c4[2], j4[2], c4[3], j4[3]);
                    cand_cx(c4[0], j4[0], c4[2], j4[2]);
                    cand_cx(c4[1], j4[1], c4[3], j4[3]);
                    cand_cx(c4[1], j4[1], c4[2], j4[2]);
                    for (int r = 0; r < p.top_k; ++r) {
                        const uint32_t mk = __reduce_max_sync(0xffffffffu, c4[0]);
                        const uint32_t me = static_cast<uint32_t>(32 * j4[0] + lane);
                        const uint32_t win =
                            __reduce_min_sync(0xffffffffu, (c4[0] == mk && mk != 0u) ? me : 0xffffffffu);
                        if (win == me) {
                            c4[0] = c4[1];
                            j4[0] = j4[1];
                            c4[1] = c4[2];
                            j4[1] = j4[2];
                            c4[2] = c4[3];
                            j4[2] = j4[3];
                            c4[3] = 0u;
                        }
                        if (lane == r) my_id = static_cast<int>(win);
                    }
                } else {
                    // this lane's kept candidates sorted best first (Batcher's
                    // odd-even merge network for 8; ties to the lower slot)
                    int cj[8];
    #pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (grp[j] < 0 || !((keep >> grp[j]) & 1u)) ck[j] = 0u;
                        cj[j] = j;
                    }
    #define GATE_CX(a, b) cand_cx(ck[a], cj[a], ck[b], cj[b])
                    GATE_CX(0, 1); GATE_CX(2, 3); GATE_CX(4, 5); GATE_CX(6, 7);
                    GATE_CX(0, 2); GATE_CX(1, 3); GATE_CX(4, 6); GATE_CX(5, 7);
                    GATE_CX(1, 2); GATE_CX(5, 6);
                    GATE_CX(0, 4); GATE_CX(1, 5); GATE_CX(2, 6); GATE_CX(3, 7);
                    GATE_CX(2, 4); GATE_CX(3, 5);
                    GATE_CX(1, 2); GATE_CX(3, 4); GATE_CX(5, 6);
    #undef GATE_CX
                    // top_k rounds: the warp's best head (largest key, then the
                    // lowest expert); the winning lane moves to its next candidate
                    for (int r = 0; r < p.top_k; ++r) {
                        const uint32_t mk = __reduce_max_sync(0xffffffffu, ck[0]);
                        const uint32_t me = static_cast<uint32_t>(32 * cj[0] + lane);
                        const uint32_t win = __reduce_min_sync(0xffffffffu, (ck[0] == mk && mk != 0u) ? me : 0xffffffffu);
                        if (win == me) {
    #pragma unroll
                            for (int j = 0; j < 7; ++j) {
                                ck[j] = ck[j + 1];
                                cj[j] = cj[j + 1];
                            }
                            ck[7] = 0u;
                        }
                        if (lane == r) my_id = static_cast<int>(win);
                    }
                }
                // gate values: the chosen affinities normalised in rank order
                const float sr = (lane < p.top_k && my_id >= 0 && my_id < p.E) ? St[my_id] : 0.0f;
                float ssum = 0.0f;
                for (int r = 0; r < p.top_k; ++r) ssum = __fadd_rn(ssum, __shfl_sync(0xffffffffu, sr, r));
                if (lane < p.top_k) {
                    const int64_t o = static_cast<int64_t>(tok0 + t) * p.top_k + lane;
                    p.ids[o] = my_id;
                    p.w[o] = __fmul_rn(__fdiv_rn(sr, ssum), p.route_scale);
                }
            }
        }
    }
    if constexpr (CS > 1) {
        // the producer and MMA warps meet the epilogue's cluster barrier
        if (warp < kGateEpiWarp0)
            asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                             "memory");
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
    if constexpr (CS > 1) cluster_sync_all();  // no CTA leaves while a peer may still read its partial logits
}

// ------------------------------------------------------------------ routing tables
//
// One thread-block cluster of kRouteCtas CTAs, each owning a contiguous
// chunk of tokens.  Each CTA counts its own chunk's selections per expert
// (shared-memory atomics: a count is the same whatever the order); after a
// cluster barrier every CTA reads all the chunks' counts through distributed
// shared memory, which gives both the totals (their exclusive scan is the
// offsets) and, per expert, the selections of the chunks before its own:
// expert e's rows for a chunk start at offsets[e] + that count.  Inside the
// chunk the rank of a selection is formed without any ordering race: tokens
// are taken kRouteThreads at a time, one per thread; each warp marks, per
// expert, the lanes that chose it (a 32-bit mask built with atomicOr), a scan
// over the warps gives each warp's base per expert, and a lane's rank is its
// warp's base plus the number of lower lanes in the mask.  A round's rows are
// gathered in shared memory expert by expert and leave as contiguous runs
// (coalesced stores).  Rows no selection reaches (a token naming an expert
// twice) get token -1 / gate 0, visible as an out-of-range id downstream.
constexpr int kRouteThreads = 512;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kRouteMaxE = 256;
constexpr int kRouteCtas = 8;  // one cluster (the portable maximum)
constexpr int kRouteMaxK = 16;
constexpr int kRouteBatch = 8;  // global loads a thread keeps in flight

struct RouteSmem {
    uint32_t mask[kRouteWarps][kRouteMaxE];
    int32_t base[kRouteWarps][kRouteMaxE];
    int32_t sel_e[kRouteThreads * kRouteMaxK];  // one round's selections, staged
    float sel_w[kRouteThreads * kRouteMaxK];
    int32_t ltok[kRouteThreads * kRouteMaxK];   // one round's rows, expert by expert
    float lw[kRouteThreads * kRouteMaxK];
    int32_t rstart[kRouteMaxE];                 // the round's first row of each expert
    int32_t rcnt[kRouteMaxE];                   // and its number of rows
    int32_t loc[kRouteMaxE];                    // where they start in ltok / lw
    int32_t mine[kRouteMaxE];  // this chunk's selections per expert (read by the whole cluster)
    int32_t total[kRouteMaxE];
    int32_t before[kRouteMaxE];
    int32_t next[kRouteMaxE];
    int32_t scan[kRouteMaxE + 1];
};

__global__ void __launch_bounds__(kRouteThreads)
    moe_route_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w, int T, int top_k, int E,
                     int chunk, int32_t* __restrict__ offsets, int32_t* __restrict__ token_of_row,
                     int32_t* __restrict__ rows_of_token, float* __restrict__ weight_of_row,
                     unsigned* __restrict__ err) {
    extern __shared__ uint8_t route_smem_raw[];
    RouteSmem& sm = *reinterpret_cast<RouteSmem*>(route_smem_raw);
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int wp = tid >> 5;
    const int me = static_cast<int>(cluster_rank());
    const int t_begin = min(T, me * chunk);
    const int t_end = min(T, t_begin + chunk);
    for (int e = tid; e < E; e += kRouteThreads) sm.mine[e] = 0;
    __syncthreads();
    grid_dependency_wait();
    allow_dependents();
    // this chunk's counts
    bool bad = false;
    const int64_t i_begin = static_cast<int64_t>(t_begin) * top_k;
    const int64_t i_end = static_cast<int64_t>(t_end) * top_k;
    for (int64_t i0 = i_begin; i0 < i_end; i0 += kRouteBatch * kRouteThreads) {
        int ev[kRouteBatch];
#pragma unroll
        for (int u = 0; u < kRouteBatch; ++u) {  // all loads first, then the counts
            const int64_t i = i0 + u * kRouteThreads + tid;
            ev[u] = i < i_end ? __ldg(ids + i) : 0;
        }
#pragma unroll
        for (int u = 0; u < kRouteBatch; ++u) {
            if (i0 + u * kRouteThreads + tid >= i_end) continue;
            if (ev[u] >= 0 && ev[u] < E) atomicAdd(&sm.mine[ev[u]], 1);
            else bad = true;
        }
    }
    __syncthreads();
    cluster_sync_all();  // every chunk's counts are complete and visible
    // totals and the counts of the chunks before this one
    const uint32_t mine0 = smem_u32(&sm.mine[0]);
    for (int e = tid; e < E; e += kRouteThreads) {
        int tot = 0, bef = 0;
        for (int c = 0; c < kRouteCtas; ++c) {
            const int v = ld_cluster_s32(mapa_rank(mine0 + 4u * static_cast<uint32_t>(e), static_cast<uint32_t>(c)));
            tot += v;
            if (c < me) bef += v;
        }
        sm.total[e] = tot;
        sm.before[e] = bef;
    }
    // the peers may leave once everyone has read their counts
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    __syncthreads();
    // exclusive scan of the totals (one warp; E <= 256)
    if (wp == 0) {
        int run = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int c = e < E ? sm.total[e] : 0;
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (e < E) sm.scan[e] = run + incl - c;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) sm.scan[E] = run;
    }
    __syncthreads();
    if (me == 0)
        for (int e = tid; e <= E; e += kRouteThreads) offsets[e] = sm.scan[e];
    for (int e = tid; e < E; e += kRouteThreads) sm.next[e] = sm.scan[e] + sm.before[e];  // this chunk's first row of e
    const uint32_t lt = (1u << lane) - 1u;
    for (int t0 = t_begin; t0 < t_end; t0 += kRouteThreads) {
        // stage the round's selections and gate values (coalesced, loads in flight together)
        const int nsel = (min(t_end, t0 + kRouteThreads) - t0) * top_k;
        const int64_t g0 = static_cast<int64_t>(t0) * top_k;
        for (int j0 = 0; j0 < nsel; j0 += kRouteBatch * kRouteThreads) {
            int ev[kRouteBatch];
            float wv[kRouteBatch];
#pragma unroll
            for (int u = 0; u < kRouteBatch; ++u) {
                const int j = j0 + u * kRouteThreads + tid;
                ev[u] = j < nsel ? __ldg(ids + g0 + j) : 0;
                wv[u] = j < nsel ? __ldg(w + g0 + j) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < kRouteBatch; ++u) {
                const int j = j0 + u * kRouteThreads + tid;
                if (j < nsel) {
                    sm.sel_e[j] = ev[u];
                    sm.sel_w[j] = wv[u];
                }
            }
        }
        for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) sm.mask[i / E][i % E] = 0u;
        __syncthreads();
        const int t = t0 + tid;
        if (t < t_end) {
            for (int k = 0; k < top_k; ++k) {
                const int e = sm.sel_e[tid * top_k + k];
                if (e >= 0 && e < E) {
                    const uint32_t old = atomicOr(&sm.mask[wp][e], 1u << lane);
                    if (old & (1u << lane)) bad = true;  // the same expert twice for one token
                }
            }
        }
        __syncthreads();
        for (int e = tid; e < E; e += kRouteThreads) {
            int run = sm.next[e];
            sm.rstart[e] = run;
            for (int q = 0; q < kRouteWarps; ++q) {
                sm.base[q][e] = run;
                run += __popc(sm.mask[q][e]);
            }
            sm.rcnt[e] = run - sm.next[e];
            sm.next[e] = run;
        }
        __syncthreads();
        // exclusive scan of the round's row counts: each expert's place in ltok / lw
        if (wp == 0) {
            int run = 0;
            for (int e0 = 0; e0 < E; e0 += 32) {
                const int e = e0 + lane;
                const int c = e < E ? sm.rcnt[e] : 0;
                int incl = c;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += v;
                }
                if (e < E) sm.loc[e] = run + incl - c;
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
        }
        __syncthreads();
        if (t < t_end) {
            for (int k = 0; k < top_k; ++k) {
                const int64_t i = static_cast<int64_t>(t) * top_k + k;
                const int e = sm.sel_e[tid * top_k + k];
                int32_t r = -1;
                if (e >= 0 && e < E) {
                    r = sm.base[wp][e] + __popc(sm.mask[wp][e] & lt);
                    const int j = sm.loc[e] + (r - sm.rstart[e]);
                    sm.ltok[j] = t;
                    sm.lw[j] = sm.sel_w[tid * top_k + k];
                }
                rows_of_token[i] = r;
            }
        }
        __syncthreads();
        // each expert's rows of the round are contiguous: one warp copies them out
        for (int e = wp; e < E; e += kRouteWarps) {
            const int n = sm.rcnt[e], r0 = sm.rstart[e], j0 = sm.loc[e];
            for (int q = lane; q < n; q += 32) {
                token_of_row[r0 + q] = sm.ltok[j0 + q];
                weight_of_row[r0 + q] = sm.lw[j0 + q];
            }
        }
        __syncthreads();
    }
    // rows no selection reached (a token naming an expert twice): token -1, gate 0
    for (int e = wp; e < E; e += kRouteWarps) {
        const int end = sm.scan[e] + sm.before[e] + sm.mine[e];
        for (int r = sm.next[e] + lane; r < end; r += 32) {
            token_of_row[r] = -1;
            weight_of_row[r] = 0.0f;
        }
    }
    if (bad) atomicOr(err, kDevErrIndex);
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace

cudaError_t launch_moe_gate(const uint16_t* x, int64_t ldx, const uint16_t* wg, const float* bias, int64_t T,
                            int64_t dim, int E, int n_groups, int topk_groups, int top_k, float route_scale,
                            int32_t* ids, float* w, const DeviceInfo& dev, cudaStream_t stream) {
    // Clusters of four CTAs per 128-token tile (a quarter of K each) while
    // the tiles fill at most two waves of the SMs that way; beyond that one
    // CTA per tile already fills the GPU without the partial-logit exchange.
    const int tiles = static_cast<int>((T + kGateM - 1) / kGateM);
    const int cs = (static_cast<int64_t>(tiles) * 4 <= 2 * static_cast<int64_t>(dev.num_sms)) ? 4 : 1;
    CUtensorMap tmX, tmW;
    cudaError_t e;
    if ((e = make_tmap_2d(&tmX, x, 2, dim, T, ldx * 2, kGateK, kGateM, 128)) != cudaSuccess) return e;
    if ((e = make_tmap_2d(&tmW, wg, 2, dim, E, dim * 2, kGateK, E, 128)) != cudaSuccess) return e;
    {
        static bool ready[64];
        if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
        if (!ready[dev.device]) {
            e = cudaFuncSetAttribute(moe_gate_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     GateLayout<1>::ALLOC);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(moe_gate_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     GateLayout<4>::ALLOC);
            if (e != cudaSuccess) return e;
            ready[dev.device] = true;
        }
    }
    GateParams p{};
    p.bias = bias;
    p.ids = ids;
    p.w = w;
    p.T = static_cast<int>(T);
    p.KB = static_cast<int>(dim / kGateK);
    p.kps = (p.KB + cs - 1) / cs;
    p.E = E;
    p.n_groups = n_groups;
    p.topk_groups = topk_groups;
    p.top_k = top_k;
    p.route_scale = route_scale;
    p.err = dev.err;
    p.timeout_ns = wait_timeout_ns();
    if (cs == 1)
        return launch_pdl(moe_gate_kernel<1>, dim3(tiles), dim3(kGateThreads), GateLayout<1>::ALLOC, stream, tmX, tmW, p);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 4;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(4 * tiles);
    cfg.blockDim = dim3(kGateThreads);
    cfg.dynamicSmemBytes = GateLayout<4>::ALLOC;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, moe_gate_kernel<4>, tmX, tmW, p);
}

cudaError_t launch_moe_route(const int32_t* ids, const float* w, int64_t T, int top_k, int E, int32_t* offsets,
                             int32_t* token_of_row, int32_t* rows_of_token, float* weight_of_row,
                             const DeviceInfo& dev, cudaStream_t stream) {
    static bool ready[64];
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    if (!ready[dev.device]) {
        const cudaError_t e = cudaFuncSetAttribute(moe_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(sizeof(RouteSmem)));
        if (e != cudaSuccess) return e;
        ready[dev.device] = true;
    }
    // one cluster; chunks of ceil(T / kRouteCtas) tokens (T == 0: the CTAs
    // still write the all-zero offsets)
    const int chunk = static_cast<int>(std::max<int64_t>(1, (T + kRouteCtas - 1) / kRouteCtas));
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kRouteCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kRouteCtas);
    cfg.blockDim = dim3(kRouteThreads);
    cfg.dynamicSmemBytes = sizeof(RouteSmem);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, moe_route_kernel, ids, w, static_cast<int>(T), top_k, E, chunk, offsets,
                              token_of_row, rows_of_token, weight_of_row, dev.err);
}

}  // namespace fp8bs
